"""Parity of the CUDA path (through the C ABI) against the fp64 oracle.

Bars: position ids bit-exact; normalised pixels within 1 bf16 ulp of the
oracle's value rounded to bf16; embeddings within a relative Frobenius error of
5e-3 per item against the float64 oracle, and within 2e-2 absolute, output cast
included, of the method-exact value: the oracle with the GEMM's input in the
model dtype (the normalised pixels rounded to bf16, as FusedInputNorm emits
them; vitfe_testutil.embed_report); cos/sin within 1e-5 absolute.
"""
import numpy as np
import pytest

import oracle
from vit_vision_encoder_fusedinputnorm_gb300 import synth
import vitfe_testutil as U

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from vit_vision_encoder_fusedinputnorm_gb300 import build
    build.build()


def _fe(wl):
    from vit_vision_encoder_fusedinputnorm_gb300.frontend import FrontEnd
    return FrontEnd.from_workload(wl)


def _report(g, wl, starts, **kw):
    """embed_report of GPU embeddings against both oracle references of the workload."""
    return U.embed_report(g, oracle.embed_workload(wl, **kw), oracle.embed_workload(wl, bf16_input=True, **kw),
                          starts)


# small seeded cases: several 128-row tiles, ragged tails, mixed stills and video
SMALL = {
    "stills_p14": (14, 256, [(1, 2, 2, 1), (1, 4, 6, 1), (1, 16, 16, 1), (1, 10, 22, 1)]),
    "mixed_p14": (14, 1280, [(2, 4, 6, 4), (1, 6, 8, 1), (3, 2, 4, 6), (1, 2, 2, 1)]),
    "video_p14": (14, 512, [(4, 8, 10, 8)]),
    "stills_p16": (16, 1152, [(1, 4, 4, 1), (1, 6, 10, 1), (2, 4, 2, 4)]),
    # all stills, five N passes: resident tiles whose passes are spread over several CTA pairs
    "allstill_p14_n1280": (14, 1280, [(1, 2, 2, 1), (1, 4, 6, 1), (1, 16, 16, 1)]),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("pad", [0, 300])
def test_embed_small_vs_oracle(name, pad):
    P, N, grids = SMALL[name]
    wl = synth.small_workload(17, grids, patch=P, hidden=N, pixels="uniform")
    fe = _fe(wl)
    b = fe.upload(wl.items)
    rows = b.live_rows + pad
    st = fe.status_tensor()
    out = fe.embed(b, rows=rows, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, -1]
    g = U.bits_to_f64(U.tensor_bits(out))
    U.check_embed(_report(g, wl, U.item_starts(wl.items), bucket_rows=rows))
    assert np.all(U.tensor_bits(out)[b.live_rows:] == 0)
    fe.close()


@pytest.mark.parametrize("name", sorted(SMALL))
def test_normalize_patchify_within_one_ulp(name):
    P, N, grids = SMALL[name]
    wl = synth.small_workload(23, grids, patch=P, hidden=N, pixels="uniform")
    fe = _fe(wl)
    b = fe.upload(wl.items)
    rows = b.live_rows + 40
    out = fe.normalize_patchify(b, rows=rows)
    got = U.tensor_bits(out)
    ref = U.f64_to_bf16_bits(oracle.normalize_patchify_workload(wl, bucket_rows=rows))
    assert got.shape == ref.shape
    assert int(U.ulp_distance(got, ref).max()) <= U.NORM_MAX_ULP
    assert np.all(got[b.live_rows:] == 0)
    fe.close()


@pytest.mark.parametrize("name", sorted(SMALL))
def test_pos_ids_and_rope(name):
    P, N, grids = SMALL[name]
    wl = synth.small_workload(5, grids, patch=P, hidden=N, head_dim=80 if P == 14 else 72)
    fe = _fe(wl)
    b = fe.upload(wl.items)
    rows = b.live_rows + 70
    pos = fe.pos_ids(b, rows=rows).cpu().numpy()
    assert np.array_equal(pos, oracle.pos_ids_workload(wl, bucket_rows=rows))
    cos, sin = fe.rope(b, wl.head_dim, wl.theta, rows=rows)
    rc, rs = oracle.rope_workload(wl, bucket_rows=rows)
    assert np.max(np.abs(cos.cpu().numpy() - rc)) <= U.ROPE_MAX_ABS
    assert np.max(np.abs(sin.cpu().numpy() - rs)) <= U.ROPE_MAX_ABS
    fe.close()


def test_one_hot_weight_returns_normalised_pixels_bit_exact():
    # W[n][k] = [k == k_n], b = 0: every output equals bf16(x) for feature k_n, which pins
    # the internal feature permutation and the row order bit-exactly against the
    # standalone normalise + patchify path.
    P, T = 14, 2
    K = 3 * T * P * P
    N = 128
    ks = np.linspace(0, K - 1, N).astype(int)
    W = np.zeros((N, K), np.uint16)
    W[np.arange(N), ks] = 0x3F80
    wl = synth.small_workload(9, [(1, 4, 6, 1), (2, 2, 4, 4), (1, 8, 2, 1)], patch=P, hidden=N)
    wl.W_bits = W
    wl.b_bits = None
    fe = _fe(wl)
    b = fe.upload(wl.items)
    emb = U.tensor_bits(fe.embed(b))
    flat = U.tensor_bits(fe.normalize_patchify(b))
    assert np.array_equal(emb, flat[:, ks])
    fe.close()


def test_still_equals_duplicated_two_frame_item():
    # A still (one stored frame) and the same frame stored twice as a t=1 video item
    # give the same embeddings up to fp32 summation order (resident vs streamed tiles).
    wl = synth.small_workload(31, [(1, 8, 16, 1)], patch=14, hidden=1280)
    px = wl.items[0].pixels
    dup = synth.Item(t=1, h=8, w=16, frames=2, pixels=np.concatenate([px, px], 0))
    fe = _fe(wl)
    a = U.tensor_bits(fe.embed(fe.upload(wl.items)))
    v = U.tensor_bits(fe.embed(fe.upload([dup])))
    d = U.ulp_distance(a, v)
    ad = np.abs(U.bits_to_f64(a) - U.bits_to_f64(v))
    # differ only by fp32 summation order: at most one bf16 ulp, or a few ulps of values
    # near zero (absolute difference at the fp32 accumulation level)
    assert np.all((d <= 1) | (ad <= 1e-5)) and np.mean(d == 0) > 0.95
    fe.close()


def test_last_round_pass_split_equals_unsplit():
    # One tile more than CTA pairs: the last round's tile has its N passes spread over
    # several pairs.  A bucket of whole rounds runs the same rows unsplit; every row's
    # embedding must be bit-identical (all stills: the same resident summation order), and
    # the split tile's rows match the oracle.
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    n = pairs + 1
    wl = synth.small_workload(47, [(1, 16, 16, 1)] * n, patch=14, hidden=1280)
    fe = _fe(wl)
    b = fe.upload(wl.items)
    assert b.live_rows == 256 * n
    a = U.tensor_bits(fe.embed(b, rows=b.live_rows))
    u = U.tensor_bits(fe.embed(b, rows=2 * 256 * pairs)[: b.live_rows])
    assert np.array_equal(a, u)
    g = U.bits_to_f64(a[-256:])
    U.check_embed(_report(g, wl, [0, 256], items=[n - 1]))
    fe.close()


def test_deterministic_rerun():
    wl = synth.make_workload(1)
    fe = _fe(wl)
    b = fe.upload(wl.items)
    x = U.tensor_bits(fe.embed(b))
    y = U.tensor_bits(fe.embed(b))
    assert np.array_equal(x, y)
    fe.close()


def test_empty_and_all_pad_calls():
    wl = synth.small_workload(3, [(1, 2, 2, 1)], patch=14, hidden=256)
    fe = _fe(wl)
    b = fe.upload(wl.items)
    b.n_items.zero_()
    st = fe.status_tensor()
    out = torch.full((300, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    fe.embed(b, rows=300, out=out, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, -1]
    assert torch.count_nonzero(out).item() == 0
    fe.embed(b, rows=0, status=st)          # nothing to write, status still set
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, -1]
    fe.close()


def test_max_items_in_one_call():
    # VITFE_MAX_ITEMS small items (stills and a few videos): every pair tile holds rows of many
    # items, and the kernels' item tables are full
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    grids = []
    for i in range(B.VITFE_MAX_ITEMS):
        if i % 16 == 5:
            grids.append((2, 2, 4, 4))                        # a short video: t = 2 of 4 frames
        else:
            grids.append((1, 2 + 2 * (i % 3), 2 + 2 * (i % 4), 1))
    wl = synth.small_workload(71, grids, patch=14, hidden=256, head_dim=80, pixels="uniform")
    fe = _fe(wl)
    b = fe.upload(wl.items)
    assert b.n_items.item() == B.VITFE_MAX_ITEMS
    rows = b.live_rows + 100
    st = fe.status_tensor()
    out, cos, sin = fe.embed_rope(b, 80, wl.theta, rows=rows, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, -1]
    rep = _report(U.bits_to_f64(U.tensor_bits(out)), wl, U.item_starts(wl.items), bucket_rows=rows)
    U.log_report(f"{B.VITFE_MAX_ITEMS} items in one call: all {rep['rows']} rows", rep)
    U.check_embed(rep)
    assert np.all(U.tensor_bits(out)[b.live_rows:] == 0)
    rc, rs = oracle.rope_workload(wl, bucket_rows=rows)
    assert np.max(np.abs(cos.cpu().numpy() - rc)) <= U.ROPE_MAX_ABS
    assert np.max(np.abs(sin.cpu().numpy() - rs)) <= U.ROPE_MAX_ABS
    fe.close()


def test_rope_side_limit():
    # an item at the largest side the RoPE tables take (positions up to 4095), one just over
    # it (rejected on the device by the fused call, its rows written as padding, but a valid
    # item for the embeddings alone), and a small one after them
    side = 4096
    wl = synth.small_workload(73, [(1, 2, side, 1), (1, 2, side + 2, 1), (1, 4, 4, 1)], patch=14, hidden=256,
                              head_dim=80, pixels="uniform")
    fe = _fe(wl)
    b = fe.upload(wl.items)
    n0, n1 = 2 * side, 2 * (side + 2)
    rows = b.live_rows + 20
    st = fe.status_tensor()
    out, cos, sin = fe.embed_rope(b, 80, wl.theta, rows=rows, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [4, 1]
    o = U.bits_to_f64(U.tensor_bits(out))
    c, sn = cos.cpu().numpy(), sin.cpu().numpy()
    assert np.all(o[n0:n0 + n1] == 0) and np.all(c[n0:n0 + n1] == 1.0) and np.all(sn[n0:n0 + n1] == 0.0)
    keep = np.r_[0:n0, n0 + n1:b.live_rows]
    ok = [0, 2]
    rep = U.embed_report(o[keep], oracle.embed_workload(wl, items=ok), oracle.embed_workload(wl, items=ok, bf16_input=True),
                         U.item_starts([wl.items[i] for i in ok]))
    U.log_report(f"item at the RoPE side limit ({side}): {rep['rows']} rows", rep)
    U.check_embed(rep)
    rc, rs = oracle.rope_workload(wl, items=ok)
    assert np.max(np.abs(c[keep] - rc)) <= U.ROPE_MAX_ABS
    assert np.max(np.abs(sn[keep] - rs)) <= U.ROPE_MAX_ABS
    # the embeddings alone take the wider item
    out2 = fe.embed(b, rows=rows, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, -1]
    o2 = U.bits_to_f64(U.tensor_bits(out2))
    U.check_embed(_report(o2, wl, U.item_starts(wl.items), bucket_rows=rows))
    fe.close()


def test_device_side_descriptor_errors_zero_the_item_rows():
    wl = synth.small_workload(13, [(1, 4, 4, 1), (1, 4, 6, 1), (1, 2, 2, 1)], patch=14, hidden=256)
    fe = _fe(wl)
    b = fe.upload(wl.items)
    good = U.tensor_bits(fe.embed(b))
    # item 1: w not a multiple of the merge size
    bad = b.host_items.copy()
    bad[1]["w"] = 5
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    it, n = B.items_tensor(bad, device="cuda")
    b.items = it
    st = fe.status_tensor()
    rows = 16 + 20 + 4
    out = fe.embed(b, rows=rows, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [4, 1]
    o = U.tensor_bits(out)
    assert np.array_equal(o[:16], good[:16])
    assert np.all(o[16:36] == 0)
    assert np.array_equal(o[36:40], good[40:44])
    # pixels beyond the buffer
    bad2 = b.host_items.copy()
    bad2[2]["pixel_offset"] = b.pixel_bytes
    b.items, _ = B.items_tensor(bad2, device="cuda")
    fe.embed(b, rows=44, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [5, 2]
    # more rows than the bucket
    b.items, _ = B.items_tensor(b.host_items, device="cuda")
    fe.embed(b, rows=30, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [5, 1]
    # count above capacity
    b.n_items.fill_(99)
    fe.embed(b, rows=44, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist()[0] == 4
    fe.close()


# --------------------------------------------------------------------------- full workloads

@pytest.mark.parametrize("cfg", [0, 1, 3])
def test_full_workload_embed(cfg):
    wl = synth.make_workload(cfg)
    fe = _fe(wl)
    b = fe.upload(wl.items)
    out = fe.embed(b)
    g = U.bits_to_f64(U.tensor_bits(out))
    rep = _report(g, wl, U.item_starts(wl.items))
    U.log_report(f"workload {cfg}: all {b.live_rows} rows", rep)
    U.check_embed(rep)
    pos = fe.pos_ids(b).cpu().numpy()
    assert np.array_equal(pos, oracle.pos_ids_workload(wl))
    cos, sin = fe.rope(b, wl.head_dim, wl.theta)
    rc, rs = oracle.rope_workload(wl)
    assert np.max(np.abs(cos.cpu().numpy() - rc)) <= U.ROPE_MAX_ABS
    assert np.max(np.abs(sin.cpu().numpy() - rs)) <= U.ROPE_MAX_ABS
    fe.close()


def test_throughput_workload_sampled():
    # 64 x 1344^2 stills, through the call and launch configuration the benchmark times
    # (vitfe_embed_rope); sampled embedding rows: both sides of every 128-row CTA tile
    # boundary plus random rows; the RoPE rows in full.
    wl = synth.make_workload(2)
    fe = _fe(wl)
    b = fe.upload(wl.items)
    st = fe.status_tensor()
    out, cos, sin = fe.embed_rope(b, wl.head_dim, wl.theta, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, -1]
    rc, rs = oracle.rope_workload(wl)
    assert np.max(np.abs(cos.cpu().numpy() - rc)) <= U.ROPE_MAX_ABS
    assert np.max(np.abs(sin.cpu().numpy() - rs)) <= U.ROPE_MAX_ABS
    del cos, sin
    rows = b.live_rows
    rng = np.random.default_rng(0)
    bnd = np.arange(128, rows, 128)
    sample = np.unique(np.concatenate([bnd, bnd - 1, rng.integers(0, rows, 8192), [0, rows - 1]]))
    g = U.bits_to_f64(U.tensor_bits(out[torch.from_numpy(sample).cuda()]))
    rep = _report(g, wl, [0, len(sample)], sample=sample)
    U.log_report(f"workload 2: {len(sample)} sampled rows (every tile boundary)", rep)
    U.check_embed(rep)
    pos = fe.pos_ids(b).cpu().numpy()
    assert np.array_equal(pos, oracle.pos_ids_workload(wl))
    flat = fe.normalize_patchify(b)
    f = U.tensor_bits(flat[torch.from_numpy(sample[:2048]).cuda()])
    # oracle rows for the sample from the items they fall in
    starts = U.item_starts(wl.items)
    ref_np = np.zeros((2048, wl.K))
    for j, r in enumerate(sample[:2048]):
        i = int(np.searchsorted(starts, r, side="right") - 1)
        it = wl.items[i]
        if j == 0 or i != last_i:
            A = oracle.normalize_patchify_item(it.pixels, it.t, it.h, it.w, patch=wl.patch, tpatch=wl.tpatch,
                                               merge=wl.merge, mean=wl.mean, std=wl.std, rescale=wl.rescale)
            last_i = i
        ref_np[j] = A[r - starts[i]]
    assert int(U.ulp_distance(f, U.f64_to_bf16_bits(ref_np)).max()) <= U.NORM_MAX_ULP
    fe.close()


def test_graph_replay_bucket_masks_pad_rows():
    # 50 varied stills (patch 16) packed into fixed 65,536-row buckets: one captured graph
    # (embed + rope) replayed per bucket; live rows equal an eager call on exactly the live
    # rows bit for bit, pad rows are masked, sampled rows match the oracle.
    wl = synth.make_workload(4)
    fe = _fe(wl)
    R = wl.bucket_rows
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    packs = [B.pack_items([wl.items[i] for i in bk], wl.patch, wl.tpatch) for bk in wl.buckets]
    cap_bytes = max(p[1].size for p in packs)
    px = torch.zeros(cap_bytes, dtype=torch.uint8, device="cuda")
    it_dev = torch.zeros(B.VITFE_MAX_ITEMS * 24, dtype=torch.uint8, device="cuda")
    n_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((R, wl.hidden), dtype=torch.bfloat16, device="cuda")
    cos = torch.empty((R, wl.head_dim // 2), dtype=torch.float32, device="cuda")
    sin = torch.empty_like(cos)
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        B.vitfe_embed(fe.h, px, cap_bytes, it_dev, n_dev, B.VITFE_MAX_ITEMS, R, out, st, s)
        B.vitfe_rope(fe.h, it_dev, n_dev, B.VITFE_MAX_ITEMS, R, wl.head_dim, wl.theta, cos, sin, None, s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        B.vitfe_embed(fe.h, px, cap_bytes, it_dev, n_dev, B.VITFE_MAX_ITEMS, R, out, st, s)
        B.vitfe_rope(fe.h, it_dev, n_dev, B.VITFE_MAX_ITEMS, R, wl.head_dim, wl.theta, cos, sin, None, s)
    rng = np.random.default_rng(4)
    for kb, (bk, (items, buf, live)) in enumerate(zip(wl.buckets, packs)):
        px[:buf.size].copy_(torch.from_numpy(buf))
        arr = np.zeros(B.VITFE_MAX_ITEMS, B.ITEM_DTYPE)
        arr[:len(items)] = items
        it_dev.copy_(torch.from_numpy(arr.view(np.uint8)))
        n_dev.fill_(len(items))
        out.fill_(3.0)
        cos.fill_(5.0)
        g.replay()
        torch.cuda.synchronize()
        assert st.cpu().tolist() == [0, -1]
        o = U.tensor_bits(out)
        assert np.all(o[live:] == 0)
        c = cos.cpu().numpy()
        assert np.all(c[live:] == 1.0) and np.all(sin.cpu().numpy()[live:] == 0.0)
        # eager call on exactly the live rows
        sub = synth.Workload(**{**wl.__dict__, "items": [wl.items[i] for i in bk], "bucket_rows": None,
                                "buckets": None})
        eb = fe.upload(sub.items)
        e = U.tensor_bits(fe.embed(eb))
        assert np.array_equal(o[:live], e)
        sample = np.unique(rng.integers(0, live, 4096))
        rep = _report(U.bits_to_f64(o[sample]), sub, [0, len(sample)], sample=sample)
        U.log_report(f"workload 4: bucket {kb} replay, {len(sample)} sampled of {live} live rows", rep)
        U.check_embed(rep)
        rc, _ = oracle.rope_workload(sub)
        assert np.max(np.abs(c[:live] - rc)) <= U.ROPE_MAX_ABS
    fe.close()


def _rope_check(fe, b, wl, head_dim, theta, rows, cos=None, sin=None):
    c, s_ = (cos, sin) if cos is not None else fe.rope(b, head_dim, theta, rows=rows)
    torch.cuda.synchronize()
    rc, rs = oracle.rope_workload(wl, bucket_rows=rows, head_dim=head_dim, theta=theta)
    assert np.max(np.abs(c.cpu().numpy() - rc)) <= U.ROPE_MAX_ABS
    assert np.max(np.abs(s_.cpu().numpy() - rs)) <= U.ROPE_MAX_ABS


def test_rope_table_first_built_inside_a_capture():
    # the first call of a (head_dim, theta) pair is captured, not run: an eager call made
    # before any replay must still build and use the right table, and the graph must
    # build its own on replay
    wl = synth.small_workload(9, [(1, 4, 6, 1), (2, 2, 4, 4)], patch=14, hidden=256, head_dim=80)
    fe = _fe(wl)
    b = fe.upload(wl.items)
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    rows = b.live_rows + 12
    cos = torch.full((rows, 40), 7.0, device="cuda")
    sin = torch.full((rows, 40), 7.0, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.vitfe_rope(fe.h, b.items, b.n_items, b.capacity, rows, 80, wl.theta, cos, sin, None, s)
    _rope_check(fe, b, wl, 80, wl.theta, rows)
    cos.fill_(7.0)
    sin.fill_(7.0)
    g.replay()
    _rope_check(fe, b, wl, 80, wl.theta, rows, cos, sin)
    fe.close()


def test_rope_tables_beyond_the_cached_slots_and_graph_reading_a_slot():
    # a graph captured on a cached pair keeps reading that pair's table after many other
    # pairs (more than the handle caches) have been used eagerly
    wl = synth.small_workload(11, [(1, 6, 4, 1), (1, 2, 2, 1)], patch=14, hidden=256, head_dim=80)
    fe = _fe(wl)
    b = fe.upload(wl.items)
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    rows = b.live_rows
    _rope_check(fe, b, wl, 80, 10000.0, rows)
    cos = torch.empty((rows, 40), device="cuda")
    sin = torch.empty((rows, 40), device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.vitfe_rope(fe.h, b.items, b.n_items, b.capacity, rows, 80, 10000.0, cos, sin, None, s)
    for hd, th in [(64, 10000.0), (80, 500.0), (72, 10000.0), (80, 1e6), (96, 10000.0), (80, 123.0), (64, 10000.0)]:
        _rope_check(fe, b, wl, hd, th, rows)
    cos.fill_(7.0)
    sin.fill_(7.0)
    g.replay()
    _rope_check(fe, b, wl, 80, 10000.0, rows, cos, sin)
    _rope_check(fe, b, wl, 80, 123.0, rows)
    fe.close()


@pytest.mark.parametrize("name", sorted(SMALL))
def test_cu_seqlens_vs_oracle(name):
    P, N, grids = SMALL[name]
    wl = synth.small_workload(3, grids, patch=P, hidden=N)
    fe = _fe(wl)
    b = fe.upload(wl.items)
    cu_ref, mx_ref = oracle.cu_seqlens_workload(wl)
    nseq = len(cu_ref) - 1
    st = fe.status_tensor()
    for pad in (0, 37):
        cap = nseq + 5
        cu, info = fe.cu_seqlens(b, cap, rows=b.live_rows + pad, status=st)
        torch.cuda.synchronize()
        assert st.cpu().tolist() == [0, -1]
        expect = np.concatenate([cu_ref, np.full(cap - nseq, cu_ref[-1])])
        assert np.array_equal(cu.cpu().numpy(), expect)
        assert info.cpu().tolist() == [nseq, mx_ref]
    fe.close()


def test_cu_seqlens_bucket_clipping_and_overflow():
    # rows below the live rows clip the last sequences; more sequences than slots fill the
    # slots and report VITFE_EDEVICE_RANGE
    wl = synth.small_workload(4, [(1, 4, 4, 1), (3, 2, 4, 6), (1, 2, 2, 1)], patch=14, hidden=256)
    fe = _fe(wl)
    b = fe.upload(wl.items)
    cu_ref, _ = oracle.cu_seqlens_workload(wl)         # [0, 16, 24, 32, 40, 44]
    st = fe.status_tensor()
    cu, info = fe.cu_seqlens(b, 8, rows=28, status=st)
    torch.cuda.synchronize()
    # item 1 keeps rows [16, 28): its groups [16, 24) and [24, 28); item 2 starts past the bucket
    assert cu_ref.tolist() == [0, 16, 24, 32, 40, 44]
    assert cu.cpu().numpy().tolist() == [0, 16, 24, 28, 28, 28, 28, 28, 28]
    assert info.cpu().tolist() == [3, 16]      # item 0 is the longest sequence
    assert st.cpu().tolist() == [5, 1]        # item 1 is the first that overflows the bucket
    cu, info = fe.cu_seqlens(b, 3, status=st)
    torch.cuda.synchronize()
    assert cu.cpu().numpy().tolist() == cu_ref[:4].tolist()
    assert int(info[0]) == 3 and st.cpu().tolist() == [5, -1]
    fe.close()


@pytest.mark.parametrize("name", sorted(SMALL))
def test_embed_rope_one_launch_equals_the_two_calls(name):
    # the fused launch writes exactly what vitfe_embed and vitfe_rope write, pad rows included
    P, N, grids = SMALL[name]
    hd = 80 if P == 14 else 72
    wl = synth.small_workload(29, grids, patch=P, hidden=N, head_dim=hd, pixels="uniform")
    fe = _fe(wl)
    b = fe.upload(wl.items)
    rows = b.live_rows + 300
    st = fe.status_tensor()
    out, cos, sin = fe.embed_rope(b, hd, wl.theta, rows=rows, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, -1]
    e = fe.embed(b, rows=rows)
    c2, s2 = fe.rope(b, hd, wl.theta, rows=rows)
    torch.cuda.synchronize()
    assert np.array_equal(U.tensor_bits(out), U.tensor_bits(e))
    assert np.array_equal(cos.cpu().numpy(), c2.cpu().numpy())
    assert np.array_equal(sin.cpu().numpy(), s2.cpu().numpy())
    rc, rs = oracle.rope_workload(wl, bucket_rows=rows)
    assert np.max(np.abs(cos.cpu().numpy() - rc)) <= U.ROPE_MAX_ABS
    assert np.max(np.abs(sin.cpu().numpy() - rs)) <= U.ROPE_MAX_ABS
    U.check_embed(_report(U.bits_to_f64(U.tensor_bits(out)), wl, U.item_starts(wl.items), bucket_rows=rows))
    fe.close()


def test_back_to_back_calls_into_one_buffer_keep_stream_order():
    # Consecutive fused calls on one stream may overlap (the next call's prologue, A
    # production and first passes run while the previous call finishes); every global write
    # of a call still lands after the previous call's.  A chain A, B, A, B ... into the same
    # outputs must leave exactly B's result, and a torch read between two calls must see the
    # first call's result.
    import torch
    wa = synth.small_workload(61, [(1, 16, 16, 1), (2, 8, 12, 4), (1, 24, 10, 1)], patch=14, hidden=1280,
                              head_dim=80, pixels="uniform")
    wb = synth.small_workload(62, [(1, 10, 30, 1), (1, 32, 16, 1), (3, 6, 8, 6)], patch=14, hidden=1280,
                              head_dim=80, pixels="uniform")
    wb.W_bits, wb.b_bits = wa.W_bits, wa.b_bits          # one handle serves both
    fe = _fe(wa)
    ba, bb = fe.upload(wa.items), fe.upload(wb.items)
    rows = max(ba.live_rows, bb.live_rows) + 200
    hd, th = 80, wa.theta
    ra = fe.embed_rope(ba, hd, th, rows=rows)
    rb = fe.embed_rope(bb, hd, th, rows=rows)
    torch.cuda.synchronize()
    ref_a = [t.clone() for t in ra]
    ref_b = [t.clone() for t in rb]
    out = torch.full_like(ref_a[0], 7.0)
    cos = torch.full_like(ref_a[1], 7.0)
    sin = torch.full_like(ref_a[2], 7.0)
    st = fe.status_tensor()
    fe.embed_rope(ba, hd, th, rows=rows, out=out, cos=cos, sin=sin, status=st)
    seen = out.clone()                                   # a torch kernel between two calls
    for k in range(7):
        fe.embed_rope(bb if k % 2 == 0 else ba, hd, th, rows=rows, out=out, cos=cos, sin=sin, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, -1]
    assert np.array_equal(U.tensor_bits(seen), U.tensor_bits(ref_a[0]))
    assert np.array_equal(U.tensor_bits(out), U.tensor_bits(ref_b[0]))
    assert np.array_equal(cos.cpu().numpy(), ref_b[1].cpu().numpy())
    assert np.array_equal(sin.cpu().numpy(), ref_b[2].cpu().numpy())
    U.check_embed(_report(U.bits_to_f64(U.tensor_bits(out)), wb, U.item_starts(wb.items), bucket_rows=rows))
    # the RoPE expansion alone right after an embedding launch (which lets the next kernel
    # start early) and in a chain of its own
    c2 = torch.full_like(ref_a[1], 7.0)
    s2 = torch.full_like(ref_a[2], 7.0)
    fe.embed_rope(ba, hd, th, rows=rows, out=out, cos=cos, sin=sin, status=st)
    for k in range(7):
        fe.rope(bb if k % 2 == 0 else ba, hd, th, rows=rows, cos=c2, sin=s2, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, -1]
    assert np.array_equal(c2.cpu().numpy(), ref_b[1].cpu().numpy())
    assert np.array_equal(s2.cpu().numpy(), ref_b[2].cpu().numpy())
    assert np.array_equal(U.tensor_bits(out), U.tensor_bits(ref_a[0]))
    fe.close()


def test_embed_rope_graph_replay_with_new_items():
    # one captured fused launch serves buckets whose items change between replays
    wl = synth.small_workload(31, [(1, 4, 6, 1), (2, 2, 4, 4), (1, 8, 8, 1)], patch=14, hidden=256, head_dim=80)
    wl2 = synth.small_workload(32, [(1, 6, 6, 1), (1, 2, 10, 1)], patch=14, hidden=256, head_dim=80)
    fe = _fe(wl)
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    R = 256
    b1 = fe.upload(wl.items, capacity=8)
    px = torch.zeros(max(b1.pixel_bytes, 1 << 20), dtype=torch.uint8, device="cuda")
    items = torch.zeros(8 * 24, dtype=torch.uint8, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((R, 256), dtype=torch.bfloat16, device="cuda")
    cos = torch.empty((R, 40), dtype=torch.float32, device="cuda")
    sin = torch.empty_like(cos)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):      # warm: builds the table outside the capture
        B.vitfe_embed_rope(fe.h, px, px.numel(), items, n, 8, R, out, 80, wl.theta, cos, sin, None, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.vitfe_embed_rope(fe.h, px, px.numel(), items, n, 8, R, out, 80, wl.theta, cos, sin, None, s)
    for w in (wl, wl2):
        recs, buf, live = B.pack_items(w.items, w.patch, w.tpatch)
        px[:buf.size].copy_(torch.from_numpy(buf))
        arr = np.zeros(8, B.ITEM_DTYPE)
        arr[:len(recs)] = recs
        items.copy_(torch.from_numpy(arr.view(np.uint8)))
        n.fill_(len(recs))
        out.fill_(3.0)
        cos.fill_(5.0)
        g.replay()
        torch.cuda.synchronize()
        eb = fe.upload(w.items)
        e = fe.embed(eb)
        c2, _ = fe.rope(eb, 80, w.theta)
        torch.cuda.synchronize()
        assert np.array_equal(U.tensor_bits(out)[:live], U.tensor_bits(e))
        assert np.all(U.tensor_bits(out)[live:] == 0)
        assert np.array_equal(cos.cpu().numpy()[:live], c2.cpu().numpy())
        assert np.all(cos.cpu().numpy()[live:] == 1.0) and np.all(sin.cpu().numpy()[live:] == 0.0)
    fe.close()


@pytest.mark.parametrize("pad", [4, 0])           # 4: 8-byte accesses; 0: 16-byte accesses where aligned
@pytest.mark.parametrize("hd,hq,hk", [(80, 16, 16), (72, 3, 5), (64, 2, 0), (8, 0, 3), (16, 1, 1), (32, 3, 2)])
def test_rope_apply_vs_oracle_in_a_packed_qkv_buffer(hd, hq, hk, pad):
    # Q and K are views into [rows][Q | K | V]; V and the padding must stay untouched
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    rng = np.random.default_rng(hd + hq)
    rows = 333
    pos = np.stack([rng.integers(0, 90, rows), rng.integers(0, 90, rows)], 1)
    pos[-5:] = -1                                       # a few bucket-pad rows (identity)
    c64, s64 = oracle.rope_tables(pos, hd, 10000.0)
    c32, s32 = c64.astype(np.float32), s64.astype(np.float32)
    width = (hq + hk + 2) * hd + pad                    # + V heads and the padding
    x = rng.standard_normal((rows, width)).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    before = U.tensor_bits(xb)
    buf = xb.cuda()
    cos_d = torch.from_numpy(c32).cuda()
    sin_d = torch.from_numpy(s32).cuda()
    q = buf if hq else None
    k = buf[:, hq * hd:] if hk else None
    B.vitfe_rope_apply(cos_d, sin_d, rows, hd, q, hq, width, k, hk, width)
    torch.cuda.synchronize()
    got = U.tensor_bits(buf)
    xin = U.bits_to_f64(before)
    for h0, nh in ((0, hq), (hq, hk)):
        if nh == 0:
            continue
        seg = xin[:, h0 * hd:(h0 + nh) * hd].reshape(rows, nh, hd)
        ref = oracle.rope_apply(seg, c32.astype(np.float64), s32.astype(np.float64)).reshape(rows, nh * hd)
        g = got[:, h0 * hd:(h0 + nh) * hd]
        assert int(U.ulp_distance(g, U.f64_to_bf16_bits(ref)).max()) <= 1
    # pad rows rotate by the identity: bit-exact; everything past Q and K untouched
    assert np.array_equal(got[-5:], before[-5:])
    assert np.array_equal(got[:, (hq + hk) * hd:], before[:, (hq + hk) * hd:])


@pytest.mark.parametrize("name", sorted(SMALL))
def test_embed_folded_vs_folded_oracle(name):
    # stills against the folded oracle (W' rounded once, identically on both sides); tiles
    # holding video rows are computed unfolded, exactly as vitfe_embed computes them
    P, N, grids = SMALL[name]
    wl = synth.small_workload(41, grids, patch=P, hidden=N, pixels="uniform")
    fe = _fe(wl)
    b = fe.upload(wl.items)
    rows = b.live_rows + 100
    st = fe.status_tensor()
    out = fe.embed_folded(b, rows=rows, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, -1]
    g = U.bits_to_f64(U.tensor_bits(out))
    ref = oracle.embed_folded_workload(wl, bucket_rows=rows)
    ref_m = oracle.embed_folded_workload(wl, bucket_rows=rows, bf16_input=True)
    starts = U.item_starts(wl.items)
    still_rows = np.zeros(rows, bool)
    for it, s0, s1 in zip(wl.items, starts[:-1], starts[1:]):
        still_rows[s0:s1] = it.frames == 1
    # a 256-row tile is folded when all of its live rows are stills
    live = b.live_rows
    tile_all_still = np.array([t < live and still_rows[t:min(t + 256, live)].all() for t in range(0, rows, 256)])
    folded_rows = np.repeat(tile_all_still, 256)[:rows] & still_rows
    exact = oracle.embed_workload(wl, bucket_rows=rows)
    exact_m = oracle.embed_workload(wl, bucket_rows=rows, bf16_input=True)
    expect = np.where(folded_rows[:, None], ref, exact)
    expect_m = np.where(folded_rows[:, None], ref_m, exact_m)
    U.check_embed(U.embed_report(g, expect, expect_m, starts))
    assert np.all(U.tensor_bits(out)[b.live_rows:] == 0)
    fe.close()


@pytest.mark.parametrize("chunks", [1, 2, 3, 7])
@pytest.mark.parametrize("name", ["mixed_p14", "stills_p16", "video_p14"])
def test_embed_rope_host_pipeline_equals_the_device_call(name, chunks):
    # host buffers in and out, the items cut into overlapped runs.  The RoPE rows equal the
    # device-buffer call's bit for bit; the embeddings meet the oracle bars (a run boundary
    # changes which rows share a 256-row tile, and with it the K summation order of stills
    # between the resident and stream paths, so bits may differ from the one-call result)
    P, N, grids = SMALL[name]
    hd = 80 if P == 14 else 72
    wl = synth.small_workload(51, grids, patch=P, hidden=N, head_dim=hd, pixels="uniform")
    fe = _fe(wl)
    out, cos, sin, st = fe.embed_rope_host(wl.items, hd, wl.theta, chunks=chunks)
    assert st.tolist() == [0, -1]
    b = fe.upload(wl.items)
    o2, c2, s2 = fe.embed_rope(b, hd, wl.theta)
    torch.cuda.synchronize()
    assert np.array_equal(cos.numpy(), c2.cpu().numpy()) and np.array_equal(sin.numpy(), s2.cpu().numpy())
    U.check_embed(_report(U.bits_to_f64(U.tensor_bits(out)), wl, U.item_starts(wl.items)))
    if chunks == 1:
        assert np.array_equal(U.tensor_bits(out), U.tensor_bits(o2))
    fe.close()


def test_embed_rope_host_reports_errors():
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    wl = synth.small_workload(52, [(1, 4, 6, 1), (1, 2, 2, 1), (1, 6, 4, 1)], patch=14, hidden=256, head_dim=80)
    fe = _fe(wl)
    items, buf, rows = B.pack_items(wl.items, 14, 2)
    out = np.zeros((rows, 256), np.uint16)
    cos = np.zeros((rows, 40), np.float32)
    sin = np.zeros((rows, 40), np.float32)
    st = np.zeros(2, np.int32)
    # pixels past the host buffer: rejected on the host, nothing copied
    with pytest.raises(B.VitfeError) as e:
        B.vitfe_embed_rope_host(fe.h, buf, buf.size - 16, items.view(np.uint8), len(items), out, 80, 1e4, cos, sin,
                                st, 2)
    assert e.value.code == 1
    # a descriptor only the device rejects (w not a multiple of the merge size): reported
    # with its index over all items, its rows zero, the others intact
    bad = items.copy()
    bad["w"][2] = 3
    bad["t"][2] = 1
    rows_bad = int(np.sum(bad["t"] * bad["h"] * bad["w"]))
    out = np.zeros((rows_bad, 256), np.uint16)
    cos = np.zeros((rows_bad, 40), np.float32)
    sin = np.zeros((rows_bad, 40), np.float32)
    B.vitfe_embed_rope_host(fe.h, buf, buf.size, bad.view(np.uint8), len(bad), out, 80, 1e4, cos, sin, st, 3)
    assert st.tolist() == [4, 2]
    assert np.all(out[rows_bad - 6 * 3:] == 0)
    fe.close()


@pytest.mark.parametrize("patch", [14, 16])
def test_bounded_wait_runs_out_and_reports_timeout(monkeypatch, patch):
    # failure detection without a fault: a handle whose weight producer issues no loads
    # (test hook) leaves the MMA's wait unsatisfied; after the short limit every role leaves,
    # the launch reports VITFE_EDEVICE_TIMEOUT, and the context keeps working (patch 16:
    # its producers also write A blocks into tensor memory)
    wl = synth.small_workload(61, [(1, 4, 6, 1), (2, 2, 4, 4)], patch=patch, hidden=256, head_dim=80)
    monkeypatch.setenv("VITFE_WAIT_LIMIT_MS", "200")
    monkeypatch.setenv("VITFE_TEST_STALL_W_LOADS", "1")
    stalled = _fe(wl)
    monkeypatch.delenv("VITFE_TEST_STALL_W_LOADS")
    monkeypatch.delenv("VITFE_WAIT_LIMIT_MS")
    b = stalled.upload(wl.items)
    st = stalled.status_tensor()
    stalled.embed(b, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [6, -1]
    stalled.close()
    # the same process and context: a normal handle still computes correct embeddings
    fe = _fe(wl)
    b = fe.upload(wl.items)
    st = fe.status_tensor()
    out = fe.embed(b, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, -1]
    U.check_embed(_report(U.bits_to_f64(U.tensor_bits(out)), wl, U.item_starts(wl.items)))
    fe.close()


SHAPES = {
    # (patch, tpatch, merge, grids (t, h, w, frames))
    "p14_t1_m2": (14, 1, 2, [(1, 4, 6, 1), (3, 2, 4, 3), (1, 6, 2, 1)]),     # generic normalise kernel
    "p16_t1_m2": (16, 1, 2, [(1, 4, 6, 1), (2, 2, 4, 2)]),                   # <16, 1> normalise kernel
    "p14_t2_m1": (14, 2, 1, [(1, 3, 5, 1), (2, 1, 3, 4), (1, 7, 1, 1)]),     # no merge grouping
    "p14_t2_m4": (14, 2, 4, [(1, 4, 8, 1), (2, 4, 4, 4)]),                   # 4 x 4 merge units
    "p8_t2_m2": (8, 2, 2, [(1, 4, 6, 1), (2, 2, 4, 4)]),                     # no embed kernel for patch 8
    # three and four temporal slices: the slices' one-step tails share one weight image
    "p14_t3_m2": (14, 3, 2, [(1, 2, 4, 1), (1, 4, 2, 3)]),
    "p14_t4_m2": (14, 4, 2, [(1, 4, 6, 1), (2, 2, 4, 8)]),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_other_patch_temporal_and_merge_shapes(name):
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    P, T, M, grids = SHAPES[name]
    wl = synth.small_workload(71, grids, patch=P, tpatch=T, merge=M, hidden=256, pixels="uniform")
    fe = _fe(wl)
    b = fe.upload(wl.items)
    rows = b.live_rows + 19
    flat = fe.normalize_patchify(b, rows=rows)
    got = U.tensor_bits(flat)
    ref = U.f64_to_bf16_bits(oracle.normalize_patchify_workload(wl, bucket_rows=rows))
    assert int(U.ulp_distance(got, ref).max()) <= U.NORM_MAX_ULP
    assert np.array_equal(fe.pos_ids(b, rows=rows).cpu().numpy(), oracle.pos_ids_workload(wl, bucket_rows=rows))
    cos, sin = fe.rope(b, wl.head_dim, wl.theta, rows=rows)
    rc, rs = oracle.rope_workload(wl, bucket_rows=rows)
    assert np.max(np.abs(cos.cpu().numpy() - rc)) <= U.ROPE_MAX_ABS
    assert np.max(np.abs(sin.cpu().numpy() - rs)) <= U.ROPE_MAX_ABS
    if P in (14, 16):
        st = fe.status_tensor()
        out = fe.embed(b, rows=rows, status=st)
        torch.cuda.synchronize()
        assert st.cpu().tolist() == [0, -1]
        e = U.bits_to_f64(U.tensor_bits(out))
        U.check_embed(_report(e, wl, U.item_starts(wl.items), bucket_rows=rows))
        assert np.all(U.tensor_bits(out)[b.live_rows:] == 0)
    else:
        with pytest.raises(B.VitfeError) as err:
            fe.embed(b, rows=rows)
        assert err.value.code == 7
    fe.close()
