"""Pins of the fp64 oracle to things other than itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
swapped channel or mean/std, a transposed axis, a wrong merge order, a wrong
rotary width) fails at least one of them:

* FusedInputNorm: hand-computed values of special parameter sets and the
  zero crossing of the real constants;
* patchify: brute-force nested-loop enumeration from the closed-form row and
  feature index on tiny position-coded items, a hand-derived golden row order,
  and the merge=1 case against plain raster img2col slicing;
* patch embed: a direct Conv3d (kernel == stride) sum on tiny items, a one-hot
  weight that must return the normalised pixels exactly, and the constant
  colour closed form;
* the model-dtype input of the GEMM (bf16_input): a one-hot weight returns the
  pixels rounded to bf16, ties go to even, exact bf16 pixels pass unchanged,
  the change is bounded by the cast's half spacings, and the constant colour
  closed form with each channel rounded by brute force;
* position ids: a hand-derived golden sequence and the closed-form index;
* RoPE: pos 0, frequency index 0, the theta^(-1/2) frequency, geometric
  frequency ratio, angle addition between neighbouring positions,
  cos^2 + sin^2 = 1, the [H || W] layout and pad rows.
"""
import math
import os

import numpy as np
import pytest

import oracle
from vit_vision_encoder_fusedinputnorm_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    return np.array(rows, dtype=np.int64)


# ---------------------------------------------------------------- normalise

def test_normalize_identity_parameters():
    v = np.arange(256, dtype=np.uint8).reshape(1, 1, 256, 1).repeat(3, axis=3)
    x = oracle.normalize(v, (0, 0, 0), (1, 1, 1), 1.0)
    assert np.array_equal(x[..., 0].ravel(), np.arange(256, dtype=np.float64))
    assert np.array_equal(x[..., 2].ravel(), np.arange(256, dtype=np.float64))


def test_normalize_minus_one_to_one():
    # mean 0.5, std 0.5 after 1/255: 0 -> -1, 255 -> +1, 51 -> -0.6.
    v = np.array([[[[0, 255, 51]]]], dtype=np.uint8)
    x = oracle.normalize(v, (0.5, 0.5, 0.5), (0.5, 0.5, 0.5), 1 / 255)
    assert np.allclose(x.ravel(), [-1.0, 1.0, -0.6], atol=1e-15)


def test_normalize_per_channel_hand_values():
    # v = 40 in every channel, mean (0, 10, 20), std (1, 2, 4), rescale 1:
    # channel 0 -> 40, channel 1 -> 15, channel 2 -> 5 (computed by hand).
    v = np.full((1, 1, 1, 3), 40, dtype=np.uint8)
    x = oracle.normalize(v, (0, 10, 20), (1, 2, 4), 1.0)
    assert x.ravel().tolist() == [40.0, 15.0, 5.0]


def test_normalize_zero_crossing_of_clip_constants():
    # mean_c / rescale = 122.78, 116.74, 104.09: the sign flips between these bytes.
    lo = np.array([[[[122, 116, 104]]]], dtype=np.uint8)
    hi = np.array([[[[123, 117, 105]]]], dtype=np.uint8)
    xl = oracle.normalize(lo, synth.QWEN_MEAN, synth.QWEN_STD, synth.RESCALE).ravel()
    xh = oracle.normalize(hi, synth.QWEN_MEAN, synth.QWEN_STD, synth.RESCALE).ravel()
    assert np.all(xl < 0) and np.all(xh > 0)
    # slope per channel is rescale / std_c
    assert np.allclose(xh - xl, [1 / 255 / 0.2686, 1 / 255 / 0.2613, 1 / 255 / 0.2758], rtol=1e-12)


def test_normalize_rejects_non_uint8():
    with pytest.raises(TypeError):
        oracle.normalize(np.zeros((1, 1, 1, 3), np.float32), (0, 0, 0), (1, 1, 1), 1.0)


# ---------------------------------------------------------------- patchify

def _brute_force_rows(x, t, h, w, P, T, m):
    """Nested loops from the closed-form indices (independent of reshape)."""
    F = x.shape[0]
    K = 3 * T * P * P
    out = np.zeros((t * h * w, K), dtype=x.dtype)
    for r in range(t * h * w):
        tg, rem = divmod(r, h * w)
        g, within = divmod(rem, m * m)
        hb, wb = divmod(g, w // m)
        mh, mw = divmod(within, m)
        hh, ww = hb * m + mh, wb * m + mw
        for c in range(3):
            for tt in range(T):
                f = 0 if F == 1 else tg * T + tt
                for ph in range(P):
                    for pw in range(P):
                        k = ((c * T + tt) * P + ph) * P + pw
                        out[r, k] = x[f, hh * P + ph, ww * P + pw, c]
    return out


@pytest.mark.parametrize("t,h,w,F,P,T,m", [
    (1, 2, 2, 1, 14, 2, 2),     # 28 x 28 still
    (1, 2, 4, 1, 14, 2, 2),     # 28 x 56
    (1, 4, 6, 1, 14, 2, 2),     # 56 x 84
    (2, 2, 4, 4, 14, 2, 2),     # 4-frame video 28 x 56
    (1, 2, 4, 1, 16, 2, 2),     # 32 x 64, patch 16
    (1, 6, 3, 1, 4, 2, 3),      # merge 3
    (3, 2, 2, 3, 4, 1, 2),      # temporal patch 1, 3 frames
])
def test_patchify_brute_force(t, h, w, F, P, T, m):
    x = synth.position_coded_image(F, h * P, w * P)
    got = oracle.patchify(x, t, h, w, P, T, m)
    exp = _brute_force_rows(x, t, h, w, P, T, m)
    assert got.shape == (t * h * w, 3 * T * P * P)
    assert np.array_equal(got, exp)


def test_patch_row_order_golden():
    g = _golden("patch_rows_h2_w4_m2.txt")
    for merge in (2, 1):
        exp = g[g[:, 0] == merge][:, 1:]
        coords = oracle.patch_coords(1, 2, 4, merge)
        assert np.array_equal(coords[:, 1:], exp)
        # and the patchified rows hold exactly those patches
        P = 2
        x = synth.position_coded_image(1, 2 * P, 4 * P)
        rows = oracle.patchify(x, 1, 2, 4, P, 2, merge)
        for r, (hh, ww) in enumerate(exp):
            blk = x[0, hh * P:(hh + 1) * P, ww * P:(ww + 1) * P, :]       # [P][P][C]
            ref = np.stack([blk, blk], 0).transpose(3, 0, 1, 2).ravel()   # (C, T, P, P)
            assert np.array_equal(rows[r], ref)


def test_patchify_merge1_is_raster_img2col():
    t, h, w, P, T = 1, 3, 5, 4, 2
    x = synth.position_coded_image(1, h * P, w * P)
    rows = oracle.patchify(x, t, h, w, P, T, 1)
    r = 0
    for hh in range(h):
        for ww in range(w):
            blk = x[0, hh * P:(hh + 1) * P, ww * P:(ww + 1) * P, :].transpose(2, 0, 1)  # C,P,P
            exp = np.stack([blk, blk], axis=1).ravel()                                 # C,T,P,P
            assert np.array_equal(rows[r], exp)
            r += 1


def test_patchify_counts_and_errors():
    x = np.zeros((1, 56, 84, 3), np.uint8)
    assert oracle.patchify(x, 1, 4, 6, 14, 2, 2).shape == (24, 1176)
    with pytest.raises(ValueError):
        oracle.patchify(np.zeros((1, 42, 84, 3), np.uint8), 1, 3, 6, 14, 2, 2)   # h not multiple of m
    with pytest.raises(ValueError):
        oracle.patchify(np.zeros((3, 28, 28, 3), np.uint8), 1, 2, 2, 14, 2, 2)   # frames != t*T


def test_workload_row_counts():
    # grid_thw counts: (H/P)(W/P) t per item.
    assert synth.make_workload(0, with_pixels=False).live_rows == 256
    assert synth.make_workload(1, with_pixels=False).live_rows == 18048
    assert synth.make_workload(2, with_pixels=False).live_rows == 589824
    w3 = synth.make_workload(3, with_pixels=False)
    assert (w3.items[0].t, w3.items[0].h, w3.items[0].w) == (16, 32, 56)
    assert w3.live_rows == 45056
    w4 = synth.make_workload(4, with_pixels=False)
    assert w4.K == 1536 and w4.hidden == 1152
    for b in w4.buckets:
        assert sum(w4.items[i].rows for i in b) <= 65536
    assert sum(len(b) for b in w4.buckets) == 50


# ---------------------------------------------------------------- embed

def _closed_form_row(tg, hh, ww, h, w, m):
    hb, mh = divmod(hh, m)
    wb, mw = divmod(ww, m)
    return ((tg * (h // m) + hb) * (w // m) + wb) * m * m + mh * m + mw


@pytest.mark.parametrize("t,h,w,F", [(1, 2, 4, 1), (2, 2, 2, 4)])
def test_embed_equals_direct_conv3d(t, h, w, F):
    P, T, m, N = 4, 2, 2, 5
    rng = np.random.default_rng(7)
    x = rng.integers(0, 256, size=(F, h * P, w * P, 3), dtype=np.uint8)
    W = synth.f32_to_bf16_bits(rng.standard_normal((N, 3 * T * P * P)).astype(np.float32) * 0.05)
    b = synth.f32_to_bf16_bits(rng.standard_normal(N).astype(np.float32) * 0.05)
    # identity normalisation (pinned above), so the conv sees the raw pixel values
    y = oracle.embed_item(x, t, h, w, W, b, patch=P, tpatch=T, merge=m, mean=(0, 0, 0),
                          std=(1, 1, 1), rescale=1.0)
    W5 = oracle.bf16_bits_to_f64(W).reshape(N, 3, T, P, P)
    conv = _direct_conv3d_float(x.astype(np.float64), t, h, w, P, T, W5,
                                oracle.bf16_bits_to_f64(b))
    for tg in range(t):
        for hh in range(h):
            for ww in range(w):
                r = _closed_form_row(tg, hh, ww, h, w, m)
                assert np.allclose(y[r], conv[tg, hh, ww], rtol=1e-12, atol=1e-12)


def _direct_conv3d_float(xf, t, h, w, P, T, W5, bias):
    F = xf.shape[0]
    X = xf.transpose(0, 3, 1, 2)
    N = W5.shape[0]
    out = np.zeros((t, h, w, N))
    for tg in range(t):
        frames = [0] * T if F == 1 else [tg * T + tt for tt in range(T)]
        for hh in range(h):
            for ww in range(w):
                blk = np.stack([X[f, :, hh * P:(hh + 1) * P, ww * P:(ww + 1) * P] for f in frames],
                               axis=1)
                for n in range(N):
                    acc = 0.0
                    for idx in np.ndindex(blk.shape):
                        acc += W5[(n,) + idx] * blk[idx]
                    out[tg, hh, ww, n] = acc + bias[n]
    return out


def test_embed_one_hot_weight_returns_pixels():
    # W[n][k] = [k == k_n], b = 0, identity normalisation: y[:, n] = A[:, k_n] = a pixel value.
    P, T, m = 4, 2, 2
    K = 3 * T * P * P
    ks = [0, 1, 17, K // 2, K - 1]
    W = np.zeros((len(ks), K), np.uint16)
    for n, k in enumerate(ks):
        W[n, k] = 0x3F80                       # bf16 1.0
    x = synth.position_coded_image(1, 2 * P, 4 * P)
    y = oracle.embed_item(x, 1, 2, 4, W, None, patch=P, tpatch=T, merge=m, mean=(0, 0, 0),
                          std=(1, 1, 1), rescale=1.0)
    for n, k in enumerate(ks):
        c, rest = divmod(k, T * P * P)
        tt, rest = divmod(rest, P * P)
        ph, pw = divmod(rest, P)
        for r in range(8):              # grid 2 x 4, merge 2: one merge row of two units
            wb, within = divmod(r, 4)
            mh, mw = divmod(within, 2)
            hh, ww = mh, wb * 2 + mw
            assert y[r, n] == x[0, hh * P + ph, ww * P + pw, c]


def test_embed_constant_colour_closed_form():
    P, T, m, N = 4, 2, 2, 6
    rng = np.random.default_rng(3)
    W = synth.f32_to_bf16_bits(rng.standard_normal((N, 3 * T * P * P)).astype(np.float32) * 0.02)
    b = synth.f32_to_bf16_bits(rng.standard_normal(N).astype(np.float32) * 0.02)
    col = (200, 17, 90)
    x = np.empty((1, 2 * P, 2 * P, 3), np.uint8)
    x[...] = col
    y = oracle.embed_item(x, 1, 2, 2, W, b, patch=P, tpatch=T, merge=m, mean=synth.QWEN_MEAN,
                          std=synth.QWEN_STD, rescale=synth.RESCALE)
    Wf = oracle.bf16_bits_to_f64(W).reshape(N, 3, -1).sum(axis=2)        # per-channel weight sums
    xc = [(col[c] / 255.0 - synth.QWEN_MEAN[c]) / synth.QWEN_STD[c] for c in range(3)]
    exp = Wf @ np.array(xc) + oracle.bf16_bits_to_f64(b)
    assert np.allclose(y, exp[None, :], rtol=1e-12, atol=1e-13)


def test_embed_linear_in_weight_and_bias():
    P, T, m = 4, 2, 2
    rng = np.random.default_rng(5)
    x = rng.integers(0, 256, size=(1, 2 * P, 2 * P, 3), dtype=np.uint8)
    W1 = synth.f32_to_bf16_bits(rng.standard_normal((3, 96)).astype(np.float32))
    W2 = synth.f32_to_bf16_bits(rng.standard_normal((3, 96)).astype(np.float32))
    kw = dict(patch=P, tpatch=T, merge=m, mean=(0.1, 0.2, 0.3), std=(0.5, 0.6, 0.7), rescale=0.01)
    y1 = oracle.embed_item(x, 1, 2, 2, W1, None, **kw)
    y2 = oracle.embed_item(x, 1, 2, 2, W2, None, **kw)
    W12 = synth.f32_to_bf16_bits(oracle.bf16_bits_to_f64(W1).astype(np.float32)
                                 + oracle.bf16_bits_to_f64(W2).astype(np.float32))
    y12 = oracle.embed_item(x, 1, 2, 2, W12, None, **kw)
    # W1 + W2 rounded to bf16: compare within bf16 rounding of the weights
    assert np.allclose(y12, y1 + y2, rtol=2e-2, atol=2e-2)


def test_embed_workload_sample_and_bucket():
    wl = synth.small_workload(11, [(1, 2, 4, 1), (2, 2, 2, 4), (1, 4, 2, 1)], patch=4, hidden=8)
    full = oracle.embed_workload(wl, bucket_rows=40)
    assert full.shape == (40, 8)
    assert np.all(full[wl.live_rows:] == 0)
    s = np.array([0, 5, 9, 8, 23, 17])
    assert np.array_equal(oracle.embed_workload(wl, sample=s), full[s])


# ---------------------------------------------------------------- the model-dtype input of the GEMM

def test_bf16_input_one_hot_returns_the_rounded_pixels():
    # a one-hot weight passes A through: with bf16_input the outputs are the normalised
    # pixels rounded to bf16 (to nearest, ties to even), and without it the exact values
    P, T, m = 4, 2, 2
    K = 3 * T * P * P
    ks = [0, 5, 47, K - 1]
    W = np.zeros((len(ks), K), np.uint16)
    W[np.arange(len(ks)), ks] = 0x3F80
    x = synth.position_coded_image(1, 2 * P, 4 * P)
    kw = dict(patch=P, tpatch=T, merge=m, mean=synth.QWEN_MEAN, std=synth.QWEN_STD, rescale=synth.RESCALE)
    exact = oracle.embed_item(x, 1, 2, 4, W, None, **kw)
    cast = oracle.embed_item(x, 1, 2, 4, W, None, bf16_input=True, **kw)
    A = oracle.normalize_patchify_item(x, 1, 2, 4, **kw)[:, ks]
    assert np.array_equal(exact, A)
    assert np.array_equal(cast, oracle.bf16_bits_to_f64(oracle.round_to_bf16_bits(A)))
    assert np.any(cast != exact)


def test_bf16_input_ties_go_to_even():
    # mean -1, std 1, rescale 1/512: x = 1 + v/512, and the bf16 spacing in [1, 2) is 4/512.
    # v = 2: halfway between 1 (even) and 1 + 4/512 -> 1; v = 6: halfway between 1 + 4/512
    # (odd) and 1 + 8/512 (even) -> 1 + 8/512; v = 1, 3: nearest; v = 4: a bf16 value
    P = 8
    vals = [2, 6, 1, 3, 4]
    x = np.zeros((1, P, P, 3), np.uint8)
    x[0, 0, :len(vals), 0] = vals
    W5 = np.zeros((len(vals), 3, P, P), np.uint16)
    for n in range(len(vals)):
        W5[n, 0, 0, n] = 0x3F80                                       # Conv3d order (c, ph, pw)
    y = oracle.embed_item(x, 1, 1, 1, W5.reshape(len(vals), -1), None, patch=P, tpatch=1, merge=1,
                          mean=(-1, -1, -1), std=(1, 1, 1), rescale=1 / 512, bf16_input=True)
    assert y[0].tolist() == [1.0, 1 + 8 / 512, 1.0, 1 + 4 / 512, 1 + 4 / 512]
    y = oracle.embed_item(x, 1, 1, 1, W5.reshape(len(vals), -1), None, patch=P, tpatch=1, merge=1,
                          mean=(-1, -1, -1), std=(1, 1, 1), rescale=1 / 512)
    assert y[0].tolist() == [1 + v / 512 for v in vals]


def test_bf16_input_changes_nothing_when_the_pixels_are_bf16_values():
    # rescale 1/256, mean 0, std 1: v / 256 has at most 8 significant bits, so the cast
    # is exact and both oracles agree bit for bit
    wl = synth.small_workload(12, [(1, 2, 4, 1), (2, 2, 2, 4)], patch=4, hidden=16)
    wl.mean, wl.std, wl.rescale = (0.0, 0.0, 0.0), (1.0, 1.0, 1.0), 1 / 256
    assert np.array_equal(oracle.embed_workload(wl, bf16_input=True), oracle.embed_workload(wl))


def test_bf16_input_difference_is_bounded_by_the_cast():
    # |y_cast - y| <= sum_k |W[n][k]| * (half a bf16 spacing at |x_k|) for every row and
    # column, and the cast moves the results (a dropped or doubled rounding would not fit)
    wl = synth.small_workload(13, [(1, 4, 6, 1), (2, 2, 2, 4)], patch=4, hidden=24)
    y = oracle.embed_workload(wl)
    yc = oracle.embed_workload(wl, bf16_input=True)
    A = np.concatenate([oracle.normalize_patchify_item(it.pixels, it.t, it.h, it.w, patch=4, tpatch=2, merge=2,
                                                       mean=wl.mean, std=wl.std, rescale=wl.rescale)
                        for it in wl.items])
    _, ex = np.frexp(np.abs(A))
    half = np.ldexp(1.0, ex - 9)
    bound = half @ np.abs(oracle.bf16_bits_to_f64(wl.W_bits)).T
    d = np.abs(yc - y)
    assert np.all(d <= bound * (1 + 1e-12))
    assert d.max() > 0.05 * bound.max()


def test_bf16_input_constant_colour_closed_form():
    P, T, m, N = 4, 2, 2, 6
    rng = np.random.default_rng(4)
    W = synth.f32_to_bf16_bits(rng.standard_normal((N, 3 * T * P * P)).astype(np.float32) * 0.02)
    b = synth.f32_to_bf16_bits(rng.standard_normal(N).astype(np.float32) * 0.02)
    col = (31, 222, 140)
    x = np.empty((1, 2 * P, 2 * P, 3), np.uint8)
    x[...] = col
    y = oracle.embed_item(x, 1, 2, 2, W, b, patch=P, tpatch=T, merge=m, mean=synth.QWEN_MEAN,
                          std=synth.QWEN_STD, rescale=synth.RESCALE, bf16_input=True)
    Wf = oracle.bf16_bits_to_f64(W).reshape(N, 3, -1).sum(axis=2)
    xc = np.array([(col[c] / 255.0 - synth.QWEN_MEAN[c]) / synth.QWEN_STD[c] for c in range(3)])
    # bf16 of each channel's value, from its own brute force over the bf16 grid near it
    xb = []
    for v in xc:
        e = math.floor(math.log2(abs(v)))
        step = 2.0 ** (e - 7)
        lo = math.floor(v / step) * step
        cands = [lo, lo + step]
        best = min(cands, key=lambda c: (abs(c - v), (round(c / step) % 2)))
        xb.append(best)
    exp = Wf @ np.array(xb) + oracle.bf16_bits_to_f64(b)
    assert np.allclose(y, exp[None, :], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- position ids

def test_pos_ids_golden():
    assert np.array_equal(oracle.pos_ids(2, 2, 4, 2), _golden("pos_ids_t2_h2_w4_m2.txt"))


@pytest.mark.parametrize("t,h,w,m", [(1, 16, 16, 2), (3, 4, 10, 2), (1, 6, 9, 3), (2, 5, 7, 1)])
def test_pos_ids_closed_form(t, h, w, m):
    p = oracle.pos_ids(t, h, w, m)
    for tg in range(t):
        for hh in range(h):
            for ww in range(w):
                r = _closed_form_row(tg, hh, ww, h, w, m)
                assert tuple(p[r]) == (hh, ww)


def test_pos_ids_agree_with_patch_coords():
    c = oracle.patch_coords(3, 4, 6, 2)
    assert np.array_equal(oracle.pos_ids(3, 4, 6, 2), c[:, 1:])


# ---------------------------------------------------------------- folded-still variant

def _bits(vals):
    return np.array(vals, np.float32).view(np.uint32) >> 16


def test_round_to_bf16_ties_to_even_and_exact_values():
    # bf16 keeps 8 significant bits: at 1.0 the spacing is 2^-7 and 1 + 2^-8 is a tie
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -30, -(1.0 + 3 * 2 ** -8),
                  0.0, 2.0 ** -100, 255.0, 257.0, 0.02])
    got = oracle.round_to_bf16_bits(x)
    expect = [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xBF82, 0x0000, int(_bits([2.0 ** -100])[0]), 0x437F, 0x4380]
    assert got[:9].tolist() == expect
    # 0.02 against a brute force over the neighbouring bf16 values (nearest, then even)
    v = 0.02
    cands = [(abs(float(np.array([c << 16], np.uint32).view(np.float32)[0]) - v), c & 1, c)
             for c in range(0x3C00, 0x3D00)]
    assert int(got[9]) == min(cands)[2]


def test_folded_weight_zero_second_slice_and_exact_sums():
    rng = np.random.default_rng(5)
    P, T, N = 14, 2, 6
    K = 3 * T * P * P
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32).view(np.uint32) >> 16
    W = W.astype(np.uint16).reshape(N, 3, T, P * P)
    Wz = W.copy()
    Wz[:, :, 1, :] = 0
    # slice 1 zero: the fold is slice 0 itself, bit for bit
    assert np.array_equal(oracle.fold_still_weight(Wz.reshape(N, K), T, P), Wz[:, :, 0, :].reshape(N, -1))
    # equal slices: the sum doubles exactly
    We = W.copy()
    We[:, :, 1, :] = We[:, :, 0, :]
    f = oracle.bf16_bits_to_f64(oracle.fold_still_weight(We.reshape(N, K), T, P))
    assert np.array_equal(f, 2 * oracle.bf16_bits_to_f64(We[:, :, 0, :].reshape(N, -1)))


def test_folded_embed_equals_step3_when_the_fold_is_exact():
    # with equal weight slices the folded weight is exact, so the folded variant of a
    # still reproduces step 3 (up to float64 summation order)
    from vit_vision_encoder_fusedinputnorm_gb300 import synth
    wl = synth.small_workload(8, [(1, 4, 6, 1), (1, 2, 2, 1)], patch=14, hidden=32, pixels="uniform")
    N, K = wl.W_bits.shape
    W = wl.W_bits.reshape(N, 3, 2, 14 * 14).copy()
    W[:, :, 1, :] = W[:, :, 0, :]
    wl.W_bits = W.reshape(N, K)
    a = oracle.embed_folded_workload(wl)
    b = oracle.embed_workload(wl)
    assert np.allclose(a, b, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- RoPE applied to Q/K

def _apply_case(seed=0, rows=7, heads=3, hd=16):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, heads, hd))
    pos = np.stack([rng.integers(0, 50, rows), rng.integers(0, 50, rows)], 1)
    c, s = oracle.rope_tables(pos, hd, 10000.0)
    return x, pos, c, s


def test_rope_apply_is_complex_rotation_of_half_pairs():
    # (x_i, x_{i+h}) as the complex number x_i + 1j*x_{i+h}, multiplied by e^{1j*angle}
    x, pos, c, s = _apply_case()
    h = x.shape[-1] // 2
    ang = np.arctan2(s, c)[:, None, :]
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * ang)
    y = oracle.rope_apply(x, c, s)
    assert np.allclose(y[..., :h], z.real, atol=1e-12) and np.allclose(y[..., h:], z.imag, atol=1e-12)


def test_rope_apply_identity_at_origin_norms_and_inverse():
    x, pos, c, s = _apply_case(1)
    h = x.shape[-1] // 2
    zero = np.zeros((len(x), 2), np.int64)
    c0, s0 = oracle.rope_tables(zero, x.shape[-1], 10000.0)
    assert np.array_equal(oracle.rope_apply(x, c0, s0), x)
    y = oracle.rope_apply(x, c, s)
    assert np.allclose(np.hypot(y[..., :h], y[..., h:]), np.hypot(x[..., :h], x[..., h:]), atol=1e-12)
    assert np.allclose(oracle.rope_apply(y, c, -s), x, atol=1e-12)


def test_rope_apply_scores_depend_on_relative_position_only():
    # <R(p) q, R(p') k> is unchanged when both positions shift by the same offset (per axis)
    rng = np.random.default_rng(2)
    hd = 16
    q = rng.standard_normal((1, 1, hd))
    k = rng.standard_normal((1, 1, hd))

    def score(pq, pk):
        cq, sq = oracle.rope_tables(np.array([pq]), hd, 100.0)
        ck, sk = oracle.rope_tables(np.array([pk]), hd, 100.0)
        return float(np.sum(oracle.rope_apply(q, cq, sq) * oracle.rope_apply(k, ck, sk)))

    base = score((3, 5), (1, 9))
    assert abs(score((13, 25), (11, 29)) - base) < 1e-9
    assert abs(score((3, 5), (2, 9)) - base) > 1e-6      # and does change with the offset


# ---------------------------------------------------------------- cu_seqlens

def test_cu_seqlens_boundaries_are_where_item_or_frame_group_changes():
    # independent construction: label every row of the packed items with (item, temporal
    # group) from the patch order itself, then take the rows where the label changes
    grids = [(1, 4, 6), (3, 2, 4), (1, 2, 2), (2, 6, 2)]
    labels = np.concatenate([np.stack([np.full(t * h * w, i), oracle.patch_coords(t, h, w, 2)[:, 0]], 1)
                             for i, (t, h, w) in enumerate(grids)])
    change = np.flatnonzero(np.any(labels[1:] != labels[:-1], axis=1)) + 1
    expect = np.concatenate([[0], change, [len(labels)]])
    cu, mx = oracle.cu_seqlens(grids)
    assert np.array_equal(cu, expect)
    assert mx == int(np.max(np.diff(expect)))


def test_cu_seqlens_stills_are_one_sequence_per_image():
    cu, mx = oracle.cu_seqlens([(1, 16, 16), (1, 4, 6), (1, 96, 96)])
    assert cu.tolist() == [0, 256, 280, 280 + 9216] and mx == 9216
    assert oracle.cu_seqlens([])[0].tolist() == [0]


# ---------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    cos, sin = oracle.rope_tables(np.zeros((3, 2), np.int64), 80, 10000.0)
    assert cos.shape == (3, 40)
    assert np.all(cos == 1.0) and np.all(sin == 0.0)


def test_rope_first_frequency_is_position():
    pos = np.array([[5, 11], [0, 95]])
    cos, sin = oracle.rope_tables(pos, 80, 10000.0)
    assert cos[0, 0] == pytest.approx(math.cos(5), abs=1e-15)
    assert sin[0, 20] == pytest.approx(math.sin(11), abs=1e-15)
    assert sin[1, 20] == pytest.approx(math.sin(95), abs=1e-15)


def test_rope_middle_frequency_closed_form():
    # head_dim 80: rotary width 40, i = 10 gives theta^(-20/40) = 1/100 for theta 1e4.
    pos = np.array([[37, 3]])
    cos, sin = oracle.rope_tables(pos, 80, 10000.0)
    assert cos[0, 10] == pytest.approx(math.cos(0.37), abs=1e-15)
    assert sin[0, 30] == pytest.approx(math.sin(0.03), abs=1e-15)


def test_rope_geometric_frequencies_and_width():
    for head_dim, ratio in [(80, 10000 ** (-1 / 20)), (72, 10000 ** (-1 / 18))]:
        cos, sin = oracle.rope_tables(np.array([[1, 1]]), head_dim, 10000.0)
        assert cos.shape[1] == head_dim // 2
        ang = np.arctan2(sin[0, :head_dim // 4], cos[0, :head_dim // 4])
        assert np.allclose(ang[1:] / ang[:-1], ratio, rtol=1e-12)


def test_rope_angle_addition_between_positions():
    pos = np.stack([np.arange(50), np.arange(50)[::-1]], 1)
    cos, sin = oracle.rope_tables(pos, 80, 10000.0)
    one_c, one_s = oracle.rope_tables(np.array([[1, 1]]), 80, 10000.0)
    h = slice(0, 20)
    # row p+1 (hpos) from row p and position 1
    nc = cos[:-1, h] * one_c[0, h] - sin[:-1, h] * one_s[0, h]
    assert np.allclose(nc, cos[1:, h], atol=1e-12)
    assert np.allclose(cos ** 2 + sin ** 2, 1.0, atol=1e-14)


def test_rope_layout_h_then_w_and_padding():
    cos, sin = oracle.rope_tables(np.array([[0, 5], [-1, -1]]), 80, 10000.0)
    assert np.all(cos[0, :20] == 1.0) and not np.any(cos[0, 20:] == 1.0)
    assert np.all(cos[1] == 1.0) and np.all(sin[1] == 0.0)


def test_rope_workload_rows_match_items():
    wl = synth.small_workload(2, [(1, 2, 4, 1), (2, 2, 2, 4)], patch=4, hidden=8)
    cos, sin = oracle.rope_workload(wl, bucket_rows=20)
    assert cos.shape == (20, 40)
    assert np.all(cos[wl.live_rows:] == 1.0)
