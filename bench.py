"""Benchmark of the fused ViT front end (patch embeddings/s, % of dense bf16 peak).

One step = one pass of the front end over 64 synthetic 1344x1344 stills
(589,824 patches): the fused normalise + patchify + patch-embed GEMM + bias and
the 2D-RoPE rows in one launch (vitfe_embed_rope), through the C ABI with
inputs resident in device memory.  Inputs (347 MB of pixels) and outputs
(1.51 GB of embeddings) exceed the 129 MB L2, so no flush is needed between
iterations.  Steps run back to back with nothing between the launches, so
consecutive launches overlap by programmatic dependent launch (the next step's
prologue, A production and first passes run while the previous step finishes;
each step's writes wait for the previous one); ``roofline.kernel_ms`` is the
time per launch over that region, ``kernel_ms_serial`` the same launch with an
event recorded between launches.  The line also carries: the same step back to back for seconds
(``sustained``, the clock under the power cap); every other workload as the
same fused call (``per_config``: one image, eight mixed images, the video
batch, and the patch-16 buckets as graph replays), each with the oracle's rate
on this host beside it; and the host-buffer path (``e2e``) with the measured
page-locked copy bandwidth that bounds it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU: one process per GPU (torchrun); every rank runs the whole workload
on its own GPU (items are independent, the weights are replicated), so scaling
is weak and there is no data-path collective.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CFG = 2
E2E_CHUNKS = 16
METRIC = "patch embeddings/sec (uint8->bf16 hidden) and % of GB300 dense bf16 peak"
UNIT = "patches/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS, bf16_tflops_sustained=1700.0), "fallback"


def datasheet_fracs(path, achieved_tflops, hbm_gbs_by_path):
    """Fractions of a datasheet's peaks, when a JSON file supplies them (nothing is
    hard-coded): {"bf16_tflops": T, "hbm_gbs": B}, either key optional.  Returns None
    without a file."""
    if not path:
        return None
    with open(path) as f:
        ds = json.load(f)
    out = {"file": os.path.basename(path)}
    if ds.get("bf16_tflops"):
        out["bf16_tflops"] = float(ds["bf16_tflops"])
        out["frac"] = achieved_tflops / float(ds["bf16_tflops"])
    if ds.get("hbm_gbs"):
        out["hbm_gbs"] = float(ds["hbm_gbs"])
        out["hbm_fracs"] = {k: v / float(ds["hbm_gbs"]) for k, v in hbm_gbs_by_path.items()}
    return out


def source_hash() -> str:
    """Hash of the embed kernel's code (comments and whitespace stripped, so that editing a
    comment does not disown the committed ncu traffic figure)."""
    import re
    h = hashlib.sha256()
    for f in ["vitfe_embed.cu", "vitfe_internal.cuh"]:
        with open(os.path.join(ROOT, "vit_vision_encoder_fusedinputnorm_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the embed kernel from the committed ncu summary, if current."""
    p = os.path.join(ROOT, "profiles", "embed_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != source_hash():
        return None
    return d.get("dram_bytes_per_launch_full")


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _oracle_strip(img: int, merge_rows: int):
    """Time the oracle on the top ``merge_rows`` merge rows of image ``img`` of the workload."""
    import dataclasses
    import oracle
    from vit_vision_encoder_fusedinputnorm_gb300 import synth
    wl = synth.make_workload(CFG, item_subset=[img])
    it = wl.items[img]
    mr = min(merge_rows, it.h // wl.merge)
    H = mr * wl.merge * wl.patch
    strip = synth.Item(t=1, h=mr * wl.merge, w=it.w, frames=1, pixels=np.ascontiguousarray(it.pixels[:, :H]))
    sub = dataclasses.replace(wl, items=[strip])
    t0 = time.perf_counter()
    oracle.embed_workload(sub)
    return strip.rows, time.perf_counter() - t0


def _cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def cpu_baseline(budget_s: float = 12.0):
    """The oracle as it stands, on this host's cores, on whole images of the workload."""
    done, t_total, i = 0, 0.0, 0
    while t_total < budget_s and i < 64:
        n, dt = _oracle_strip(i, 10 ** 6)
        done += n
        t_total += dt
        i += 1
    return {"value": done / t_total, "unit": UNIT, "cores": _cores(), "kind": "oracle",
            "sample": f"{i} whole images of 64 ({done} patches): fp64 numpy oracle "
                      f"(normalise, patchify, BLAS GEMM), {t_total:.1f} s"}


def world_max(x: float, world: int, device) -> float:
    """The slowest replica's figure: max over the ranks of the process group."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(rows_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job patches/s: every rank embeds its own copy of the workload (replicas, weak
    scaling), so the job processes world * rows per step in the slowest rank's time."""
    return world * rows_per_rank / (ms_per_step / 1e3)


def run_reference(args, rank, world):
    """The oracle timed as the reference arm, on this host's cores.  Each step is a bounded
    sample of the workload (the top merge rows of one image), sized so that the whole run
    stays within about two minutes; ms_per_step and rows_per_step are the sample's own."""
    if rank != 0:
        return 0
    per_step = max(0.2, 100.0 / (args.steps + args.warmup))
    n, dt = _oracle_strip(0, 4)                    # calibration
    merge_rows = max(1, min(48, int(4 * per_step / max(dt, 1e-3))))
    for w in range(args.warmup):
        _oracle_strip(w % 64, merge_rows)
    rows_done, t_done = 0, 0.0
    for k in range(args.steps):
        n, dt = _oracle_strip(k % 64, merge_rows)
        rows_done += n
        t_done += dt
    v = rows_done / t_done
    strip_rows = rows_done // args.steps
    part = "the whole image" if merge_rows >= 48 else f"its top {merge_rows} merge rows"
    sample = (f"each step: one 1344x1344 image of the workload, {part} ({strip_rows} patches), fp64 numpy "
              f"oracle (normalise, patchify, BLAS GEMM)")
    line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_done / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "64 x 1344x1344 uint8 stills, patch 14, tpatch 2, merge 2, K 1176, N 1280",
                       "rows_per_step": strip_rows,
                       "step": "a bounded sample: one strip of one image per step (rows_per_step patches)"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": _cores(), "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def oracle_items_rate(wl, budget_s: float):
    """The oracle as it stands on whole items of a workload, in order, until about
    ``budget_s`` seconds (at least one item): (patches/s, rows, items timed, seconds)."""
    import dataclasses
    import oracle
    rows, t, n = 0, 0.0, 0
    for it in wl.items:
        sub = dataclasses.replace(wl, items=[it], bucket_rows=None, buckets=None)
        t0 = time.perf_counter()
        oracle.embed_workload(sub)
        t += time.perf_counter() - t0
        rows += it.rows
        n += 1
        if t >= budget_s:
            break
    return rows / t, rows, n, t


def kernel_only(args):
    """Small case for ncu captures: one entry point on the first ``images`` images."""
    import torch
    from vit_vision_encoder_fusedinputnorm_gb300 import build as vbuild
    from vit_vision_encoder_fusedinputnorm_gb300 import synth
    from vit_vision_encoder_fusedinputnorm_gb300.frontend import FrontEnd
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    vbuild.build()
    if args.cfg == 4:
        # the patch-16 workload: its first 65,536-row bucket of stills
        wl = synth.make_workload(4)
        wl.items = [wl.items[i] for i in wl.buckets[0]]
    else:
        wl = synth.make_workload(args.cfg, item_subset=list(range(args.images)))
        wl.items = wl.items[:args.images]
    fe = FrontEnd.from_workload(wl)
    b = fe.upload(wl.items)
    st = fe.status_tensor()
    bufs = {}
    for i in range(args.warmup + args.launches):
        if args.kernel_only == "embed":
            bufs["o"] = fe.embed(b, out=bufs.get("o"), status=st)
        elif args.kernel_only == "embed_rope":
            o, c, s_ = fe.embed_rope(b, wl.head_dim, wl.theta, out=bufs.get("o"), cos=bufs.get("c"),
                                     sin=bufs.get("s"), status=st)
            bufs["o"], bufs["c"], bufs["s"] = o, c, s_
        elif args.kernel_only == "rope":
            c, s_ = fe.rope(b, wl.head_dim, wl.theta, cos=bufs.get("c"), sin=bufs.get("s"), status=st)
            bufs["c"], bufs["s"] = c, s_
        elif args.kernel_only == "rope_apply":
            if "qkv" not in bufs:
                bufs["c"], bufs["s"] = fe.rope(b, wl.head_dim, wl.theta, status=st)
                bufs["qkv"] = torch.zeros((b.live_rows, 3 * wl.hidden), dtype=torch.bfloat16, device="cuda")
            heads = wl.hidden // wl.head_dim
            q = bufs["qkv"]
            B.vitfe_rope_apply(bufs["c"], bufs["s"], b.live_rows, wl.head_dim, q, heads, 3 * wl.hidden,
                               q[:, wl.hidden:], heads, 3 * wl.hidden)
        else:
            bufs["o"] = fe.normalize_patchify(b, out=bufs.get("o"), status=st)
    torch.cuda.synchronize()
    if st.cpu().tolist() != [0, -1]:
        raise RuntimeError(f"device status {st.cpu().tolist()}")
    fe.close()
    return 0


def link_bandwidth(torch, dev, host_in, host_out, stream):
    """Page-locked host <-> device copy bandwidth on this machine (cudaMemcpyAsync through torch):
    up alone, down alone, and both at once on two streams.  GB/s, best of three."""
    d_in = torch.empty(host_in.numel(), dtype=torch.uint8, device=dev)
    d_out = torch.empty(host_out.numel() * host_out.element_size(), dtype=torch.uint8, device=dev)
    h_out = host_out.view(-1).view(torch.uint8)
    h_in = host_in.view(-1).view(torch.uint8)
    s2 = torch.cuda.Stream(device=dev)

    def run(up, down):
        best = float("inf")
        for _ in range(3):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            if up:
                with torch.cuda.stream(stream):
                    d_in.copy_(h_in, non_blocking=True)
            if down:
                with torch.cuda.stream(s2):
                    h_out.copy_(d_out, non_blocking=True)
            torch.cuda.synchronize(dev)
            best = min(best, time.perf_counter() - t0)
        return best

    t_up, t_down, t_both = run(True, False), run(False, True), run(True, True)
    nb_in, nb_out = h_in.numel(), h_out.numel()
    del d_in, d_out
    return {"h2d_gbs": nb_in / t_up / 1e9, "d2h_gbs": nb_out / t_down / 1e9,
            "both_gbs": (nb_in + nb_out) / t_both / 1e9, "both_ms": t_both * 1e3}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--sustain-s", type=float, default=2.0,
                    help="seconds of back-to-back steps for the sustained-clock figure (0: skip)")
    ap.add_argument("--oracle-budget-s", type=float, default=5.0,
                    help="seconds of oracle time per workload in the per-workload table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--datasheet", default=None,
                    help="JSON file with datasheet peaks ({\"bf16_tflops\": ..., \"hbm_gbs\": ...}); "
                         "adds fractions of them to the line")
    ap.add_argument("--cfg", type=int, default=CFG,
                    help="--kernel-only workload: 2 (first --images stills of the throughput set) or 4 (patch-16 bucket)")
    ap.add_argument("--kernel-only", choices=["embed", "embed_rope", "rope", "rope_apply", "normalize_patchify"],
                    help="profiling mode: launch one entry point on a subset of the images, print nothing")
    ap.add_argument("--images", type=int, default=64, help="images of the workload (profiling mode)")
    ap.add_argument("--launches", type=int, default=3, help="launches after warm-up (profiling mode)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.kernel_only:
        return kernel_only(args)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import torch.distributed as dist
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    from vit_vision_encoder_fusedinputnorm_gb300 import build as vbuild
    from vit_vision_encoder_fusedinputnorm_gb300 import synth
    from vit_vision_encoder_fusedinputnorm_gb300.frontend import FrontEnd

    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        vbuild.build()
    if world > 1:
        dist.barrier()
    B.load()

    wl = synth.make_workload(CFG)
    fe = FrontEnd.from_workload(wl, device=f"cuda:{local}")
    batch = fe.upload(wl.items)
    rows = batch.live_rows
    N, K = wl.hidden, wl.K
    out = torch.empty((rows, N), dtype=torch.bfloat16, device=dev)
    cos = torch.empty((rows, wl.head_dim // 2), dtype=torch.float32, device=dev)
    sin = torch.empty_like(cos)
    st = torch.zeros(2, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(ev=None):
        # the whole hot path in one launch: embeddings and the RoPE rows of the same items
        if ev is not None:
            ev[0].record(stream)
        B.vitfe_embed_rope(fe.h, batch.pixels, batch.pixel_bytes, batch.items, batch.n_items, batch.capacity,
                           rows, out, wl.head_dim, wl.theta, cos, sin, st, stream)
        if ev is not None:
            ev[1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    if st.cpu().tolist() != [0, -1]:
        raise RuntimeError(f"device status {st.cpu().tolist()}")

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # nothing between the launches: consecutive steps overlap by programmatic dependent launch
    # (the next step's prologue, A production and first passes run while the previous one
    # finishes; each step's writes wait for the previous step)
    t0.record(stream)
    for i in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    total_ms = world_max(t0.elapsed_time(t1), world, dev)
    ms_step = total_ms / args.steps
    # the step is one embed_kernel<14> launch: its time per launch over the timed region
    embed_ms = t0.elapsed_time(t1) / args.steps
    # the same launch serialised (an event recorded between launches stops the overlap)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            step(evs[i])
    torch.cuda.synchronize(dev)
    embed_serial_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    value = replica_value(rows, world, ms_step)

    # the same step back to back for seconds: the clock settles where the power cap puts it
    sustained = None
    if args.sustain_s > 0:
        n_sus = max(10, int(args.sustain_s / (ms_step / 1e3)))
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        smp = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
        if smp:
            smp.start()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        s0.record(stream)
        for _ in range(n_sus):
            step()
        s1.record(stream)
        torch.cuda.synchronize(dev)
        sus_clocks = smp.stop() if smp else None
        sus_ms = world_max(s0.elapsed_time(s1), world, dev) / n_sus
        sustained = {"steps": n_sus, "ms_per_step": sus_ms, "patches_per_s": replica_value(rows, world, sus_ms),
                     "clocks": sus_clocks}

    # end to end through the host-buffer entry point (vitfe_embed_rope_host): page-locked
    # pixels and descriptors in, embeddings and cos/sin out, the copies overlapped with the
    # launches in runs of consecutive images; wall clock around the (synchronous) call
    items_np, buf_np, _ = B.pack_items(wl.items, wl.patch, wl.tpatch)
    host_px = torch.from_numpy(buf_np).pin_memory()
    host_items = torch.from_numpy(np.ascontiguousarray(items_np).view(np.uint8)).pin_memory()
    host_out = torch.empty((rows, N), dtype=torch.bfloat16).pin_memory()
    host_cos = torch.empty(cos.shape, dtype=torch.float32).pin_memory()
    host_sin = torch.empty(sin.shape, dtype=torch.float32).pin_memory()
    host_st = torch.zeros(2, dtype=torch.int32)
    h2d = host_px.numel() + host_items.numel()
    d2h = host_out.numel() * 2 + host_cos.numel() * 4 * 2 + 8

    def e2e_step():
        B.vitfe_embed_rope_host(fe.h, host_px, host_px.numel(), host_items, len(items_np), host_out, wl.head_dim,
                                wl.theta, host_cos, host_sin, host_st, E2E_CHUNKS)

    e2e_step()
    if host_st.tolist() != [0, -1]:
        raise RuntimeError(f"device status {host_st.tolist()}")
    if world > 1:
        dist.barrier()
    t_e2e = time.perf_counter()
    for _ in range(args.e2e_steps):
        e2e_step()
    e2e_ms = world_max((time.perf_counter() - t_e2e) * 1e3 / args.e2e_steps, world, dev)

    def timed(fn, n=8, skip=3):
        ts = []
        with torch.cuda.stream(stream):
            for i in range(n):
                a0 = torch.cuda.Event(enable_timing=True)
                a1 = torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                fn()
                a1.record(stream)
                a1.synchronize()
                if i >= skip:
                    ts.append(a0.elapsed_time(a1))
        return statistics.median(ts)

    def looped(fn, n=50, warm=5):
        """Mean time per launch over a back-to-back loop (steady-state bandwidth of the
        short HBM-bound kernels, whose launch gaps the isolated timing would count)."""
        with torch.cuda.stream(stream):
            for _ in range(warm):
                fn()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(n):
                fn()
            a1.record(stream)
            a1.synchronize()
        return a0.elapsed_time(a1) / n

    # the two calls the fused launch replaces, and the RoPE expansion alone (HBM-write bound)
    def unfused():
        B.vitfe_embed(fe.h, batch.pixels, batch.pixel_bytes, batch.items, batch.n_items, batch.capacity, rows,
                      out, st, stream)
        B.vitfe_rope(fe.h, batch.items, batch.n_items, batch.capacity, rows, wl.head_dim, wl.theta, cos, sin,
                     None, stream)

    unfused_ms = timed(unfused)
    # the folded-still variant (an approximation: the summed weight slices are rounded once
    # to bf16), timed for reference only; it is never the headline
    folded_ms = timed(lambda: B.vitfe_embed_folded(fe.h, batch.pixels, batch.pixel_bytes, batch.items,
                                                   batch.n_items, batch.capacity, rows, out, None, stream))
    def rope_call():
        B.vitfe_rope(fe.h, batch.items, batch.n_items, batch.capacity, rows, wl.head_dim, wl.theta, cos, sin,
                     None, stream)

    rope_iso_ms = timed(rope_call)
    rope_ms = looped(rope_call)

    # standalone normalise + patchify (HBM-bound side path), timed alone
    flat = torch.empty((rows, K), dtype=torch.bfloat16, device=dev)
    def np_call():
        B.vitfe_normalize_patchify(fe.h, batch.pixels, batch.pixel_bytes, batch.items, batch.n_items,
                                   batch.capacity, rows, flat, None, stream)

    np_iso_ms = timed(np_call)
    np_ms = looped(np_call)
    np_bytes = batch.pixel_bytes + rows * K * 2

    # RoPE applied to Q and K (16 + 16 heads of 80, views into a packed [rows][Q | K | V]
    # buffer), from the step's cos/sin tables: HBM bound, in place
    heads = N // wl.head_dim
    qkv = torch.zeros((rows, 3 * N), dtype=torch.bfloat16, device=dev)
    def apply_call():
        B.vitfe_rope_apply(cos, sin, rows, wl.head_dim, qkv, heads, 3 * N, qkv[:, N:], heads, 3 * N, stream)

    apply_iso_ms = timed(apply_call)
    apply_ms = looped(apply_call)
    apply_bytes = rows * (2 * heads * wl.head_dim * 2 * 2 + wl.head_dim // 2 * 4 * 2)
    del qkv
    del flat

    pk, pk_kind = peaks()
    burst = float(pk["bf16_tflops"])

    # every other workload, as the fused call a user makes (device-resident inputs), with the
    # oracle on this host's cores beside it
    per_config = {}
    cores = _cores()
    for cfg in (0, 1, 3):
        wlc = synth.make_workload(cfg)
        fec = FrontEnd.from_workload(wlc, device=f"cuda:{local}")
        bc = fec.upload(wlc.items)
        oc, cc, sc = fec.embed_rope(bc, wlc.head_dim, wlc.theta)

        def call_c():
            B.vitfe_embed_rope(fec.h, bc.pixels, bc.pixel_bytes, bc.items, bc.n_items, bc.capacity, bc.live_rows,
                               oc, wlc.head_dim, wlc.theta, cc, sc, None, stream)

        ms_c = looped(call_c)
        iso_c = timed(call_c)
        fl = 2.0 * bc.live_rows * wlc.K * wlc.hidden
        entry = {"rows": bc.live_rows, "ms": ms_c, "isolated_ms": iso_c, "patches_per_s": bc.live_rows / (ms_c / 1e3),
                 "tflops": fl / (ms_c / 1e3) / 1e12, "frac_of_burst": fl / (ms_c / 1e3) / 1e12 / burst}
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            rate, orows, nit, ot = oracle_items_rate(wlc, args.oracle_budget_s)
            entry["oracle"] = {"patches_per_s": rate, "cores": cores,
                               "sample": f"{nit} of {len(wlc.items)} items, {orows} patches, {ot:.1f} s"}
        per_config[str(cfg)] = entry
        del oc, cc, sc
        fec.close()

    # workload 4 as the serving path runs it: one captured graph of the fused call over the
    # fixed 65,536-row bucket, replayed once per bucket of the 50 requests
    wl4 = synth.make_workload(4)
    fe4 = FrontEnd.from_workload(wl4, device=f"cuda:{local}")
    packs = [B.pack_items([wl4.items[i] for i in bk], wl4.patch, wl4.tpatch) for bk in wl4.buckets]
    R4 = wl4.bucket_rows
    px4 = torch.zeros(max(p[1].size for p in packs), dtype=torch.uint8, device=dev)
    it4 = torch.zeros(B.VITFE_MAX_ITEMS * 24, dtype=torch.uint8, device=dev)
    n4 = torch.zeros(1, dtype=torch.int32, device=dev)
    gout = torch.empty((R4, wl4.hidden), dtype=torch.bfloat16, device=dev)
    gcos = torch.empty((R4, wl4.head_dim // 2), dtype=torch.float32, device=dev)
    gsin = torch.empty_like(gcos)

    def fused4():
        B.vitfe_embed_rope(fe4.h, px4, px4.numel(), it4, n4, B.VITFE_MAX_ITEMS, R4, gout, wl4.head_dim, wl4.theta,
                           gcos, gsin, None, stream)

    with torch.cuda.stream(stream):
        fused4()                       # builds the RoPE table outside the capture
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fused4()
    buckets4, live4, t4 = [], 0, 0.0
    for items, buf, live in packs:
        px4[:buf.size].copy_(torch.from_numpy(buf))
        arr = np.zeros(B.VITFE_MAX_ITEMS, B.ITEM_DTYPE)
        arr[:len(items)] = items
        it4.copy_(torch.from_numpy(arr.view(np.uint8)))
        n4.fill_(len(items))
        torch.cuda.synchronize(dev)
        ms_b = looped(graph.replay, n=20, warm=3)
        iso_b = timed(graph.replay)
        fl = 2.0 * live * wl4.K * wl4.hidden
        buckets4.append({"live_rows": live, "ms": ms_b, "isolated_ms": iso_b,
                         "tflops": fl / (ms_b / 1e3) / 1e12, "frac_of_burst": fl / (ms_b / 1e3) / 1e12 / burst})
        live4 += live
        t4 += ms_b
    entry4 = {"rows": live4, "bucket_rows": R4, "replays": len(packs), "ms": t4,
              "patches_per_s": live4 / (t4 / 1e3),
              "tflops": 2.0 * live4 * wl4.K * wl4.hidden / (t4 / 1e3) / 1e12,
              "frac_of_burst": 2.0 * live4 * wl4.K * wl4.hidden / (t4 / 1e3) / 1e12 / burst, "buckets": buckets4}
    # the same three buckets as direct calls back to back, each with its own buffers (no
    # graph): consecutive calls overlap by programmatic dependent launch, graph replays do not
    dsets = []
    for items, buf, live in packs:
        arr = np.zeros(B.VITFE_MAX_ITEMS, B.ITEM_DTYPE)
        arr[:len(items)] = items
        dsets.append((torch.from_numpy(buf).to(dev), torch.from_numpy(arr.view(np.uint8)).to(dev),
                      torch.tensor([len(items)], dtype=torch.int32, device=dev),
                      torch.empty((R4, wl4.hidden), dtype=torch.bfloat16, device=dev),
                      torch.empty((R4, wl4.head_dim // 2), dtype=torch.float32, device=dev),
                      torch.empty((R4, wl4.head_dim // 2), dtype=torch.float32, device=dev)))

    def direct4():
        for dpx, dit, dn, dout, dcos, dsin in dsets:
            B.vitfe_embed_rope(fe4.h, dpx, dpx.numel(), dit, dn, B.VITFE_MAX_ITEMS, R4, dout, wl4.head_dim,
                               wl4.theta, dcos, dsin, None, stream)

    ms_d = looped(direct4, n=20, warm=3)
    entry4["direct_calls"] = {"ms": ms_d, "patches_per_s": live4 / (ms_d / 1e3),
                              "tflops": 2.0 * live4 * wl4.K * wl4.hidden / (ms_d / 1e3) / 1e12,
                              "frac_of_burst": 2.0 * live4 * wl4.K * wl4.hidden / (ms_d / 1e3) / 1e12 / burst,
                              "how": "the three buckets as direct calls back to back, each on its own buffers "
                                     "(consecutive calls overlap by programmatic dependent launch)"}
    del dsets
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, orows, nit, ot = oracle_items_rate(wl4, args.oracle_budget_s)
        entry4["oracle"] = {"patches_per_s": rate, "cores": cores,
                            "sample": f"{nit} of {len(wl4.items)} items, {orows} patches, {ot:.1f} s"}
    per_config["4"] = entry4
    del gout, gcos, gsin, graph, px4
    fe4.close()

    link = link_bandwidth(torch, dev, host_px, host_out, stream)
    # the copies' floor: the download alone, the upload alone, or both directions sharing the link
    link_floor_ms = max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9),
                        (h2d + d2h) / (link["both_gbs"] * 1e9)) * 1e3

    flops = 2.0 * rows * K * N
    achieved = flops / (embed_ms / 1e3) / 1e12
    peak = float(pk["bf16_tflops"])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "64 x 1344x1344 uint8 stills, patch 14, tpatch 2, merge 2, K 1176, N 1280, "
                               "RoPE head_dim 80", "rows_per_step": rows,
                   "step": "vitfe_embed_rope: embeddings + RoPE rows in one launch (C ABI, device-resident inputs)",
                   "l2": "inputs (347 MB) and outputs (1.5 GB) exceed L2; no flush",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(),
                     "peak_kind": f"{pk_kind} bf16 burst",
                     "kernel": "embed_kernel<14>", "flops_per_launch": flops,
                     "kernel_ms": embed_ms,
                     "kernel_ms_how": "per launch over the timed region (one launch per step; consecutive "
                                      "launches overlap by programmatic dependent launch)",
                     "kernel_ms_serial": embed_serial_ms},
        "datasheet": datasheet_fracs(args.datasheet, achieved, {
            "rope": rows * wl.head_dim // 2 * 4 * 2 / (rope_ms / 1e3) / 1e9,
            "rope_apply_qk": apply_bytes / (apply_ms / 1e3) / 1e9,
            "normalize_patchify": np_bytes / (np_ms / 1e3) / 1e9}),
        "side_paths": {"timing": ("rope, rope_apply_qk and normalize_patchify (HBM bound): mean over a "
                                  "back-to-back loop of 50 launches, like the step; their *_isolated_ms and the "
                                  "other side paths: median of isolated launches, each waited for before the "
                                  "next (the GPU idles between them, so launch latency counts and the clock "
                                  "recovers)"),
                       "unfused_embed_then_rope_ms": unfused_ms,
                       "folded_still_variant": {"ms": folded_ms, "patches_per_s": world * rows / (folded_ms / 1e3),
                                                "note": "approximation (W slices summed, rounded once to bf16); "
                                                        "K 588 for stills; not the method's exact result"},
                       "rope_ms": rope_ms,
                       "rope_isolated_ms": rope_iso_ms,
                       "rope_gbs": rows * wl.head_dim // 2 * 4 * 2 / (rope_ms / 1e3) / 1e9,
                       "rope_frac_hbm": rows * wl.head_dim // 2 * 4 * 2 / (rope_ms / 1e3) / 1e9 / float(pk["hbm_gbs"]),
                       "rope_apply_qk_ms": apply_ms,
                       "rope_apply_qk_isolated_ms": apply_iso_ms,
                       "rope_apply_qk_gbs": apply_bytes / (apply_ms / 1e3) / 1e9,
                       "rope_apply_qk_frac_hbm": apply_bytes / (apply_ms / 1e3) / 1e9 / float(pk["hbm_gbs"]),
                       "normalize_patchify_ms": np_ms,
                       "normalize_patchify_isolated_ms": np_iso_ms,
                       "normalize_patchify_gbs": np_bytes / (np_ms / 1e3) / 1e9,
                       "normalize_patchify_frac_hbm": np_bytes / (np_ms / 1e3) / 1e9 / float(pk["hbm_gbs"])},
        "e2e": {"value": world * rows / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "how": f"vitfe_embed_rope_host, page-locked host buffers, {E2E_CHUNKS} overlapped runs, wall clock",
                "link_gbs": link, "link_floor_ms": link_floor_ms, "frac_link": link_floor_ms / e2e_ms},
        "per_config": per_config,
        "sustained": None if sustained is None else dict(
            sustained, tflops=flops / (sustained["ms_per_step"] / 1e3) / 1e12,
            frac_of_sustained=flops / (sustained["ms_per_step"] / 1e3) / 1e12 / float(
                pk.get("bf16_tflops_sustained", peak)),
            frac_of_burst=flops / (sustained["ms_per_step"] / 1e3) / 1e12 / peak,
            mhz_x_ms=(sustained["clocks"] or {}).get("sm_mhz", float("nan")) * sustained["ms_per_step"]),
        # per step: one embed_kernel launch that also writes the RoPE rows (the position
        # table stays cached in the handle after the first warm-up step built it)
        "gpu_launches": 1 * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    fe.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
