"""Comparison helpers shared by the GPU parity tests (test-side code only)."""
from __future__ import annotations

import numpy as np

import oracle

EMBED_REL_FROB = 5e-3     # max relative Frobenius error per item (against the float64 oracle)
EMBED_MAX_ABS = 2e-2      # max absolute error (against the method-exact value, see embed_report)
ROPE_MAX_ABS = 1e-5       # cos/sin, fp32
NORM_MAX_ULP = 1          # normalised pixels, bf16 ulps


def tensor_bits(t) -> np.ndarray:
    """Raw 16-bit patterns of a bf16 torch tensor, copied to the host."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return oracle.bf16_bits_to_f64(bits)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 to the nearest bf16 (ties to even), exactly."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32).view(np.uint32).astype(np.int64)
    base = (f & 0xFFFF0000)
    cands = np.stack([base - 0x10000, base, base + 0x10000], axis=-1)
    sign = (f & 0x80000000)
    # keep candidates inside the same sign class
    cands = np.where((cands & 0x80000000) != sign[..., None], base[..., None], cands) & 0xFFFFFFFF
    vals = (cands.astype(np.uint32)).view(np.float32).astype(np.float64)
    d = np.abs(vals - x[..., None])
    best = np.argmin(d, axis=-1)
    dmin = np.take_along_axis(d, best[..., None], -1)[..., 0]
    bits = np.take_along_axis(cands, best[..., None], -1)[..., 0]
    # ties: prefer even mantissa
    tie = (np.sum(d == dmin[..., None], axis=-1) > 1)
    if np.any(tie):
        for idx in zip(*np.nonzero(tie)):
            opts = cands[idx][d[idx] == dmin[idx]]
            even = [o for o in opts if ((o >> 16) & 1) == 0]
            bits[idx] = even[0] if even else opts[0]
    return (bits >> 16).astype(np.uint16)


def ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(ordered(a_bits) - ordered(b_bits))


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |x| (the largest error of rounding x to bf16)."""
    _, ex = np.frexp(np.abs(np.asarray(x, dtype=np.float64)))
    return np.ldexp(1.0, ex - 9)


def rne_bf16_values(x: np.ndarray) -> np.ndarray:
    """float64 values rounded to the nearest bf16 value (ties to even), as float64.

    With x = m * 2^e (0.5 <= |m| < 1), bf16 keeps rint(m * 2^8) * 2^(e - 8); exact for
    the normal range, which every embedding value is in (zero stays zero).
    """
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(m * 256.0), e - 8)


def beyond_rounding(g: np.ndarray, y: np.ndarray) -> np.ndarray:
    """Distance from y to the set of reals that round (to nearest) to the bf16 value g.

    0 when rounding y gives g.  Otherwise it is how far a value that rounds to g must be
    from y at least, i.e. a lower bound on the error of whatever was rounded to give g.
    """
    g = np.asarray(g, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    sgn = np.where(g < 0, -1.0, 1.0)
    ga, ya = np.abs(g), sgn * y
    m, e = np.frexp(ga)
    above = np.ldexp(1.0, e - 9)                            # half the spacing above |g|
    below = np.where(m == 0.5, above / 2, above)            # at a power of two the spacing halves
    d = ya - ga
    out = np.where(d > 0, d - above, -d - below)
    out = np.where(ga == 0, np.abs(y), out)
    return np.maximum(out, 0.0)


def embed_report(gpu: np.ndarray, ref: np.ndarray, ref_m: np.ndarray, starts) -> dict:
    """Errors of GPU embeddings (float64 values of the bf16 outputs) on the live rows.

    ref:   the float64 oracle (normalised pixels unrounded);
    ref_m: the oracle with the GEMM's input in the model dtype (``bf16_input``): the
           normalised pixels rounded to bf16 as FusedInputNorm emits them, GEMM and bias
           exact.  This is the method's result before its output cast to bf16.
    starts: item row boundaries (rows past starts[-1] are pad rows, checked elsewhere).

    rel         max over items of ||gpu - ref||_F / ||ref||_F           (bar 5e-3)
    max_abs     max |gpu - ref_m|                                       (bar 2e-2)
    raw_max_abs max |gpu - ref|: adds the method's own bf16 cast of the normalised pixels
    max_y       max |ref|
    cast        max |ref_m - ref|: what that cast alone moves (both sides oracle)
    out_round   max |bf16(ref_m) - ref_m|: the output cast of the method-exact value
    acc         max beyond_rounding(gpu, ref_m): a lower bound on how far the GPU's fp32
                sum, before its output cast, lies from the exact sum
    flips       outputs where gpu != bf16(ref_m)
    """
    live = int(starts[-1])
    rep = {"rows": live, "rel": 0.0, "max_abs": 0.0, "raw_max_abs": 0.0, "max_y": 0.0, "cast": 0.0,
           "out_round": 0.0, "acc": 0.0, "flips": 0}
    for s, e in zip(starts[:-1], starts[1:]):
        if e <= s:
            continue
        d = gpu[s:e] - ref[s:e]
        nr = np.linalg.norm(ref[s:e])
        rel = np.linalg.norm(d) / nr if nr > 0 else np.linalg.norm(d)
        rep["rel"] = max(rep["rel"], float(rel))
    for s in range(0, live, 8192):
        e = min(live, s + 8192)
        g, y, ym = gpu[s:e], ref[s:e], ref_m[s:e]
        r = rne_bf16_values(ym)
        rep["max_abs"] = max(rep["max_abs"], float(np.max(np.abs(g - ym))))
        rep["raw_max_abs"] = max(rep["raw_max_abs"], float(np.max(np.abs(g - y))))
        rep["max_y"] = max(rep["max_y"], float(np.max(np.abs(y))))
        rep["cast"] = max(rep["cast"], float(np.max(np.abs(ym - y))))
        rep["out_round"] = max(rep["out_round"], float(np.max(np.abs(r - ym))))
        rep["acc"] = max(rep["acc"], float(np.max(beyond_rounding(g, ym))))
        rep["flips"] += int(np.count_nonzero(g != r))
    return rep


def check_embed(rep: dict) -> None:
    """The embedding bars: relative Frobenius error against the float64 oracle, and the
    absolute error against the method-exact value (output cast included, no allowance)."""
    assert rep["rel"] <= EMBED_REL_FROB and rep["max_abs"] <= EMBED_MAX_ABS, rep


def log_report(name: str, rep: dict) -> None:
    """Print a parity report; with VITFE_PARITY_LOG set, also append it there as JSON."""
    import json
    import os
    line = json.dumps({"case": name, **rep})
    print(line)
    path = os.environ.get("VITFE_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")


def item_starts(items) -> np.ndarray:
    return np.concatenate([[0], np.cumsum([it.t * it.h * it.w for it in items])]).astype(np.int64)
