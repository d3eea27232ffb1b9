"""Comparison helpers shared by the GPU parity tests (test-side code only)."""
from __future__ import annotations

import numpy as np

import oracle

EMBED_REL_FROB = 5e-3     # max relative Frobenius error per item
EMBED_MAX_ABS = 2e-2      # max absolute error
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


def embed_errors(gpu: np.ndarray, ref: np.ndarray, starts) -> tuple:
    """(max relative Frobenius error over items, max abs error beyond the bf16 output rounding).

    The embeddings are bf16 by definition, so rounding the exact value to the output
    type alone costs up to half a bf16 ulp (0.0156 for |y| in [4, 8), 0.031 above 8);
    the absolute bound is applied to what remains after that rounding allowance.
    """
    worst_rel, worst_abs = 0.0, 0.0
    for s, e in zip(starts[:-1], starts[1:]):
        if e <= s:
            continue
        d = gpu[s:e] - ref[s:e]
        nr = np.linalg.norm(ref[s:e])
        rel = np.linalg.norm(d) / nr if nr > 0 else np.linalg.norm(d)
        worst_rel = max(worst_rel, float(rel))
        allow = np.maximum(bf16_half_ulp(ref[s:e]), bf16_half_ulp(gpu[s:e]))
        worst_abs = max(worst_abs, float(np.max(np.abs(d) - allow)))
    return worst_rel, worst_abs


def raw_max_abs(gpu: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(gpu - ref)))


def item_starts(items) -> np.ndarray:
    return np.concatenate([[0], np.cumsum([it.t * it.h * it.w for it in items])]).astype(np.int64)
