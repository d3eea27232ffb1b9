"""Plain fp64 CPU oracle of the Qwen-VL vision-tower front end.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module.  The product path (the CUDA library
and its Python binding) never imports, calls or links anything here, and this
module imports nothing from the product.

What it computes, step by step, with the passage each step follows:

1. FusedInputNorm: x = (v * rescale - mean_c) / std_c for every uint8 pixel v
   of channel c.  "PR #55370 完整报告" ([Bugfix] Make mm_device_do_normalize
   encoder-cudagraph safe), section 实现拆解 item 2: the vision tower's
   ``forward`` first runs ``FusedInputNorm`` on integer pixels, doing
   "rescale + normalize" and emitting the model dtype; section 评论区精华
   item 1: the input contract is uint8.
2. Patchify in merge order: cut each frame into patch x patch patches, put each
   merge x merge group of neighbouring patches consecutively, flatten each
   patch to C*T*P*P features.  "vLLM 多模态推理｜ViT 性能优化", §2.2
   (multimodal input encoding, step (1)) and §3.2 (the flatten_patches shapes
   for images and videos).  A still is replicated over the temporal patch.
3. Patch embedding: a Conv3d whose kernel equals its stride, computed as the
   img2col GEMM  y = A W^T + b  with W the Conv3d weight [N][C][T][P][P]
   flattened to [N][C*T*P*P].  Same page, §3.2.
4. 2D position ids: (hpos, wpos) per patch, regrouped by spatial-merge unit,
   repeated over the t temporal groups.  Same page, §3.3 step 2.
5. 2D-RoPE tables: inverse frequencies of a rotary embedding of width
   rotary_dim = head_dim / 2 (theta^(-2i/rotary_dim), i < rotary_dim/2);
   each row is [cos(hpos*w_i) ... || cos(wpos*w_i) ...], likewise for sin.
   Same page, §3.3 steps 1, 3 and 5.

6. Attention sequence boundaries: one sequence per temporal group of each item,
   h*w tokens long, in item order.  Same page, §3.4 (cu_seqlens) read with
   §3.3 (the encoder models single images and frames).
7. RoPE applied to Q/K in each vision block (same page, §3.3 step 6), in the
   rotate-half form: feature i of a head and feature i + head_dim/2 rotate as
   one pair by the angle of table column i.
8. A folded-still variant of step 3 (not part of the method; reported on its
   own): a still's equal temporal slices of A multiply the summed weight
   slices rounded once to bf16.

Precision.  Everything is float64, with one option: FusedInputNorm emits the
model dtype (step 1's source, 实现拆解 item 2), bf16 here, so the GEMM of the
method receives the normalised pixels rounded to bf16.  ``bf16_input=True``
(embedding functions) applies exactly that rounding (to nearest, ties to even)
to A before the exact float64 GEMM; the default leaves A unrounded.  The first
is the method's own result before its output cast, the second the plain
mathematical value; the parity tests compare against both.

Readings where the pages are silent (each also listed in the design notes):
the first step's order is rescale, subtract the mean, divide by std; the
rotary width is head_dim / 2; a padded bucket's rows past the live rows are
embedding 0, cos 1, sin 0, position id -1.

Every function is pinned by the non-GPU tests against closed forms, brute
force on tiny inputs and invariants (see tests/test_oracle_pins.py).
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "bf16_bits_to_f64", "normalize", "patchify", "normalize_patchify_item",
    "embed_rows", "embed_item", "embed_workload", "pos_ids", "rope_tables",
    "rope_workload", "pos_ids_workload", "normalize_patchify_workload", "cu_seqlens",
    "cu_seqlens_workload", "rope_apply", "round_to_bf16_bits", "fold_still_weight", "embed_folded_item",
    "embed_folded_workload",
    "patch_coords", "to_model_dtype",
]


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float64: the top 16 bits of an fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# 1. FusedInputNorm
# ---------------------------------------------------------------------------

def normalize(pixels: np.ndarray, mean: Sequence[float], std: Sequence[float],
              rescale: float) -> np.ndarray:
    """(v * rescale - mean_c) / std_c in float64; channels are the last axis.

    "PR #55370 完整报告", 实现拆解 item 2 (rescale + normalize of integer
    pixels inside the tower's forward).
    """
    if pixels.dtype != np.uint8:
        raise TypeError("FusedInputNorm takes uint8 pixels only")
    v = pixels.astype(np.float64)
    mean = np.asarray(mean, dtype=np.float64)
    std = np.asarray(std, dtype=np.float64)
    return (v * float(rescale) - mean) / std


# ---------------------------------------------------------------------------
# 2. patchify in merge order
# ---------------------------------------------------------------------------

def patchify(x: np.ndarray, t: int, h: int, w: int, patch: int, tpatch: int,
             merge: int) -> np.ndarray:
    """Literal reshape/transpose of one item's frames into flatten_patches.

    x: [F][H][W][C] (any dtype), F == 1 (a still, replicated over the temporal
    patch, t must be 1) or F == t * tpatch.  Returns [t*h*w][C*T*P*P] with rows
    in merge order (t, h/m, w/m, m, m) and features in (C, T, P, P) order.

    "vLLM 多模态推理｜ViT 性能优化", §2.2 step (1) and §3.2.
    """
    F, H, W, C = x.shape
    if H != h * patch or W != w * patch:
        raise ValueError("frame size does not match the grid")
    if h % merge or w % merge:
        raise ValueError("grid not a multiple of the merge size")
    X = np.transpose(x, (0, 3, 1, 2))                      # [F][C][H][W]
    if F == 1 and t == 1:
        X = np.repeat(X, tpatch, axis=0)                   # still -> T identical frames
    if X.shape[0] != t * tpatch:
        raise ValueError("frame count does not match t * tpatch")
    X = X.reshape(t, tpatch, C, h // merge, merge, patch, w // merge, merge, patch)
    #              0    1     2     3        4      5       6        7      8
    X = X.transpose(0, 3, 6, 4, 7, 2, 1, 5, 8)             # t, hb, wb, mh, mw, C, T, ph, pw
    return X.reshape(t * h * w, C * tpatch * patch * patch)


def patch_coords(t: int, h: int, w: int, merge: int) -> np.ndarray:
    """Per row of an item, (tg, hh, ww): its temporal group and patch position.

    Built by the same reshape/transpose as ``patchify`` applied to index grids,
    so that the two always agree; pinned against the closed-form row index.
    """
    tg = np.broadcast_to(np.arange(t)[:, None, None], (t, h, w))
    hh = np.broadcast_to(np.arange(h)[None, :, None], (t, h, w))
    ww = np.broadcast_to(np.arange(w)[None, None, :], (t, h, w))

    def order(a):
        a = a.reshape(t, h // merge, merge, w // merge, merge)
        return a.transpose(0, 1, 3, 2, 4).reshape(-1)

    return np.stack([order(tg), order(hh), order(ww)], axis=1)


def normalize_patchify_item(item_pixels: np.ndarray, t: int, h: int, w: int, *, patch: int,
                            tpatch: int, merge: int, mean, std, rescale) -> np.ndarray:
    """flatten_patches (fp64) of one item: normalise, then patchify."""
    return patchify(normalize(item_pixels, mean, std, rescale), t, h, w, patch, tpatch, merge)


def to_model_dtype(x: np.ndarray) -> np.ndarray:
    """The normalised pixels as FusedInputNorm hands them on: rounded to the nearest bf16
    (ties to even), returned as float64.

    "PR #55370 完整报告", 实现拆解 item 2: the norm emits the model dtype.
    """
    return bf16_bits_to_f64(round_to_bf16_bits(x))


# ---------------------------------------------------------------------------
# 3. patch embedding (img2col GEMM)
# ---------------------------------------------------------------------------

def embed_rows(A: np.ndarray, W_bits: np.ndarray, b_bits: Optional[np.ndarray]) -> np.ndarray:
    """y = A W^T + b in float64; W, b are the bf16 parameters widened exactly.

    "vLLM 多模态推理｜ViT 性能优化", §3.2 (Conv3d with kernel == stride as one
    large matrix product with the weight viewed as a 2-D matrix).
    """
    Wf = bf16_bits_to_f64(W_bits)
    y = np.asarray(A, dtype=np.float64) @ Wf.T
    if b_bits is not None:
        y = y + bf16_bits_to_f64(b_bits)[None, :]
    return y


def embed_item(item_pixels, t, h, w, W_bits, b_bits, *, patch, tpatch, merge, mean, std,
               rescale, rows: Optional[np.ndarray] = None, bf16_input: bool = False) -> np.ndarray:
    """Embeddings of one item (optionally only the given local rows).

    bf16_input: the GEMM receives the normalised pixels in the model dtype
    (``to_model_dtype``) instead of unrounded.
    """
    A = normalize_patchify_item(item_pixels, t, h, w, patch=patch, tpatch=tpatch, merge=merge,
                                mean=mean, std=std, rescale=rescale)
    if rows is not None:
        A = A[np.asarray(rows)]
    if bf16_input:
        A = to_model_dtype(A)
    return embed_rows(A, W_bits, b_bits)


def _item_starts(items) -> np.ndarray:
    rows = [it.t * it.h * it.w for it in items]
    return np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)


def embed_workload(wl, items: Optional[Sequence[int]] = None, bucket_rows: Optional[int] = None,
                   sample: Optional[np.ndarray] = None, bf16_input: bool = False) -> np.ndarray:
    """Embeddings of the items ``items`` (default: all) packed in order.

    With ``bucket_rows`` the result has that many rows and the pad rows are 0.
    With ``sample`` (global row indices into the packed output) only those rows
    are returned, in the given order.  ``bf16_input`` as in ``embed_item``.
    """
    idx = list(range(len(wl.items))) if items is None else list(items)
    its = [wl.items[i] for i in idx]
    starts = _item_starts(its)
    live = int(starts[-1])
    total = live if bucket_rows is None else int(bucket_rows)
    common = dict(patch=wl.patch, tpatch=wl.tpatch, merge=wl.merge, mean=wl.mean,
                  std=wl.std, rescale=wl.rescale, bf16_input=bf16_input)
    if sample is None:
        out = np.zeros((total, wl.hidden), dtype=np.float64)
        for j, it in enumerate(its):
            out[starts[j]:starts[j + 1]] = embed_item(it.pixels, it.t, it.h, it.w, wl.W_bits,
                                                      wl.b_bits, **common)
        return out
    sample = np.asarray(sample, dtype=np.int64)
    out = np.zeros((len(sample), wl.hidden), dtype=np.float64)
    for j, it in enumerate(its):
        sel = np.nonzero((sample >= starts[j]) & (sample < starts[j + 1]))[0]
        if len(sel) == 0:
            continue
        out[sel] = embed_item(it.pixels, it.t, it.h, it.w, wl.W_bits, wl.b_bits,
                              rows=sample[sel] - starts[j], **common)
    return out


# ---------------------------------------------------------------------------
# 3c. folded-still variant (an approximation of step 3, reported on its own)
# ---------------------------------------------------------------------------

def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 of float64 values, ties to even, in one rounding (bit patterns).

    bf16 keeps 8 significant bits: with x = m * 2^e (0.5 <= |m| < 1, frexp), the
    result is rint(m * 2^8) * 2^(e - 8), rint rounding half to even; both steps
    are exact in float64.  Normal-range inputs only (the folded weights and the
    normalised pixels; zero stays zero).
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    r = np.ldexp(np.rint(m * 256.0), e - 8)
    nz = r != 0
    if np.any(np.abs(r[nz]) < 2.0 ** -126) or not np.all(np.isfinite(r)):
        raise ValueError("outside the normal bf16 range")
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def fold_still_weight(W_bits: np.ndarray, tpatch: int, patch: int) -> np.ndarray:
    """W' [N][3*P*P] (bf16 bits, (c, ph, pw) order): the temporal slices of W summed.

    A still repeats one frame over the temporal patch (§3.2), so its T slices of
    A are equal and  sum_s A_s W_s^T = A_0 (sum_s W_s)^T  exactly; the variant
    stores sum_s W_s rounded once to bf16 and halves the GEMM's K.  Only that one
    rounding differs from step 3.  The sum of bf16 values is exact in float64 and
    is rounded to bf16 directly.
    """
    N = W_bits.shape[0]
    Wf = bf16_bits_to_f64(W_bits).reshape(N, 3, tpatch, patch, patch)
    return round_to_bf16_bits(Wf.sum(axis=2).reshape(N, 3 * patch * patch))


def embed_folded_item(item_pixels, t, h, w, W_bits, b_bits, Wf_bits, *, patch, tpatch, merge, mean,
                      std, rescale, still: bool, bf16_input: bool = False) -> np.ndarray:
    """Embeddings of one item in the folded-still variant: a still uses temporal
    slice 0 of A against W' (fold_still_weight); a video uses step 3 unchanged.
    ``bf16_input`` as in ``embed_item``."""
    A = normalize_patchify_item(item_pixels, t, h, w, patch=patch, tpatch=tpatch, merge=merge,
                                mean=mean, std=std, rescale=rescale)
    if bf16_input:
        A = to_model_dtype(A)
    if not still:
        return embed_rows(A, W_bits, b_bits)
    A4 = A.reshape(A.shape[0], 3, tpatch, patch * patch)
    A0 = A4[:, :, 0, :].reshape(A.shape[0], 3 * patch * patch)
    return embed_rows(A0, Wf_bits, b_bits)


def embed_folded_workload(wl, bucket_rows: Optional[int] = None, bf16_input: bool = False) -> np.ndarray:
    Wf = fold_still_weight(wl.W_bits, wl.tpatch, wl.patch)
    starts = _item_starts(wl.items)
    total = int(starts[-1]) if bucket_rows is None else int(bucket_rows)
    out = np.zeros((total, wl.hidden), dtype=np.float64)
    for j, it in enumerate(wl.items):
        out[starts[j]:starts[j + 1]] = embed_folded_item(
            it.pixels, it.t, it.h, it.w, wl.W_bits, wl.b_bits, Wf, patch=wl.patch, tpatch=wl.tpatch,
            merge=wl.merge, mean=wl.mean, std=wl.std, rescale=wl.rescale, still=(it.frames == 1),
            bf16_input=bf16_input)
    return out


def normalize_patchify_workload(wl, items=None, bucket_rows=None) -> np.ndarray:
    """flatten_patches (fp64) of the packed items; pad rows are 0."""
    idx = list(range(len(wl.items))) if items is None else list(items)
    its = [wl.items[i] for i in idx]
    starts = _item_starts(its)
    total = int(starts[-1]) if bucket_rows is None else int(bucket_rows)
    out = np.zeros((total, wl.K), dtype=np.float64)
    for j, it in enumerate(its):
        out[starts[j]:starts[j + 1]] = normalize_patchify_item(
            it.pixels, it.t, it.h, it.w, patch=wl.patch, tpatch=wl.tpatch, merge=wl.merge,
            mean=wl.mean, std=wl.std, rescale=wl.rescale)
    return out


# ---------------------------------------------------------------------------
# 3b. attention sequence boundaries
# ---------------------------------------------------------------------------

def cu_seqlens(grids: Sequence[Tuple[int, int, int]]) -> Tuple[np.ndarray, int]:
    """(cu_seqlens int64 [n_seq + 1], longest sequence) of items with grids (t, h, w).

    "vLLM 多模态推理｜ViT 性能优化", §3.4: cu_seqlens records where each image's
    tokens start and end, so the encoder's attention keeps images apart.  The
    encoder models single images and single frames (§3.3), so each of an item's
    t temporal groups is one sequence of h*w tokens, in item order.
    """
    lens = []
    for t, h, w in grids:
        lens.extend([h * w] * t)
    cu = np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))]).astype(np.int64)
    return cu, (max(lens) if lens else 0)


def cu_seqlens_workload(wl, items=None) -> Tuple[np.ndarray, int]:
    idx = list(range(len(wl.items))) if items is None else list(items)
    return cu_seqlens([(wl.items[i].t, wl.items[i].h, wl.items[i].w) for i in idx])


# ---------------------------------------------------------------------------
# 4. 2D position ids
# ---------------------------------------------------------------------------

def pos_ids(t: int, h: int, w: int, merge: int) -> np.ndarray:
    """(hpos, wpos) per patch in merge order, tiled over t: int64 [t*h*w][2].

    "vLLM 多模态推理｜ViT 性能优化", §3.3 step 2: hpos/wpos over the h x w grid,
    regrouped so each merge unit is consecutive, the pair stacked and the T
    temporal groups concatenated.
    """
    hpos = np.repeat(np.arange(h)[:, None], w, axis=1)     # hpos[i][j] = i
    wpos = np.repeat(np.arange(w)[None, :], h, axis=0)     # wpos[i][j] = j

    def merge_order(a):
        return a.reshape(h // merge, merge, w // merge, merge).transpose(0, 2, 1, 3).reshape(-1)

    pid = np.stack([merge_order(hpos), merge_order(wpos)], axis=1)
    return np.tile(pid, (t, 1)).astype(np.int64)


def pos_ids_workload(wl, items=None, bucket_rows=None) -> np.ndarray:
    idx = list(range(len(wl.items))) if items is None else list(items)
    parts = [pos_ids(wl.items[i].t, wl.items[i].h, wl.items[i].w, wl.merge) for i in idx]
    p = np.concatenate(parts, axis=0) if parts else np.zeros((0, 2), np.int64)
    if bucket_rows is not None:
        pad = np.full((int(bucket_rows) - len(p), 2), -1, dtype=np.int64)
        p = np.concatenate([p, pad], axis=0)
    return p


# ---------------------------------------------------------------------------
# 5. 2D-RoPE cos/sin tables
# ---------------------------------------------------------------------------

def rope_tables(pos: np.ndarray, head_dim: int, theta: float) -> Tuple[np.ndarray, np.ndarray]:
    """cos, sin float64 [rows][head_dim/2] = [f(hpos*w_i) || f(wpos*w_i)].

    rotary_dim = head_dim / 2 and w_i = theta^(-2i/rotary_dim) for
    i < rotary_dim / 2.  "vLLM 多模态推理｜ViT 性能优化", §3.3 steps 1 (the
    cos/sin cache), 3 (look up hpos and wpos, concatenate H then W) and 5
    (items concatenated).  Rows with position -1 (bucket padding) are the
    identity rotation: cos 1, sin 0.
    """
    if head_dim % 4:
        raise ValueError("head_dim must be a multiple of 4")
    d = head_dim // 2
    i = np.arange(head_dim // 4, dtype=np.float64)
    omega = np.power(float(theta), -2.0 * i / d)
    pos = np.asarray(pos)
    ph = pos[:, 0:1].astype(np.float64)
    pw = pos[:, 1:2].astype(np.float64)
    cos = np.concatenate([np.cos(ph * omega), np.cos(pw * omega)], axis=1)
    sin = np.concatenate([np.sin(ph * omega), np.sin(pw * omega)], axis=1)
    pad = pos[:, 0] < 0
    cos[pad] = 1.0
    sin[pad] = 0.0
    return cos, sin


def rope_apply(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """RoPE applied to one projection (Q or K), float64 [rows][heads][head_dim].

    "vLLM 多模态推理｜ViT 性能优化", §3.3 step 6 ("apply RoPE to Q/K in every
    VisionBlock").  The tables are [rows][head_dim/2] (the [H || W] layout of
    step 3); the page does not spell the rotation out, and this takes the
    rotate-half form of a head_dim-wide rotary embedding whose two halves repeat
    the table: with h = head_dim / 2, c = cos[r][i], s = sin[r][i],
        y[i]     = x[i] * c - x[i + h] * s
        y[i + h] = x[i + h] * c + x[i] * s        (i < h)
    for every head.
    """
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    if cos.shape[-1] != h or sin.shape[-1] != h:
        raise ValueError("tables must be [rows][head_dim/2]")
    c = np.asarray(cos, dtype=np.float64)[:, None, :]
    s = np.asarray(sin, dtype=np.float64)[:, None, :]
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_workload(wl, items=None, bucket_rows=None, head_dim=None, theta=None):
    p = pos_ids_workload(wl, items, bucket_rows)
    return rope_tables(p, wl.head_dim if head_dim is None else head_dim,
                       wl.theta if theta is None else theta)
