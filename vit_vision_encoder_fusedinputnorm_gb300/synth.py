"""Seeded synthetic workloads for the vision-tower front end.

This module only *draws inputs*: uint8 pixel frames, the Conv3d patch-embed
weight and bias (as bf16 bit patterns) and the per-item grids.  It holds none
of the method's arithmetic (no normalisation, no patch ordering, no GEMM, no
RoPE), so both the CUDA path and the CPU oracle can be fed from it.

The shapes and value distributions follow the five workloads the front end is
measured on:

* ``c0``  one 224x224 still, pixels uniform in [0, 255];
* ``c1``  eight stills of mixed sizes, smooth gradient + Gaussian noise;
* ``c2``  64 stills of 1344x1344 (the throughput workload);
* ``c3``  a 32-frame 448x784 video with random-walk drift, plus four 896x896
          stills, packed in one call;
* ``c4``  50 stills of random sizes (multiples of 32 in [256, 1536]) packed
          greedily into fixed buckets of 65,536 patch rows, patch 16.

Stand-ins for the pages' real inputs (document pages, mixed photos, videos),
which are not available here.  Readings of details the pages leave open:

* "smooth gradient field": base_c(y, x) = 255 * (a_c * y/(H-1) + (1-a_c) *
  x/(W-1)) with a = (0.25, 0.5, 0.75), plus N(0, 12^2) noise, rounded half to
  even and clipped to [0, 255];
* "random-walk drift (step sigma 4)": frame 0 as above (unclipped float
  field s_0), then s_f = s_{f-1} + N(0, 4^2) per pixel; each stored frame is
  clip(rint(s_f));
* sizes are read as H x W;
* weights W ~ N(0, 0.02) and bias b ~ N(0, 0.02), rounded to bf16 (RNE).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np

# Normalisation constants of the Qwen-VL image processor (CLIP statistics, to the
# four decimals the measured workloads state).
QWEN_MEAN = (0.4815, 0.4578, 0.4082)
QWEN_STD = (0.2686, 0.2613, 0.2758)
RESCALE = 1.0 / 255.0

BUCKET_ROWS_C4 = 65536


@dataclasses.dataclass
class Item:
    """One image or video: grid (t, h, w) in patches and its stored frames.

    ``frames == 1`` marks a still that the temporal patch replicates; a video
    stores ``t * tpatch`` frames.  ``pixels`` is uint8 [frames][H][W][3].
    """
    t: int
    h: int
    w: int
    frames: int
    pixels: Optional[np.ndarray] = None

    @property
    def rows(self) -> int:
        return self.t * self.h * self.w


@dataclasses.dataclass
class Workload:
    name: str
    patch: int
    tpatch: int
    merge: int
    hidden: int
    head_dim: int
    theta: float
    mean: Tuple[float, float, float]
    std: Tuple[float, float, float]
    rescale: float
    items: List[Item]
    W_bits: np.ndarray          # uint16 [hidden][3*tpatch*patch*patch], Conv3d weight flattened (C,T,P,P)
    b_bits: np.ndarray          # uint16 [hidden]
    bucket_rows: Optional[int] = None   # fixed padded bucket size (graph replay), else None
    buckets: Optional[List[List[int]]] = None  # item indices per bucket

    @property
    def K(self) -> int:
        return 3 * self.tpatch * self.patch * self.patch

    @property
    def live_rows(self) -> int:
        return sum(it.rows for it in self.items)


# --------------------------------------------------------------------------
# bit-level helpers (input encoding only)
# --------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); finite inputs only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# pixel fields
# --------------------------------------------------------------------------

def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(list(key))


def uniform_image(rng: np.random.Generator, H: int, W: int) -> np.ndarray:
    return rng.integers(0, 256, size=(1, H, W, 3), dtype=np.uint8)


def _gradient_field(H: int, W: int) -> np.ndarray:
    a = np.array([0.25, 0.5, 0.75], dtype=np.float32)
    yy = (np.arange(H, dtype=np.float32) / max(H - 1, 1))[:, None, None]
    xx = (np.arange(W, dtype=np.float32) / max(W - 1, 1))[None, :, None]
    return 255.0 * (a * yy + (1.0 - a) * xx)          # [H][W][3] float32


def _quantise(s: np.ndarray) -> np.ndarray:
    return np.clip(np.rint(s), 0, 255).astype(np.uint8)


def gradient_noise_image(rng: np.random.Generator, H: int, W: int, sigma: float = 12.0) -> np.ndarray:
    s = _gradient_field(H, W) + sigma * rng.standard_normal((H, W, 3), dtype=np.float32)
    return _quantise(s)[None]


def random_walk_video(rng: np.random.Generator, F: int, H: int, W: int,
                      sigma0: float = 12.0, step: float = 4.0) -> np.ndarray:
    out = np.empty((F, H, W, 3), dtype=np.uint8)
    s = _gradient_field(H, W) + sigma0 * rng.standard_normal((H, W, 3), dtype=np.float32)
    out[0] = _quantise(s)
    for f in range(1, F):
        s = s + step * rng.standard_normal((H, W, 3), dtype=np.float32)
        out[f] = _quantise(s)
    return out


def weights(seed: int, hidden: int, K: int, sigma: float = 0.02) -> Tuple[np.ndarray, np.ndarray]:
    rng = _rng(seed, 0)
    W = f32_to_bf16_bits(sigma * rng.standard_normal((hidden, K), dtype=np.float32))
    b = f32_to_bf16_bits(sigma * rng.standard_normal((hidden,), dtype=np.float32))
    return W, b


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

C1_SIZES = [(224, 224), (448, 448), (672, 1008), (1008, 672),
            (336, 896), (896, 336), (560, 560), (1344, 756)]


def still(rng, H, W, P, kind="gradient") -> Item:
    px = uniform_image(rng, H, W) if kind == "uniform" else gradient_noise_image(rng, H, W)
    return Item(t=1, h=H // P, w=W // P, frames=1, pixels=px)


def c4_sizes(seed: int = 1004, n: int = 50) -> List[Tuple[int, int]]:
    rng = _rng(seed, 2)
    choices = np.arange(256, 1536 + 1, 32)
    H = rng.choice(choices, size=n)
    W = rng.choice(choices, size=n)
    return [(int(h), int(w)) for h, w in zip(H, W)]


def pack_buckets(rows: Sequence[int], bucket: int) -> List[List[int]]:
    """Greedy in-order packing of items into buckets of at most ``bucket`` rows."""
    out: List[List[int]] = [[]]
    used = 0
    for i, r in enumerate(rows):
        if r > bucket:
            raise ValueError("item larger than the bucket")
        if used + r > bucket:
            out.append([])
            used = 0
        out[-1].append(i)
        used += r
    return out


def make_workload(cfg: int, seed: Optional[int] = None, with_pixels: bool = True,
                  item_subset: Optional[Sequence[int]] = None) -> Workload:
    """Build workload ``cfg`` (0..4).  ``item_subset`` restricts which items get pixels."""
    seed = 1000 + cfg if seed is None else seed
    P, T, m = (16, 2, 2) if cfg == 4 else (14, 2, 2)
    hidden = 1152 if cfg == 4 else 1280
    head_dim = 72 if cfg == 4 else 80
    K = 3 * T * P * P
    Wb, bb = weights(seed, hidden, K)

    specs: List[Tuple[str, int, int, int]] = []   # (kind, F, H, W)
    if cfg == 0:
        specs = [("uniform", 1, 224, 224)]
    elif cfg == 1:
        specs = [("gradient", 1, H, W) for H, W in C1_SIZES]
    elif cfg == 2:
        specs = [("gradient", 1, 1344, 1344)] * 64
    elif cfg == 3:
        specs = [("video", 32, 448, 784)] + [("gradient", 1, 896, 896)] * 4
    elif cfg == 4:
        specs = [("gradient", 1, H, W) for H, W in c4_sizes(seed)]
    else:
        raise ValueError(cfg)

    items: List[Item] = []
    for i, (kind, F, H, W) in enumerate(specs):
        if kind == "video":
            it = Item(t=F // T, h=H // P, w=W // P, frames=F)
        else:
            it = Item(t=1, h=H // P, w=W // P, frames=1)
        if with_pixels and (item_subset is None or i in item_subset):
            rng = _rng(seed, 1, i)
            if kind == "uniform":
                it.pixels = uniform_image(rng, H, W)
            elif kind == "video":
                it.pixels = random_walk_video(rng, F, H, W)
            else:
                it.pixels = gradient_noise_image(rng, H, W)
        items.append(it)

    wl = Workload(name=f"c{cfg}", patch=P, tpatch=T, merge=m, hidden=hidden,
                  head_dim=head_dim, theta=10000.0, mean=QWEN_MEAN, std=QWEN_STD,
                  rescale=RESCALE, items=items, W_bits=Wb, b_bits=bb)
    if cfg == 4:
        wl.bucket_rows = BUCKET_ROWS_C4
        wl.buckets = pack_buckets([it.rows for it in items], BUCKET_ROWS_C4)
    return wl


def position_coded_image(F: int, H: int, W: int) -> np.ndarray:
    """uint8 frames whose value encodes (frame, y, x, channel): any misplaced pixel shows."""
    f = np.arange(F)[:, None, None, None]
    y = np.arange(H)[None, :, None, None]
    x = np.arange(W)[None, None, :, None]
    c = np.arange(3)[None, None, None, :]
    return ((7 * x + 13 * y + 29 * c + 31 * f) % 256).astype(np.uint8)


def small_workload(seed: int, grids: Sequence[Tuple[int, int, int, int]], patch: int = 14,
                   tpatch: int = 2, merge: int = 2, hidden: int = 256, head_dim: int = 80,
                   pixels: str = "uniform") -> Workload:
    """A small seeded workload with explicit grids (t, h, w, frames) for parity tests."""
    K = 3 * tpatch * patch * patch
    Wb, bb = weights(seed, hidden, K)
    items = []
    for i, (t, h, w, F) in enumerate(grids):
        rng = _rng(seed, 1, i)
        H, Wd = h * patch, w * patch
        if pixels == "uniform":
            px = rng.integers(0, 256, size=(F, H, Wd, 3), dtype=np.uint8)
        elif pixels == "coded":
            px = position_coded_image(F, H, Wd)
        else:
            px = gradient_noise_image(rng, H, Wd) if F == 1 else random_walk_video(rng, F, H, Wd)
        items.append(Item(t=t, h=h, w=w, frames=F, pixels=px))
    return Workload(name="small", patch=patch, tpatch=tpatch, merge=merge, hidden=hidden,
                    head_dim=head_dim, theta=10000.0, mean=QWEN_MEAN, std=QWEN_STD,
                    rescale=RESCALE, items=items, W_bits=Wb, b_bits=bb)
