"""Torch-side owner of a libvitfe handle and of the device buffers around it.

PyTorch only provides device memory and streams here; every step of the front
end runs in the library's CUDA kernels (see ``binding``).
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

from . import binding as B


@dataclasses.dataclass
class Batch:
    """Items resident on the device: packed uint8 pixels + vitfe_item table."""
    pixels: "object"        # torch uint8 [pixel_bytes] (device)
    pixel_bytes: int
    items: "object"         # torch uint8 [capacity * 24] (device)
    n_items: "object"       # torch int32 [1] (device)
    capacity: int
    live_rows: int
    host_items: np.ndarray


class FrontEnd:
    def __init__(self, mean, std, rescale, patch, tpatch, merge, hidden, W_bits, b_bits=None,
                 device: str = "cuda:0", stream=None):
        import torch
        self.torch = torch
        self.device = torch.device(device)
        self.patch, self.tpatch, self.merge, self.hidden = patch, tpatch, merge, hidden
        Wt = self._bf16(W_bits)
        bt = None if b_bits is None else self._bf16(b_bits)
        with torch.cuda.device(self.device):
            self.h = B.vitfe_create(mean, std, rescale, patch, tpatch, merge, hidden, Wt, bt,
                                    stream if stream is not None else torch.cuda.current_stream(self.device))
        self.K = B.vitfe_feature_dim(self.h)

    def _bf16(self, x):
        torch = self.torch
        if isinstance(x, np.ndarray):
            t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(self.device)
            return t.view(torch.bfloat16)
        return x.to(self.device).contiguous()

    @classmethod
    def from_workload(cls, wl, device: str = "cuda:0"):
        return cls(wl.mean, wl.std, wl.rescale, wl.patch, wl.tpatch, wl.merge, wl.hidden, wl.W_bits,
                   wl.b_bits, device=device)

    def close(self):
        if getattr(self, "h", None):
            B.vitfe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ data
    def upload(self, item_list: Sequence, capacity: Optional[int] = None, pinned: bool = False) -> Batch:
        torch = self.torch
        items, buf, rows = B.pack_items(item_list, self.patch, self.tpatch)
        px = torch.from_numpy(buf)
        if pinned:
            px = px.pin_memory()
        px = px.to(self.device, non_blocking=pinned)
        it, n = B.items_tensor(items, capacity, device=self.device)
        return Batch(px, int(buf.size), it, n, max(len(items), capacity or 0), rows, items)

    def status_tensor(self):
        return self.torch.full((2,), -7, dtype=self.torch.int32, device=self.device)

    def _stream(self, stream):
        return stream if stream is not None else self.torch.cuda.current_stream(self.device)

    # ------------------------------------------------------------------ calls
    def embed(self, b: Batch, rows: Optional[int] = None, out=None, status=None, stream=None):
        torch = self.torch
        rows = b.live_rows if rows is None else rows
        if out is None:
            out = torch.empty((rows, self.hidden), dtype=torch.bfloat16, device=self.device)
        B.vitfe_embed(self.h, b.pixels, b.pixel_bytes, b.items, b.n_items, b.capacity, rows, out, status,
                      self._stream(stream))
        return out

    def normalize_patchify(self, b: Batch, rows: Optional[int] = None, out=None, status=None, stream=None):
        torch = self.torch
        rows = b.live_rows if rows is None else rows
        if out is None:
            out = torch.empty((rows, self.K), dtype=torch.bfloat16, device=self.device)
        B.vitfe_normalize_patchify(self.h, b.pixels, b.pixel_bytes, b.items, b.n_items, b.capacity, rows, out,
                                   status, self._stream(stream))
        return out

    def embed_rope_host(self, item_list, head_dim: int, theta: float, chunks: int = 16, pinned: bool = True):
        """Host in, host out, copies overlapped (vitfe_embed_rope_host): (out, cos, sin, status)
        as torch CPU tensors (page-locked when ``pinned``)."""
        torch = self.torch
        items, buf, rows = B.pack_items(item_list, self.patch, self.tpatch)
        px = torch.from_numpy(buf)
        if pinned:
            px = px.pin_memory()
        it = torch.from_numpy(np.ascontiguousarray(items).view(np.uint8))
        out = torch.empty((rows, self.hidden), dtype=torch.bfloat16, pin_memory=pinned)
        cos = torch.empty((rows, head_dim // 2), dtype=torch.float32, pin_memory=pinned)
        sin = torch.empty((rows, head_dim // 2), dtype=torch.float32, pin_memory=pinned)
        st = torch.zeros(2, dtype=torch.int32)
        B.vitfe_embed_rope_host(self.h, px, px.numel(), it, len(items), out, head_dim, theta, cos, sin, st, chunks)
        return out, cos, sin, st

    def embed_folded(self, b: Batch, rows: Optional[int] = None, out=None, status=None, stream=None):
        """The folded-still variant of embed (an approximation; see vitfe_embed_folded)."""
        torch = self.torch
        rows = b.live_rows if rows is None else rows
        if out is None:
            out = torch.empty((rows, self.hidden), dtype=torch.bfloat16, device=self.device)
        B.vitfe_embed_folded(self.h, b.pixels, b.pixel_bytes, b.items, b.n_items, b.capacity, rows, out, status,
                             self._stream(stream))
        return out

    def embed_rope(self, b: Batch, head_dim: int, theta: float, rows: Optional[int] = None, out=None, cos=None,
                   sin=None, status=None, stream=None):
        """embed + rope in one launch: (out, cos, sin)."""
        torch = self.torch
        rows = b.live_rows if rows is None else rows
        if out is None:
            out = torch.empty((rows, self.hidden), dtype=torch.bfloat16, device=self.device)
        if cos is None:
            cos = torch.empty((rows, head_dim // 2), dtype=torch.float32, device=self.device)
        if sin is None:
            sin = torch.empty((rows, head_dim // 2), dtype=torch.float32, device=self.device)
        B.vitfe_embed_rope(self.h, b.pixels, b.pixel_bytes, b.items, b.n_items, b.capacity, rows, out, head_dim,
                           theta, cos, sin, status, self._stream(stream))
        return out, cos, sin

    def rope(self, b: Batch, head_dim: int, theta: float, rows: Optional[int] = None, cos=None, sin=None,
             status=None, stream=None):
        torch = self.torch
        rows = b.live_rows if rows is None else rows
        if cos is None:
            cos = torch.empty((rows, head_dim // 2), dtype=torch.float32, device=self.device)
        if sin is None:
            sin = torch.empty((rows, head_dim // 2), dtype=torch.float32, device=self.device)
        B.vitfe_rope(self.h, b.items, b.n_items, b.capacity, rows, head_dim, theta, cos, sin, status,
                     self._stream(stream))
        return cos, sin

    def cu_seqlens(self, b: Batch, max_seqs: int, rows: Optional[int] = None, out=None, info=None, status=None,
                   stream=None):
        """(cu_seqlens int32 [max_seqs + 1], seq_info int32 [2] = {sequences, longest})."""
        torch = self.torch
        rows = b.live_rows if rows is None else rows
        if out is None:
            out = torch.empty(max_seqs + 1, dtype=torch.int32, device=self.device)
        if info is None:
            info = torch.empty(2, dtype=torch.int32, device=self.device)
        B.vitfe_cu_seqlens(self.h, b.items, b.n_items, b.capacity, rows, max_seqs, out, info, status,
                           self._stream(stream))
        return out, info

    def pos_ids(self, b: Batch, rows: Optional[int] = None, out=None, status=None, stream=None):
        torch = self.torch
        rows = b.live_rows if rows is None else rows
        if out is None:
            out = torch.empty((rows, 2), dtype=torch.int32, device=self.device)
        B.vitfe_pos_ids(self.h, b.items, b.n_items, b.capacity, rows, out, status, self._stream(stream))
        return out
