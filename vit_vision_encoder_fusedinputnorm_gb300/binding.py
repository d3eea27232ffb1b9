"""ctypes binding of libvitfe (argument marshalling only).

Every computation happens in the CUDA library; this module converts torch
tensors / ints to the pointers and sizes the C ABI takes.  There is no CPU
fallback: if the shared library is missing or cannot be loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libvitfe.so")

VITFE_MAX_ITEMS = 256
VITFE_ROPE_MAX_SIDE = 4096

STATUS_NAMES = {0: "VITFE_OK", 1: "VITFE_EINVAL", 2: "VITFE_ENOMEM", 3: "VITFE_ECUDA",
                4: "VITFE_EDEVICE_DESC", 5: "VITFE_EDEVICE_RANGE", 6: "VITFE_EDEVICE_TIMEOUT",
                7: "VITFE_EUNSUPPORTED"}

# exported symbols of include/vitfe.h
EXPORTS = ["vitfe_create", "vitfe_destroy", "vitfe_embed", "vitfe_embed_rope", "vitfe_embed_rope_host",
           "vitfe_embed_folded", "vitfe_rope", "vitfe_normalize_patchify",
           "vitfe_pos_ids", "vitfe_cu_seqlens", "vitfe_rope_apply", "vitfe_rope_noalloc",
           "vitfe_items_from_grid",
           "vitfe_feature_dim", "vitfe_status_str"]

ITEM_DTYPE = np.dtype([("pixel_offset", "<i8"), ("t", "<i4"), ("h", "<i4"), ("w", "<i4"),
                       ("frames", "<i4")])
assert ITEM_DTYPE.itemsize == 24


class VitfeItem(ctypes.Structure):
    _fields_ = [("pixel_offset", ctypes.c_int64), ("t", ctypes.c_int32), ("h", ctypes.c_int32),
                ("w", ctypes.c_int32), ("frames", ctypes.c_int32)]


class VitfeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)}")
        self.code = code


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once; raises OSError when it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"libvitfe not built ({path} missing): run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I32, I64, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.vitfe_create.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(F32), ctypes.POINTER(F32), F32,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P]
    lib.vitfe_create.restype = ctypes.c_int
    lib.vitfe_destroy.argtypes = [P]
    lib.vitfe_destroy.restype = None
    lib.vitfe_embed.argtypes = [P, P, I64, P, P, I32, I64, P, P, P]
    lib.vitfe_embed.restype = ctypes.c_int
    lib.vitfe_embed_rope.argtypes = [P, P, I64, P, P, I32, I64, P, ctypes.c_int, F32, P, P, P, P]
    lib.vitfe_embed_rope.restype = ctypes.c_int
    lib.vitfe_embed_rope_host.argtypes = [P, P, I64, P, I32, P, ctypes.c_int, F32, P, P, P, I32]
    lib.vitfe_embed_rope_host.restype = ctypes.c_int
    lib.vitfe_embed_folded.argtypes = [P, P, I64, P, P, I32, I64, P, P, P]
    lib.vitfe_embed_folded.restype = ctypes.c_int
    lib.vitfe_rope.argtypes = [P, P, P, I32, I64, ctypes.c_int, F32, P, P, P, P]
    lib.vitfe_rope.restype = ctypes.c_int
    lib.vitfe_rope_noalloc.argtypes = [ctypes.c_int, ctypes.c_int, P, P, I32, I64, ctypes.c_int, F32, P, P, P, P]
    lib.vitfe_rope_noalloc.restype = ctypes.c_int
    lib.vitfe_normalize_patchify.argtypes = [P, P, I64, P, P, I32, I64, P, P, P]
    lib.vitfe_normalize_patchify.restype = ctypes.c_int
    lib.vitfe_pos_ids.argtypes = [P, P, P, I32, I64, P, P, P]
    lib.vitfe_pos_ids.restype = ctypes.c_int
    lib.vitfe_cu_seqlens.argtypes = [P, P, P, I32, I64, I32, P, P, P, P]
    lib.vitfe_cu_seqlens.restype = ctypes.c_int
    lib.vitfe_rope_apply.argtypes = [P, P, I64, ctypes.c_int, P, I32, I64, P, I32, I64, P]
    lib.vitfe_rope_apply.restype = ctypes.c_int
    lib.vitfe_items_from_grid.argtypes = [P, P, I32, ctypes.c_int, ctypes.c_int, P,
                                          ctypes.POINTER(I64), ctypes.POINTER(I64)]
    lib.vitfe_items_from_grid.restype = ctypes.c_int
    lib.vitfe_feature_dim.argtypes = [P]
    lib.vitfe_feature_dim.restype = ctypes.c_int
    lib.vitfe_status_str.argtypes = [ctypes.c_int]
    lib.vitfe_status_str.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(x) -> Optional[int]:
    """Device/host pointer of a torch tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _hptr(x) -> Optional[int]:
    """Address of a host buffer: numpy array, torch CPU tensor, int, or None."""
    if x is None or isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return int(x.ctypes.data)
    return int(x.data_ptr())


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise VitfeError(fn, code)


# --------------------------------------------------------------------------
# the C entry points, same names
# --------------------------------------------------------------------------

def vitfe_create(mean: Sequence[float], std: Sequence[float], rescale: float, patch: int, tpatch: int,
                 merge: int, hidden: int, W, b=None, stream=None) -> int:
    lib = load()
    h = ctypes.c_void_p()
    m = (ctypes.c_float * 3)(*[float(v) for v in mean])
    s = (ctypes.c_float * 3)(*[float(v) for v in std])
    _check("vitfe_create", lib.vitfe_create(ctypes.byref(h), m, s, float(rescale), int(patch), int(tpatch),
                                            int(merge), int(hidden), _ptr(W), _ptr(b), _stream(stream)))
    return int(h.value)


def vitfe_destroy(h: int) -> None:
    load().vitfe_destroy(h)


def vitfe_embed(h, pixels, pixel_bytes, items, n_items, max_items, rows, out, status=None, stream=None) -> None:
    _check("vitfe_embed", load().vitfe_embed(h, _ptr(pixels), int(pixel_bytes), _ptr(items), _ptr(n_items),
                                             int(max_items), int(rows), _ptr(out), _ptr(status),
                                             _stream(stream)))


def vitfe_embed_rope_host(h, pixels, pixel_bytes, items, n_items, out, head_dim, theta, cos, sin, status=None,
                          chunks=16) -> None:
    """Host buffers (numpy arrays, torch CPU tensors or int addresses)."""
    _check("vitfe_embed_rope_host",
           load().vitfe_embed_rope_host(h, _hptr(pixels), int(pixel_bytes), _hptr(items), int(n_items), _hptr(out),
                                        int(head_dim), float(theta), _hptr(cos), _hptr(sin), _hptr(status),
                                        int(chunks)))


def vitfe_embed_folded(h, pixels, pixel_bytes, items, n_items, max_items, rows, out, status=None,
                       stream=None) -> None:
    _check("vitfe_embed_folded",
           load().vitfe_embed_folded(h, _ptr(pixels), int(pixel_bytes), _ptr(items), _ptr(n_items),
                                     int(max_items), int(rows), _ptr(out), _ptr(status), _stream(stream)))


def vitfe_embed_rope(h, pixels, pixel_bytes, items, n_items, max_items, rows, out, head_dim, theta, cos, sin,
                     status=None, stream=None) -> None:
    _check("vitfe_embed_rope",
           load().vitfe_embed_rope(h, _ptr(pixels), int(pixel_bytes), _ptr(items), _ptr(n_items), int(max_items),
                                   int(rows), _ptr(out), int(head_dim), float(theta), _ptr(cos), _ptr(sin),
                                   _ptr(status), _stream(stream)))


def vitfe_rope(h, items, n_items, max_items, rows, head_dim, theta, cos, sin, status=None, stream=None) -> None:
    _check("vitfe_rope", load().vitfe_rope(h, _ptr(items), _ptr(n_items), int(max_items), int(rows),
                                           int(head_dim), float(theta), _ptr(cos), _ptr(sin), _ptr(status),
                                           _stream(stream)))


def vitfe_rope_noalloc(tpatch, merge, items, n_items, max_items, rows, head_dim, theta, cos, sin, status=None,
                       stream=None) -> None:
    _check("vitfe_rope_noalloc", load().vitfe_rope_noalloc(int(tpatch), int(merge), _ptr(items), _ptr(n_items),
                                                           int(max_items), int(rows), int(head_dim),
                                                           float(theta), _ptr(cos), _ptr(sin), _ptr(status),
                                                           _stream(stream)))


def vitfe_normalize_patchify(h, pixels, pixel_bytes, items, n_items, max_items, rows, out, status=None,
                             stream=None) -> None:
    _check("vitfe_normalize_patchify",
           load().vitfe_normalize_patchify(h, _ptr(pixels), int(pixel_bytes), _ptr(items), _ptr(n_items),
                                           int(max_items), int(rows), _ptr(out), _ptr(status), _stream(stream)))


def vitfe_pos_ids(h, items, n_items, max_items, rows, pos, status=None, stream=None) -> None:
    _check("vitfe_pos_ids", load().vitfe_pos_ids(h, _ptr(items), _ptr(n_items), int(max_items), int(rows),
                                                 _ptr(pos), _ptr(status), _stream(stream)))


def vitfe_cu_seqlens(h, items, n_items, max_items, rows, max_seqs, cu_seqlens, seq_info, status=None,
                     stream=None) -> None:
    _check("vitfe_cu_seqlens", load().vitfe_cu_seqlens(h, _ptr(items), _ptr(n_items), int(max_items), int(rows),
                                                       int(max_seqs), _ptr(cu_seqlens), _ptr(seq_info),
                                                       _ptr(status), _stream(stream)))


def vitfe_rope_apply(cos, sin, rows, head_dim, q, heads_q, q_row_stride, k, heads_k, k_row_stride,
                     stream=None) -> None:
    _check("vitfe_rope_apply", load().vitfe_rope_apply(_ptr(cos), _ptr(sin), int(rows), int(head_dim), _ptr(q),
                                                       int(heads_q), int(q_row_stride), _ptr(k), int(heads_k),
                                                       int(k_row_stride), _stream(stream)))


def vitfe_items_from_grid(grid_thw: np.ndarray, is_still: Optional[np.ndarray], patch: int,
                          tpatch: int) -> Tuple[np.ndarray, int, int]:
    """Host helper: item descriptors (numpy, ITEM_DTYPE), total rows, pixel bytes."""
    lib = load()
    g = np.ascontiguousarray(grid_thw, dtype=np.int32).reshape(-1, 3)
    n = g.shape[0]
    st = None if is_still is None else np.ascontiguousarray(is_still, dtype=np.uint8)
    items = np.zeros(n, dtype=ITEM_DTYPE)
    rows = ctypes.c_int64()
    nbytes = ctypes.c_int64()
    _check("vitfe_items_from_grid",
           lib.vitfe_items_from_grid(g.ctypes.data if n else None, None if st is None else st.ctypes.data, n,
                                     int(patch), int(tpatch), items.ctypes.data if n else None,
                                     ctypes.byref(rows), ctypes.byref(nbytes)))
    return items, int(rows.value), int(nbytes.value)


def vitfe_feature_dim(h) -> int:
    return int(load().vitfe_feature_dim(h))


def vitfe_status_str(code: int) -> str:
    return load().vitfe_status_str(int(code)).decode()


# --------------------------------------------------------------------------
# marshalling helpers for torch callers (tests, bench, smoke)
# --------------------------------------------------------------------------

def pack_items(item_list, patch: int, tpatch: int):
    """Pack items (objects with t, h, w, frames, pixels) into one host byte buffer.

    Returns (items ITEM_DTYPE array, uint8 pixel buffer, total rows); offsets come
    from vitfe_items_from_grid (16-byte aligned).
    """
    grid = np.array([[it.t, it.h, it.w] for it in item_list], dtype=np.int32).reshape(-1, 3)
    still = np.array([1 if it.frames == 1 else 0 for it in item_list], dtype=np.uint8)
    items, rows, nbytes = vitfe_items_from_grid(grid, still, patch, tpatch)
    buf = np.zeros(max(nbytes, 16), dtype=np.uint8)
    for rec, it in zip(items, item_list):
        if it.pixels is None:
            continue
        flat = np.ascontiguousarray(it.pixels, dtype=np.uint8).reshape(-1)
        o = int(rec["pixel_offset"])
        buf[o:o + flat.size] = flat
    return items, buf, rows


def items_tensor(items: np.ndarray, capacity: Optional[int] = None, device="cuda"):
    """Device byte tensor holding vitfe_item[capacity] (unused slots zero) and int32 count."""
    import torch
    cap = len(items) if capacity is None else int(capacity)
    arr = np.zeros(max(cap, 1), dtype=ITEM_DTYPE)
    arr[:len(items)] = items
    t = torch.from_numpy(arr.view(np.uint8).copy()).to(device)
    n = torch.tensor([len(items)], dtype=torch.int32, device=device)
    return t, n
