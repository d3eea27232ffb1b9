"""C-ABI checks that need no GPU: the library loads, exports every symbol that
include/vitfe.h declares, and its host-only logic behaves (argument validation
that returns before any CUDA call, item packing)."""
import ctypes
import os
import re

import numpy as np
import pytest

from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
from vit_vision_encoder_fusedinputnorm_gb300 import build as vbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    vbuild.build()
    return B.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "vitfe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vitfe_[a-z_]+)\s*\(", src)))


def test_header_declares_expected_entry_points():
    assert _declared_functions() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_item_struct_layout():
    assert ctypes.sizeof(B.VitfeItem) == 24
    assert B.ITEM_DTYPE.itemsize == 24
    assert B.VitfeItem.t.offset == 8 and B.VitfeItem.frames.offset == 20


def test_status_strings(lib):
    for code in range(8):
        assert B.vitfe_status_str(code)
    assert "unknown" in B.vitfe_status_str(99)


def test_items_from_grid_packs_aligned(lib):
    grid = np.array([[1, 16, 16], [16, 32, 56], [1, 4, 6]], np.int32)
    still = np.array([1, 0, 1], np.uint8)
    items, rows, nbytes = B.vitfe_items_from_grid(grid, still, 14, 2)
    assert rows == 256 + 16 * 32 * 56 + 24
    assert list(items["frames"]) == [1, 32, 1]
    sizes = [1 * 224 * 224 * 3, 32 * 448 * 784 * 3, 56 * 84 * 3]
    off = 0
    for it, sz in zip(items, sizes):
        assert it["pixel_offset"] == off and off % 16 == 0
        off += (sz + 15) // 16 * 16
    assert nbytes == off


def test_items_from_grid_default_still_rule_and_errors(lib):
    items, rows, _ = B.vitfe_items_from_grid(np.array([[1, 2, 2], [2, 2, 2]], np.int32), None, 14, 2)
    assert list(items["frames"]) == [1, 4]
    with pytest.raises(B.VitfeError):
        B.vitfe_items_from_grid(np.array([[2, 2, 2]], np.int32), np.array([1], np.uint8), 14, 2)
    with pytest.raises(B.VitfeError):
        B.vitfe_items_from_grid(np.array([[1, -2, 2]], np.int32), None, 14, 2)


def test_create_rejects_bad_normalisation_before_touching_the_device(lib):
    # std <= 0, non-finite mean, zero rescale: no identity default, EINVAL.
    for mean, std, rs in [((0.5, 0.5, 0.5), (0.5, 0.0, 0.5), 1 / 255),
                          ((float("nan"), 0.5, 0.5), (0.5, 0.5, 0.5), 1 / 255),
                          ((0.5, 0.5, 0.5), (0.5, 0.5, 0.5), 0.0)]:
        with pytest.raises(B.VitfeError) as e:
            B.vitfe_create(mean, std, rs, 14, 2, 2, 1280, 16)
        assert e.value.code == 1
    for args in [(0, 2, 2, 1280), (14, 0, 2, 1280), (14, 2, 2, 1000), (14, 2, 0, 1280)]:
        with pytest.raises(B.VitfeError) as e:
            B.vitfe_create((0.5,) * 3, (0.5,) * 3, 1 / 255, *args, 16)
        assert e.value.code == 1
    with pytest.raises(B.VitfeError):
        B.vitfe_create((0.5,) * 3, (0.5,) * 3, 1 / 255, 14, 2, 2, 1280, None)


def test_calls_reject_null_handle(lib):
    for fn, args in [(B.vitfe_embed, (None, 16, 100, 16, 16, 1, 10, 16)),
                     (B.vitfe_rope, (None, 16, 16, 1, 10, 80, 1e4, 16, 16)),
                     (B.vitfe_pos_ids, (None, 16, 16, 1, 10, 16)),
                     (B.vitfe_cu_seqlens, (None, 16, 16, 1, 10, 8, 16, 16)),
                     (B.vitfe_embed_rope, (None, 16, 100, 16, 16, 1, 10, 16, 80, 1e4, 16, 16)),
                     (B.vitfe_embed_folded, (None, 16, 100, 16, 16, 1, 10, 16)),
                     (B.vitfe_normalize_patchify, (None, 16, 100, 16, 16, 1, 10, 16))]:
        with pytest.raises(B.VitfeError) as e:
            fn(*args)
        assert e.value.code == 1


def test_rope_apply_rejects_bad_shapes_before_launching(lib):
    # host validation only: nothing is launched, so any pointer values work here
    bad = [(16, 16, 10, 84, 16, 2, 168, 16, 2, 168),      # head_dim not a multiple of 8
           (16, 16, 10, 80, 16, 2, 100, 16, 2, 160),      # q stride below heads * head_dim
           (16, 16, 10, 80, 16, 2, 162, 16, 2, 160),      # q stride not a multiple of 4
           (16, 16, 10, 80, 12, 2, 160, 16, 2, 160),      # q not 8-byte aligned
           (24, 16, 10, 80, 16, 2, 160, 16, 2, 160),      # cos not 16-byte aligned
           (16, 16, -1, 80, 16, 2, 160, 16, 2, 160),      # negative rows
           (16, 16, 10, 80, None, 2, 160, 16, 2, 160)]    # heads but no pointer
    for args in bad:
        with pytest.raises(B.VitfeError) as e:
            B.vitfe_rope_apply(*args)
        assert e.value.code == 1


def test_noalloc_rope_rejects_sizes_beyond_its_static_table(lib):
    # head_dim above 128 does not fit the fixed scratch table: a clear error, nothing launched
    with pytest.raises(B.VitfeError) as e:
        B.vitfe_rope_noalloc(2, 2, 16, 16, 1, 10, 256, 1e4, 16, 16)
    assert e.value.code == 7
    with pytest.raises(B.VitfeError) as e:
        B.vitfe_rope_noalloc(2, 2, 16, 16, 1, 10, 84, 1e4, 16, 16)      # not a multiple of 8
    assert e.value.code == 1
