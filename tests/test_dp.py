"""Data-parallel sharding of the front end ("vLLM 多模态推理｜ViT 性能优化" §3.1): the
balance by patch count and the all-gather back to input order, on the CPU (gloo ranks)."""
import itertools
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

from vit_vision_encoder_fusedinputnorm_gb300 import dp


def test_worked_example_of_the_pages():
    # 4 images of [1000, 100, 200, 50] patches on 2 GPUs: image 0 alone on GPU 0, images
    # 1, 2, 3 (350 patches) on GPU 1
    a = dp.assign_by_patches([1000, 100, 200, 50], 2)
    assert a == [[0], [1, 2, 3]]
    assert dp.rank_rows([1000, 100, 200, 50], a) == [1000, 350]


def test_every_item_once_and_single_rank():
    p = [5, 0, 7, 7, 3]
    a = dp.assign_by_patches(p, 3)
    assert sorted(i for lst in a for i in lst) == list(range(len(p)))
    assert all(lst == sorted(lst) for lst in a)
    assert dp.assign_by_patches(p, 1) == [list(range(len(p)))]
    assert dp.assign_by_patches([], 2) == [[], []]
    with pytest.raises(ValueError):
        dp.assign_by_patches([1], 0)


@pytest.mark.parametrize("seed", range(20))
def test_largest_first_is_within_the_known_bound_of_the_best_split(seed):
    # largest-first greedy keeps the busiest rank within (4/3 - 1/(3m)) of the best split;
    # the best split by brute force over every assignment of up to 7 items
    rng = np.random.default_rng(seed)
    n, m = int(rng.integers(1, 8)), int(rng.integers(2, 4))
    p = [int(x) for x in rng.integers(1, 2000, n)]
    got = max(dp.rank_rows(p, dp.assign_by_patches(p, m)))
    best = min(max(sum(p[i] for i in range(n) if c[i] == r) for r in range(m))
               for c in itertools.product(range(m), repeat=n))
    assert got <= (4 / 3 - 1 / (3 * m)) * best + 1e-9


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rows_of(item, n, width, dtype):
    # rows that name their item and position in columns of small integers (exact in bf16):
    # item, row % 256, row // 256, then the column index
    r = torch.arange(n)
    x = torch.arange(width, dtype=torch.float32)[None, :].repeat(n, 1)
    x[:, 0] = float(item)
    x[:, 1] = (r % 256).float()
    x[:, 2] = (r // 256).float()
    return x.to(dtype)


def _rank(rank, world, port, patches, width, dtype, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        a = dp.assign_by_patches(patches, world)
        mine = [_rows_of(i, patches[i], width, dtype) for i in a[rank]]
        local = torch.cat(mine) if mine else torch.empty((0, width), dtype=dtype)
        out = dp.gather_in_input_order(local, patches, a)
        results[rank] = out.float().numpy()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("patches,dtype", [
    ([1000, 100, 200, 50], torch.bfloat16),
    ([7, 3, 0, 12, 5, 5], torch.float32),
    ([9], torch.bfloat16),                    # one rank gets no item
])
def test_gather_restores_the_input_order_on_two_gloo_ranks(patches, dtype):
    world, width = 2, 6
    results = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), patches, width, dtype, results), nprocs=world, join=True)
    want = torch.cat([_rows_of(i, n, width, dtype) for i, n in enumerate(patches)]).float().numpy()
    for r in range(world):
        assert np.array_equal(results[r], want)


def _single(rank, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=0, world_size=1)
    try:
        patches = [3, 5]
        a = dp.assign_by_patches(patches, 1)
        local = torch.cat([_rows_of(i, n, 4, torch.float32) for i, n in enumerate(patches)])
        results["same"] = bool(torch.equal(dp.gather_in_input_order(local, patches, a), local))
        try:
            dp.gather_in_input_order(local[:-1], patches, a)
            results["short"] = "no error"
        except ValueError:
            results["short"] = "ValueError"
        try:
            dp.gather_in_input_order(local, patches, [[0], [1]])
            results["lists"] = "no error"
        except ValueError:
            results["lists"] = "ValueError"
    finally:
        dist.destroy_process_group()


def test_gather_on_one_rank_is_the_identity_and_checks_its_arguments():
    results = mp.Manager().dict()
    mp.spawn(_single, args=(_free_port(), results), nprocs=1, join=True)
    assert results["same"] is True
    assert results["short"] == "ValueError"   # local rows must match the rank's items
    assert results["lists"] == "ValueError"   # one item list per rank
