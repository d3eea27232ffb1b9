"""The allocation-free RoPE entry point against the oracle and the handle path.

vitfe_rope_noalloc is for callers that may not allocate device memory: code
whose device memory is all reserved up front by a pool it does not own (a
serving runtime that carves up the GPU at start-up), or a process that is not
allowed to call cudaMalloc once it is serving, because an allocation there can
fail or stall the other work sharing the GPU.  Creating a handle allocates, so
such callers cannot use vitfe_rope; this entry point runs the same kernels with
their scratch table in a fixed device array instead.  This file is collected
last on purpose, so that a run that stops at the first failure has already run
every other test.
"""
import numpy as np
import pytest

import oracle
from vit_vision_encoder_fusedinputnorm_gb300 import synth
import vitfe_testutil as U

pytestmark = pytest.mark.gpu


def test_noalloc_rope_matches_the_oracle_and_the_handle_path_on_two_calls_in_a_row():
    import torch
    from vit_vision_encoder_fusedinputnorm_gb300 import binding as B
    from vit_vision_encoder_fusedinputnorm_gb300 import build
    from vit_vision_encoder_fusedinputnorm_gb300.frontend import FrontEnd

    build.build()
    # two different calls in a row: the second must not see anything left by the first
    cases = [
        (synth.small_workload(41, [(1, 16, 16, 1), (2, 4, 6, 4), (1, 10, 22, 1)], patch=14, hidden=256,
                              head_dim=80), 80, 300),
        (synth.small_workload(42, [(1, 6, 10, 1), (3, 8, 4, 6)], patch=16, hidden=256, head_dim=72), 72, 64),
    ]
    for wl, head_dim, pad in cases:
        fe = FrontEnd.from_workload(wl)
        b = fe.upload(wl.items)
        rows = b.live_rows + pad
        ref_cos, ref_sin = fe.rope(b, head_dim, wl.theta, rows=rows)
        cos = torch.full((rows, head_dim // 2), 9.0, dtype=torch.float32, device="cuda")
        sin = torch.full_like(cos, 9.0)
        st = torch.full((2,), -7, dtype=torch.int32, device="cuda")
        B.vitfe_rope_noalloc(wl.tpatch, wl.merge, b.items, b.n_items, b.capacity, rows, head_dim, wl.theta,
                             cos, sin, st, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert st.cpu().tolist() == [0, -1]
        c, s = cos.cpu().numpy(), sin.cpu().numpy()
        # the oracle's tables (pad rows: identity), within the cos/sin bar
        oc, os_ = oracle.rope_workload(wl, bucket_rows=rows, head_dim=head_dim, theta=wl.theta)
        assert np.max(np.abs(c - oc)) <= U.ROPE_MAX_ABS
        assert np.max(np.abs(s - os_)) <= U.ROPE_MAX_ABS
        assert np.all(c[b.live_rows:] == 1.0) and np.all(s[b.live_rows:] == 0.0)
        # the same kernels as the handle path: bit for bit
        assert np.array_equal(c.view(np.uint32), ref_cos.cpu().numpy().view(np.uint32))
        assert np.array_equal(s.view(np.uint32), ref_sin.cpu().numpy().view(np.uint32))
        fe.close()
