"""moe_route_noalloc: the routing front end for callers that cannot allocate
device memory (for example a plugin handed only its input and output buffers,
or a path that must not call cudaMalloc after start-up).  Its scratch is a
static device array inside the library, so the caller passes only inputs and
outputs.

The GPU test calls it twice in a row, through the C ABI, on two different
problems and compares each result with what moe_forward (which uses a caller
workspace) computes for the same inputs.  This file is collected last on
purpose."""
import ctypes

import numpy as np
import pytest
import torch

import moe_inputs as MI
import precision_moe_grouped_gb300 as P
from precision_moe_grouped_gb300 import _lib as L


def _forward_front(case):
    """ids, weights, offsets, row_of as moe_forward computes them."""
    from gpu_helpers import GpuRun
    run = GpuRun(case)
    assert run.status == 0
    return run.ids, run.weights, run.offsets, run.row_of


def _noalloc(case):
    cfg, T = case.cfg, case.T
    dev = torch.device("cuda:0")
    k, E = cfg.top_k, cfg.num_experts
    ids = torch.full((T, k), -1, dtype=torch.int32, device=dev)
    wts = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
    rows = torch.full((T, k), -1, dtype=torch.int32, device=dev)
    s = P.shape(T, E, k, cfg.hidden, cfg.inter)
    logits = case.logits.to(dev)
    rc = P.load().moe_route_noalloc(ctypes.byref(s), logits.data_ptr(), ids.data_ptr(),
                                    wts.data_ptr(), offs.data_ptr(), rows.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == L.MOE_OK, P.load().moe_last_error()
    torch.cuda.synchronize()
    return ids.cpu().numpy(), wts.cpu().numpy(), offs.cpu().numpy(), rows.cpu().numpy()


@pytest.mark.gpu
def test_noalloc_route_matches_forward_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    P.load()
    cases = [MI.make_case(MI.custom_config(8, 2, 256, 128), 200, seed=71),
             MI.make_case(MI.custom_config(16, 4, 256, 128), 37, seed=72)]
    for case in cases:                        # two calls in a row, different shapes
        got = _noalloc(case)
        ref = _forward_front(case)
        np.testing.assert_array_equal(got[0], ref[0])                 # ids
        np.testing.assert_allclose(got[1], ref[1], rtol=3e-6, atol=1e-7)  # weights
        np.testing.assert_array_equal(got[2], ref[2])                 # offsets
        np.testing.assert_array_equal(got[3], ref[3])                 # row_of


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    import os
    if not os.path.exists(L.LIB_PATH):
        from precision_moe_grouped_gb300 import build
        try:
            build.build()
        except (RuntimeError, FileNotFoundError) as e:
            pytest.skip(f"cannot build libmoe.so here: {e}")
    lib = P.load()
    s = P.shape(1 << 20, 1024, 8, 128, 128)       # histogram alone exceeds 4 MiB
    rc = lib.moe_route_noalloc(ctypes.byref(s), None, None, None, None, None, None)
    assert rc == L.MOE_ERR_WORKSPACE_TOO_SMALL
    assert b"static scratch" in lib.moe_last_error()
    assert lib.moe_route_noalloc(ctypes.byref(P.shape(0, 8, 2, 128, 128)),
                                 None, None, None, None, None, None) == L.MOE_OK
