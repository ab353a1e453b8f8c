"""moe_route_noalloc: the routing front end for callers that cannot allocate
device memory (for example a plugin handed only its input and output buffers,
or a path that must not call cudaMalloc after start-up).  Its scratch is a
static device array inside the library, so the caller passes only inputs and
outputs.

The GPU test calls it several times in a row, through the C ABI, on
different problems (up to the largest one the static array holds) and
compares each result with the CPU oracle's routing and expansion and with
what moe_forward (which uses a caller workspace) computes for the same
inputs.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import moe_inputs as MI
import precision_moe_grouped_gb300 as P
from precision_moe_grouped_gb300 import _lib as L


def _forward_front(case):
    """ids, weights, offsets, row_of as moe_forward computes them."""
    from gpu_helpers import DeviceRun
    run = DeviceRun(case)
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


def _oracle_front(case):
    """ids, weights, offsets, row_of from the CPU oracle's routing and
    expansion (softmax top-k renormalised; stable expert-major rows)."""
    from oracle import moe as M
    ids, w = M.route(case.logits.cpu().numpy(), case.cfg.top_k)
    rt = M.expand(ids, w, case.cfg.num_experts)
    return rt.ids, rt.weights, rt.offsets, rt.row_of


def _scratch_bytes(T, E, k):
    """Scratch moe_route_noalloc carves for a shape (the layout noalloc.cu
    documents: per-chunk histogram, counts, row map, tile list, tile count,
    each rounded up to 256 bytes)."""
    up = lambda v: (v + 255) // 256 * 256      # noqa: E731
    R, chunks = T * k, (T + 31) // 32
    tiles = R // 32 + min(E, R) + 1
    off = up(chunks * E * 4)
    off = up(off + E * 4)
    off = up(off + R * 4)
    off = up(off + tiles * 16)
    return up(off + 16)


def _largest_tokens(E, k):
    lo, hi = 1, 1 << 20
    while lo < hi:
        m = (lo + hi + 1) // 2
        lo, hi = (m, hi) if _scratch_bytes(m, E, k) <= L.MOE_NOALLOC_SCRATCH_BYTES else (lo, m - 1)
    return lo


def _check(got, ref):
    np.testing.assert_array_equal(got[0], ref[0])                      # ids
    np.testing.assert_allclose(got[1], ref[1], rtol=3e-6, atol=1e-7)   # weights
    np.testing.assert_array_equal(got[2], ref[2])                      # offsets
    np.testing.assert_array_equal(got[3], ref[3])                      # row_of


@pytest.mark.gpu
def test_noalloc_route_matches_forward_and_oracle_on_consecutive_calls():
    """Consecutive calls on different shapes share the one static array:
    small decode-like shapes (the one-kernel small-batch path of the forward
    serves the same inputs), the DeepSeek-V3 routing shape at T = 2048 (E =
    256, top-8: the multi-chunk route, scan and rank kernels) and the largest
    token count whose scratch still fits the array.  Each result must equal
    the oracle's routing and expansion; the first three also moe_forward's
    front end."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    P.load()
    t_max = _largest_tokens(256, 8)
    assert _scratch_bytes(t_max + 1, 256, 8) > L.MOE_NOALLOC_SCRATCH_BYTES
    cases = [MI.make_case(MI.custom_config(8, 2, 256, 128), 200, seed=71),
             MI.make_case(MI.custom_config(16, 4, 256, 128), 37, seed=72),
             MI.make_case(MI.custom_config(256, 8, 256, 128), 2048, seed=73),
             MI.make_case(MI.custom_config(256, 8, 128, 128), t_max, seed=74, experts=[])]
    for i, case in enumerate(cases):
        got = _noalloc(case)
        _check(got, _oracle_front(case))
        if i < 3:
            _check(got, _forward_front(case))
    # a second call on an earlier shape after the largest one: the array's
    # leftover contents from the larger call must not leak into the result
    _check(_noalloc(cases[0]), _oracle_front(cases[0]))


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
