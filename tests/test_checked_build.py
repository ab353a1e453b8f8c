"""The bounds-checked debug build (libmoe_checked.so, -DMOE_CHECKS).

It validates the device-built work map (tile count and every tile entry)
where the GEMMs read it, so that a wrong map turns into the status
MOE_ERR_DEVICE_CHECK instead of an out-of-range access.  CPU: it builds and
exports every declared symbol.  GPU: a subset of the parity tests runs
against it in a child process (MOE_CHECKED=1 picks the library at import)
and must give the same results with device status 0; inside that child the
status words that carry the limits hold R and E."""
import ctypes
import os
import subprocess
import sys

import pytest

from precision_moe_grouped_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# parity tests that together reach every GEMM kernel: the one-CTA FP8 GEMM in
# all its tile variants, the CTA-pair GEMM, the MXFP8 and the W4A16 GEMMs
CHECKED_SUBSET = [
    "tests/test_gpu_parity.py::test_tiny_config_full",
    "tests/test_gpu_parity.py::test_several_tiles_ragged",
    "tests/test_gpu_parity.py::test_degenerate_routing",
    "tests/test_gpu_parity.py::test_empty_experts",
    "tests/test_gpu_parity.py::test_zero_tokens_is_noop",
    "tests/test_gpu_pair.py::test_pair_tiles_split_and_tails",
    "tests/test_gpu_mxfp8.py::test_mx_several_tiles_ragged",
    "tests/test_gpu_w4a16.py::test_w16_ragged_tiles",
    "tests/test_checked_build.py::test_limits_recorded_in_checked_build",
]


def test_checked_build_exports_every_symbol():
    from precision_moe_grouped_gb300 import build
    try:
        path = build.build(checks=True)
    except (RuntimeError, FileNotFoundError) as e:  # no nvcc on this machine
        pytest.skip(f"cannot build libmoe_checked.so here: {e}")
    assert os.path.basename(path) == "libmoe_checked.so"
    lib = ctypes.CDLL(path)
    for name in L.EXPORTS:
        assert hasattr(lib, name), name
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [ctypes.c_int32]
    assert b"bounds check" in lib.moe_status_string(L.MOE_ERR_DEVICE_CHECK)


@pytest.mark.gpu
def test_limits_recorded_in_checked_build():
    """Runs only inside the checked child process: the forward's first kernel
    wrote R = T * k and E to status words 2 and 3, and no check fired."""
    if not L.CHECKED:
        pytest.skip("runs in the MOE_CHECKED=1 child process")
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_inputs as MI
    from gpu_helpers import DeviceRun
    cfg = MI.CONFIGS["tiny"]
    for T in (1, 37, 300):
        run = DeviceRun(MI.make_case(cfg, T))
        assert run.status == 0
        assert list(run.ints("status", 4)[2:]) == [T * cfg.top_k, cfg.num_experts]


@pytest.mark.gpu
def test_parity_subset_on_checked_build():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if L.CHECKED:
        pytest.skip("already the checked child process")
    from precision_moe_grouped_gb300 import build
    build.build(checks=True)
    env = dict(os.environ, MOE_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p",
                        "no:cacheprovider", *CHECKED_SUBSET], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout, r.stdout[-2000:]
