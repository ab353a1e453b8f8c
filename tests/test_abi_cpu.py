"""CPU-side checks of the C ABI: the library builds, loads and exports every
function include/moe.h declares; host-only entry points (workspace size and
layout) and argument validation work without a GPU (validation returns
before any CUDA call)."""
import ctypes
import os
import re

import pytest

import precision_moe_grouped_gb300 as P
from precision_moe_grouped_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from precision_moe_grouped_gb300 import build
        try:
            build.build()
        except (RuntimeError, FileNotFoundError) as e:  # no nvcc on this machine
            pytest.skip(f"cannot build libmoe.so here: {e}")
    return P.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    decl = declared_functions()
    assert len(decl) >= 10
    for name in decl:
        assert hasattr(lib, name), name
    assert set(decl) == set(L.EXPORTS)
    assert b"sm_103a" in lib.moe_version()


def _shape(T=16, E=8, k=2, H=256, I=128):
    return P.shape(T, E, k, H, I)


def test_workspace_size_and_layout(lib):
    s = _shape(4096, 256, 8, 7168, 2048)
    n = P.workspace_size(s)
    lay = P.workspace_layout(s)
    assert n == lay.total and n % 256 == 0
    R = 4096 * 8
    offs = [("status", 16), ("ids", R * 4), ("weights", R * 4), ("row_of", R * 4),
            ("counts", 256 * 4), ("offsets", 257 * 4), ("chunk_counts", 128 * 256 * 4),
            ("token_slot", R * 4), ("tiles", lay.max_tiles * 16), ("xq", R * 7168),
            ("x_scale", R * 4), ("h", R * 2048 * 2), ("hq", R * 2048), ("h_scale", R * 4),
            ("y", R * 7168 * 2), ("x_stage", 4096 * 7168 * 2), ("logits_stage", 4096 * 256 * 4),
            ("out_stage", 4096 * 7168 * 2)]
    end = 0
    for name, size in offs:
        o = getattr(lay, name)
        assert o % 256 == 0 and o >= end, name
        end = o + size
    assert end <= n
    assert lay.num_chunks == 128
    # the tile bound covers the worst case of the decode tiling
    assert lay.max_tiles >= R // 32 + 256


def test_workspace_layout_mxfp8(lib):
    """W8A8 adds the E8M0 block-scale regions (row-major and per-tile); the
    W4A8 layout gives them no bytes."""
    T, E, k, H, I = 4096, 256, 8, 7168, 2048
    s, R = _shape(T, E, k, H, I), T * k
    l0, l2 = P.workspace_layout(s, 0), P.workspace_layout(s, 2)
    assert l2.max_tiles == l0.max_tiles
    sizes = [("tile_plan", E * 8), ("x_sf", R * H // 32), ("h_sf", R * I // 32),
             ("x_sf_tiled", l2.max_tiles * (H // 128) * 1024),
             ("h_sf_tiled", l2.max_tiles * (I // 128) * 1024)]
    end = l2.out_stage
    for name, size in sizes:
        o = getattr(l2, name)
        assert o % 256 == 0 and o >= end, name
        end = o + size
    assert end <= l2.total == P.workspace_size(s, 2)
    assert l0.x_sf == l0.h_sf == l0.x_sf_tiled == l0.h_sf_tiled   # zero-size in W4A8
    assert l0.total < l2.total


@pytest.mark.parametrize("bad", [dict(T=-1), dict(E=0), dict(k=0), dict(k=9, E=8), dict(k=33, E=64),
                                 dict(H=100), dict(I=96), dict(E=2000),
                                 dict(E=1024, I=8192, H=16384)])
def test_workspace_size_rejects_bad_shapes(lib, bad):
    kw = dict(T=16, E=8, k=2, H=256, I=128)
    kw.update(bad)
    assert P.workspace_size(_shape(**kw)) == 0
    assert P.workspace_size(_shape(), 7) == 0


def test_weight_box_coordinates_stay_32_bit(lib):
    """E * 2I * H / 128 weight-box rows must fit a 32-bit TMA coordinate:
    the largest shape just below the limit is accepted, the next one not."""
    ok = _shape(T=1, E=1023, k=1, H=16384, I=8192)       # 1023 * 2^14 * 2^7 < 2^31
    assert P.workspace_size(ok) > 0
    bad = _shape(T=1, E=1024, k=1, H=16384, I=8192)      # exactly 2^31
    assert P.workspace_size(bad) == 0
    L_ = L.WsLayout()
    assert lib.moe_workspace_layout(ctypes.byref(bad), 0, ctypes.byref(L_)) == \
        L.MOE_ERR_UNSUPPORTED
    assert b"32-bit" in lib.moe_last_error()
    # work items: (R/16 + E + 1) * 2I/128 with R = 2^31 - 1 expanded rows
    many = _shape(T=(1 << 31) - 1, E=8, k=1, H=256, I=1 << 14)
    assert P.workspace_size(many) == 0 and b"work items" in lib.moe_last_error()


def _fwd(lib, s, ptrs, nbytes, mode=0, opts=None):
    args = [ctypes.byref(s), mode] + list(ptrs) + [nbytes, None]
    if opts is None:
        return lib.moe_forward(*args)
    return lib.moe_forward_ex(*args, ctypes.byref(opts))


def test_forward_validation_without_gpu(lib):
    s = _shape()
    need = P.workspace_size(s)
    good = [0x100000 * (i + 1) for i in range(8)]
    assert _fwd(lib, s, [None] + good[1:], need) == L.MOE_ERR_INVALID_ARG
    mis = list(good)
    mis[0] += 8                                         # x not 16-byte aligned
    assert _fwd(lib, s, mis, need) == L.MOE_ERR_MISALIGNED
    mis = list(good)
    mis[2] += 32                                        # w1 not 256-byte aligned
    assert _fwd(lib, s, mis, need) == L.MOE_ERR_MISALIGNED
    assert _fwd(lib, s, good, need - 1) == L.MOE_ERR_WORKSPACE_TOO_SMALL
    # W4A16 keeps two FP8 terms per expanded element: the W4A8 workspace is
    # too small for it
    assert P.workspace_size(s, 1) > need
    assert _fwd(lib, s, good, need, mode=1) == L.MOE_ERR_WORKSPACE_TOO_SMALL
    assert _fwd(lib, s, good, need, mode=2) == L.MOE_ERR_WORKSPACE_TOO_SMALL
    assert _fwd(lib, s, good, need, mode=5) == L.MOE_ERR_INVALID_ARG
    assert _fwd(lib, _shape(H=200), good, need) == L.MOE_ERR_MISALIGNED
    assert _fwd(lib, s, good, need, opts=P.options(tile_variant=99)) == L.MOE_ERR_INVALID_ARG
    assert _fwd(lib, s, good, need, opts=P.options(tile_variant=-1)) == L.MOE_ERR_INVALID_ARG
    o = P.options()
    o.reserved[0] = 1
    assert _fwd(lib, s, good, need, opts=o) == L.MOE_ERR_INVALID_ARG
    assert _fwd(lib, s, good, need, opts=P.options(gather_x=2)) == L.MOE_ERR_INVALID_ARG
    assert _fwd(lib, s, good, need, opts=P.options(fuse_combine=3)) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_last_error()                          # a message was recorded
    # zero tokens: a no-op that succeeds without touching the device
    assert _fwd(lib, _shape(T=0), [None] * 8, 0) == L.MOE_OK
    assert lib.moe_forward(None, 0, *([None] * 8), 0, None) == L.MOE_ERR_INVALID_ARG


def test_prepare_and_misc_validation_without_gpu(lib):
    s = _shape()
    p = [0x100000 * (i + 1) for i in range(8)]
    assert lib.moe_prepare_weights(ctypes.byref(s), 0, None, *p[1:], None) == L.MOE_ERR_INVALID_ARG
    alias = list(p)
    alias[4] = alias[0]
    assert lib.moe_prepare_weights(ctypes.byref(s), 0, *alias, None) == L.MOE_ERR_INVALID_ARG
    for mode in (1, 2):   # W4A16 and W8A8 validate their arguments the same way
        assert lib.moe_prepare_weights(ctypes.byref(s), mode, *alias, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_prepare_weights(ctypes.byref(s), 7, *p, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_timeout(None, 10, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_timeout(0x100000, 0, None) == L.MOE_ERR_INVALID_ARG
    st = ctypes.c_int32(0)
    assert lib.moe_read_device_status(None, None, ctypes.byref(st)) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_status_string(-6) == b"device-side wait timed out"


def _steps(lib, s, n, ptrs, x, lg, out, nbytes, opts=None):
    arr = lambda v: (ctypes.c_void_p * len(v))(*v) if v is not None else None
    return lib.moe_forward_host_steps(ctypes.byref(s), 0, n, arr(x), arr(lg), *ptrs, arr(out),
                                      0x200000, nbytes, None,
                                      ctypes.byref(opts) if opts is not None else None)


def test_steps_workspace_and_validation_without_gpu(lib):
    """moe_forward_host_steps: its workspace is moe_forward's plus a second
    staging set (x, logits, out of one step, each 256-byte aligned); argument
    errors return before any CUDA call."""
    T, E, H = 16, 8, 256
    s = _shape(T, E, 2, H, 128)
    up = lambda n: (n + 255) // 256 * 256
    need = P.steps_workspace_size(s)
    assert need == P.workspace_size(s) + up(T * H * 2) + up(T * E * 4) + up(T * H * 2)
    assert P.steps_workspace_size(s, 1) > need           # W4A16's larger workspace
    assert P.steps_workspace_size(_shape(H=200)) == 0
    w = [0x100000 * (i + 1) for i in range(4)]
    hx, hl, ho = [0x7000] * 3, [0x8000] * 3, [0x9000] * 3
    assert _steps(lib, s, -1, w, hx, hl, ho, need) == L.MOE_ERR_INVALID_ARG
    assert _steps(lib, s, 0, w, None, None, None, 0) == L.MOE_OK
    assert _steps(lib, _shape(T=0), 3, w, None, None, None, 0) == L.MOE_OK
    assert _steps(lib, s, 3, w, None, hl, ho, need) == L.MOE_ERR_INVALID_ARG
    assert _steps(lib, s, 3, w, hx, hl, [0x9000, None, 0x9000], need) == L.MOE_ERR_INVALID_ARG
    assert _steps(lib, s, 3, w, hx, hl, ho, P.workspace_size(s)) == \
        L.MOE_ERR_WORKSPACE_TOO_SMALL
    mis = list(w)
    mis[1] += 32                                          # w1_sf not 256-byte aligned
    assert _steps(lib, s, 3, mis, hx, hl, ho, need) == L.MOE_ERR_MISALIGNED
    ev = (ctypes.c_void_p * 9)(*([0x10] * 9))
    o = P.options(stage_events=ev)
    assert _steps(lib, s, 3, w, hx, hl, ho, need, opts=o) == L.MOE_ERR_INVALID_ARG
    assert b"stage_events" in lib.moe_last_error()


def test_no_device_gives_cuda_error(lib):
    """Valid arguments on a machine without a GPU: the first CUDA call fails
    and every entry point that reaches one returns MOE_ERR_CUDA with a
    message, before any memory is touched.  Skipped where a GPU exists (the
    pointers here are not device memory)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: these pointers must not reach it")
    s = _shape()
    good = [0x100000 * (i + 1) for i in range(8)]
    assert _fwd(lib, s, good, P.workspace_size(s)) == L.MOE_ERR_CUDA
    assert lib.moe_last_error()
    assert lib.moe_prepare_weights(ctypes.byref(s), 0, *good, None) == L.MOE_ERR_CUDA
    assert lib.moe_selftest_timeout(0x100000, 10, None) == L.MOE_ERR_CUDA
    hx = (ctypes.c_void_p * 2)(0x7000, 0x7000)
    assert lib.moe_forward_host_steps(ctypes.byref(s), 0, 2, hx, hx, *good[:4], hx, 0x200000,
                                      P.steps_workspace_size(s), None, None) == L.MOE_ERR_CUDA
    st = ctypes.c_int32(0)
    assert lib.moe_read_device_status(0x100000, None, ctypes.byref(st)) == L.MOE_ERR_CUDA
