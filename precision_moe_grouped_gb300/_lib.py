"""ctypes binding of libmoe.so (include/moe.h).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  If the
library is not built, loading fails loudly -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
# MOE_CHECKED=1 selects the bounds-checked debug build (build(checks=True))
CHECKED = os.environ.get("MOE_CHECKED", "0") == "1"
LIB_PATH = os.path.join(PKG, "libmoe_checked.so" if CHECKED else "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_MISALIGNED = -3
MOE_ERR_WORKSPACE_TOO_SMALL = -4
MOE_ERR_CUDA = -5
MOE_ERR_DEVICE_TIMEOUT = -6
MOE_ERR_DEVICE_CHECK = -7

MOE_W4A8_MXFP4_FP8 = 0
MOE_W4A16_MXFP4_BF16 = 1
MOE_W8A8_MXFP8 = 2

# every symbol include/moe.h declares
EXPORTS = ("moe_workspace_size", "moe_workspace_layout", "moe_prepare_weights", "moe_forward",
           "moe_forward_ex", "moe_forward_host", "moe_read_device_status",
           "moe_selftest_timeout", "moe_last_error", "moe_stage_name", "moe_status_string",
           "moe_version", "moe_route_noalloc", "moe_steps_workspace_size",
           "moe_forward_host_steps")

MOE_NOALLOC_SCRATCH_BYTES = 4 << 20

MOE_NUM_STAGES = 8
MOE_SMALL_BATCH_TOKENS = 256


MOE_TINY_BATCH_TOKENS = 32


def kernels_per_forward(num_tokens: int, mode: int = 0) -> int:
    """Kernels one forward launches (0 for an empty batch): W4A8 batches of
    <= 32 tokens route and expand in one kernel, batches of <= 256 tokens in
    two, larger ones in three (routing, scan, scatter); then GEMM1, the h
    quantisation, GEMM2 and the combine."""
    if num_tokens == 0:
        return 0
    if mode == 0 and num_tokens <= MOE_TINY_BATCH_TOKENS:
        return 5
    return 6 if num_tokens <= MOE_SMALL_BATCH_TOKENS else 7


class MoeShape(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32)]


class MoeOptions(ctypes.Structure):
    _fields_ = [("tile_variant", ctypes.c_int32), ("timeout_ms", ctypes.c_int32),
                ("stage_events", ctypes.c_void_p), ("prefetch_stages", ctypes.c_int32),
                ("gather_x", ctypes.c_int32), ("fuse_combine", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 1)]


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "status", "ids", "weights", "row_of", "counts", "offsets", "chunk_counts", "token_slot",
        "tiles", "xq", "x_scale", "h", "hq", "h_scale", "y", "x_stage", "logits_stage",
        "out_stage", "tile_plan", "x_sf", "h_sf", "x_sf_tiled", "h_sf_tiled", "total")] + [("max_tiles", ctypes.c_int32), ("num_chunks", ctypes.c_int32),
                                  ("reserved", ctypes.c_int32 * 6)]


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"moe error {code}: {msg}")
        self.code = code


_lib = None


def load() -> ctypes.CDLL:
    """Load libmoe.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as "
                           f"g; g.build()\"` first (there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    shp = ctypes.POINTER(MoeShape)
    lib.moe_workspace_size.argtypes = [shp, i32]
    lib.moe_workspace_size.restype = sz
    lib.moe_workspace_layout.argtypes = [shp, i32, ctypes.POINTER(WsLayout)]
    lib.moe_workspace_layout.restype = i32
    lib.moe_prepare_weights.argtypes = [shp, i32] + [vp] * 9
    lib.moe_prepare_weights.restype = i32
    lib.moe_forward.argtypes = [shp, i32] + [vp] * 8 + [sz, vp]
    lib.moe_forward.restype = i32
    lib.moe_forward_ex.argtypes = [shp, i32] + [vp] * 8 + [sz, vp, ctypes.POINTER(MoeOptions)]
    lib.moe_forward_ex.restype = i32
    lib.moe_forward_host.argtypes = [shp, i32] + [vp] * 8 + [sz, vp, ctypes.POINTER(MoeOptions)]
    lib.moe_forward_host.restype = i32
    lib.moe_steps_workspace_size.argtypes = [shp, i32]
    lib.moe_steps_workspace_size.restype = sz
    lib.moe_forward_host_steps.argtypes = ([shp, i32, i32, vp, vp] + [vp] * 6 +
                                           [sz, vp, ctypes.POINTER(MoeOptions)])
    lib.moe_forward_host_steps.restype = i32
    lib.moe_read_device_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
    lib.moe_read_device_status.restype = i32
    lib.moe_selftest_timeout.argtypes = [vp, i32, vp]
    lib.moe_selftest_timeout.restype = i32
    for f in ("moe_last_error", "moe_version"):
        getattr(lib, f).argtypes = []
        getattr(lib, f).restype = ctypes.c_char_p
    lib.moe_route_noalloc.argtypes = [shp, vp, vp, vp, vp, vp, vp]
    lib.moe_route_noalloc.restype = i32
    lib.moe_stage_name.argtypes = [i32]
    lib.moe_stage_name.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [i32]
    lib.moe_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def check(rc: int) -> None:
    if rc != MOE_OK:
        lib = load()
        raise MoeError(rc, (lib.moe_last_error() or b"").decode() or
                       lib.moe_status_string(rc).decode())


def shape(T: int, E: int, k: int, H: int, I: int) -> MoeShape:
    return MoeShape(T, E, k, H, I)


def options(tile_variant: int = 0, timeout_ms: int = 0, stage_events=None,
            prefetch_stages: int = 0, gather_x: int = 0, fuse_combine: int = 0) -> MoeOptions:
    """stage_events: None, or a ctypes array of MOE_NUM_STAGES + 1 cudaEvent_t
    handles (e.g. from stage_event_array())."""
    o = MoeOptions()
    o.tile_variant, o.timeout_ms, o.prefetch_stages = tile_variant, timeout_ms, prefetch_stages
    o.gather_x, o.fuse_combine = gather_x, fuse_combine
    o.stage_events = ctypes.cast(stage_events, ctypes.c_void_p) if stage_events is not None else None
    return o


def stage_names() -> list:
    lib = load()
    return [lib.moe_stage_name(i).decode() for i in range(MOE_NUM_STAGES)]


def stage_event_array(events) -> "ctypes.Array":
    """ctypes array of the raw cudaEvent_t handles of torch.cuda.Event objects."""
    assert len(events) == MOE_NUM_STAGES + 1
    return (ctypes.c_void_p * len(events))(*[int(e.cuda_event) for e in events])


def workspace_size(s: MoeShape, mode: int = MOE_W4A8_MXFP4_FP8) -> int:
    return int(load().moe_workspace_size(ctypes.byref(s), mode))


def steps_workspace_size(s: MoeShape, mode: int = MOE_W4A8_MXFP4_FP8) -> int:
    """Workspace bytes of forward_host_steps (moe_steps_workspace_size)."""
    return int(load().moe_steps_workspace_size(ctypes.byref(s), mode))


def workspace_layout(s: MoeShape, mode: int = MOE_W4A8_MXFP4_FP8) -> WsLayout:
    L = WsLayout()
    check(load().moe_workspace_layout(ctypes.byref(s), mode, ctypes.byref(L)))
    return L


# ------------------------------------------------------------ tensor checks
# The C ABI takes raw pointers and cannot tell a host buffer, a wrong dtype or
# a strided view from a valid device tensor; a wrong one would be read as
# device memory.  The binding therefore checks every tensor it marshals
# (placement, device, dtype, contiguity, shape or size) and raises
# MoeError(MOE_ERR_INVALID_ARG) before any library call.

def _bad(msg: str):
    raise MoeError(MOE_ERR_INVALID_ARG, msg)


def _check_tensor(t, name: str, *, cuda: bool, dtype=None, itemsize: int | None = None,
                  shape=None, numel: int | None = None, device: int | None = None) -> None:
    if t is None:
        _bad(f"{name} is None")
    if bool(t.is_cuda) != cuda:
        _bad(f"{name} must be a {'CUDA' if cuda else 'host (CPU)'} tensor, got {t.device}")
    if cuda and device is not None and t.device.index != device:
        _bad(f"{name} is on {t.device}, the current device is cuda:{device}")
    if dtype is not None and t.dtype != dtype:
        _bad(f"{name} must be {dtype}, got {t.dtype}")
    if itemsize is not None and t.element_size() != itemsize:
        _bad(f"{name} must have {itemsize}-byte elements, got {t.dtype}")
    if not t.is_contiguous():
        _bad(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        _bad(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if numel is not None and t.numel() != numel:
        _bad(f"{name} must hold {numel} elements, got {t.numel()}")


def weight_numels(s: MoeShape, mode: int) -> tuple:
    """Elements (bytes) of w1, w1_sf, w2, w2_sf: MXFP4 codes two per byte
    (MXFP8: one E4M3 byte each) and one E8M0 byte per 32 K."""
    E, H, I = s.num_experts, s.hidden, s.inter
    per = 1 if mode == MOE_W8A8_MXFP8 else 2
    return (E * 2 * I * H // per, E * 2 * I * H // 32, E * H * I // per, E * H * I // 32)


def _check_mode(mode: int) -> None:
    if mode not in (MOE_W4A8_MXFP4_FP8, MOE_W4A16_MXFP4_BF16, MOE_W8A8_MXFP8):
        _bad(f"quant_mode {mode} unknown")


def _check_weights(s: MoeShape, mode: int, tensors, names, device) -> None:
    for t, name, n in zip(tensors, names, weight_numels(s, mode)):
        _check_tensor(t, name, cuda=True, itemsize=1, numel=n, device=device)


def validate_forward(s: MoeShape, mode: int, x, logits, w1_p, w1_sf_p, w2_p, w2_sf_p, out,
                     workspace, host: bool = False, device: int | None = None) -> None:
    """Checks the tensors of forward() (host=False) or forward_host()
    (host=True: x, logits and out on the host).  `device`: the current CUDA
    device index every device tensor must live on."""
    import torch
    _check_mode(mode)
    T, E, H = s.num_tokens, s.num_experts, s.hidden
    dev = not host
    _check_tensor(x, "x", cuda=dev, dtype=torch.bfloat16, shape=(T, H), device=device)
    _check_tensor(logits, "logits", cuda=dev, dtype=torch.float32, shape=(T, E), device=device)
    _check_tensor(out, "out", cuda=dev, dtype=torch.bfloat16, shape=(T, H), device=device)
    _check_weights(s, mode, (w1_p, w1_sf_p, w2_p, w2_sf_p), ("w1", "w1_sf", "w2", "w2_sf"),
                   device)
    _check_tensor(workspace, "workspace", cuda=True, device=device)


def _current_device() -> int | None:
    """Index of the current CUDA device (None without one: every tensor then
    fails the placement check)."""
    import torch
    return torch.cuda.current_device() if torch.cuda.is_available() else None


def _stream(stream) -> int:
    if stream is not None:
        return int(stream)
    import torch
    return int(torch.cuda.current_stream().cuda_stream)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def prepare_weights(s: MoeShape, w1, w1_sf, w2, w2_sf, w1_p, w1_sf_p, w2_p, w2_sf_p,
                    mode: int = MOE_W4A8_MXFP4_FP8, stream=None) -> None:
    _check_mode(mode)
    dev = _current_device()
    names = ("w1", "w1_sf", "w2", "w2_sf")
    _check_weights(s, mode, (w1, w1_sf, w2, w2_sf), names, dev)
    _check_weights(s, mode, (w1_p, w1_sf_p, w2_p, w2_sf_p), [n + "_p" for n in names], dev)
    check(load().moe_prepare_weights(ctypes.byref(s), mode, *(_ptr(t) for t in (
        w1, w1_sf, w2, w2_sf, w1_p, w1_sf_p, w2_p, w2_sf_p)), _stream(stream)))


def forward(s: MoeShape, x, logits, w1_p, w1_sf_p, w2_p, w2_sf_p, out, workspace,
            mode: int = MOE_W4A8_MXFP4_FP8, opts: MoeOptions | None = None, stream=None,
            validate: bool = True) -> None:
    """validate=False skips the tensor checks (a few microseconds of host time)
    for a caller that reuses tensors it has already passed once with checks."""
    lib = load()
    if validate:
        validate_forward(s, mode, x, logits, w1_p, w1_sf_p, w2_p, w2_sf_p, out, workspace,
                         device=_current_device())
    nbytes = workspace.numel() * workspace.element_size()
    args = [ctypes.byref(s), mode, _ptr(x), _ptr(logits), _ptr(w1_p), _ptr(w1_sf_p), _ptr(w2_p),
            _ptr(w2_sf_p), _ptr(out), _ptr(workspace), nbytes, _stream(stream)]
    if opts is None:
        check(lib.moe_forward(*args))
    else:
        check(lib.moe_forward_ex(*args, ctypes.byref(opts)))


def forward_host(s: MoeShape, x_host, logits_host, w1_p, w1_sf_p, w2_p, w2_sf_p, out_host,
                 workspace, mode: int = MOE_W4A8_MXFP4_FP8, opts: MoeOptions | None = None,
                 stream=None, validate: bool = True) -> None:
    if validate:
        validate_forward(s, mode, x_host, logits_host, w1_p, w1_sf_p, w2_p, w2_sf_p, out_host,
                         workspace, host=True, device=_current_device())
    nbytes = workspace.numel() * workspace.element_size()
    check(load().moe_forward_host(ctypes.byref(s), mode, _ptr(x_host), _ptr(logits_host),
                                  _ptr(w1_p), _ptr(w1_sf_p), _ptr(w2_p), _ptr(w2_sf_p),
                                  _ptr(out_host), _ptr(workspace), nbytes, _stream(stream),
                                  ctypes.byref(opts) if opts is not None else None))


def forward_host_steps(s: MoeShape, x_hosts, logits_hosts, w1_p, w1_sf_p, w2_p, w2_sf_p,
                       out_hosts, workspace, mode: int = MOE_W4A8_MXFP4_FP8,
                       opts: MoeOptions | None = None, stream=None,
                       validate: bool = True) -> None:
    """len(x_hosts) forwards, step i from host tensors x_hosts[i],
    logits_hosts[i] into out_hosts[i], copies overlapped with the computation
    (moe_forward_host_steps; page-locked host tensors for the overlap).  The
    workspace holds steps_workspace_size(s, mode) bytes."""
    n = len(x_hosts)
    if len(logits_hosts) != n or len(out_hosts) != n:
        _bad("x_hosts, logits_hosts and out_hosts must have the same length")
    if validate:
        dev = _current_device()
        for i in range(n):
            validate_forward(s, mode, x_hosts[i], logits_hosts[i], w1_p, w1_sf_p, w2_p, w2_sf_p,
                             out_hosts[i], workspace, host=True, device=dev)
    xs = (ctypes.c_void_p * max(n, 1))(*[_ptr(t) for t in x_hosts])
    ls = (ctypes.c_void_p * max(n, 1))(*[_ptr(t) for t in logits_hosts])
    os_ = (ctypes.c_void_p * max(n, 1))(*[_ptr(t) for t in out_hosts])
    nbytes = workspace.numel() * workspace.element_size()
    check(load().moe_forward_host_steps(ctypes.byref(s), mode, n, xs, ls, _ptr(w1_p),
                                        _ptr(w1_sf_p), _ptr(w2_p), _ptr(w2_sf_p), os_,
                                        _ptr(workspace), nbytes, _stream(stream),
                                        ctypes.byref(opts) if opts is not None else None))


def read_device_status(workspace, stream=None) -> int:
    _check_tensor(workspace, "workspace", cuda=True, device=_current_device())
    v = ctypes.c_int32(0)
    check(load().moe_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(v)))
    return int(v.value)


def selftest_timeout(workspace, timeout_us: int, stream=None) -> None:
    _check_tensor(workspace, "workspace", cuda=True, device=_current_device())
    check(load().moe_selftest_timeout(_ptr(workspace), timeout_us, _stream(stream)))


def route_noalloc(s: MoeShape, logits, ids, weights, offsets, row_of, stream=None) -> None:
    """Routing front end (ids, weights, offsets, row map) using the library's
    static device scratch instead of a workspace; see moe_route_noalloc in
    include/moe.h for the size limit and the no-overlap rule."""
    import torch
    dev = _current_device()
    T, E, k = s.num_tokens, s.num_experts, s.top_k
    _check_tensor(logits, "logits", cuda=True, dtype=torch.float32, shape=(T, E), device=dev)
    for t, name, dt, shp in ((ids, "ids", torch.int32, (T, k)), (weights, "weights", torch.float32,
                              (T, k)), (offsets, "offsets", torch.int32, (E + 1,)),
                             (row_of, "row_of", torch.int32, (T, k))):
        _check_tensor(t, name, cuda=True, dtype=dt, shape=shp, device=dev)
    check(load().moe_route_noalloc(ctypes.byref(s), _ptr(logits), _ptr(ids), _ptr(weights),
                                   _ptr(offsets), _ptr(row_of), _stream(stream)))
