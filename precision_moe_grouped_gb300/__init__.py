"""GB300-native fused MXFP4 x FP8 mixture-of-experts forward.

The compute path is libmoe.so (csrc/, C ABI in include/moe.h): hand-written
sm_103a CUDA kernels for routing, the expert-sorted scatter with per-token
FP8 quantisation, two tcgen05 block-scaled grouped GEMMs (SwiGLU and the
token scale fused in GEMM1's epilogue), the FP8 quantisation of h and the
top-k combine.  This package only marshals torch tensors into that ABI.
"""
from __future__ import annotations

from . import _lib
from ._lib import (MOE_W4A8_MXFP4_FP8, MOE_W4A16_MXFP4_BF16, MOE_W8A8_MXFP8, MoeError,
                   MoeOptions, MoeShape, WsLayout, forward, forward_host, forward_host_steps,
                   load, options, prepare_weights, read_device_status, selftest_timeout, shape,
                   steps_workspace_size, workspace_layout, workspace_size)

__all__ = ["FusedMoE", "MoeError", "MoeOptions", "MoeShape", "WsLayout", "forward",
           "forward_host", "forward_host_steps", "load", "options", "prepare_weights",
           "read_device_status", "selftest_timeout", "shape", "steps_workspace_size",
           "workspace_layout", "workspace_size",
           "MOE_W4A8_MXFP4_FP8", "MOE_W4A16_MXFP4_BF16", "MOE_W8A8_MXFP8"]


class FusedMoE:
    """Prepared expert weights on one GPU plus a reusable workspace.

    w1 uint8 [E, 2I, H/2], w1_sf uint8 [E, 2I, H/32], w2 uint8 [E, H, I/2],
    w2_sf uint8 [E, H, I/32] (MXFP4: E2M1 codes two per byte, low nibble =
    even K index; E8M0 scale per 32 K); in the W8A8 mode w1 [E, 2I, H] and
    w2 [E, H, I] hold E4M3 codes.  Rows 0..I-1 of w1 are the gate
    projection, I..2I-1 the up projection."""

    def __init__(self, w1, w1_sf, w2, w2_sf, top_k: int, mode: int = MOE_W4A8_MXFP4_FP8):
        import torch
        E, I2, Hk = w1.shape   # Hk = H/2 packed E2M1 bytes, or H E4M3 bytes (W8A8)
        H = Hk if mode == MOE_W8A8_MXFP8 else Hk * 2
        self.E, self.I, self.H, self.top_k, self.mode = E, I2 // 2, H, top_k, mode
        self.device = w1.device
        self.w1_p = torch.empty_like(w1)
        self.w1_sf_p = torch.empty_like(w1_sf)
        self.w2_p = torch.empty_like(w2)
        self.w2_sf_p = torch.empty_like(w2_sf)
        prepare_weights(self.shape(0), w1, w1_sf, w2, w2_sf, self.w1_p, self.w1_sf_p, self.w2_p,
                        self.w2_sf_p, mode)
        self._ws = None
        self._steps_ws = None

    def shape(self, T: int) -> MoeShape:
        return shape(T, self.E, self.top_k, self.H, self.I)

    def workspace(self, T: int):
        import torch
        need = workspace_size(self.shape(T), self.mode)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    def __call__(self, x, logits, out=None, opts: MoeOptions | None = None):
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=self.device)
        ws = self.workspace(T)
        forward(self.shape(T), x, logits, self.w1_p, self.w1_sf_p, self.w2_p, self.w2_sf_p, out,
                ws, self.mode, opts)
        return out

    def host_steps(self, xs, logits, outs=None, opts: MoeOptions | None = None):
        """Forwards of host (CPU) tensors xs[i] [T, H] bf16 and logits[i]
        [T, E] float32, one per step, with the host<->device copies
        overlapped with the neighbouring steps' computation
        (moe_forward_host_steps; page-locked tensors for the overlap).
        Returns the host outputs, complete when the current stream reaches
        this point."""
        import torch
        T = xs[0].shape[0]
        if outs is None:
            outs = [torch.empty((T, self.H), dtype=torch.bfloat16, pin_memory=True)
                    for _ in xs]
        need = steps_workspace_size(self.shape(T), self.mode)
        if self._steps_ws is None or self._steps_ws.numel() < need:
            self._steps_ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        forward_host_steps(self.shape(T), xs, logits, self.w1_p, self.w1_sf_p, self.w2_p,
                           self.w2_sf_p, outs, self._steps_ws, self.mode, opts)
        return outs
