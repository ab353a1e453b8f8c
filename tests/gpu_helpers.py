"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and read its intermediates back from the workspace; run the oracle on the
same seeded inputs."""
from __future__ import annotations

import os

import numpy as np
import torch

import moe_inputs as MI
import precision_moe_grouped_gb300 as P
from oracle import moe as M


def max_err_ok(got, ref, max_rel=2e-2, mean_rel=5e-3):
    """Output tolerance: max|err| <= max_rel * max|ref| and
    sum|err| / sum|ref| <= mean_rel."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    mx = float(err.max()) if err.size else 0.0
    ref_max = float(np.abs(ref).max()) if ref.size else 0.0
    mean = float(err.sum() / max(np.abs(ref).sum(), 1e-30))
    ok = mx <= max_rel * ref_max + 1e-30 and mean <= mean_rel
    return ok, dict(max_err=mx, ref_max=ref_max, mean_rel=mean)


class ExpertView:
    """Indexable view of one expert tensor living on the GPU; copies an expert
    to the host on first use (the oracle indexes weights by expert)."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.shape = tuple(t.shape)
        self._cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self._cache:
            self._cache[e] = self.t[e].cpu().numpy()
        return self._cache[e]


def oracle_weights(case: MI.MoeCase) -> M.Weights:
    if case.w1.is_cuda:
        return M.Weights(ExpertView(case.w1), ExpertView(case.w1_sf), ExpertView(case.w2),
                         ExpertView(case.w2_sf), mode=case.mode)
    return M.Weights(case.w1.numpy(), case.w1_sf.numpy(), case.w2.numpy(), case.w2_sf.numpy(),
                     mode=case.mode)


def x_bits(case: MI.MoeCase) -> np.ndarray:
    return case.x.view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceRun:
    """One forward through the C ABI with every intermediate read back."""

    def __init__(self, case: MI.MoeCase, variant: int = 0, moe: P.FusedMoE | None = None,
                 gather_x: int = 0, fuse_combine: int = 0, ws=None):
        dev = torch.device("cuda:0")
        cfg = case.cfg
        self.case = case
        T, E, k, H, I = case.T, cfg.num_experts, cfg.top_k, cfg.hidden, cfg.inter
        self.mode = mode = case.mode
        self.moe = moe or P.FusedMoE(case.w1.to(dev), case.w1_sf.to(dev), case.w2.to(dev),
                                     case.w2_sf.to(dev), k, mode=mode)
        x = case.x.to(dev)
        logits = case.logits.to(dev)
        s = P.shape(T, E, k, H, I)
        self.ws = ws if ws is not None else torch.zeros(max(P.workspace_size(s, mode), 256),
                                                        dtype=torch.uint8, device=dev)
        self.out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=dev)
        opts = P.options(tile_variant=variant, gather_x=gather_x, fuse_combine=fuse_combine)
        P.forward(s, x, logits, self.moe.w1_p, self.moe.w1_sf_p, self.moe.w2_p,
                  self.moe.w2_sf_p, self.out, self.ws, mode=mode, opts=opts)
        torch.cuda.synchronize()
        self.status = P.read_device_status(self.ws)
        self.L = P.workspace_layout(s, mode)
        self.T, self.E, self.k, self.H, self.I, self.R = T, E, k, H, I, T * k
        # W4A16: the activations and h are stored as two FP8 terms (hi | lo)
        self.terms = 2 if mode == MI.QUANT_W4A16 else 1

    def _view(self, off, n, dtype):
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).cpu()

    def ints(self, name, n):
        return self._view(getattr(self.L, name), n, torch.int32).numpy()

    def floats(self, name, n):
        return self._view(getattr(self.L, name), n, torch.float32).numpy()

    @property
    def ids(self):
        return self.ints("ids", self.R).reshape(self.T, self.k)

    @property
    def weights(self):
        return self.floats("weights", self.R).reshape(self.T, self.k)

    @property
    def row_of(self):
        return self.ints("row_of", self.R).reshape(self.T, self.k)

    @property
    def counts(self):
        return self.ints("counts", self.E)

    @property
    def offsets(self):
        return self.ints("offsets", self.E + 1)

    @property
    def token_slot(self):
        return self.ints("token_slot", self.R)

    @property
    def xq(self):
        """FP8 codes of the expanded rows, [R, H] (W4A16: [R, 2H], hi | lo)."""
        w = self.terms * self.H
        return self._view(self.L.xq, self.R * w, torch.uint8).numpy().reshape(self.R, w)

    @property
    def x_scale(self):
        return self.floats("x_scale", self.R)

    def bytes_(self, name, n):
        return self._view(getattr(self.L, name), n, torch.uint8).numpy()

    @property
    def x_sf(self):
        """MXFP8 and W4A16 modes: E8M0 block scales of xq, [R, H/32] (W4A16:
        [R, 2H/32])."""
        n = self.terms * self.H // 32
        return self.bytes_("x_sf", self.R * n).reshape(self.R, n)

    @property
    def h_sf(self):
        """MXFP8 and W4A16 modes: E8M0 block scales of hq, [R, I/32] (W4A16:
        [R, 2I/32])."""
        n = self.terms * self.I // 32
        return self.bytes_("h_sf", self.R * n).reshape(self.R, n)

    @property
    def tile_plan(self):
        return self.ints("tile_plan", 2 * self.E).reshape(self.E, 2)

    @property
    def h(self):
        return self._view(self.L.h, self.R * self.I, torch.bfloat16).float().numpy().reshape(
            self.R, self.I)

    @property
    def hq(self):
        w = self.terms * self.I
        return self._view(self.L.hq, self.R * w, torch.uint8).numpy().reshape(self.R, w)

    @property
    def h_scale(self):
        return self.floats("h_scale", self.R)

    @property
    def y(self):
        return self._view(self.L.y, self.R * self.H, torch.bfloat16).float().numpy().reshape(
            self.R, self.H)

    @property
    def num_tiles(self):
        return int(self.ints("status", 2)[1])

    @property
    def tiles(self):
        return self.ints("tiles", 4 * self.num_tiles).reshape(-1, 4)

    def out_np(self):
        return self.out.float().cpu().numpy()


def dump(name: str, **arrays):
    """Save arrays for offline inspection when MOE_DUMP_DIR is set."""
    d = os.environ.get("MOE_DUMP_DIR")
    if d:
        os.makedirs(d, exist_ok=True)
        np.savez_compressed(os.path.join(d, f"{name}.npz"), **arrays)
