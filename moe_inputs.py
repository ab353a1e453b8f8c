"""Seeded synthetic inputs for the fused MoE forward (tests and bench).

This module only draws random numbers and lays them out in the C ABI's user
layout; it computes none of the forward.  Both the CPU oracle and the CUDA
path consume what it returns, so neither depends on the other.

Recipe (the pages benchmark DeepSeek-V3 / V4-Pro shaped MoE layers but ship
no data; these synthetic tensors stand in for real activations and weights):
  x       ~ N(0, 1), rounded to bf16                      [T, H]
  logits  ~ N(0, 1) float32                               [T, E]
            (Zipf mode adds b_e = -s * ln(rank_e) with ranks a seeded
             permutation of 1..E, so expert popularity falls off as Zipf(s))
  weights ~ N(0, 0.02) float32, stored as MXFP4: per 32-element block along
            K, scale X = 2^(floor(log2 amax) - 2) (byte = exponent + 127; an
            all-zero block gets byte 127) and E2M1 codes = round-to-nearest-
            even(v / X) saturated to +-6, two codes per byte, low nibble =
            even K index.  (MXFP8 weights for the W8A8 mode: X = 2^(floor(log2
            amax) - 8), E4M3 codes.)  This weight encoding is model
            preprocessing, not a step of the forward: both sides decode the
            same bytes.
Seeds: seed(config, T) = 1234 + 17 * config_index + T.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

QUANT_W4A8, QUANT_W4A16, QUANT_W8A8 = 0, 1, 2


@dataclass(frozen=True)
class MoeConfig:
    name: str
    index: int
    num_experts: int
    top_k: int
    hidden: int
    inter: int
    tokens: tuple
    mode: int = QUANT_W4A8
    zipf: float = 0.0


CONFIGS = {
    "tiny": MoeConfig("tiny", 0, 8, 2, 256, 128, (16,)),
    "w4a16": MoeConfig("w4a16", 1, 64, 4, 2048, 1024, (256,), mode=QUANT_W4A16),
    "dsv3": MoeConfig("dsv3", 2, 256, 8, 7168, 2048, (1, 8, 64, 512, 4096)),
    "v4pro": MoeConfig("v4pro", 3, 384, 6, 7168, 3072, (1, 16, 128, 1024, 8192)),
    "mxfp8_zipf": MoeConfig("mxfp8_zipf", 4, 256, 8, 7168, 2048, (4096,),
                            mode=QUANT_W8A8, zipf=1.2),
    # DeepSeek-V3 layer shape with 32 experts: at T=512 each expert gets the
    # same ~128 rows as the full layer at T=4096, in 0.75 GB of weights (used
    # for profiler captures that must stay small)
    "dsv3_e32": MoeConfig("dsv3_e32", 5, 32, 8, 7168, 2048, (512,)),
    # the MXFP8 Zipf workload's shape with 32 experts, for the same purpose
    "mxfp8_e32": MoeConfig("mxfp8_e32", 6, 32, 8, 7168, 2048, (512,), mode=QUANT_W8A8,
                           zipf=1.2),
}


def seed_for(cfg: MoeConfig, tokens: int) -> int:
    return 1234 + 17 * cfg.index + tokens


def _e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """E2M1 codes (uint8, 0..15) of values already divided by the block scale;
    round to nearest, ties to the even code, saturate at 6."""
    a = v.abs()
    # grid 0, .5, 1, 1.5, 2, 3, 4, 6; midpoint b between codes i and i+1 goes
    # to the even code: strict '>' when i is even, '>=' when i is odd
    mag = ((a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8)
           + (a > 1.25).to(torch.uint8) + (a >= 1.75).to(torch.uint8)
           + (a > 2.5).to(torch.uint8) + (a >= 3.5).to(torch.uint8)
           + (a > 5.0).to(torch.uint8))
    sign = (v < 0).to(torch.uint8) << 3
    return mag | sign


def _block_exponent(amax: torch.Tensor, emax: int) -> torch.Tensor:
    """floor(log2 amax) - emax as int32 (amax > 0), 0 where amax == 0."""
    safe = torch.where(amax > 0, amax, torch.ones_like(amax))
    _, e2 = torch.frexp(safe)
    e = (e2 - 1 - emax).clamp(-127, 127)
    return torch.where(amax > 0, e, torch.zeros_like(e)).to(torch.int32)


def quantize_mxfp4(w: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """float32 [..., N, K] -> (packed uint8 [..., N, K/2], scales uint8 [..., N, K/32])."""
    shp = w.shape
    blk = w.reshape(*shp[:-1], shp[-1] // 32, 32)
    e = _block_exponent(blk.abs().amax(-1), 2)
    v = blk / torch.ldexp(torch.ones_like(e, dtype=torch.float32), e)[..., None]
    codes = _e2m1_codes(v).reshape(shp)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    return packed.contiguous(), (e + 127).to(torch.uint8).contiguous()


def quantize_mxfp8_weights(w: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """float32 [..., N, K] -> (E4M3 bytes [..., N, K], scales uint8 [..., N, K/32])."""
    shp = w.shape
    blk = w.reshape(*shp[:-1], shp[-1] // 32, 32)
    e = _block_exponent(blk.abs().amax(-1), 8)
    v = blk / torch.ldexp(torch.ones_like(e, dtype=torch.float32), e)[..., None]
    codes = v.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.reshape(shp).contiguous(), (e + 127).to(torch.uint8).contiguous()


@dataclass
class MoeCase:
    cfg: MoeConfig
    T: int
    x: torch.Tensor        # bf16 [T, H]
    logits: torch.Tensor   # float32 [T, E]
    w1: torch.Tensor       # uint8, user layout
    w1_sf: torch.Tensor
    w2: torch.Tensor
    w2_sf: torch.Tensor

    @property
    def mode(self) -> int:
        return self.cfg.mode


def expert_weights(cfg: MoeConfig, seed: int, e: int, device: str = "cpu"):
    """(w1, w1_sf, w2, w2_sf) of expert e, drawn from the expert's own seed."""
    quant = quantize_mxfp8_weights if cfg.mode == QUANT_W8A8 else quantize_mxfp4
    E, H, I = cfg.num_experts, cfg.hidden, cfg.inter
    ge = torch.Generator(device=device).manual_seed(seed * 1000003 + 7919 * e + 1)
    a = torch.randn((2 * I, H), generator=ge, device=device, dtype=torch.float32) * 0.02
    w1, w1_sf = quant(a)
    b = torch.randn((H, I), generator=ge, device=device, dtype=torch.float32) * 0.02
    w2, w2_sf = quant(b)
    return w1, w1_sf, w2, w2_sf


def make_activations(cfg: MoeConfig, T: int, device: str = "cpu", seed: int | None = None):
    """(x bf16 [T, H], logits float32 [T, E]) of the seeded case."""
    seed = seed_for(cfg, T) if seed is None else seed
    g = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn((T, cfg.hidden), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    logits = torch.randn((T, cfg.num_experts), generator=g, device=device, dtype=torch.float32)
    if cfg.zipf > 0:
        ranks = torch.randperm(cfg.num_experts, generator=g, device=device).to(torch.float32) + 1.0
        logits = logits - cfg.zipf * torch.log(ranks)[None, :]
    return x, logits


def make_case(cfg: MoeConfig, T: int, device: str = "cpu", seed: int | None = None,
              experts: list | None = None) -> MoeCase:
    """Draw one seeded case.  Weights are drawn expert by expert from a
    per-expert seed, so any subset ``experts`` can be regenerated alone (the
    other experts' weights are then left zero)."""
    seed = seed_for(cfg, T) if seed is None else seed
    E, H, I = cfg.num_experts, cfg.hidden, cfg.inter
    x, logits = make_activations(cfg, T, device, seed)
    kdiv = 1 if cfg.mode == QUANT_W8A8 else 2
    w1 = torch.zeros((E, 2 * I, H // kdiv), dtype=torch.uint8, device=device)
    w2 = torch.zeros((E, H, I // kdiv), dtype=torch.uint8, device=device)
    w1_sf = torch.full((E, 2 * I, H // 32), 127, dtype=torch.uint8, device=device)
    w2_sf = torch.full((E, H, I // 32), 127, dtype=torch.uint8, device=device)
    for e in (range(E) if experts is None else experts):
        w1[e], w1_sf[e], w2[e], w2_sf[e] = expert_weights(cfg, seed, e, device)
    return MoeCase(cfg=cfg, T=T, x=x, logits=logits, w1=w1, w1_sf=w1_sf, w2=w2, w2_sf=w2_sf)


def custom_config(num_experts: int, top_k: int, hidden: int, inter: int,
                  mode: int = QUANT_W4A8, zipf: float = 0.0, name: str = "custom") -> MoeConfig:
    return MoeConfig(name, 9, num_experts, top_k, hidden, inter, (), mode=mode, zipf=zipf)
