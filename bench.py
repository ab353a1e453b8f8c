#!/usr/bin/env python
"""Throughput of the fused MXFP4 x FP8 MoE forward on GB300 (one JSON line).

Workload (default): the DeepSeek-V3-shaped MoE layer -- E=256 experts, top-8
softmax routing, H=7168, I=2048, SwiGLU -- at T=4096 tokens, MXFP4 expert
weights and runtime per-token FP8 activations, synthetic seeded inputs
(moe_inputs.py).  One step = one full forward (routing, scatter + FP8
quantisation, GEMM1 + SwiGLU, h quantisation, GEMM2, combine) through the C
ABI, inputs resident in HBM.  The same metric is also reported end to end
(`e2e`: host activations copied in and the output copied out inside the
timed region), per kernel (CUDA events the library records between its
launches), as a roofline fraction, and over the T sweep 1..4096.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

N > 1 (launched under torch.distributed.run) runs independent replicas, one
per GPU (the forward has no exchange step on one GPU): value = all tokens
processed / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused-MoE tokens/s + TFLOP/s at DSV3 shape, T=1..4096; % of roofline"
UNIT = "tokens/s"
FP8_OVER_BF16 = 2.0          # nominal dense FP8 : BF16 tensor-rate ratio on GB300
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="dsv3")
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--sweep-steps", type=int, default=30)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-modes", action="store_true",
                    help="skip the W4A16 and MXFP8 workloads")
    ap.add_argument("--variant", type=int, default=0,
                    help="GEMM tile variant (moe_options.tile_variant): 0 auto, 1-6 forced")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    return dict(FALLBACK), "fallback"


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as td
            td.init_process_group(backend=backend)
            self.pg = td

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def done(self):
        if self.pg:
            self.pg.destroy_process_group()


class Clocks:
    """nvidia-smi clock / throttle samples over a region (every 100 ms)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.25)

    def stop(self) -> dict:
        time.sleep(0.15)
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                c = [x.strip() for x in line.split(",")]
                if len(c) < 9:
                    continue
                try:
                    sm.append(float(c[1]))
                    smax.append(float(c[2]))
                except ValueError:
                    continue
                for n, v in zip(names, c[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def source_hash(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


GEMM_SOURCES = ["precision_moe_grouped_gb300/csrc/gemm.cu",
                "precision_moe_grouped_gb300/csrc/gemm_pair.cu",
                "precision_moe_grouped_gb300/csrc/gemm_common.cuh",
                "precision_moe_grouped_gb300/csrc/ptx.cuh"]
KERNEL_SOURCES = {
    "gemm1": GEMM_SOURCES,
    "gemm2": GEMM_SOURCES,
    "combine": ["precision_moe_grouped_gb300/csrc/rowops.cu"],
    "hquant": ["precision_moe_grouped_gb300/csrc/rowops.cu"],
    "quant_scatter": ["precision_moe_grouped_gb300/csrc/route.cu"],
}


def ncu_traffic(stage: str, cfg_name: str, T: int):
    """DRAM bytes per launch of `stage` from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p) or stage not in KERNEL_SOURCES:
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(f"{stage}:{cfg_name}:{T}")
    if not rec or rec.get("source_sha") != source_hash(KERNEL_SOURCES[stage]):
        return None
    return rec.get("dram_bytes_per_launch")


def alg_cost(stage: str, cfg, T: int, n_touched: int, mode: int = 0):
    """Algorithmic (bytes, flops) of one launch of `stage` in quantisation
    `mode` (0 W4A8, 1 W4A16, 2 W8A8): weights are packed E2M1 (0.5 B) or
    E4M3 (1 B) per element plus one scale byte per 32; the expanded
    activations and h are E4M3 (+ a row scale, or a scale byte per 32 in
    W8A8), or in W4A16 two E4M3 terms with a scale byte per 32 each (the
    bf16 values split for the FP8 tensor cores)."""
    E, k, H, I = cfg.num_experts, cfg.top_k, cfg.hidden, cfg.inter
    R = T * k
    wb = 1.0 if mode == 2 else 0.5
    w1 = 2 * I * H * (wb + 1 / 32)
    w2 = H * I * (wb + 1 / 32)
    act = {0: 1.0, 1: 2 * (1 + 1 / 32), 2: 1 + 1 / 32}[mode]   # bytes per element
    rs = 4 if mode == 0 else 0                                  # row-scale bytes
    table = {
        "route": (T * E * 4 + R * 8, 0),
        "scan": (2 * 4 * E * -(-T // 32), 0),     # per-chunk counts in, chunk bases out
        "rank": (R * 12, 0),
        "quant_scatter": (T * H * 2 + R * H * act + R * rs, 0),
        "gemm1": (n_touched * w1 + R * H * act + R * rs + R * I * 2, 2.0 * R * H * 2 * I),
        "hquant": (R * I * 2 + R * I * act + R * rs, 0),
        "gemm2": (n_touched * w2 + R * I * act + R * rs + R * H * 2, 2.0 * R * I * H),
        "combine": (R * H * 2 + R * 8 + T * H * 2, 0),
    }
    return table[stage]


# Per quantisation mode: the arithmetic the GEMMs compute in, and the
# weight encoding of the synthetic data.
MODE_DTYPE = {0: "fp8e4m3 x fp4e2m1 (mxf8f6f4), fp32 accumulate",
              1: "bf16 activations as two fp8e4m3 terms x fp4e2m1 (mxf8f6f4, MX block "
                 "scales), fp32 accumulate",
              2: "fp8e4m3 x fp8e4m3 (mxf8f6f4, MX block scales), fp32 accumulate"}
MODE_WEIGHTS = {0: "MXFP4", 1: "MXFP4", 2: "MXFP8"}
MODE_NAME = {0: "MXFP4xFP8", 1: "MXFP4xBF16", 2: "MXFP8xMXFP8"}


# model whose MoE layer shape a configuration copies (H, I, E, k)
SHAPE_NAMES = {(7168, 2048, 256, 8): "DeepSeek-V3-shaped ", (7168, 3072, 384, 6):
               "DeepSeek-V4-Pro-shaped "}


def workload_config(cfg, T: int) -> dict:
    """The `config` keys both arms report for the same workload."""
    mode = cfg.mode
    model = SHAPE_NAMES.get((cfg.hidden, cfg.inter, cfg.num_experts, cfg.top_k), "")
    return {"workload": f"{model}MoE layer E={cfg.num_experts} top-{cfg.top_k} "
                        f"H={cfg.hidden} I={cfg.inter} SwiGLU, T={T}, {MODE_NAME[mode]}"
                        + (f", Zipf({cfg.zipf}) routing" if cfg.zipf else ""),
            "num_tokens": T, "num_experts": cfg.num_experts, "top_k": cfg.top_k,
            "hidden": cfg.hidden, "inter": cfg.inter}


def fused_roofline(cfg, T, n_touched, t_s, pk, mode=0):
    """Roofline of the whole forward: max(touched weight+scale + activation
    bytes / HBM, FLOPs / tensor peak): the FP8 peak for W4A8 and W8A8, the
    bf16 peak for W4A16 (a bf16 product; run as two FP8 MMAs, it takes the
    same tensor time)."""
    E, k, H, I = cfg.num_experts, cfg.top_k, cfg.hidden, cfg.inter
    w_bytes = 1.0 if mode == 2 else 0.5          # E4M3 or packed E2M1 per weight
    bytes_ = n_touched * 3 * I * H * (w_bytes + 1 / 32) + T * H * 2 + T * E * 4 + T * H * 2
    flops = 2.0 * T * k * 3 * I * H
    t_mem = bytes_ / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops"] * (1.0 if mode == 1 else FP8_OVER_BF16) * 1e12)
    return {"bytes": bytes_, "flops": flops, "t_hbm_us": t_mem * 1e6, "t_tensor_us": t_tc * 1e6,
            "bound": "hbm" if t_mem >= t_tc else "tensor",
            "frac": max(t_mem, t_tc) / t_s, "hbm_frac": t_mem / t_s, "tensor_frac": t_tc / t_s}


# ------------------------------------------------------------------ our arm
def run_ours(args, dist: Dist):
    import torch

    import moe_inputs as MI
    import precision_moe_grouped_gb300 as P

    torch.cuda.set_device(dist.local)
    dist.init("nccl")
    dev = torch.device("cuda", dist.local)
    cfg = MI.CONFIGS[args.config]
    T = args.tokens
    K, W = args.steps, args.warmup
    pk, pk_src = peaks()
    mode = cfg.mode
    case = MI.make_case(cfg, T, device=f"cuda:{dist.local}")
    moe = P.FusedMoE(case.w1, case.w1_sf, case.w2, case.w2_sf, cfg.top_k, mode=mode)
    del case.w1, case.w1_sf, case.w2, case.w2_sf
    torch.cuda.synchronize()
    x, logits = case.x, case.logits
    out = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device=dev)
    s = moe.shape(T)
    ws = moe.workspace(T)
    stream = torch.cuda.current_stream()
    nst = P._lib.MOE_NUM_STAGES
    names = P._lib.stage_names()

    # the binding's tensor checks run once here, not inside the timed loops
    P._lib.validate_forward(s, mode, x, logits, moe.w1_p, moe.w1_sf_p, moe.w2_p, moe.w2_sf_p,
                            out, ws, device=torch.cuda.current_device())

    def fwd(opts=None):
        P.forward(s, x, logits, moe.w1_p, moe.w1_sf_p, moe.w2_p, moe.w2_sf_p, out, ws,
                  mode=mode, opts=opts, validate=False)

    base = P.options(tile_variant=args.variant)
    for _ in range(max(W, 3)):
        fwd(base)
    torch.cuda.synchronize()
    if P.read_device_status(ws) != 0:
        raise RuntimeError("device status error after warm-up")
    lay = P.workspace_layout(s, mode)
    counts = ws[lay.counts:lay.counts + 4 * cfg.num_experts].view(torch.int32).cpu().numpy()
    n_touched = int((counts > 0).sum())

    # Timed region: K forwards, nothing else on the stream (events recorded
    # between the library's kernels would break its programmatic-launch
    # overlap, so per-kernel times come from a second pass below).
    clocks = Clocks(dist.local)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        fwd(base)
    t1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop()
    ms_local = t0.elapsed_time(t1) / K
    ms = dist.max(ms_local)
    if P.read_device_status(ws) != 0:
        raise RuntimeError("device status error in timed region")
    gpu_launches = P._lib.kernels_per_forward(T, mode) * K

    # Kernel timing pass: the same K forwards with CUDA events the library
    # records on its stream before its first kernel and after each kernel.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(K)]
    for row in evs:
        for e in row:
            e.record(stream)          # creates the event handles up front
    arrays = [P._lib.stage_event_array(row) for row in evs]
    opts = [P.options(tile_variant=args.variant, stage_events=a) for a in arrays]
    torch.cuda.synchronize()
    for i in range(K):
        fwd(opts[i])
    torch.cuda.synchronize()
    stage_ms = {names[j]: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K))
                for j in range(nst)}

    # end to end: host activations in, output out, inside the timed region,
    # through the multi-step host entry point: step i's inputs are copied in
    # and step i-1's output copied out (DMA, two copy streams) while step i
    # computes, through two device staging sets; three input and output sets
    # rotate, so no step reads the inputs the step before it read.
    xh = [x.cpu().pin_memory() for _ in range(3)]
    lh = [logits.cpu().pin_memory() for _ in range(3)]
    ohs = [torch.empty((T, cfg.hidden), dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    ws_steps = torch.empty(P.steps_workspace_size(s, mode), dtype=torch.uint8, device=dev)
    for i in range(3):
        P._lib.validate_forward(s, mode, xh[i], lh[i], moe.w1_p, moe.w1_sf_p, moe.w2_p,
                                moe.w2_sf_p, ohs[i], ws_steps, host=True,
                                device=torch.cuda.current_device())

    def steps(n):
        P.forward_host_steps(s, [xh[i % 3] for i in range(n)], [lh[i % 3] for i in range(n)],
                             moe.w1_p, moe.w1_sf_p, moe.w2_p, moe.w2_sf_p,
                             [ohs[i % 3] for i in range(n)], ws_steps, mode=mode, opts=base,
                             validate=False)
    steps(2)
    torch.cuda.synchronize()
    dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    steps(K)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = dist.max(e0.elapsed_time(e1) / K)
    for oh in ohs[:min(K, 3)]:   # the output sets the timed steps wrote
        assert torch.equal(oh.to(dev), out), "host-buffer forward disagrees with device forward"
    del ws_steps

    # the single-step host call for comparison: page-locked buffers read and
    # written in place by the kernels over the host link
    oh = ohs[0]
    for i in range(2):
        P.forward_host(s, xh[i % 3], lh[i % 3], moe.w1_p, moe.w1_sf_p, moe.w2_p, moe.w2_sf_p, oh,
                       ws, mode=mode, opts=base, validate=False)
    torch.cuda.synchronize()
    dist.barrier()
    e0.record(stream)
    for i in range(K):
        P.forward_host(s, xh[i % 3], lh[i % 3], moe.w1_p, moe.w1_sf_p, moe.w2_p, moe.w2_sf_p, oh,
                       ws, mode=mode, opts=base, validate=False)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e_single = dist.max(e0.elapsed_time(e1) / K)
    assert torch.equal(oh.to(dev), out), "host-buffer forward disagrees with device forward"
    del xh, lh, ohs

    # dominant kernel and its roofline
    dom = max(stage_ms, key=stage_ms.get)
    dbytes, dflops = alg_cost(dom, cfg, T, n_touched, mode)
    dsec = stage_ms[dom] / 1e3
    t_mem = dbytes / (pk["hbm_gbs"] * 1e9)
    # burst peak: the timed region is K forwards of a few ms each, far from
    # the seconds-long loop the sustained figure was measured over
    tc_peak = pk["bf16_tflops"] * (1.0 if mode == 1 else FP8_OVER_BF16)
    t_tc = dflops / (tc_peak * 1e12)
    if t_tc > t_mem:
        roof = {"bound": "tensor", "achieved": dflops / dsec / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": dbytes / dsec / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = ncu_traffic(dom, cfg.name, T)
    roof.update({"kernel": dom, "alg_bytes_per_launch": dbytes, "alg_flops_per_launch": dflops,
                 "ms_per_launch": stage_ms[dom], "peak_source": pk_src,
                 "tensor_frac": (dflops / dsec / 1e12) / tc_peak if dflops else 0.0,
                 "hbm_frac": dbytes / dsec / 1e9 / pk["hbm_gbs"]})

    fr = fused_roofline(cfg, T, n_touched, ms / 1e3, pk, mode)
    wbytes = (1.0 if mode == 2 else 0.5) + 1 / 32
    result = {
        "metric": METRIC, "value": dist.world * T / (ms / 1e3), "unit": UNIT,
        "n_gpus": dist.world, "steps": K, "warmup": W, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": MODE_DTYPE[mode],
        "data": "synthetic (seeded N(0,1) activations/logits, N(0,0.02) weights as "
                f"{MODE_WEIGHTS[mode]})" + (f", Zipf({cfg.zipf}) routing skew" if cfg.zipf else ""),
        "config": {**workload_config(cfg, T), "parallelism": f"replicas x{dist.world}",
                   "l2": "no flush: the touched expert weights per step "
                         f"({n_touched * 3 * cfg.inter * cfg.hidden * wbytes / 1e9:.2f} GB) "
                         "exceed the 129 MB L2",
                   "tile_variant": args.variant},
        "tflops": fr["flops"] / (ms / 1e3) / 1e12,
        "fused_roofline": fr,
        "roofline": roof,
        "stage_ms": stage_ms,
        "stage_ms_note": "per-kernel CUDA-event times from a second pass of the same K steps "
                         "(events between kernels add launch gaps; the headline value is "
                         "timed without them)",
        "e2e": {"value": dist.world * T / (ms_e2e / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": T * cfg.hidden * 2 + T * cfg.num_experts * 4,
                "d2h_bytes_per_step": T * cfg.hidden * 2, "ms_per_step": ms_e2e,
                "transfer": "page-locked host buffers; one moe_forward_host_steps call for "
                            "the K steps: each step's inputs copied in and its output copied "
                            "out by DMA on two copy streams, overlapped with the neighbouring "
                            "steps' computation (two device staging sets; 3 rotating input and "
                            "output sets)",
                "single_call": {"value": dist.world * T / (ms_e2e_single / 1e3),
                                "ms_per_step": ms_e2e_single,
                                "transfer": "moe_forward_host per step: page-locked buffers "
                                            "read and written in place by the kernels over "
                                            "the host link"}},
        "gpu_launches": gpu_launches,
        "clocks": clk,
        "experts_touched": n_touched,
    }

    if not args.no_sweep:
        result["sweep"] = sweep(args, cfg, moe, x, logits, dist, pk)
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(cfg, T, x, logits)
    del moe, ws, out, case
    torch.cuda.empty_cache()
    if not args.no_sweep and args.config == "dsv3":
        result["v4pro_sweep"] = v4pro_sweep(args, dist, pk)
    if not args.no_other_modes:
        result["other_modes"] = other_modes(args, dist, pk)
    dist.done()
    return result


def other_modes(args, dist, pk):
    """The other quantisation modes on their own workloads (device-resident
    inputs, CUDA events, 16 rotating token sets where the tokens allow):
    W4A16 (MXFP4 x bf16) at E=64/top-4/H=2048/I=1024/T=256, and MXFP8 x MXFP8
    with Zipf(1.2) routing skew at E=256/top-8/H=7168/I=2048/T=4096."""
    import torch

    import moe_inputs as MI
    import precision_moe_grouped_gb300 as P
    res = []
    stream = torch.cuda.current_stream()
    for name, T in (("w4a16", 256), ("mxfp8_zipf", 4096)):
        cfg = MI.CONFIGS[name]
        nsets = 16 if T <= 512 else 1
        case = MI.make_case(cfg, T * nsets, device=f"cuda:{dist.local}")
        moe = P.FusedMoE(case.w1, case.w1_sf, case.w2, case.w2_sf, cfg.top_k, mode=cfg.mode)
        del case.w1, case.w1_sf, case.w2, case.w2_sf
        sets = [(case.x[i * T:(i + 1) * T].contiguous(),
                 case.logits[i * T:(i + 1) * T].contiguous()) for i in range(nsets)]
        s = moe.shape(T)
        ws = moe.workspace(T)
        out = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device=case.x.device)

        for xs, ls in sets:
            P._lib.validate_forward(s, cfg.mode, xs, ls, moe.w1_p, moe.w1_sf_p, moe.w2_p,
                                    moe.w2_sf_p, out, ws, device=torch.cuda.current_device())

        def fwd(i):
            xs, ls = sets[i % nsets]
            P.forward(s, xs, ls, moe.w1_p, moe.w1_sf_p, moe.w2_p, moe.w2_sf_p, out, ws,
                      mode=cfg.mode, validate=False)
        lay = P.workspace_layout(s, cfg.mode)
        touched, empty = [], []
        for i in range(max(3, nsets)):
            fwd(i)
            torch.cuda.synchronize()
            c = ws[lay.counts:lay.counts + 4 * cfg.num_experts].view(torch.int32)
            touched.append(int((c > 0).sum().item()))
            empty.append(int((c == 0).sum().item()))
        status = P.read_device_status(ws)
        dist.barrier()
        steps = 20
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            fwd(i)
        b.record(stream)
        torch.cuda.synchronize()
        ms = dist.max(a.elapsed_time(b) / steps)
        n_t = sum(touched) / len(touched)
        fr = fused_roofline(cfg, T, n_t, ms / 1e3, pk, cfg.mode)
        res.append({"workload": f"{name}: E={cfg.num_experts} top-{cfg.top_k} H={cfg.hidden} "
                                f"I={cfg.inter} T={T}" + (f" zipf={cfg.zipf}" if cfg.zipf else ""),
                    "mode": {0: "W4A8", 1: "W4A16", 2: "W8A8 (MXFP8)"}[cfg.mode],
                    "ms": ms, "tokens_s": dist.world * T / (ms / 1e3),
                    "tflops": fr["flops"] / (ms / 1e3) / 1e12, "experts_touched": n_t,
                    "experts_empty": sum(empty) / len(empty), "roofline_frac": fr["frac"],
                    "bound": fr["bound"], "hbm_frac": fr["hbm_frac"],
                    "tensor_frac": fr["tensor_frac"],
                    "tensor_peak": "bf16" if cfg.mode == 1 else "fp8 (2 x measured bf16)",
                    "token_sets": nsets, "device_status": status})
        del moe, ws, out, case, sets
        torch.cuda.empty_cache()
    return res


def sweep(args, cfg, moe, x_all, lg_all, dist, pk):
    """Each T of the configuration's sweep, with 16 rotating token sets (so
    successive steps route to different experts and do not reuse L2)."""
    import torch

    import precision_moe_grouped_gb300 as P
    res = []
    stream = torch.cuda.current_stream()
    T_all = x_all.shape[0]
    for T in cfg.tokens:
        nsets = max(1, min(16, T_all // T))
        sets = [(x_all[i * T:(i + 1) * T].contiguous(), lg_all[i * T:(i + 1) * T].contiguous())
                for i in range(nsets)]
        s = moe.shape(T)
        ws = moe.workspace(T) if T == T_all else torch.empty(
            P.workspace_size(s), dtype=torch.uint8, device=x_all.device)
        out = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device=x_all.device)
        o = P.options(tile_variant=args.variant)

        for xs, ls in sets:
            P._lib.validate_forward(s, cfg.mode, xs, ls, moe.w1_p, moe.w1_sf_p, moe.w2_p,
                                    moe.w2_sf_p, out, ws, device=torch.cuda.current_device())

        def fwd(i):
            xs, ls = sets[i % nsets]
            P.forward(s, xs, ls, moe.w1_p, moe.w1_sf_p, moe.w2_p, moe.w2_sf_p, out, ws,
                      mode=cfg.mode, opts=o, validate=False)
        for i in range(5):
            fwd(i)
        torch.cuda.synchronize()
        lay = P.workspace_layout(s, cfg.mode)
        touched = []
        for i in range(nsets):
            fwd(i)
            torch.cuda.synchronize()
            c = ws[lay.counts:lay.counts + 4 * cfg.num_experts].view(torch.int32)
            touched.append(int((c > 0).sum().item()))
        dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(args.sweep_steps):
            fwd(i)
        b.record(stream)
        torch.cuda.synchronize()
        ms = dist.max(a.elapsed_time(b) / args.sweep_steps)
        n_t = sum(touched) / len(touched)
        fr = fused_roofline(cfg, T, n_t, ms / 1e3, pk, cfg.mode)
        # per-kernel times: a separate pass with the library's stage events
        nst = P._lib.MOE_NUM_STAGES
        names = P._lib.stage_names()
        n_ev = min(args.sweep_steps, 10)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)]
               for _ in range(n_ev)]
        for row in evs:
            for e in row:
                e.record(stream)
        arrays = [P._lib.stage_event_array(row) for row in evs]
        torch.cuda.synchronize()
        for i in range(n_ev):
            xs, ls = sets[i % nsets]
            P.forward(s, xs, ls, moe.w1_p, moe.w1_sf_p, moe.w2_p, moe.w2_sf_p, out, ws,
                      mode=cfg.mode, validate=False,
                      opts=P.options(tile_variant=args.variant, stage_events=arrays[i]))
        torch.cuda.synchronize()
        stage_us = {names[j]: round(1e3 * statistics.mean(
            evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n_ev)), 2) for j in range(nst)}
        res.append({"T": T, "ms": ms, "tokens_s": dist.world * T / (ms / 1e3),
                    "tflops": fr["flops"] / (ms / 1e3) / 1e12, "experts_touched": n_t,
                    "roofline_frac": fr["frac"], "bound": fr["bound"],
                    "hbm_frac": fr["hbm_frac"], "tensor_frac": fr["tensor_frac"],
                    "t_roofline_us": max(fr["t_hbm_us"], fr["t_tensor_us"]),
                    "token_sets": nsets, "stage_us": stage_us})
        if ws is not moe.workspace(T_all):
            del ws
    return res


def v4pro_sweep(args, dist, pk):
    """The DeepSeek-V4-Pro-shaped layer (E=384, top-6, H=7168, I=3072) over
    its T sweep 1..8192, on device-resident inputs: seeded activations for
    8192 tokens, cut into up to 16 rotating token sets for the small T."""
    import torch

    import moe_inputs as MI
    import precision_moe_grouped_gb300 as P
    cfg = MI.CONFIGS["v4pro"]
    T_all = max(cfg.tokens)
    case = MI.make_case(cfg, T_all, device=f"cuda:{dist.local}")
    moe = P.FusedMoE(case.w1, case.w1_sf, case.w2, case.w2_sf, cfg.top_k, mode=cfg.mode)
    del case.w1, case.w1_sf, case.w2, case.w2_sf
    torch.cuda.synchronize()
    res = sweep(args, cfg, moe, case.x, case.logits, dist, pk)
    del moe, case
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ oracle timing
# The oracle's full forward at these sizes runs for minutes (each touched
# expert's weights are decoded to float64 once, ~0.5 s per DSV3 expert), so
# its T-token time is extrapolated from timed parts, each run through the
# oracle's own routines in the order forward() runs them:
#   t(T) = T * t_token + n_touched * t_expert
# t_token: the steps whose cost grows with the tokens (routing, expansion,
#   activation quantisation, gather and decode of the expanded rows, combine),
#   timed on the first n_tok tokens and divided by n_tok;
# t_expert: one touched expert's steps at its full-T row count (decode of its
#   w1 and w2, GEMM1, token scale, SwiGLU, h quantisation, GEMM2, row scale),
#   the mean over a seeded sample of the touched experts.
# tests/test_bench_accounting.py checks that these parts, run for every
# expert, reproduce forward()'s outputs.

def oracle_token_part(xb, lg, top_k, num_experts, mode):
    """forward()'s token-linear steps on the given tokens (x as raw bf16
    bits, logits float32): returns (routing, decoded expanded rows a1, the
    per-row activation scales of W4A8 or None, out)."""
    import numpy as np

    from oracle import formats as F
    from oracle import moe as M
    x_all = F.bf16_bits_to_f32(xb)
    ids, w = M.route(lg, top_k)
    rt = M.expand(ids, w, num_experts)
    xs = None
    if mode == M.QUANT_W4A8:
        tq, ts = M.quantize_rows_fp8(x_all)
        xs = ts[rt.token_of_row]
        a1 = F.e4m3_decode(tq[rt.token_of_row])
    elif mode == M.QUANT_W8A8:
        tq, ts = M.quantize_rows_mxfp8(x_all)
        a1 = F.mxfp8_dequant(tq[rt.token_of_row], ts[rt.token_of_row])
    else:
        a1 = x_all[rt.token_of_row].astype(np.float64)
    y = np.zeros((int(rt.offsets[-1]), x_all.shape[1]), np.float32)
    out = M.combine(w, y, rt.row_of)
    return rt, a1, xs, out


def oracle_expert_part(W, e, a1_rows, xs_rows, mode):
    """forward()'s steps for expert e on its expanded rows: GEMM1 (+ token
    scale), SwiGLU, h quantisation, GEMM2 (+ row scale).  Returns y rows."""
    import numpy as np

    from oracle import formats as F
    from oracle import moe as M
    acc = M._exact_dot_f32(a1_rows, W.dense(1, e))
    if mode == M.QUANT_W4A8:
        acc = M.apply_row_scale(acc, xs_rows)
    h = M.swiglu_bf16(acc)
    hs = None
    if mode == M.QUANT_W4A8:
        hq, hs = M.quantize_rows_fp8(h)
        a2 = F.e4m3_decode(hq)
    elif mode == M.QUANT_W8A8:
        hq, hsb = M.quantize_rows_mxfp8(h)
        a2 = F.mxfp8_dequant(hq, hsb)
    else:
        a2 = h.astype(np.float64)
    y = M._exact_dot_f32(a2, W.dense(2, e))
    if mode == M.QUANT_W4A8:
        y = M.apply_row_scale(y, hs)
    return y


class OracleCost:
    """Host inputs and timed parts of the oracle for a T-token workload.

    prepare(): full-T routing (untimed; it gives the touched experts and
    their row counts), the token-linear part timed on the first n_tok
    tokens, and the inputs of n_exp seeded touched experts (weights
    regenerated from the per-expert seeds: the same bytes as the GPU run)."""

    def __init__(self, cfg, T, x, logits, n_tok, n_exp):
        import numpy as np
        import torch

        import moe_inputs as MI
        from oracle import formats as F
        from oracle import moe as M
        self.cfg, self.T, self.mode = cfg, T, cfg.mode
        xb = x.cpu().view(torch.int16).numpy().view(np.uint16)
        lg = logits.cpu().numpy().astype(np.float32)
        k, E = cfg.top_k, cfg.num_experts
        ids, w = M.route(lg, k)
        rt = M.expand(ids, w, E)
        self.n_touched = int((rt.counts > 0).sum())
        self.n_tok = min(T, n_tok)
        t = time.perf_counter()
        oracle_token_part(xb[:self.n_tok], lg[:self.n_tok], k, E, self.mode)
        self.t_token = (time.perf_counter() - t) / self.n_tok
        touched = np.flatnonzero(rt.counts > 0)
        rng = np.random.default_rng(MI.seed_for(cfg, T))
        self.experts = [int(e) for e in rng.choice(touched, size=min(n_exp, touched.size),
                                                   replace=False)]
        dev = "cuda" if x.is_cuda else "cpu"
        x_all = F.bf16_bits_to_f32(xb)
        kd = 1 if self.mode == M.QUANT_W8A8 else 2
        H, I = cfg.hidden, cfg.inter
        self.jobs = []
        for e in self.experts:
            wts = [t_.cpu().numpy()[None] for t_ in
                   MI.expert_weights(cfg, MI.seed_for(cfg, T), e, dev)]
            W = M.Weights(wts[0], wts[1], wts[2], wts[3], mode=self.mode)
            toks = rt.token_of_row[rt.offsets[e]:rt.offsets[e + 1]]
            xs = None
            if self.mode == M.QUANT_W4A8:
                tq, xs = M.quantize_rows_fp8(x_all[toks])
                a1 = F.e4m3_decode(tq)
            elif self.mode == M.QUANT_W8A8:
                tq, ts = M.quantize_rows_mxfp8(x_all[toks])
                a1 = F.mxfp8_dequant(tq, ts)
            else:
                a1 = x_all[toks].astype(np.float64)
            assert W.w1.shape[1:] == (2 * I, H // kd)
            self.jobs.append((W, a1, xs, len(toks)))
        self.t_expert = []

    def run_expert(self, i):
        """Times one sampled expert's part (job i mod n_exp); returns seconds."""
        W, a1, xs, _ = self.jobs[i % len(self.jobs)]
        t = time.perf_counter()
        oracle_expert_part(W, 0, a1, xs, self.mode)
        dt = time.perf_counter() - t
        self.t_expert.append(dt)
        return dt

    def seconds(self):
        """Extrapolated time of the oracle's T-token forward."""
        te = statistics.mean(self.t_expert)
        return self.T * self.t_token + self.n_touched * te

    def describe(self):
        te = statistics.mean(self.t_expert)
        rows = [j[3] for j in self.jobs]
        return (f"extrapolated: t(T) = T x t_token + n_touched x t_expert = {self.T} x "
                f"{self.t_token * 1e3:.3f} ms + {self.n_touched} x {te * 1e3:.1f} ms; t_token "
                f"timed on the first {self.n_tok} tokens (routing, expansion, quantisation, "
                f"row gather and decode, combine), t_expert the mean of {len(self.t_expert)} "
                f"timed passes over {len(self.jobs)} sampled touched experts (rows {rows}: "
                f"w1/w2 decode, GEMM1, SwiGLU, h quantisation, GEMM2); numpy, BLAS matmuls "
                f"may use all listed cores")


def cpu_baseline(cfg, T, x, logits, n_tok=256, n_exp=4):
    """The oracle, as it stands, timed on the host cores (extrapolated to T)."""
    t0 = time.perf_counter()
    oc = OracleCost(cfg, T, x, logits, n_tok, n_exp)
    for i in range(len(oc.jobs)):
        oc.run_expert(i)
    sec = oc.seconds()
    return {"value": T / sec, "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "extrapolated": True, "sample": oc.describe(),
            "t_forward_s": sec, "wall_s": time.perf_counter() - t0}


def run_reference(args, dist: Dist):
    """The oracle (CPU) on the same workload: the warm-up prepares the
    inputs and times the token-linear part; each timed step runs one sampled
    touched expert's part; the value is T over the extrapolated T-token
    time (OracleCost)."""
    if dist.rank != 0:
        return None
    import moe_inputs as MI
    cfg = MI.CONFIGS[args.config]
    T = args.tokens
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x, logits = MI.make_activations(cfg, T, dev)
    oc = OracleCost(cfg, T, x, logits, n_tok=256, n_exp=4)
    for i in range(args.warmup):
        oc.run_expert(i)
    oc.t_expert.clear()
    t = time.perf_counter()
    for i in range(max(1, args.steps)):
        oc.run_expert(i)
    dt = time.perf_counter() - t
    v = T / oc.seconds()
    return {"metric": METRIC, "value": v, "unit": UNIT, "impl": "reference", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / max(1, args.steps) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32",
            "data": "synthetic", "config": {**workload_config(cfg, T), "parallelism": "replicas x1"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
                             "kind": "oracle", "extrapolated": True, "sample": oc.describe()},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    dist = Dist()
    if args.impl == "reference":
        res = run_reference(args, dist)
    else:
        res = run_ours(args, dist)
    if res is not None and dist.rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
