"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bit-exact: routing ids, per-expert counts/offsets, the expanded-row maps,
the FP8 activation codes and the per-token scales.  Floating point (routing
weights, h, y, output): max|err| <= 2e-2 * max|ref| and
sum|err| / sum|ref| <= 5e-3 (outputs in bf16)."""
import numpy as np
import pytest
import torch

import moe_inputs as MI
import precision_moe_grouped_gb300 as P
from oracle import moe as M

from gpu_helpers import DeviceRun, dump, max_err_ok, oracle_weights, x_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    P.load()


def check_front(run: DeviceRun, rt: M.Routing, tq: np.ndarray, ts: np.ndarray, rows=None):
    """Bit-exact checks of routing, expansion and FP8 activation quantisation
    (rows: optional subset of expanded rows to compare codes on)."""
    np.testing.assert_array_equal(run.ids, rt.ids)
    np.testing.assert_array_equal(run.counts, rt.counts)
    np.testing.assert_array_equal(run.offsets, rt.offsets)
    np.testing.assert_array_equal(run.row_of, rt.row_of)
    ts_gpu = run.token_slot
    np.testing.assert_array_equal(ts_gpu // run.k, rt.token_of_row)
    np.testing.assert_array_equal(ts_gpu % run.k, rt.slot_of_row)
    np.testing.assert_allclose(run.weights, rt.weights, rtol=3e-6, atol=1e-7)
    np.testing.assert_array_equal(run.x_scale, ts[rt.token_of_row])
    xq = run.xq
    sel = np.arange(run.R) if rows is None else np.asarray(rows)
    np.testing.assert_array_equal(xq[sel], tq[rt.token_of_row[sel]])


def check_tiles(run: DeviceRun, bn: int):
    """The work map covers every expanded row exactly once, in expert order,
    with tiles of at most bn rows."""
    tiles = run.tiles
    covered = np.zeros(run.R, np.int32)
    off = run.offsets
    for e, r0, n, _ in tiles:
        assert 0 < n <= bn
        assert off[e] <= r0 and r0 + n <= off[e + 1]
        covered[r0:r0 + n] += 1
    assert np.all(covered == 1)


def full_parity(case, variant=0, name="case"):
    run = DeviceRun(case, variant=variant)
    assert run.status == 0
    fw = M.forward(x_bits(case), case.logits.cpu().numpy(), oracle_weights(case),
                   case.cfg.top_k)
    tq, ts = M.quantize_rows_fp8(
        np.asarray(case.x.float().cpu().numpy(), np.float32))
    try:
        check_front(run, fw.routing, tq, ts)
        # GEMM2's FP8 operand: the oracle's quantiser applied to the GPU's
        # own h gives the same codes and scales bit for bit (h itself is a
        # tolerance item, so the codes are compared against its quantisation)
        hq_ref, hs_ref = M.quantize_rows_fp8(run.h.astype(np.float32))
        np.testing.assert_array_equal(run.hq, hq_ref)
        np.testing.assert_array_equal(run.h_scale, hs_ref)
        ok_h, st_h = max_err_ok(run.h, fw.h)
        ok_y, st_y = max_err_ok(run.y, fw.y)
        ok_o, st_o = max_err_ok(run.out_np(), fw.out)
        assert ok_h, ("h", st_h)
        assert ok_y, ("y", st_y)
        assert ok_o, ("out", st_o)
    except AssertionError:
        dump(name, h=run.h, h_ref=fw.h, y=run.y, y_ref=fw.y, out=run.out_np(), out_ref=fw.out,
             xq=run.xq, xq_ref=fw.xq, ids=run.ids, ids_ref=fw.routing.ids, tiles=run.tiles,
             hq=run.hq, hq_ref=fw.hq, hs=run.h_scale, hs_ref=fw.h_scale, g_ref=fw.g)
        raise
    return run, fw


def test_tiny_config_full():
    cfg = MI.CONFIGS["tiny"]
    run, _ = full_parity(MI.make_case(cfg, 16), name="tiny")
    check_tiles(run, 32)


@pytest.mark.parametrize("variant", [1, 2, 3, 4, 5])
def test_several_tiles_ragged(variant):
    """Many token tiles per expert (decode variant), ragged tails, several
    weight M-tiles and K stages."""
    cfg = MI.custom_config(8, 2, 512, 256)
    run, _ = full_parity(MI.make_case(cfg, 200, seed=7), variant=variant, name=f"ragged{variant}")
    check_tiles(run, {1: 32, 2: 224, 3: 16, 4: 224, 5: 160}[variant])


@pytest.mark.parametrize("variant", [2, 4, 5])
def test_expert_split_over_tiles_prefill(variant):
    """Experts with > 224 rows split into balanced tiles (prefill variants)."""
    cfg = MI.custom_config(4, 2, 256, 128)
    run, _ = full_parity(MI.make_case(cfg, 700, seed=9), variant=variant, name=f"split{variant}")
    assert run.counts.max() > 224
    check_tiles(run, 160 if variant == 5 else 224)


def test_variants_agree_bitwise():
    cfg = MI.custom_config(8, 2, 256, 128)
    case = MI.make_case(cfg, 96, seed=13)
    a = DeviceRun(case, variant=1)
    for v in (2, 3, 4, 5):
        b = DeviceRun(case, variant=v, moe=a.moe)
        np.testing.assert_array_equal(a.out_np(), b.out_np())


def test_deterministic():
    cfg = MI.custom_config(16, 4, 256, 256)
    case = MI.make_case(cfg, 64, seed=21)
    a = DeviceRun(case)
    b = DeviceRun(case, moe=a.moe)
    np.testing.assert_array_equal(a.out_np(), b.out_np())


@pytest.mark.parametrize("E,k,T", [(1, 1, 5), (4, 4, 33), (32, 1, 7), (16, 16, 3)])
def test_degenerate_routing(E, k, T):
    """One expert; every expert selected (k = E); k = 1; more experts than rows."""
    cfg = MI.custom_config(E, k, 128, 128)
    full_parity(MI.make_case(cfg, T, seed=31 + T), name=f"degen{E}_{k}_{T}")


@pytest.mark.parametrize("T", [32, 33])
def test_tiny_batch_boundary(T):
    """T = 32 routes, expands and quantises in one kernel; T = 33 takes the
    two-kernel small-batch path.  Both must match the oracle bit for bit on
    the front end."""
    cfg = MI.custom_config(64, 8, 256, 128)
    run, _ = full_parity(MI.make_case(cfg, T, seed=61 + T), name=f"tiny_boundary{T}")
    check_tiles(run, 16 if run.R / 64 <= 8 else 32)


def test_many_experts_and_top32():
    """The routing limits: E = 1024 experts (32 logits per lane) and top-32."""
    cfg = MI.custom_config(1024, 32, 128, 128)
    full_parity(MI.make_case(cfg, 20, seed=71), name="e1024_k32")


def test_zero_rows_and_ties():
    cfg = MI.custom_config(8, 2, 256, 128)
    case = MI.make_case(cfg, 24, seed=41)
    case.x[3] = 0                      # amax = 0: s = 1, zero codes
    case.x[5, 7] = -0.0
    case.logits[4] = 0.0               # all-equal logits: lowest indices win
    case.logits[6, 2] = case.logits[6, 5] = case.logits[6].max() + 1.0
    run, fw = full_parity(case, name="zeros_ties")
    assert run.x_scale[run.row_of[3, 0]] == 1.0
    np.testing.assert_array_equal(run.ids[4], [0, 1])
    np.testing.assert_array_equal(run.ids[6], [2, 5])


def test_empty_experts():
    cfg = MI.custom_config(16, 2, 256, 128)
    case = MI.make_case(cfg, 40, seed=43)
    case.logits[:, 3:9] -= 50.0        # experts 3..8 never chosen
    run, _ = full_parity(case, name="empty")
    assert np.all(run.counts[3:9] == 0)


def test_zero_tokens_is_noop():
    cfg = MI.custom_config(8, 2, 256, 128)
    case = MI.make_case(cfg, 4)
    dev = torch.device("cuda:0")
    moe = P.FusedMoE(case.w1.to(dev), case.w1_sf.to(dev), case.w2.to(dev), case.w2_sf.to(dev), 2)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=dev)
    lg = torch.empty((0, 8), dtype=torch.float32, device=dev)
    out = moe(x, lg)
    torch.cuda.synchronize()
    assert out.shape == (0, 256)


def test_prepare_weights_layout():
    """moe_prepare_weights moves rows and scale bytes exactly as documented."""
    cfg = MI.custom_config(3, 2, 256, 256)
    case = MI.make_case(cfg, 1, seed=3)
    dev = torch.device("cuda:0")
    moe = P.FusedMoE(case.w1.to(dev), case.w1_sf.to(dev), case.w2.to(dev), case.w2_sf.to(dev), 2)
    torch.cuda.synchronize()
    E, I, H = 3, 256, 256
    w1, sf1 = case.w1.numpy(), case.w1_sf.numpy()
    src = np.empty(2 * I, np.int64)
    for p in range(2 * I):
        mt, r = divmod(p, 128)
        q, i = divmod(r, 32)
        f = 64 * mt + 16 * q + (i & 15)
        src[p] = f if i < 16 else I + f

    def blocked(w, rows_src, M, K):
        """[E, M, K/2] -> boxes [E, M/128, K/128, 128 rows, 64 bytes]."""
        wp = w[:, rows_src].reshape(E, M // 128, 128, K // 128, 64)
        return wp.transpose(0, 1, 3, 2, 4).reshape(E, -1)
    np.testing.assert_array_equal(moe.w1_p.cpu().numpy().reshape(E, -1),
                                  blocked(w1, src, 2 * I, H))
    np.testing.assert_array_equal(moe.w2_p.cpu().numpy().reshape(E, -1),
                                  blocked(case.w2.numpy(), np.arange(H), H, I))

    def relayout(sf, rows_src, M, K):
        out = np.empty((E, M // 128, K // 128, 32, 4, 4), np.uint8)
        for mt in range(M // 128):
            for ks in range(K // 128):
                for l in range(32):
                    for i in range(4):
                        out[:, mt, ks, l, i, :] = sf[:, rows_src[mt * 128 + 32 * i + l],
                                                     4 * ks:4 * ks + 4]
        return out.reshape(E, -1)
    np.testing.assert_array_equal(moe.w1_sf_p.cpu().numpy().reshape(E, -1),
                                  relayout(sf1, src, 2 * I, H))
    np.testing.assert_array_equal(moe.w2_sf_p.cpu().numpy().reshape(E, -1),
                                  relayout(case.w2_sf.numpy(), np.arange(H), H, I))


@pytest.mark.parametrize("mode", [MI.QUANT_W4A8, MI.QUANT_W4A16, MI.QUANT_W8A8])
@pytest.mark.parametrize("T", [1, 50, 300])
@pytest.mark.parametrize("pinned", ["all", "none", "x_only"])
def test_forward_host_matches_device_path(mode, T, pinned):
    """moe_forward_host reads page-locked host buffers in place (over the host
    link) and stages the others through the workspace; every combination
    gives the device-buffer forward's output bit for bit, on the tiny, small
    and large-batch front ends."""
    cfg = MI.custom_config(8, 2, 256, 128, mode=mode)
    case = MI.make_case(cfg, T, seed=17)
    run = DeviceRun(case)
    s = P.shape(T, 8, 2, 256, 128)
    pin = {"all": (True, True, True), "none": (False, False, False),
           "x_only": (True, False, False)}[pinned]
    xh, lh = case.x.clone(), case.logits.clone()
    oh = torch.empty((T, 256), dtype=torch.bfloat16)
    xh, lh, oh = [t.pin_memory() if p else t for t, p in zip((xh, lh, oh), pin)]
    ws = torch.zeros(P.workspace_size(s, mode), dtype=torch.uint8, device="cuda:0")
    P.forward_host(s, xh, lh, run.moe.w1_p, run.moe.w1_sf_p, run.moe.w2_p, run.moe.w2_sf_p, oh,
                   ws, mode=mode)
    torch.cuda.synchronize()
    assert P.read_device_status(ws) == 0
    np.testing.assert_array_equal(oh.float().numpy(), run.out_np())


@pytest.mark.parametrize("mode", [MI.QUANT_W4A8, MI.QUANT_W4A16, MI.QUANT_W8A8])
@pytest.mark.parametrize("T,n_steps", [(1, 5), (50, 2), (300, 3), (300, 1)])
def test_forward_host_steps_match_device_path(mode, T, n_steps):
    """moe_forward_host_steps: step i's inputs come in, and step i-1's output
    goes out, on copy streams of their own through two device staging sets
    while step i computes; every step's output equals the device-buffer
    forward of its own inputs, bit for bit (distinct inputs per step, so a
    staging set read by the wrong step shows)."""
    cfg = MI.custom_config(8, 2, 256, 128, mode=mode)
    cases = [MI.make_case(cfg, T, seed=31 + i) for i in range(n_steps)]
    run0 = DeviceRun(cases[0])
    refs = [run0.out_np()] + [DeviceRun(c, moe=run0.moe).out_np() for c in cases[1:]]
    s = P.shape(T, 8, 2, 256, 128)
    xs = [c.x.clone().pin_memory() for c in cases]
    ls = [c.logits.clone().pin_memory() for c in cases]
    outs = [torch.full((T, 256), float("nan"), dtype=torch.bfloat16).pin_memory()
            for _ in range(n_steps)]
    assert P.steps_workspace_size(s, mode) > P.workspace_size(s, mode)
    ws = torch.zeros(P.steps_workspace_size(s, mode), dtype=torch.uint8, device="cuda:0")
    m = run0.moe
    P.forward_host_steps(s, xs, ls, m.w1_p, m.w1_sf_p, m.w2_p, m.w2_sf_p, outs, ws, mode=mode)
    torch.cuda.current_stream().synchronize()
    assert P.read_device_status(ws) == 0
    for i in range(n_steps):
        np.testing.assert_array_equal(outs[i].float().numpy(), refs[i])


def test_forward_host_steps_with_gather():
    """The multi-step host entry point with gather_x = 1 (T > 256, W4A8): the
    staged x is on the device, so the expansion writes token-major rows and
    GEMM1 gathers them; every step equals the expanded-copy device forward."""
    cfg = MI.custom_config(8, 2, 256, 128)
    cases = [MI.make_case(cfg, 300, seed=81 + i) for i in range(3)]
    run0 = DeviceRun(cases[0])
    refs = [run0.out_np()] + [DeviceRun(c, moe=run0.moe).out_np() for c in cases[1:]]
    s = P.shape(300, 8, 2, 256, 128)
    xs = [c.x.clone().pin_memory() for c in cases]
    ls = [c.logits.clone().pin_memory() for c in cases]
    outs = [torch.empty((300, 256), dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    ws = torch.zeros(P.steps_workspace_size(s), dtype=torch.uint8, device="cuda:0")
    m = run0.moe
    P.forward_host_steps(s, xs, ls, m.w1_p, m.w1_sf_p, m.w2_p, m.w2_sf_p, outs, ws,
                         opts=P.options(gather_x=1))
    torch.cuda.current_stream().synchronize()
    assert P.read_device_status(ws) == 0
    for o, r in zip(outs, refs):
        np.testing.assert_array_equal(o.float().numpy(), r)


def test_fused_moe_host_steps():
    """FusedMoE.host_steps: the convenience wrapper of the multi-step host
    entry point returns each step's output equal to FusedMoE.__call__'s."""
    cfg = MI.custom_config(8, 2, 256, 128)
    cases = [MI.make_case(cfg, 64, seed=95 + i) for i in range(3)]
    m = P.FusedMoE(cases[0].w1.cuda(), cases[0].w1_sf.cuda(), cases[0].w2.cuda(),
                   cases[0].w2_sf.cuda(), 2)
    refs = [m(c.x.cuda(), c.logits.cuda()).cpu() for c in cases]
    outs = m.host_steps([c.x.pin_memory() for c in cases], [c.logits.pin_memory() for c in cases])
    torch.cuda.current_stream().synchronize()
    for o, r in zip(outs, refs):
        assert torch.equal(o, r)


def test_forward_host_steps_pageable_and_short_workspace():
    """Pageable host buffers give the same outputs (the copies just do not
    overlap); the workspace of a single forward is too small."""
    cfg = MI.custom_config(8, 2, 256, 128)
    cases = [MI.make_case(cfg, 40, seed=51 + i) for i in range(3)]
    run0 = DeviceRun(cases[0])
    refs = [run0.out_np()] + [DeviceRun(c, moe=run0.moe).out_np() for c in cases[1:]]
    s = P.shape(40, 8, 2, 256, 128)
    outs = [torch.empty((40, 256), dtype=torch.bfloat16) for _ in range(3)]
    m = run0.moe
    small = torch.zeros(P.workspace_size(s), dtype=torch.uint8, device="cuda:0")
    with pytest.raises(P.MoeError):
        P.forward_host_steps(s, [c.x for c in cases], [c.logits for c in cases], m.w1_p,
                             m.w1_sf_p, m.w2_p, m.w2_sf_p, outs, small)
    ws = torch.zeros(P.steps_workspace_size(s), dtype=torch.uint8, device="cuda:0")
    P.forward_host_steps(s, [c.x for c in cases], [c.logits for c in cases], m.w1_p, m.w1_sf_p,
                         m.w2_p, m.w2_sf_p, outs, ws)
    torch.cuda.current_stream().synchronize()
    for o, r in zip(outs, refs):
        np.testing.assert_array_equal(o.float().numpy(), r)


@pytest.mark.parametrize("T", [300, 700])
def test_gather_x_matches_expanded_copy(T):
    """gather_x = 1 (W4A8, more than 256 tokens): the expansion writes each
    token's FP8 row once, token-major in the xq region, and GEMM1 gathers
    its tiles' rows by token with TMA gather4.  The token rows equal the
    oracle's per-token quantisation, every expanded row keeps its scale,
    and h, hq and the output equal the expanded-copy forward's bit for bit
    (tiles that split an expert, ragged tails of 1..15 padded rows)."""
    cfg = MI.custom_config(8, 2, 256, 128)
    case = MI.make_case(cfg, T, seed=71)
    a = DeviceRun(case)
    b = DeviceRun(case, moe=a.moe, gather_x=1)
    assert b.status == 0
    tq, ts = M.quantize_rows_fp8(np.asarray(case.x.float().cpu().numpy(), np.float32))
    np.testing.assert_array_equal(b.xq[:T], tq)
    np.testing.assert_array_equal(b.x_scale, a.x_scale)
    np.testing.assert_array_equal(b.row_of, a.row_of)
    np.testing.assert_array_equal(b.h, a.h)
    np.testing.assert_array_equal(b.hq, a.hq)
    np.testing.assert_array_equal(b.out_np(), a.out_np())


def test_gather_x_dsv3_T4096_sampled():
    """The DSV3 layer at T=4096 with gather_x = 1: output tokens on a sample
    equal the expanded-copy forward's, bit for bit."""
    case = MI.make_case(MI.CONFIGS["dsv3"], 4096, device="cuda")
    a = DeviceRun(case)
    b = DeviceRun(case, moe=a.moe, gather_x=1)
    assert b.status == 0
    rng = np.random.default_rng(3)
    toks = rng.choice(4096, 64, replace=False)
    np.testing.assert_array_equal(b.out_np()[toks], a.out_np()[toks])


@pytest.mark.parametrize("mode", [MI.QUANT_W4A8, MI.QUANT_W4A16, MI.QUANT_W8A8])
@pytest.mark.parametrize("T", [1, 50, 300, 700])
def test_fused_combine_matches_combine_kernel(mode, T):
    """fuse_combine = 1: GEMM2's epilogue forms the top-k combine (the last
    of a token's k slots to finish a 32-column segment sums the k rows of y
    in slot order) and no combine kernel runs.  The output equals the
    combine kernel's bit for bit, on a workspace that starts as garbage (the
    front end clears the counters) and again on the same workspace (every
    counter was reset by its last arrival)."""
    cfg = MI.custom_config(8, 2, 256, 128, mode=mode)
    case = MI.make_case(cfg, T, seed=91)
    a = DeviceRun(case)
    s = P.shape(T, 8, 2, 256, 128)
    ws = torch.full((P.workspace_size(s, mode),), 0x5A, dtype=torch.uint8, device="cuda:0")
    b = DeviceRun(case, moe=a.moe, fuse_combine=1, ws=ws)
    assert b.status == 0
    np.testing.assert_array_equal(b.out_np(), a.out_np())
    c = DeviceRun(case, moe=a.moe, fuse_combine=1, ws=ws)
    np.testing.assert_array_equal(c.out_np(), a.out_np())


def test_fused_combine_dsv3_T4096():
    """The DSV3 layer at T=4096 with the combine in GEMM2's epilogue: the whole
    output equals the combine kernel's, bit for bit."""
    case = MI.make_case(MI.CONFIGS["dsv3"], 4096, device="cuda")
    a = DeviceRun(case)
    b = DeviceRun(case, moe=a.moe, fuse_combine=1)
    assert b.status == 0
    assert torch.equal(a.out, b.out)


def test_device_timeout_status_and_recovery():
    """A bounded wait that nothing satisfies returns an error status; the
    context stays usable for the next forward."""
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda:0")
    P.selftest_timeout(ws, 2000)
    torch.cuda.synchronize()
    assert P.read_device_status(ws) == P._lib.MOE_ERR_DEVICE_TIMEOUT
    cfg = MI.CONFIGS["tiny"]
    full_parity(MI.make_case(cfg, 16), name="after_timeout")


def test_invalid_args_on_device():
    """Well-formed tensors with a short workspace: the library's own check
    fires; malformed tensors are stopped by the binding before the call."""
    s = P.shape(4, 8, 2, 256, 128)
    dev = "cuda:0"
    ws = torch.zeros(P.workspace_size(s) - 256, dtype=torch.uint8, device=dev)
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device=dev)
    lg = torch.zeros((4, 8), dtype=torch.float32, device=dev)
    out = torch.empty((4, 256), dtype=torch.bfloat16, device=dev)
    w = [torch.zeros(n, dtype=torch.uint8, device=dev) for n in P._lib.weight_numels(s, 0)]
    with pytest.raises(P.MoeError) as ei:
        P.forward(s, x, lg, *w, out, ws)
    assert ei.value.code == P._lib.MOE_ERR_WORKSPACE_TOO_SMALL
    for bad in (dict(mode=7), dict(x=x.float()), dict(x=x.cpu()), dict(lg=lg[:2]),
                dict(out=out.t().contiguous().t())):
        a = dict(x=x, lg=lg, out=out, mode=0)
        a.update(bad)
        with pytest.raises(P.MoeError) as ei:
            P.forward(s, a["x"], a["lg"], *w, a["out"], ws, mode=a["mode"])
        assert ei.value.code == P._lib.MOE_ERR_INVALID_ARG


# ------------------------------------------------------------------ full sizes
def _sampled_parity(cfg, T, n_sample, variant=0):
    """Full-size run in the bench's launch configuration; S1-S3 (ids,
    offsets, row maps, every expanded row's FP8 codes and scales) checked
    bit-exactly, the output on a seeded token sample (a token's output
    depends only on its own inputs)."""
    case = MI.make_case(cfg, T, device="cuda")
    run = DeviceRun(case, variant=variant)
    assert run.status == 0
    rt, tq, ts = M.route_and_quantize(x_bits(case), case.logits.cpu().numpy(), cfg.top_k)
    check_front(run, rt, tq, ts)        # every expanded row's codes, bit for bit
    rng = np.random.default_rng(T)
    toks = np.sort(rng.choice(T, size=min(T, n_sample), replace=False))
    fw = M.forward(x_bits(case), case.logits.cpu().numpy(), oracle_weights(case), cfg.top_k,
                   tokens=toks)
    ok, st = max_err_ok(run.out_np()[toks], fw.out)
    if not ok:
        dump(f"{cfg.name}_{T}", out=run.out_np()[toks], out_ref=fw.out, toks=toks)
    assert ok, st
    return run


@pytest.mark.parametrize("T", [1, 8, 64, 512, 4096])
def test_dsv3_sizes(T):
    _sampled_parity(MI.CONFIGS["dsv3"], T, n_sample=4 if T > 8 else T)


@pytest.mark.parametrize("T", [1, 16, 128, 1024, 8192])
def test_v4pro_sizes(T):
    _sampled_parity(MI.CONFIGS["v4pro"], T, n_sample=3 if T > 1 else 1)


@pytest.mark.parametrize("T,E", [(8, 64), (100, 64), (1100, 256)])
def test_nan_logits_route_in_range(T, E):
    """NaN router logits (one NaN, half NaN, and a whole NaN row), on the
    tiny, small and large-batch front ends: every routed id stays in [0, E)
    and a token's ids stay distinct; a NaN ranks as -inf (so each row's ids
    equal the oracle's routing of the logits with NaN replaced by -inf); the
    expansion of those ids, every FP8 code and scale, and the outputs of the
    tokens with finite logits match the oracle."""
    k = 8
    cfg = MI.custom_config(E, k, 256, 128)
    case = MI.make_case(cfg, T, seed=91 + T)
    nan = float("nan")
    case.logits[1, 5] = nan
    case.logits[3, ::2] = nan
    case.logits[T - 2] = nan
    run = DeviceRun(case)
    assert run.status == 0
    ids = run.ids
    assert ids.min() >= 0 and ids.max() < E
    assert all(len(set(r)) == k for r in ids.tolist())
    lg = case.logits.cpu().numpy()
    ref_ids, ref_w = M.route(np.where(np.isnan(lg), -np.inf, lg), k)
    np.testing.assert_array_equal(ids, ref_ids)
    finite = np.flatnonzero(~np.isnan(lg).any(axis=1))
    np.testing.assert_allclose(run.weights[finite], ref_w[finite], rtol=3e-6, atol=1e-7)
    rt = M.expand(ids, run.weights, E)
    tq, ts = M.quantize_rows_fp8(np.asarray(case.x.float().cpu().numpy(), np.float32))
    check_front(run, M.Routing(ids=rt.ids, weights=run.weights, counts=rt.counts,
                               offsets=rt.offsets, row_of=rt.row_of,
                               token_of_row=rt.token_of_row, slot_of_row=rt.slot_of_row,
                               expert_of_row=rt.expert_of_row), tq, ts)
    fw = M.forward(x_bits(case), lg, oracle_weights(case), k, tokens=finite)
    ok, st = max_err_ok(run.out_np()[finite], fw.out)
    assert ok, st


def test_scan_stages_counts_in_several_batches():
    """The large-batch scan stages the per-chunk expert counts in shared
    memory batches; with 1024 experts a batch holds 48 chunks, so T = 2000
    tokens (63 chunks) take two batches.  Offsets, row maps and codes stay
    bit-exact."""
    cfg = MI.custom_config(1024, 2, 128, 128)
    run, _ = full_parity(MI.make_case(cfg, 2000, seed=97), name="scan_batches")
    check_tiles(run, 160)


@pytest.mark.parametrize("T", [40, 400])
def test_long_h_rows_take_the_register_quantisation(T):
    """I = 4224 (> 4096): the h quantisation keeps its register form instead
    of staging 8 rows in shared memory; T = 400 also takes the large-batch
    expansion.  (The scatter kernel's register form, for rows it does not
    stage, runs in the page-locked host-buffer tests.)  Every code and scale
    is bit-exact, the outputs within the tolerance."""
    cfg = MI.custom_config(8, 2, 256, 4224)
    full_parity(MI.make_case(cfg, T, seed=77 + T), name=f"long_h_{T}")
