"""The forward captured into a CUDA graph (the decode fast path of a serving
stack replays one graph per step): the captured launches -- programmatic
dependent launches included -- replay to exactly the eager result, and a
replay after new inputs are copied into the captured buffers matches an
eager run on those inputs.  One case per front-end path: the one-kernel
tiny batch (T <= 32), the small-batch expansion (T <= 256) and the
multi-kernel expansion."""
import pytest
import torch

import moe_inputs as MI
import precision_moe_grouped_gb300 as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    P.load()


@pytest.mark.parametrize("mode", [MI.QUANT_W4A8, MI.QUANT_W8A8, MI.QUANT_W4A16])
@pytest.mark.parametrize("T", [1, 64, 1100])
def test_forward_replays_from_cuda_graph(T, mode):
    cfg = MI.custom_config(16, 4, 256, 256, mode=mode)
    a = MI.make_case(cfg, T, seed=3, device="cuda")
    b = MI.make_case(cfg, T, seed=4, device="cuda")
    moe = P.FusedMoE(a.w1, a.w1_sf, a.w2, a.w2_sf, cfg.top_k, mode=mode)
    s = moe.shape(T)
    ws = moe.workspace(T)
    x = a.x.clone()
    logits = a.logits.clone()
    out = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    ref_a = moe(a.x, a.logits)          # eager runs (they also set kernel attributes)
    ref_b = moe(b.x, b.logits)
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side), torch.cuda.graph(g, stream=side):
        P.forward(s, x, logits, moe.w1_p, moe.w1_sf_p, moe.w2_p, moe.w2_sf_p, out, ws,
                  mode=mode)
    g.replay()
    torch.cuda.synchronize()
    assert P.read_device_status(ws) == 0
    assert torch.equal(out, ref_a)

    x.copy_(b.x)
    logits.copy_(b.logits)
    g.replay()
    torch.cuda.synchronize()
    assert P.read_device_status(ws) == 0
    assert torch.equal(out, ref_b)
