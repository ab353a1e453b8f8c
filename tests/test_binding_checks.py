"""The Python binding's tensor checks (CPU, no GPU needed).

The C ABI takes raw pointers, so the binding checks each tensor's placement,
device, dtype, contiguity and shape before any library call.  These tests
run the checks on the generator's own tensors for every quantisation mode,
with the tensors that belong on the GPU presented as CUDA tensors by a thin
view, so the accepting path is covered here too and not only the rejecting
one."""
import pytest
import torch

import moe_inputs as MI
import precision_moe_grouped_gb300 as P
from precision_moe_grouped_gb300 import _lib as L


class OnCuda:
    """A CPU tensor seen as a CUDA tensor on device `index`: exposes only the
    attributes the binding's checks read."""
    is_cuda = True

    def __init__(self, t: torch.Tensor, index: int = 0):
        self.t, self.index = t, index

    @property
    def device(self):
        return torch.device("cuda", self.index)

    @property
    def dtype(self):
        return self.t.dtype

    @property
    def shape(self):
        return self.t.shape

    def is_contiguous(self):
        return self.t.is_contiguous()

    def numel(self):
        return self.t.numel()

    def element_size(self):
        return self.t.element_size()


def _case(mode, T=5):
    cfg = MI.custom_config(8, 2, 256, 128, mode=mode)
    case = MI.make_case(cfg, T, experts=[0])
    s = P.shape(T, 8, 2, 256, 128)
    # what FusedMoE allocates for the prepared weights
    prepared = [OnCuda(torch.empty_like(w)) for w in (case.w1, case.w1_sf, case.w2, case.w2_sf)]
    ws = OnCuda(torch.empty(64, dtype=torch.uint8))
    out = torch.empty((T, 256), dtype=torch.bfloat16)
    return s, case, prepared, ws, out


MODES = [MI.QUANT_W4A8, MI.QUANT_W4A16, MI.QUANT_W8A8]


@pytest.mark.parametrize("mode", MODES)
def test_generator_tensors_pass(mode):
    s, case, w, ws, out = _case(mode)
    L.validate_forward(s, mode, OnCuda(case.x), OnCuda(case.logits), *w, OnCuda(out), ws,
                       device=0)
    L.validate_forward(s, mode, case.x, case.logits, *w, out, ws, host=True, device=0)
    assert [t.numel() for t in w] == list(L.weight_numels(s, mode))


@pytest.mark.parametrize("mode", MODES)
def test_malformed_tensors_are_rejected(mode):
    s, case, w, ws, out = _case(mode)
    x, lg, o = OnCuda(case.x), OnCuda(case.logits), OnCuda(out)
    bad = {
        "host x": dict(x=case.x),
        "fp32 x": dict(x=OnCuda(case.x.float())),
        "strided x": dict(x=OnCuda(case.x.t().contiguous().t())),
        "short logits": dict(lg=OnCuda(case.logits[:2])),
        "bf16 logits": dict(lg=OnCuda(case.logits.bfloat16())),
        "out on another device": dict(o=OnCuda(out, index=1)),
        "wrong w1 size": dict(w1=OnCuda(torch.empty(10, dtype=torch.uint8))),
        "2-byte w2_sf": dict(w2_sf=OnCuda(w[3].t.view(torch.int16))),
        "missing workspace": dict(ws=None),
        "host workspace": dict(ws=ws.t),
        "unknown mode": dict(mode=7),
    }
    for why, change in bad.items():
        a = dict(x=x, lg=lg, o=o, w1=w[0], w1_sf=w[1], w2=w[2], w2_sf=w[3], ws=ws, mode=mode)
        a.update(change)
        with pytest.raises(P.MoeError) as ei:
            L.validate_forward(s, a["mode"], a["x"], a["lg"], a["w1"], a["w1_sf"], a["w2"],
                               a["w2_sf"], a["o"], a["ws"], device=0)
        assert ei.value.code == L.MOE_ERR_INVALID_ARG, why


def test_host_entry_wants_host_activations():
    s, case, w, ws, out = _case(MI.QUANT_W4A8)
    with pytest.raises(P.MoeError) as ei:
        L.validate_forward(s, 0, OnCuda(case.x), case.logits, *w, out, ws, host=True, device=0)
    assert ei.value.code == L.MOE_ERR_INVALID_ARG and "host" in str(ei.value)


def test_forward_rejects_cpu_tensors_before_the_library():
    """On a machine without a GPU every tensor fails the placement check, so
    nothing reaches the C ABI."""
    s, case, w, ws, out = _case(MI.QUANT_W4A8)
    with pytest.raises(P.MoeError) as ei:
        P.forward(s, case.x, case.logits, *(t.t for t in w), out, ws.t)
    assert ei.value.code == L.MOE_ERR_INVALID_ARG and "CUDA" in str(ei.value)
    with pytest.raises(P.MoeError):
        P.read_device_status(ws.t)
