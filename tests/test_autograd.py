"""The autograd wrapper: gradients that flow through ``torch.autograd`` are the ones the C ABI
backward computes, and they match the fp64 oracle."""
import pytest
import torch

from gqa_flashattention_backward_gb300 import gqa_attention
from gqa_flashattention_backward_gb300 import workloads as W
from tests._util import assert_close, f64, oracle_full

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [
    lambda: W.shrink(W.mha_causal(), name="ag_mha", B=1, Hq=2, Hkv=2, S=300),
    lambda: W.shrink(W.sink_window(), name="ag_sink", Hq=4, Hkv=2, S=333, window=100),
])
def test_autograd_matches_oracle(make):
    w = make()
    inputs = W.make_inputs(w)
    q, k, v, do, sink = inputs
    dev = torch.device("cuda")
    qd, kd, vd = (x.to(dev).requires_grad_(True) for x in (q, k, v))
    sd = sink.to(dev).requires_grad_(True) if sink is not None else None
    o = gqa_attention(qd, kd, vd, causal=w.causal, window=w.window, scale=w.resolved_scale, sink=sd)
    o.backward(do.to(dev))
    torch.cuda.synchronize()
    ref = oracle_full(w, inputs)
    assert_close(f"{w.name}:o", f64(o), ref["o"])
    assert_close(f"{w.name}:dq", f64(qd.grad), ref["dq"])
    assert_close(f"{w.name}:dk", f64(kd.grad), ref["dk"])
    assert_close(f"{w.name}:dv", f64(vd.grad), ref["dv"])
    if sd is not None:
        assert sd.grad is not None and sd.grad.dtype == torch.float32
        assert_close(f"{w.name}:dsink", f64(sd.grad), ref["dsink"])
