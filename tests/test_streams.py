"""Problems in flight at the same time on two CUDA streams, each call with its own workspace: the
library keeps no state between calls outside the workspace (tensor maps are built per call, the
error word and the accumulators live in the workspace), so concurrent problems must not disturb one
another.  Each stream's results are compared with the fp64 oracle; the deterministic mode must give
bit-identical results on both streams."""
import pytest
import torch

from gqa_flashattention_backward_gb300 import attention_backward, attention_forward
from gqa_flashattention_backward_gb300 import workloads as W
from tests._util import assert_close, f64, oracle_full

pytestmark = pytest.mark.gpu


def _device_inputs(w):
    q, k, v, do, sink = W.make_inputs(w)
    dev = torch.device("cuda")
    return tuple(x.to(dev) for x in (q, k, v, do)) + ((sink.to(dev) if sink is not None else None),)


def _launch(w, d, **kw):
    """Forward then backward on the current stream, no synchronisation."""
    q, k, v, do, sink = d
    args = dict(causal=w.causal, window=w.window, scale=w.resolved_scale, sink=sink)
    o, lse = attention_forward(q, k, v, **args)
    res = attention_backward(q, k, v, o, lse, do, **args, **kw)
    res["o"], res["lse"] = o, lse
    return res


def _check(w, res, ref):
    assert_close(f"{w.name}:o", f64(res["o"]), ref["o"])
    assert_close(f"{w.name}:lse", f64(res["lse"]), ref["lse"], rtol=1e-3, atol=1e-3)
    for n in ("dq", "dk", "dv"):
        assert_close(f"{w.name}:{n}", f64(res[n]), ref[n])
    if w.sink:
        assert_close(f"{w.name}:dsink", f64(res["dsink"]), ref["dsink"])


def test_two_problems_on_two_streams():
    wa = W.Workload("stream_a", 80, B=2, Hq=4, Hkv=2, S=700, Dqk=64, Dv=64, dtype=torch.float16)
    wb = W.Workload("stream_b", 81, B=1, Hq=8, Hkv=2, S=520, Dqk=128, Dv=128, dtype=torch.bfloat16,
                    window=200, sink=True)
    refs = {w.name: oracle_full(w, W.make_inputs(w)) for w in (wa, wb)}
    da, db = _device_inputs(wa), _device_inputs(wb)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    out = []
    for _ in range(3):  # interleaved submissions, so the two streams' kernels overlap
        with torch.cuda.stream(sa):
            ra = _launch(wa, da)
        with torch.cuda.stream(sb):
            rb = _launch(wb, db)
        out.append((ra, rb))
    torch.cuda.synchronize()
    for ra, rb in out:
        _check(wa, ra, refs[wa.name])
        _check(wb, rb, refs[wb.name])


def test_deterministic_identical_across_streams():
    w = W.Workload("stream_det", 82, B=1, Hq=8, Hkv=2, S=600, Dqk=128, Dv=128, dtype=torch.bfloat16)
    d = _device_inputs(w)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(2)]
    res = []
    for s in streams:
        with torch.cuda.stream(s):
            res.append(_launch(w, d, deterministic=True))
    torch.cuda.synchronize()
    for n in ("dq", "dk", "dv"):
        assert torch.equal(res[0][n].view(torch.int16), res[1][n].view(torch.int16)), n
    _check(w, res[0], oracle_full(w, W.make_inputs(w)))
