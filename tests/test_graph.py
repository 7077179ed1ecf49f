"""The backward captured as one CUDA graph: replays equal the eager calls (bit for bit in the
deterministic mode, also after new inputs are copied in place) and the oracle."""
import pytest
import torch

from gqa_flashattention_backward_gb300 import GraphedBackward, attention_backward, attention_forward
from gqa_flashattention_backward_gb300 import workloads as W
from tests._util import assert_close, f64, oracle_full

pytestmark = pytest.mark.gpu


def _setup(w, seed=None):
    q, k, v, do, sink = (x.cuda() if x is not None else None for x in W.make_inputs(w, seed))
    kw = dict(causal=w.causal, window=w.window, scale=w.resolved_scale, sink=sink)
    o, lse = attention_forward(q, k, v, **kw)
    return q, k, v, o, lse, do, kw


@pytest.mark.parametrize("deterministic", [True, False])
def test_graph_replay_matches_eager_and_oracle(deterministic):
    w = W.shrink(W.sink_window(), name="graph_sink", Hq=8, Hkv=2, S=384, window=150)
    q, k, v, o, lse, do, kw = _setup(w)
    gb = GraphedBackward(q, k, v, o, lse, do, deterministic=deterministic, **kw)
    for seed in (None, 77):  # the second round copies new inputs into the captured tensors
        if seed is not None:
            q2, k2, v2, o2, lse2, do2, kw2 = _setup(w, seed)
            for dst, src in ((q, q2), (k, k2), (v, v2), (o, o2), (lse, lse2), (do, do2), (kw["sink"], kw2["sink"])):
                dst.copy_(src)
        res = {n: t.clone() for n, t in gb.replay().items()}
        eager = attention_backward(q, k, v, o, lse, do, deterministic=deterministic, **kw)
        torch.cuda.synchronize()
        for n in ("dq", "dk", "dv", "delta", "dsink"):
            if deterministic:
                assert torch.equal(res[n], eager[n]), n
            else:
                assert_close(f"graph:{n}", f64(res[n]), f64(eager[n]), rtol=1e-3, atol=1e-5)
    inputs = tuple(t.cpu() for t in (q, k, v, do)) + (kw["sink"].cpu(),)
    ref = oracle_full(w, inputs)
    for n in ("dq", "dk", "dv", "dsink"):
        assert_close(f"graph:{n}", f64(res[n]), ref[n])
