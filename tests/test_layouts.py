"""General memory layouts: BSHD views, packed THD for variable-length batches and mixed layouts
run through the kernels with their strides (no copies) and must match the fp64 oracle computed
on the same values."""
import pytest
import torch

from gqa_flashattention_backward_gb300 import _native as nat
from gqa_flashattention_backward_gb300 import attention_backward, attention_forward
from gqa_flashattention_backward_gb300 import workloads as W
from tests._util import assert_close, f64, oracle_full

pytestmark = pytest.mark.gpu


def bshd(x):
    """The same [B, H, S, D] values stored batch, sequence, head, dim (a view, nothing copied later)."""
    return x.transpose(1, 2).contiguous().cuda().transpose(1, 2)


def thd(x):
    """[1, H, T, D] values stored token-major, as packed variable-length batches usually are."""
    assert x.shape[0] == 1
    return x[0].transpose(0, 1).contiguous().cuda().transpose(0, 1).unsqueeze(0)


def bhsd(x):
    return x.contiguous().cuda()


def _run(w, inputs, lay_q, lay_kv, lay_do, **mode):
    q, k, v, do, sink = inputs
    qd, kd, vd, dod = lay_q(q), lay_kv(k), lay_kv(v), lay_do(do)
    sd = sink.cuda() if sink is not None else None
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device="cuda") if w.cu_seqlens is not None else None
    kw = dict(causal=w.causal, window=w.window, scale=w.resolved_scale, sink=sd, cu_seqlens=cu,
              max_seqlen=w.max_seqlen if cu is not None else None)
    o, lse = attention_forward(qd, kd, vd, **kw)
    assert o.stride() == attention_layout_stride(qd, w.Dv), (o.stride(), qd.stride())
    res = attention_backward(qd, kd, vd, o, lse, dod, **kw, **mode)
    torch.cuda.synchronize()
    for n, ref in (("dq", qd), ("dk", kd), ("dv", vd)):
        assert nat.tensor_strides(res[n]) == nat.tensor_strides(ref) or res[n].shape[-1] != ref.shape[-1], n
    res["o"], res["lse"] = o, lse
    return res


def attention_layout_stride(ref, last):
    """Strides of an output laid out like `ref` with head dim `last`."""
    order = sorted(range(3), key=lambda i: -ref.stride(i))
    sizes = {i: ref.shape[i] for i in range(3)}
    st, acc = {}, last
    for i in reversed(order):
        st[i] = acc
        acc *= sizes[i]
    return (st[0], st[1], st[2], 1)


def _check(w, res, ref):
    assert_close(f"{w.name}:o", f64(res["o"]), ref["o"])
    assert_close(f"{w.name}:lse", f64(res["lse"]), ref["lse"], rtol=1e-3, atol=1e-3)
    for n in ("dq", "dk", "dv"):
        assert_close(f"{w.name}:{n}", f64(res[n]), ref[n])
    if w.sink:
        assert_close(f"{w.name}:dsink", f64(res["dsink"]), ref["dsink"])


CASES = {
    "mha64": lambda: W.shrink(W.mha_causal(), name="lay_mha64", B=2, Hq=4, Hkv=2, S=300),
    "sink128": lambda: W.shrink(W.sink_window(), name="lay_sink128", B=2, Hq=4, Hkv=2, S=260, window=100),
    "long192": lambda: W.shrink(W.long_context(), name="lay_long192", B=2, Hq=4, Hkv=1, S=200),
}


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("mode", ["default", "deterministic", "atomic"])
def test_bshd_everywhere(case, mode):
    w = CASES[case]()
    inputs = W.make_inputs(w)
    ref = oracle_full(w, inputs)
    kw = {"default": {}, "deterministic": dict(deterministic=True),
          "atomic": dict(group_mode=nat.GQA_GROUP_ATOMIC)}[mode]
    res = _run(w, inputs, bshd, bshd, bshd, **kw)
    _check(w, res, ref)


def test_mixed_layouts():
    w = CASES["mha64"]()
    inputs = W.make_inputs(w)
    ref = oracle_full(w, inputs)
    _check(w, _run(w, inputs, bshd, bhsd, bshd), ref)
    _check(w, _run(w, inputs, bhsd, bshd, bhsd), ref)


@pytest.mark.parametrize("dims", [(64, 64), (128, 128)])
def test_packed_thd_varlen(dims):
    dqk, dv = dims
    w = W.Workload(f"lay_thd{dqk}", 31, B=1, Hq=4, Hkv=2, S=465, Dqk=dqk, Dv=dv, dtype=torch.bfloat16,
                   varlen_lengths=[130, 1, 0, 257, 77])
    inputs = W.make_inputs(w)
    ref = oracle_full(w, inputs)
    _check(w, _run(w, inputs, thd, thd, thd), ref)
