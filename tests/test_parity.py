"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on
the same seeded, rounded inputs, element by element, at sizes the oracle
finishes in seconds that still span several tiles and a ragged tail."""
import numpy as np
import pytest
import torch

from gqa_flashattention_backward_gb300 import _native as nat
from gqa_flashattention_backward_gb300 import workloads as W
from tests._util import assert_close, f64, gpu_run, oracle_full

pytestmark = pytest.mark.gpu


def _cases():
    return {
        "tiny": W.tiny(),
        "tiny_ragged": W.shrink(W.tiny(), name="tiny_ragged", S=300),
        "mha": W.shrink(W.mha_causal(), name="mha_small", B=2, Hq=2, Hkv=2, S=520),
        "varlen": W.shrink(W.varlen(), name="varlen_small", Hq=8, Hkv=2, S=849,
                           varlen_lengths=[130, 1, 0, 257, 384, 77]),
        # skewed packing: a long sequence first and late, short and empty ones between (the longest-first
        # schedule of the main kernel reorders these items)
        "varlen_skewed": W.shrink(W.varlen(), name="varlen_skewed", Hq=4, Hkv=1, S=9337,
                                  varlen_lengths=[4096, 64, 64, 64, 3000, 1, 0, 2048]),
        "sink_window": W.shrink(W.sink_window(), name="sink_window_small", Hq=8, Hkv=1, S=600, window=200),
        "long_context": W.shrink(W.long_context(), name="long_context_small", Hq=4, Hkv=1, S=450),
        "noncausal64": W.Workload("noncausal64", 10, B=1, Hq=2, Hkv=1, S=300, Dqk=64, Dv=64,
                                  dtype=torch.float16, causal=False),
        "noncausal128": W.Workload("noncausal128", 11, B=1, Hq=2, Hkv=2, S=260, Dqk=128, Dv=128,
                                   dtype=torch.bfloat16, causal=False),
    }


CASES = _cases()
_oracle_cache = {}


def _oracle(name):
    if name not in _oracle_cache:
        w = CASES[name]
        inputs = W.make_inputs(w)
        _oracle_cache[name] = (inputs, oracle_full(w, inputs))
    return _oracle_cache[name]


def _compare(w, res, ref, names=("dq", "dk", "dv")):
    for n in names:
        assert_close(f"{w.name}:{n}", f64(res[n]), ref[n])
    if w.sink:
        assert_close(f"{w.name}:dsink", f64(res["dsink"]), ref["dsink"])


@pytest.mark.parametrize("name", list(CASES))
def test_forward(name):
    w = CASES[name]
    inputs, ref = _oracle(name)
    res = gpu_run(w, inputs)
    assert_close(f"{name}:o", f64(res["o"]), ref["o"])
    assert_close(f"{name}:lse", f64(res["lse"]), ref["lse"], rtol=1e-3, atol=1e-3)


MODES = {
    "tmem_v4": dict(group_mode=nat.GQA_GROUP_TMEM, red_mode=nat.GQA_RED_V4),
    "tmem_scalar": dict(group_mode=nat.GQA_GROUP_TMEM, red_mode=nat.GQA_RED_SCALAR),
    "tmem_bulk": dict(group_mode=nat.GQA_GROUP_TMEM, red_mode=nat.GQA_RED_BULK),
    "atomic_v4": dict(group_mode=nat.GQA_GROUP_ATOMIC, red_mode=nat.GQA_RED_V4),
    "atomic_scalar": dict(group_mode=nat.GQA_GROUP_ATOMIC, red_mode=nat.GQA_RED_SCALAR),
    "atomic_bulk": dict(group_mode=nat.GQA_GROUP_ATOMIC, red_mode=nat.GQA_RED_BULK),
    "deterministic": dict(deterministic=True),
}


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("name", list(CASES))
def test_backward(name, mode):
    w = CASES[name]
    inputs, ref = _oracle(name)
    res = gpu_run(w, inputs, **MODES[mode])
    _compare(w, res, ref)
    assert_close(f"{name}:delta", f64(res["delta"]), ref["delta"])


@pytest.mark.parametrize("name", ["tiny_ragged", "varlen", "sink_window", "long_context"])
def test_backward_isolated_from_forward(name):
    """The backward fed the oracle's own O (rounded) and LSE."""
    w = CASES[name]
    inputs, ref = _oracle(name)
    res = gpu_run(w, inputs, o_lse=(torch.from_numpy(ref["o"]), torch.from_numpy(ref["lse"])))
    _compare(w, res, ref)


@pytest.mark.parametrize("name", ["tiny_ragged", "varlen", "long_context"])
def test_deterministic_bit_identical(name):
    w = CASES[name]
    inputs, _ = _oracle(name)
    outs = [gpu_run(w, inputs, deterministic=True) for _ in range(3)]
    for n in ("dq", "dk", "dv"):
        a = outs[0][n].view(torch.int16)
        for o in outs[1:]:
            assert torch.equal(a, o[n].view(torch.int16)), n


@pytest.mark.parametrize("case", ["mha", "varlen"])
def test_no_accumulation_variant_runs(case):
    """The benchmark-only store mode (d=64 tensor-store and d=128 bulk-store paths): dK / dV are
    unaffected by the dQ mode and must still match; dQ is only required to be finite."""
    w = CASES[case]
    inputs, ref = _oracle(case)
    res = gpu_run(w, inputs, red_mode=nat.GQA_RED_NONE)
    for n in ("dk", "dv"):
        assert_close(f"{case}:none:{n}", f64(res[n]), ref[n])
    assert torch.isfinite(res["dq"].float()).all()


def test_single_token_and_empty_sequences():
    w = W.Workload("edge", 12, B=1, Hq=4, Hkv=2, S=5, Dqk=64, Dv=64, dtype=torch.float16,
                   varlen_lengths=[0, 1, 0, 4, 0])
    inputs = W.make_inputs(w)
    ref = oracle_full(w, inputs)
    for mode in ("tmem_v4", "atomic_v4", "deterministic"):
        res = gpu_run(w, inputs, **MODES[mode])
        assert_close("edge:o", f64(res["o"]), ref["o"])
        _compare(w, res, ref)


def test_sequence_longer_than_max_is_reported():
    dev = torch.device("cuda")
    S = 300
    q = torch.randn(1, 2, S, 64, device=dev, dtype=torch.float16)
    k = torch.randn(1, 1, S, 64, device=dev, dtype=torch.float16)
    v = torch.randn(1, 1, S, 64, device=dev, dtype=torch.float16)
    cu = torch.tensor([0, 100, 300], dtype=torch.int32, device=dev)
    p = nat.make_params(1, 2, 1, S, 64, 64, torch.float16, cu_seqlens=cu, max_seqlen=150)
    ws = nat.alloc_workspace(p)
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, S, device=dev)
    nat.fwd(p, q, k, v, None, o, lse, ws)
    status, site = nat.get_device_error(ws)
    assert status == nat.GQA_ERR_DEVICE_INPUT, (status, hex(site))
    assert nat.get_device_error(ws)[0] == nat.GQA_OK  # reading clears it


def test_wait_timeout_is_reported_and_context_survives():
    p = nat.make_params(1, 1, 1, 128, 64, 64, torch.float16)
    ws = nat.alloc_workspace(p)
    try:
        nat.set_wait_limit(20000)  # cycles
        nat.selftest_wait_timeout(ws)
        status, site = nat.get_device_error(ws)
        assert status == nat.GQA_ERR_DEVICE_TIMEOUT
        assert site & 0xFF == 0x7E
    finally:
        nat.set_wait_limit(0)
    # the context is still usable
    w = CASES["tiny"]
    inputs, ref = _oracle("tiny")
    res = gpu_run(w, inputs)
    _compare(w, res, ref)
