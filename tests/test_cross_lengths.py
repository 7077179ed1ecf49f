"""Keys fewer or more than queries (chunked prefill, a KV cache, cross-attention): the causal
diagonal is aligned at the bottom right (query i of a sequence with Lq queries and Lk keys sees
key j iff j <= i + Lk - Lq).  GPU against the fp64 oracle, which was pinned on its own for this
(finite differences, brute force, PyTorch autograd, the decode case, rows that see no key)."""
import numpy as np
import pytest
import torch

from gqa_flashattention_backward_gb300 import _native as nat
from gqa_flashattention_backward_gb300 import workloads as W
from tests._util import assert_close, f64, gpu_run, oracle_full

pytestmark = pytest.mark.gpu


def _compare(w, res, ref):
    lse, rlse = f64(res["lse"]), ref["lse"]
    empty = np.isneginf(rlse)  # query rows that see no key (and no sink)
    assert np.array_equal(np.isneginf(lse), empty), f"{w.name}: rows without keys differ"
    assert_close(f"{w.name}:lse", lse[~empty], rlse[~empty], rtol=1e-3, atol=1e-3)
    assert_close(f"{w.name}:o", f64(res["o"]), ref["o"])
    for n in ("dq", "dk", "dv"):
        assert_close(f"{w.name}:{n}", f64(res[n]), ref[n])
    if w.sink:
        assert_close(f"{w.name}:dsink", f64(res["dsink"]), ref["dsink"])


CASES = {
    "prefill64": lambda: W.Workload("x_prefill64", 40, B=2, Hq=4, Hkv=2, S=200, Sk=456, Dqk=64, Dv=64,
                                    dtype=torch.float16),
    "morequeries64": lambda: W.Workload("x_moreq64", 41, B=2, Hq=4, Hkv=2, S=456, Sk=200, Dqk=64, Dv=64,
                                        dtype=torch.float16),
    "morequeries64_sink": lambda: W.Workload("x_moreq64s", 42, B=1, Hq=4, Hkv=1, S=300, Sk=130, Dqk=64, Dv=64,
                                             dtype=torch.float16, sink=True),
    "varlen128_window": lambda: W.Workload("x_var128", 43, B=1, Hq=4, Hkv=2, S=272, Sk=501, Dqk=128, Dv=128,
                                           dtype=torch.bfloat16, window=100, varlen_lengths=[130, 1, 77, 64],
                                           varlen_lengths_k=[300, 1, 0, 200]),
    "cross128_noncausal": lambda: W.Workload("x_cross128", 44, B=2, Hq=4, Hkv=4, S=150, Sk=333, Dqk=128, Dv=128,
                                             dtype=torch.float16, causal=False, sink=True),
    "prefill192": lambda: W.Workload("x_prefill192", 45, B=1, Hq=4, Hkv=1, S=130, Sk=260, Dqk=192, Dv=128,
                                     dtype=torch.bfloat16, qkv_std=0.5),
    "decode64": lambda: W.Workload("x_decode64", 46, B=2, Hq=8, Hkv=2, S=1, Sk=300, Dqk=64, Dv=64,
                                   dtype=torch.float16),
    # the forward's first pair of 128-row query tiles: the first tile sees no key, the second some
    "morequeries128": lambda: W.Workload("x_moreq128", 47, B=1, Hq=4, Hkv=2, S=300, Sk=130, Dqk=128, Dv=128,
                                         dtype=torch.bfloat16),
    "morequeries192_sink": lambda: W.Workload("x_moreq192s", 48, B=1, Hq=4, Hkv=1, S=300, Sk=100, Dqk=192,
                                              Dv=128, dtype=torch.bfloat16, sink=True, qkv_std=0.5),
}


@pytest.mark.parametrize("case", list(CASES))
def test_cross_lengths(case):
    w = CASES[case]()
    inputs = W.make_inputs(w)
    ref = oracle_full(w, inputs)
    _compare(w, gpu_run(w, inputs), ref)


@pytest.mark.parametrize("mode", ["deterministic", "atomic"])
@pytest.mark.parametrize("case", ["prefill64", "morequeries64", "varlen128_window"])
def test_cross_lengths_other_modes(case, mode):
    w = CASES[case]()
    inputs = W.make_inputs(w)
    ref = oracle_full(w, inputs)
    kw = dict(deterministic=True) if mode == "deterministic" else dict(group_mode=nat.GQA_GROUP_ATOMIC)
    _compare(w, gpu_run(w, inputs, **kw), ref)


# ---------------------------------------------------------------- right window (non-causal local attention)
LOCAL = {
    "twosided64": lambda: W.Workload("l_two64", 50, B=2, Hq=4, Hkv=2, S=300, Dqk=64, Dv=64, dtype=torch.float16,
                                     causal=False, window=65, window_right=40),
    "rightonly128_sink": lambda: W.Workload("l_right128", 51, B=1, Hq=4, Hkv=2, S=260, Dqk=128, Dv=128,
                                            dtype=torch.bfloat16, causal=False, window_right=100, sink=True),
    "twosided64_prefill": lambda: W.Workload("l_two64x", 52, B=1, Hq=4, Hkv=1, S=200, Sk=330, Dqk=64, Dv=64,
                                             dtype=torch.float16, causal=False, window=80, window_right=50),
    "twosided128_varlen": lambda: W.Workload("l_var128", 53, B=1, Hq=4, Hkv=2, S=207, Sk=260, Dqk=128, Dv=128,
                                             dtype=torch.bfloat16, causal=False, window=50, window_right=30,
                                             varlen_lengths=[130, 77], varlen_lengths_k=[200, 60]),
    "twosided192": lambda: W.Workload("l_two192", 54, B=1, Hq=4, Hkv=1, S=260, Dqk=192, Dv=128,
                                      dtype=torch.bfloat16, causal=False, window=60, window_right=40, qkv_std=0.5),
}


@pytest.mark.parametrize("case", list(LOCAL))
def test_right_window(case):
    w = LOCAL[case]()
    inputs = W.make_inputs(w)
    ref = oracle_full(w, inputs)
    _compare(w, gpu_run(w, inputs), ref)


@pytest.mark.parametrize("mode", ["deterministic", "atomic"])
def test_right_window_other_modes(mode):
    w = LOCAL["twosided64_prefill"]()
    inputs = W.make_inputs(w)
    ref = oracle_full(w, inputs)
    kw = dict(deterministic=True) if mode == "deterministic" else dict(group_mode=nat.GQA_GROUP_ATOMIC)
    _compare(w, gpu_run(w, inputs, **kw), ref)
