"""Packed batches with many sequences: up to 256 sequences the main kernel runs them longest first,
through an order the preprocess writes into the workspace; above that it takes them in packing
order.  Both sides of that boundary, and a batch of 600 short sequences (empty and one-token ones
among them), in several accumulation modes, against the fp64 oracle: the forward's O and LSE, and the
backward on the same stored O and LSE on both sides."""
import random

import pytest
import torch

from gqa_flashattention_backward_gb300 import _native as nat
from gqa_flashattention_backward_gb300 import workloads as W
from tests._util import assert_close, f64, gpu_run, oracle_backward_on_stored, oracle_full

pytestmark = pytest.mark.gpu


def _lengths(n, seed, hi):
    rng = random.Random(seed)
    out = [rng.choice([0, 1, rng.randint(2, hi), rng.randint(2, hi)]) for _ in range(n)]
    out[n // 2] = hi  # one long sequence in the middle of the packing
    return out


CASES = {
    "n256_d64": (W.Workload("many256", 90, B=1, Hq=4, Hkv=2, S=0, Dqk=64, Dv=64, dtype=torch.float16,
                            varlen_lengths=_lengths(256, 1, 150)), {}),
    "n257_d64": (W.Workload("many257", 91, B=1, Hq=4, Hkv=2, S=0, Dqk=64, Dv=64, dtype=torch.float16,
                            varlen_lengths=_lengths(257, 2, 150)), {}),
    "n600_d128_window_sink": (W.Workload("many600", 92, B=1, Hq=4, Hkv=1, S=0, Dqk=128, Dv=128,
                                         dtype=torch.bfloat16, window=40, sink=True,
                                         varlen_lengths=_lengths(600, 3, 200)), {}),
    "n300_d64_atomic": (W.Workload("many300a", 93, B=1, Hq=4, Hkv=2, S=0, Dqk=64, Dv=64, dtype=torch.float16,
                                   varlen_lengths=_lengths(300, 4, 120)),
                        dict(group_mode=nat.GQA_GROUP_ATOMIC)),
    "n300_d192_deterministic": (W.Workload("many300d", 94, B=1, Hq=4, Hkv=1, S=0, Dqk=192, Dv=128,
                                           dtype=torch.bfloat16, qkv_std=0.5, varlen_lengths=_lengths(300, 5, 140)),
                                dict(deterministic=True)),
}
for _w, _ in CASES.values():
    _w.S = sum(_w.varlen_lengths)


@pytest.mark.parametrize("case", list(CASES))
def test_many_sequences(case):
    w, mode = CASES[case]
    inputs = W.make_inputs(w)
    ref = oracle_full(w, inputs)
    res = gpu_run(w, inputs, **mode)
    assert_close(f"{case}:o", f64(res["o"]), ref["o"])
    assert_close(f"{case}:lse", f64(res["lse"]), ref["lse"], rtol=1e-3, atol=1e-3)
    # the backward on the same stored O and LSE on both sides
    ref_b = oracle_backward_on_stored(w, inputs, ref)
    res_b = gpu_run(w, inputs, o_lse=(ref["o"], ref["lse"]), **mode)
    for n in ("dq", "dk", "dv"):
        assert_close(f"{case}:{n}", f64(res_b[n]), ref_b[n])
    if w.sink:
        assert_close(f"{case}:dsink", f64(res_b["dsink"]), ref_b["dsink"])
