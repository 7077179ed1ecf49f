"""Seeded random configurations: head dims, dtypes, group sizes, masks (causal, sliding window,
two-sided and right-only local windows, none), sinks, packed batches with empty and one-token
sequences, keys fewer or more than queries, input scales and every reduction mode, drawn together
so that combinations no hand-written case names are exercised; some draws also take a softmax scale
other than 1/sqrt(Dqk).  Each is run forward and backward
through the C ABI and compared element by element with the fp64 oracle on the same rounded
inputs: O and LSE from the GPU forward against the oracle's (rows that see no key, possible when keys
are fewer than queries, must have LSE = -inf on both sides), and the backward against the oracle
backward on the same stored O and LSE.  A CPU test checks first that the library's parameter validation accepts every drawn
configuration, so that a GPU failure is a numerical one."""
import random

import numpy as np
import pytest
import torch

from gqa_flashattention_backward_gb300 import _native as nat
from gqa_flashattention_backward_gb300 import workloads as W
from tests._util import assert_close, f64, gpu_run, oracle_backward_on_stored, oracle_full

SEED = 5281
COUNT = 24
DIMS = [(64, 64), (128, 128), (192, 128)]
MASKS = ["causal", "causal_window", "full", "two_sided", "right_only", "causal"]
MODES = [
    dict(group_mode=nat.GQA_GROUP_TMEM, red_mode=nat.GQA_RED_V4),
    dict(group_mode=nat.GQA_GROUP_TMEM, red_mode=nat.GQA_RED_SCALAR),
    dict(group_mode=nat.GQA_GROUP_TMEM, red_mode=nat.GQA_RED_BULK),
    dict(group_mode=nat.GQA_GROUP_ATOMIC, red_mode=nat.GQA_RED_V4),
    dict(group_mode=nat.GQA_GROUP_ATOMIC, red_mode=nat.GQA_RED_BULK),
    dict(deterministic=True),
]


def _lengths(rng, n, lo, hi):
    """n sequence lengths, about one in five empty and one in eight a single token."""
    out = []
    for _ in range(n):
        u = rng.random()
        out.append(0 if u < 0.2 else 1 if u < 0.32 else rng.randint(lo, hi))
    return out


def _draw(rng, i):
    dqk, dv = rng.choice(DIMS)
    dtype = rng.choice([torch.float16, torch.bfloat16])
    hkv = rng.choice([1, 2])
    hq = hkv * rng.choice([1, 2, 4])
    mask = MASKS[i % len(MASKS)]
    causal = mask in ("causal", "causal_window")
    window = rng.randint(1, 300) if mask in ("causal_window", "two_sided") else 0
    window_right = rng.randint(1, 200) if mask in ("two_sided", "right_only") else 0
    kw = dict(Dqk=dqk, Dv=dv, dtype=dtype, Hq=hq, Hkv=hkv, causal=causal, window=window,
              window_right=window_right, sink=rng.random() < 0.4,
              qkv_std=rng.choice([0.5, 1.0, 1.0, 2.0]))
    cross = rng.random() < 0.35  # keys fewer or more than queries
    if rng.random() < 0.35:  # packed batch
        n = rng.randint(1, 5)
        lq = _lengths(rng, n, 2, 300)
        if max(lq) == 0:
            lq[rng.randrange(n)] = rng.randint(2, 300)
        kw.update(B=1, S=sum(lq), varlen_lengths=lq)
        if cross:
            lk = _lengths(rng, n, 2, 300)
            if sum(lk) == 0:
                lk[0] = rng.randint(2, 300)
            kw.update(Sk=sum(lk), varlen_lengths_k=lk)
    else:
        s = rng.randint(1, 400)
        kw.update(B=rng.choice([1, 2]), S=s)
        if cross:
            kw.update(Sk=rng.randint(1, 450))
    mode = (i // len(MASKS) + i) % len(MODES)
    # a softmax scale other than 1/sqrt(Dqk) now and then (logits stay well conditioned: their standard
    # deviation is at most qkv_std^2 * 1.5 = 6)
    mult = rng.choice([1.0, 1.0, 0.5, 1.5])
    if mult != 1.0:
        kw.update(scale=mult * dqk ** -0.5)
    return W.Workload(f"rand{i}", 300 + i, **kw), mode


def _configs():
    rng = random.Random(SEED)
    return [_draw(rng, i) for i in range(COUNT)]


CONFIGS = _configs()


def _id(c):
    w, mode = c
    parts = [f"d{w.Dqk}", "bf16" if w.dtype == torch.bfloat16 else "fp16", f"g{w.Hq // w.Hkv}",
             f"S{w.S}", f"Sk{w.key_len}"]
    if w.varlen_lengths:
        parts.append("packed")
    parts.append("causal" if w.causal else "noncausal")
    if w.window:
        parts.append(f"w{w.window}")
    if w.window_right:
        parts.append(f"wr{w.window_right}")
    if w.sink:
        parts.append("sink")
    if w.scale is not None:
        parts.append(f"x{w.scale * w.Dqk ** 0.5:g}")
    parts.append(f"m{mode}")
    return "-".join(parts)


def _params(w, mode):
    cu = torch.zeros(len(w.varlen_lengths) + 1, dtype=torch.int32) if w.varlen_lengths else None
    cuk = torch.zeros(len(w.varlen_lengths_k) + 1, dtype=torch.int32) if w.varlen_lengths_k else None
    return nat.make_params(w.B, w.Hq, w.Hkv, w.S, w.Dqk, w.Dv, w.dtype, causal=w.causal, window=w.window,
                           scale=w.resolved_scale, cu_seqlens=cu, max_seqlen=w.max_seqlen if cu is not None else None,
                           Sk=w.key_len, cu_seqlens_k=cuk, max_seqlen_k=w.max_seqlen_k if cuk is not None else None,
                           window_right=w.window_right, **MODES[mode]), (cu, cuk)


def test_draws_cover_the_space():
    """The fixed seed reaches every head dim, both dtypes, every mask kind, sinks, packed and
    cross-length problems and every reduction mode."""
    ws = [w for w, _ in CONFIGS]
    assert {(w.Dqk, w.Dv) for w in ws} == set(DIMS)
    assert {w.dtype for w in ws} == {torch.float16, torch.bfloat16}
    assert {m for _, m in CONFIGS} == set(range(len(MODES)))
    assert any(w.sink for w in ws) and any(w.varlen_lengths for w in ws)
    assert any(w.key_len != w.S for w in ws)
    assert any(w.causal and w.window for w in ws) and any(w.window and w.window_right for w in ws)
    assert any(not w.causal and not w.window and w.window_right for w in ws)
    assert any(not w.causal and not w.window and not w.window_right for w in ws)
    assert any(w.varlen_lengths and 0 in w.varlen_lengths for w in ws)
    assert any(w.scale is not None for w in ws)


@pytest.mark.parametrize("cfg", CONFIGS, ids=_id)
def test_params_accepted(cfg):
    """Validation only reads the struct (the sequence-offset arrays are CPU tensors here: only their
    addresses are checked): a zero workspace size would mean the draw is not a valid problem."""
    w, mode = cfg
    p, _keep = _params(w, mode)
    assert nat.workspace_size(p) > 0


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", CONFIGS, ids=_id)
def test_random_config(cfg):
    w, mode = cfg
    inputs = W.make_inputs(w)
    ref = oracle_full(w, inputs)
    # forward: O and LSE against the oracle's
    res = gpu_run(w, inputs, **MODES[mode])
    lse, rlse = f64(res["lse"]), ref["lse"]
    empty = np.isneginf(rlse)
    assert np.array_equal(np.isneginf(lse), empty), f"{w.name}: rows without keys differ"
    assert_close(f"{w.name}:lse", lse[~empty], rlse[~empty], rtol=1e-3, atol=1e-3)
    assert_close(f"{w.name}:o", f64(res["o"]), ref["o"])
    # backward: both sides on the same stored O and LSE
    ref_b = oracle_backward_on_stored(w, inputs, ref)
    res_b = gpu_run(w, inputs, o_lse=(ref["o"], ref["lse"]), **MODES[mode])
    for n in ("dq", "dk", "dv"):
        assert_close(f"{w.name}:{n}", f64(res_b[n]), ref_b[n])
    if w.sink:
        assert_close(f"{w.name}:dsink", f64(res_b["dsink"]), ref_b["dsink"])
