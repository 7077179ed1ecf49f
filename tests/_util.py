"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the fp64 oracle on the same rounded inputs, compare with the tolerance
max|gpu - ref| <= 2e-2 * max|ref| + 1e-3 (per tensor)."""
from __future__ import annotations

import numpy as np
import torch

from gqa_flashattention_backward_gb300 import _native as nat
from gqa_flashattention_backward_gb300 import attention_backward, attention_forward
from oracle import oracle as orc

RTOL_MAX = 2e-2
ATOL = 1e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def assert_close(name, got, ref, rtol=RTOL_MAX, atol=ATOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref).max() if ref.size else 0.0
    bound = rtol * (np.abs(ref).max() if ref.size else 0.0) + atol
    assert err <= bound, f"{name}: max|err| {err:.3e} > {bound:.3e} (max|ref| {np.abs(ref).max():.3e})"
    return err, bound


def problem_of(w) -> orc.Problem:
    return orc.Problem(B=w.B, Hq=w.Hq, Hkv=w.Hkv, S=w.S, Dqk=w.Dqk, Dv=w.Dv, causal=w.causal, window=w.window,
                       scale=w.resolved_scale, cu_seqlens=w.cu_seqlens, Sk=w.key_len, cu_seqlens_k=w.cu_seqlens_k,
                       window_right=w.window_right)


def gpu_run(w, inputs, *, group_mode=nat.GQA_GROUP_TMEM, red_mode=None, deterministic=False,
            o_lse=None):
    """Forward then backward on the GPU.  o_lse: optional (o, lse) CPU tensors to feed the backward."""
    q, k, v, do, sink = inputs
    dev = torch.device("cuda")
    qd, kd, vd, dod = (x.to(dev).contiguous() for x in (q, k, v, do))
    sd = sink.to(dev) if sink is not None else None
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev) if w.cu_seqlens is not None else None
    cuk = torch.tensor(w.cu_seqlens_k, dtype=torch.int32, device=dev) if w.cu_seqlens_k is not None else None
    kw = dict(causal=w.causal, window=w.window, scale=w.resolved_scale, sink=sd, cu_seqlens=cu,
              max_seqlen=w.max_seqlen if cu is not None else None, cu_seqlens_k=cuk,
              max_seqlen_k=w.max_seqlen_k if cuk is not None else None, window_right=w.window_right)
    o, lse = attention_forward(qd, kd, vd, **kw)
    if o_lse is not None:  # isolate the backward: feed it the oracle's O (rounded) and LSE
        o = torch.as_tensor(o_lse[0]).to(w.dtype).to(dev).contiguous()
        lse = torch.as_tensor(o_lse[1]).to(torch.float32).to(dev).contiguous()
    res = attention_backward(qd, kd, vd, o, lse, dod, group_mode=group_mode, red_mode=red_mode,
                             deterministic=deterministic, **kw)
    torch.cuda.synchronize()
    res["o"], res["lse"] = o, lse
    return res


def oracle_full(w, inputs):
    q, k, v, do, sink = inputs
    pb = problem_of(w)
    sink64 = f64(sink) if sink is not None else None
    o, lse = orc.forward(pb, f64(q), f64(k), f64(v), sink64)
    g = orc.backward(pb, f64(q), f64(k), f64(v), o, lse, f64(do), sink64)
    g["o"], g["lse"] = o, lse
    return g



def oracle_backward_on_stored(w, inputs, ref):
    """The oracle backward on the O the GPU backward reads: the oracle's O rounded to the input dtype
    (and its LSE).  Delta is defined on O as stored (tilelang-ascend PR #1638 "Add GQA Sink Backward
    BHSD", 4->2 commit: Phase0(Delta) = sum(O*dO)); with few keys per row, or many rows in dsink, the
    rounding of O alone moves dQ, dK and dsink past 2e-2 max|ref| in bf16, so a backward check that
    should see only the kernels' own arithmetic gives both sides the same stored O."""
    q, k, v, do, sink = inputs
    o_st = f64(torch.as_tensor(ref["o"]).to(w.dtype))
    sink64 = f64(sink) if sink is not None else None
    g = orc.backward(problem_of(w), f64(q), f64(k), f64(v), o_st, ref["lse"], f64(do), sink64)
    return g
