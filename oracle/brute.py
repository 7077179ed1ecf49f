"""Second, independent fp64 reference: materialises the full S x S score matrix.

TEST INFRASTRUCTURE ONLY (tiny inputs).  Written separately from gqa_oracle.c:
the mask is built as a boolean matrix, the softmax is taken over an explicit
extra sink column, and GQA is handled by expanding K/V to one copy per query
head, running plain multi-head attention head by head and summing the per-head
dK/dV over each group (the group reduction of tilelang PR #1093, "accumulate
locally, write once", done here the obvious way).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np


def mask_matrix(S: int, causal: bool, window: int, cu_seqlens: Optional[Sequence[int]], Sk: Optional[int] = None,
                cu_seqlens_k: Optional[Sequence[int]] = None, window_right: int = 0) -> np.ndarray:
    """allowed[i, j] for query row i and key row j: same sequence, and with local indices
    il, jl and the sequence's lengths Lq, Lk, causal jl <= il + Lk - Lq, window il + Lk - Lq - jl < W,
    right window jl - (il + Lk - Lq) < Wr."""
    Sk = Sk or S
    cu_q = list(cu_seqlens) if cu_seqlens is not None else [0, S]
    cu_k = list(cu_seqlens_k) if cu_seqlens_k is not None else (list(cu_seqlens) if cu_seqlens is not None
                                                                 else [0, Sk])
    seq_q, loc_q, off_q = np.full(S, -1), np.zeros(S, dtype=np.int64), np.zeros(S, dtype=np.int64)
    seq_k, loc_k = np.full(Sk, -2), np.zeros(Sk, dtype=np.int64)
    for s in range(len(cu_q) - 1):
        lq, lk = cu_q[s + 1] - cu_q[s], cu_k[s + 1] - cu_k[s]
        seq_q[cu_q[s]:cu_q[s + 1]] = s
        loc_q[cu_q[s]:cu_q[s + 1]] = np.arange(lq)
        off_q[cu_q[s]:cu_q[s + 1]] = lk - lq
        seq_k[cu_k[s]:cu_k[s + 1]] = s
        loc_k[cu_k[s]:cu_k[s + 1]] = np.arange(lk)
    diag = (loc_q + off_q)[:, None]  # each query's key diagonal
    jl = loc_k[None, :]
    allowed = seq_q[:, None] == seq_k[None, :]
    if causal:
        allowed &= jl <= diag
    if window > 0:
        allowed &= (diag - jl) < window
    if window_right > 0 and not causal:
        allowed &= (jl - diag) < window_right
    return allowed


def mha_head(q, k, v, dout, scale, allowed, sink: Optional[float]):
    """One head of plain attention, forward + backward, all matrices explicit.

    Returns a dict with O, LSE, P, p_sink, dP, dS, Delta, dQ, dK, dV, dsink.
    """
    S = scale * (q @ k.T)                        # [Sq, Sk]
    S = np.where(allowed, S, -np.inf)
    cols = S if sink is None else np.concatenate([S, np.full((S.shape[0], 1), sink)], axis=1)
    m = cols.max(axis=1, keepdims=True)
    empty = ~np.isfinite(m)                      # a query row that sees nothing (no key, no sink)
    m = np.where(empty, 0.0, m)
    e = np.exp(cols - m)
    z = e.sum(axis=1, keepdims=True)
    with np.errstate(divide="ignore"):
        lse = (m + np.log(z))[:, 0]
    probs = np.where(z > 0, e / np.where(z > 0, z, 1.0), 0.0)
    P = probs[:, :S.shape[1]]
    p_sink = probs[:, S.shape[1]] if sink is not None else np.zeros(S.shape[0])
    O = P @ v
    Delta = (dout * O).sum(axis=1)
    dP = dout @ v.T
    dS = P * (dP - Delta[:, None]) * scale
    dQ = dS @ k
    dK = dS.T @ q
    dV = P.T @ dout
    dsink = -(p_sink * Delta).sum()
    return dict(O=O, LSE=lse, P=P, p_sink=p_sink, dP=dP, dS=dS, Delta=Delta, dQ=dQ, dK=dK, dV=dV, dsink=dsink)


def gqa(q, k, v, dout, scale, causal=True, window=0, cu_seqlens=None, sink=None, cu_seqlens_k=None, window_right=0):
    """Full GQA forward+backward for [B,H,S,D] float64 arrays via per-head MHA (k, v may have
    another length Sk)."""
    B, Hq, S, _ = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    allowed = mask_matrix(S, causal, window, cu_seqlens, Sk, cu_seqlens_k, window_right)
    out = dict(
        o=np.zeros((B, Hq, S, v.shape[3])), lse=np.zeros((B, Hq, S)), delta=np.zeros((B, Hq, S)),
        dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v), dsink=np.zeros(Hq),
        P=np.zeros((B, Hq, S, Sk)), dS=np.zeros((B, Hq, S, Sk)), dP=np.zeros((B, Hq, S, Sk)),
        p_sink=np.zeros((B, Hq, S)),
    )
    for b in range(B):
        for h in range(Hq):
            kh = np.repeat(k[b], G, axis=0)[h]   # expanded K/V: query head h reads kv head h // G
            vh = np.repeat(v[b], G, axis=0)[h]
            r = mha_head(q[b, h], kh, vh, dout[b, h], scale, allowed, None if sink is None else float(sink[h]))
            out["o"][b, h] = r["O"]
            out["lse"][b, h] = r["LSE"]
            out["delta"][b, h] = r["Delta"]
            out["dq"][b, h] = r["dQ"]
            out["dk"][b, h // G] += r["dK"]
            out["dv"][b, h // G] += r["dV"]
            out["dsink"][h] += r["dsink"]
            out["P"][b, h] = r["P"]
            out["dS"][b, h] = r["dS"]
            out["dP"][b, h] = r["dP"]
            out["p_sink"][b, h] = r["p_sink"]
    return out
