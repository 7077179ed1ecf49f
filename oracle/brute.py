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


def mask_matrix(S: int, causal: bool, window: int, cu_seqlens: Optional[Sequence[int]]) -> np.ndarray:
    """allowed[i, j] for query row i and key row j."""
    seq = np.zeros(S, dtype=np.int64)
    if cu_seqlens is not None:
        cu = list(cu_seqlens)
        for s in range(len(cu) - 1):
            seq[cu[s]:cu[s + 1]] = s
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    allowed = seq[:, None] == seq[None, :]
    if causal:
        allowed &= j <= i
    if window > 0:
        allowed &= (i - j) < window
    return allowed


def mha_head(q, k, v, dout, scale, allowed, sink: Optional[float]):
    """One head of plain attention, forward + backward, all matrices explicit.

    Returns a dict with O, LSE, P, p_sink, dP, dS, Delta, dQ, dK, dV, dsink.
    """
    S = scale * (q @ k.T)                        # [Sq, Sk]
    S = np.where(allowed, S, -np.inf)
    cols = S if sink is None else np.concatenate([S, np.full((S.shape[0], 1), sink)], axis=1)
    m = cols.max(axis=1, keepdims=True)
    e = np.exp(cols - m)
    z = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(z))[:, 0]
    probs = e / z
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


def gqa(q, k, v, dout, scale, causal=True, window=0, cu_seqlens=None, sink=None):
    """Full GQA forward+backward for [B,H,S,D] float64 arrays via per-head MHA."""
    B, Hq, S, _ = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    allowed = mask_matrix(S, causal, window, cu_seqlens)
    out = dict(
        o=np.zeros((B, Hq, S, v.shape[3])), lse=np.zeros((B, Hq, S)), delta=np.zeros((B, Hq, S)),
        dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v), dsink=np.zeros(Hq),
        P=np.zeros((B, Hq, S, S)), dS=np.zeros((B, Hq, S, S)), dP=np.zeros((B, Hq, S, S)),
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
