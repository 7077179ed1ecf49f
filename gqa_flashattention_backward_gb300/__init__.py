"""GB300 (sm_103a) grouped-query FlashAttention forward and backward.

The computation lives in ``libgqa_attn.so`` (hand-written CUDA behind the C ABI
of ``include/gqa_attn.h``); this package only marshals PyTorch device tensors
into those calls.  The two helpers below chain the entry points in the order
the C ABI prescribes:

* :func:`attention_forward`  -> ``gqa_attn_fwd``
* :func:`attention_backward` -> ``gqa_attn_bwd_preprocess``, ``gqa_attn_bwd``,
  ``gqa_attn_bwd_postprocess`` and (with a sink) ``gqa_attn_dsink``.
* :func:`gqa_attention` -> both, as a ``torch.autograd.Function`` (O from the
  forward, dQ / dK / dV / dsink from the backward when autograd asks for them).
* :class:`GraphedBackward` -> the backward chain of fixed shapes captured once as a
  CUDA graph and replayed with one launch (small, launch-bound problems).

Tensors have shape q [B,Hq,S,Dqk], k [B,Hkv,S,Dqk], v [B,Hkv,S,Dv], o/dout [B,Hq,S,Dv]
and any layout whose head dim is contiguous (BHSD, a BSHD view ``x.transpose(1, 2)``, packed
THD for varlen as ``x.permute(1, 0, 2).unsqueeze(0)``): the strides go to the kernels, nothing
is copied; outputs take the layout of the matching input.  Packed variable-length batches use
B=1 and ``cu_seqlens``.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _native as native
from ._native import (GQA_GROUP_ATOMIC, GQA_GROUP_TMEM, GQA_RED_BULK, GQA_RED_NONE, GQA_RED_SCALAR,
                      GQA_RED_V4, GqaError)

__all__ = [
    "attention_forward", "attention_backward", "gqa_attention", "GqaAttentionFunction", "GraphedBackward",
    "preferred_red_mode", "native", "GqaError", "GQA_GROUP_TMEM", "GQA_GROUP_ATOMIC",
    "GQA_RED_V4", "GQA_RED_BULK", "GQA_RED_SCALAR", "GQA_RED_NONE",
]


def preferred_red_mode(Dqk: int) -> int:
    """The fastest measured reduction for every supported head dim: the bulk reduce of
    whole tiles staged in shared memory."""
    return GQA_RED_BULK


def _validate(q, k, v, **named):
    """What the C ABI cannot see through its raw pointers: every tensor's dtype, shape and device.
    `named`: any of o, do, dq, dk, dv (q's dtype), lse, delta (fp32 [B, Hq, S], contiguous), sink,
    dsink (fp32 [Hq], contiguous), cu_seqlens, cu_seqlens_k (int32, 1-D, contiguous); None is skipped.
    Raises ValueError naming the first tensor that does not fit."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, S, D]")
    B, Hq, S, Dqk = q.shape
    Hkv, Sk, Dv = k.shape[1], k.shape[2], v.shape[3]
    if k.shape[0] != B or k.shape[3] != Dqk or tuple(v.shape[:3]) != (B, Hkv, Sk):
        raise ValueError(f"k {tuple(k.shape)} and v {tuple(v.shape)} do not match q {tuple(q.shape)}: "
                         "expected k [B, Hkv, Sk, Dqk] and v [B, Hkv, Sk, Dv]")
    f32 = torch.float32
    want = dict(o=((B, Hq, S, Dv), q.dtype, False), do=((B, Hq, S, Dv), q.dtype, False),
                dq=((B, Hq, S, Dqk), q.dtype, False), dk=((B, Hkv, Sk, Dqk), q.dtype, False),
                dv=((B, Hkv, Sk, Dv), q.dtype, False), lse=((B, Hq, S), f32, True), delta=((B, Hq, S), f32, True),
                sink=((Hq,), f32, True), dsink=((Hq,), f32, True), cu_seqlens=(None, torch.int32, True),
                cu_seqlens_k=(None, torch.int32, True))
    for name, t in named.items():
        if t is None:
            continue
        shape, dtype, contiguous = want[name]
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
        if t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        if shape is None:  # sequence offsets: nseq + 1 entries
            if t.dim() != 1 or t.numel() < 2:
                raise ValueError(f"{name} must be 1-D with at least two offsets")
        elif tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
        if contiguous and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    cu, cuk = named.get("cu_seqlens"), named.get("cu_seqlens_k")
    if cuk is not None and (cu is None or cuk.numel() != cu.numel()):
        raise ValueError("cu_seqlens_k needs cu_seqlens with as many offsets")


def _params(q, k, v, causal, window, scale, cu_seqlens, max_seqlen, group_mode=GQA_GROUP_TMEM,
            red_mode=None, deterministic=False, cu_seqlens_k=None, max_seqlen_k=None, window_right=0, **tensors):
    """`tensors`: any of o, do, dq, dk, dv whose layouts the call uses.  k / v may have another
    length than q (k.shape[2]): the causal diagonal is then aligned at the bottom right."""
    B, Hq, S, Dqk = q.shape
    if red_mode is None:
        red_mode = preferred_red_mode(Dqk)
    Hkv, Dv = k.shape[1], v.shape[3]
    for t in (q, k, v):
        if not (t.is_cuda and t.dtype == q.dtype):
            raise ValueError("q, k, v must be CUDA tensors of one dtype")
    named = dict(q=q, k=k, v=v, **{n: t for n, t in tensors.items() if t is not None})
    strides = {n: native.tensor_strides(t) for n, t in named.items()}
    return native.make_params(B, Hq, Hkv, S, Dqk, Dv, q.dtype, causal=causal, window=window, scale=scale,
                              cu_seqlens=cu_seqlens, max_seqlen=max_seqlen, group_mode=group_mode,
                              red_mode=red_mode, deterministic=deterministic, strides=strides, Sk=k.shape[2],
                              cu_seqlens_k=cu_seqlens_k, max_seqlen_k=max_seqlen_k, window_right=window_right)


def _empty_like_layout(ref: torch.Tensor, last_dim: int) -> torch.Tensor:
    """An uninitialised [B, H, S, last_dim] tensor whose dims are ordered in memory like ref's."""
    order = sorted(range(3), key=lambda i: -ref.stride(i))  # outermost first
    shape = [ref.shape[i] for i in order] + [last_dim]
    t = torch.empty(shape, dtype=ref.dtype, device=ref.device)
    inv = [order.index(i) for i in range(3)] + [3]
    return t.permute(*inv)


def attention_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, causal: bool = True, window: int = 0,
                      scale: Optional[float] = None, sink: Optional[torch.Tensor] = None,
                      cu_seqlens: Optional[torch.Tensor] = None, max_seqlen: Optional[int] = None,
                      cu_seqlens_k: Optional[torch.Tensor] = None, max_seqlen_k: Optional[int] = None,
                      window_right: int = 0, workspace: Optional[torch.Tensor] = None):
    """Returns (o, lse): o [B,Hq,S,Dv] in q's dtype, lse [B,Hq,S] fp32 (natural log, sink included)."""
    _validate(q, k, v, sink=sink, cu_seqlens=cu_seqlens, cu_seqlens_k=cu_seqlens_k)
    B, Hq, S, _ = q.shape
    o = _empty_like_layout(q, v.shape[3])
    p = _params(q, k, v, causal, window, scale, cu_seqlens, max_seqlen, cu_seqlens_k=cu_seqlens_k,
                max_seqlen_k=max_seqlen_k, window_right=window_right, o=o)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    ws = workspace if workspace is not None else native.alloc_workspace(p, q.device)
    native.fwd(p, q, k, v, sink, o, lse, ws)
    return o, lse


def attention_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
                       dout: torch.Tensor, *, causal: bool = True, window: int = 0, scale: Optional[float] = None,
                       sink: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None,
                       max_seqlen: Optional[int] = None, group_mode: int = GQA_GROUP_TMEM,
                       red_mode: Optional[int] = None, deterministic: bool = False,
                       cu_seqlens_k: Optional[torch.Tensor] = None, max_seqlen_k: Optional[int] = None,
                       window_right: int = 0, workspace: Optional[torch.Tensor] = None,
                       out: Optional[dict] = None) -> dict:
    """Returns dict(dq, dk, dv, delta[, dsink]).  `out` may hold preallocated tensors of the same names.
    red_mode None picks :func:`preferred_red_mode`."""
    res = dict(out) if out else {}
    _validate(q, k, v, o=o, do=dout, lse=lse, sink=sink, cu_seqlens=cu_seqlens, cu_seqlens_k=cu_seqlens_k,
              **{n: t for n, t in res.items() if n in ("dq", "dk", "dv", "delta", "dsink")})
    B, Hq, S, Dqk = q.shape
    Hkv, Dv = k.shape[1], v.shape[3]
    dev = q.device
    if "dq" not in res:
        res["dq"] = _empty_like_layout(q, Dqk)
    if "dk" not in res:
        res["dk"] = _empty_like_layout(k, Dqk)
    if "dv" not in res:
        res["dv"] = _empty_like_layout(v, Dv)
    p = _params(q, k, v, causal, window, scale, cu_seqlens, max_seqlen, group_mode, red_mode, deterministic,
                cu_seqlens_k=cu_seqlens_k, max_seqlen_k=max_seqlen_k, window_right=window_right, o=o, do=dout,
                dq=res["dq"], dk=res["dk"], dv=res["dv"])
    if "delta" not in res:
        res["delta"] = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    if sink is not None and "dsink" not in res:
        res["dsink"] = torch.empty((Hq,), dtype=torch.float32, device=dev)
    ws = workspace if workspace is not None else native.alloc_workspace(p, dev)
    native.bwd_preprocess(p, o, dout, lse, res["delta"], ws)
    native.bwd(p, q, k, v, dout, res["dq"], res["dk"], res["dv"], ws)
    native.bwd_postprocess(p, res["dq"], res["dk"], res["dv"], ws)
    if sink is not None:
        native.dsink(p, sink, lse, res["delta"], res["dsink"])
    return res


class GqaAttentionFunction(torch.autograd.Function):
    """Autograd wrapper: the forward saves Q, K, V, O and LSE; the backward runs the four
    backward entry points on them.  Every step runs in the CUDA library."""

    @staticmethod
    def forward(ctx, q, k, v, sink, causal, window, scale, cu_seqlens, max_seqlen, deterministic, cu_seqlens_k=None,
                max_seqlen_k=None, window_right=0):
        o, lse = attention_forward(q, k, v, causal=causal, window=window, scale=scale, sink=sink,
                                   cu_seqlens=cu_seqlens, max_seqlen=max_seqlen, cu_seqlens_k=cu_seqlens_k,
                                   max_seqlen_k=max_seqlen_k, window_right=window_right)
        ctx.save_for_backward(q, k, v, o, lse, sink)
        ctx.opts = dict(causal=causal, window=window, scale=scale, cu_seqlens=cu_seqlens, max_seqlen=max_seqlen,
                        deterministic=deterministic, cu_seqlens_k=cu_seqlens_k, max_seqlen_k=max_seqlen_k,
                        window_right=window_right)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, sink = ctx.saved_tensors
        g = attention_backward(q, k, v, o, lse, do.contiguous(), sink=sink, **ctx.opts)
        dsink = g.get("dsink") if sink is not None and ctx.needs_input_grad[3] else None
        return g["dq"], g["dk"], g["dv"], dsink, None, None, None, None, None, None, None, None, None


def gqa_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, causal: bool = True, window: int = 0,
                  scale: Optional[float] = None, sink: Optional[torch.Tensor] = None,
                  cu_seqlens: Optional[torch.Tensor] = None, max_seqlen: Optional[int] = None,
                  deterministic: bool = False, cu_seqlens_k: Optional[torch.Tensor] = None,
                  max_seqlen_k: Optional[int] = None, window_right: int = 0) -> torch.Tensor:
    """Differentiable grouped-query attention: returns O [B,Hq,S,Dv]; ``O.backward(dO)`` fills
    q.grad, k.grad, v.grad (and sink.grad, fp32) through the backward kernels."""
    return GqaAttentionFunction.apply(q, k, v, sink, causal, window, scale, cu_seqlens, max_seqlen, deterministic,
                                      cu_seqlens_k, max_seqlen_k, window_right)


class GraphedBackward:
    """The backward of fixed shapes (preprocess, main kernel, postprocess and, with a sink, the sink
    gradient) captured once as a CUDA graph; :meth:`replay` runs all of it with one graph launch on
    the current stream.  The graph reads and writes the very tensors it was built with: copy new
    q, k, v, o, lse, dout (and sink) into them in place before a replay; the results are in
    :attr:`out` (dq, dk, dv, delta[, dsink]).  Keyword arguments are those of attention_backward."""

    def __init__(self, q, k, v, o, lse, dout, **kw):
        if "out" in kw or "workspace" in kw:
            raise ValueError("GraphedBackward owns its outputs and workspace")
        self.tensors = (q, k, v, o, lse, dout)
        self.kw = kw  # keeps sink / cu_seqlens alive: the graph holds their addresses
        B, Hq, S, Dqk = q.shape
        self.out = dict(dq=_empty_like_layout(q, Dqk), dk=_empty_like_layout(k, Dqk),
                        dv=_empty_like_layout(v, v.shape[3]),
                        delta=torch.empty((B, Hq, S), dtype=torch.float32, device=q.device))
        if kw.get("sink") is not None:
            self.out["dsink"] = torch.empty((Hq,), dtype=torch.float32, device=q.device)
        p = _params(q, k, v, kw.get("causal", True), kw.get("window", 0), kw.get("scale"), kw.get("cu_seqlens"),
                    kw.get("max_seqlen"), kw.get("group_mode", GQA_GROUP_TMEM), kw.get("red_mode"),
                    kw.get("deterministic", False), cu_seqlens_k=kw.get("cu_seqlens_k"),
                    max_seqlen_k=kw.get("max_seqlen_k"), window_right=kw.get("window_right", 0))
        self.workspace = native.alloc_workspace(p, q.device)
        side = torch.cuda.Stream(device=q.device)
        side.wait_stream(torch.cuda.current_stream(q.device))
        with torch.cuda.stream(side):  # one eager run first: kernel attributes, lazy module loading
            self._run()
        torch.cuda.current_stream(q.device).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        # the library does host-side setup (tensor maps, kernel attributes) between its launches
        with torch.cuda.graph(self.graph, capture_error_mode="relaxed"):
            self._run()

    def _run(self):
        q, k, v, o, lse, dout = self.tensors
        attention_backward(q, k, v, o, lse, dout, workspace=self.workspace, out=self.out, **self.kw)

    def replay(self) -> dict:
        self.graph.replay()
        return self.out
