"""ctypes front-end of the fp64 C oracle (gqa_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module.  It shares no code with the
CUDA path: inputs arrive as numpy arrays (already rounded to the input dtype by
the caller and upcast to float64), outputs are float64.

Every function here follows the definitions written at the top of
``gqa_oracle.c`` (forward with attention sink: tilelang-ascend PR #1638; the
backward formulas k1..k5 and "Kernel 9: Dsink" of the same PR; the group
mapping ``bx // groups`` of tilelang PR #1093).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB = os.path.join(_HERE, "libgqa_oracle.so")
# Another build of gqa_oracle.c to load instead of the one above: the mutation test points this at
# copies with a mistake planted in them and checks that the oracle's pins reject every one.
_LIB_OVERRIDE = os.environ.get("GQA_ORACLE_LIB")


def build_oracle(force: bool = False) -> str:
    """Compile gqa_oracle.c into oracle/libgqa_oracle.so (plain gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("S", ctypes.c_int),
        ("Dqk", ctypes.c_int), ("Dv", ctypes.c_int), ("causal", ctypes.c_int), ("window", ctypes.c_int),
        ("scale", ctypes.c_double), ("nseq", ctypes.c_int),
        ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)), ("sink", ctypes.POINTER(ctypes.c_double)),
        ("Sk", ctypes.c_int), ("cu_seqlens_k", ctypes.POINTER(ctypes.c_int32)), ("window_right", ctypes.c_int),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(_LIB_OVERRIDE or build_oracle())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        pp = ctypes.POINTER(_Problem)
        _lib.oracle_forward.argtypes = [pp, dp, dp, dp, dp, dp]
        _lib.oracle_backward.argtypes = [pp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
        _lib.oracle_delta.argtypes = [pp, dp, dp, dp]
        _lib.oracle_sample_rows.argtypes = [pp, dp, dp, dp, dp, ctypes.c_int, ip, ip, ip, dp, dp, dp, dp]
        _lib.oracle_sample_cols.argtypes = [pp, dp, dp, dp, dp, ctypes.c_int, ip, ip, ip, dp, dp]
        _lib.oracle_row_stats.argtypes = [pp, dp, dp, dp, dp, ctypes.c_int, ip, ip, ip, dp, dp]
        _lib.oracle_cols_with_stats.argtypes = [pp, dp, dp, dp, dp, dp, dp, ctypes.c_int, ip, ip, ip, dp, dp]
        _lib.oracle_dsink.argtypes = [pp, dp, dp, dp]
    return _lib


@dataclass
class Problem:
    """Shapes and masking of one attention problem (layout [B, H, S, D]; k / v have Sk rows).

    With Sk != S (or key offsets cu_seqlens_k different from cu_seqlens) the causal diagonal
    is aligned at the bottom right: query i of a sequence sees key j iff j <= i + (Lk - Lq)."""
    B: int
    Hq: int
    Hkv: int
    S: int
    Dqk: int
    Dv: int
    causal: bool = True
    window: int = 0
    scale: Optional[float] = None
    cu_seqlens: Optional[Sequence[int]] = None
    Sk: Optional[int] = None
    cu_seqlens_k: Optional[Sequence[int]] = None
    window_right: int = 0   # > 0 (not causal): keys j with j - (i + Lk - Lq) < window_right

    def resolved_scale(self) -> float:
        return float(self.scale) if self.scale is not None else 1.0 / np.sqrt(self.Dqk)

    @property
    def key_len(self) -> int:
        return int(self.Sk) if self.Sk else int(self.S)


def _dp(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a: np.ndarray):
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _mk(pb: Problem, sink: Optional[np.ndarray], keep: list):
    st = _Problem()
    st.B, st.Hq, st.Hkv, st.S, st.Dqk, st.Dv = pb.B, pb.Hq, pb.Hkv, pb.S, pb.Dqk, pb.Dv
    st.causal = int(bool(pb.causal))
    st.window = int(pb.window)
    st.scale = pb.resolved_scale()
    if pb.cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(pb.cu_seqlens, dtype=np.int32))
        keep.append(cu)
        st.nseq = len(cu) - 1
        st.cu_seqlens = _ip(cu)
    else:
        st.nseq = 0
        st.cu_seqlens = ctypes.POINTER(ctypes.c_int32)()
    if sink is not None:
        s = np.ascontiguousarray(sink, dtype=np.float64)
        keep.append(s)
        st.sink = _dp(s)
    else:
        st.sink = ctypes.POINTER(ctypes.c_double)()
    st.Sk = pb.key_len
    st.window_right = int(pb.window_right)
    if pb.cu_seqlens_k is not None:
        ck = np.ascontiguousarray(np.asarray(pb.cu_seqlens_k, dtype=np.int32))
        keep.append(ck)
        st.cu_seqlens_k = _ip(ck)
    else:
        st.cu_seqlens_k = ctypes.POINTER(ctypes.c_int32)()
    return st


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def forward(pb: Problem, q, k, v, sink=None):
    """O [B,Hq,S,Dv] and LSE [B,Hq,S] (natural log, sink included)."""
    lib, keep = _load(), []
    q, k, v = _f64(q), _f64(k), _f64(v)
    st = _mk(pb, sink, keep)
    o = np.zeros((pb.B, pb.Hq, pb.S, pb.Dv))
    lse = np.zeros((pb.B, pb.Hq, pb.S))
    lib.oracle_forward(ctypes.byref(st), _dp(q), _dp(k), _dp(v), _dp(o), _dp(lse))
    return o, lse


def backward(pb: Problem, q, k, v, o, lse, dout, sink=None):
    """dict with delta, dq, dk, dv and (with a sink) dsink."""
    lib, keep = _load(), []
    q, k, v, o, lse, dout = map(_f64, (q, k, v, o, lse, dout))
    st = _mk(pb, sink, keep)
    delta = np.zeros((pb.B, pb.Hq, pb.S))
    dq = np.zeros((pb.B, pb.Hq, pb.S, pb.Dqk))
    dk = np.zeros((pb.B, pb.Hkv, pb.key_len, pb.Dqk))
    dv = np.zeros((pb.B, pb.Hkv, pb.key_len, pb.Dv))
    dsink = np.zeros(pb.Hq)
    lib.oracle_backward(ctypes.byref(st), _dp(q), _dp(k), _dp(v), _dp(o), _dp(lse), _dp(dout), _dp(delta),
                        _dp(dq), _dp(dk), _dp(dv), _dp(dsink))
    out = dict(delta=delta, dq=dq, dk=dk, dv=dv)
    if sink is not None:
        out["dsink"] = dsink
    return out


def sample_rows(pb: Problem, q, k, v, dout, bs, hs, is_, sink=None):
    """Exact LSE, O, Delta, dQ at the listed query rows (b, h, i)."""
    lib, keep = _load(), []
    q, k, v, dout = map(_f64, (q, k, v, dout))
    st = _mk(pb, sink, keep)
    bs, hs, is_ = (np.ascontiguousarray(x, dtype=np.int32) for x in (bs, hs, is_))
    n = len(bs)
    lse = np.zeros(n)
    o = np.zeros((n, pb.Dv))
    delta = np.zeros(n)
    dq = np.zeros((n, pb.Dqk))
    lib.oracle_sample_rows(ctypes.byref(st), _dp(q), _dp(k), _dp(v), _dp(dout), n, _ip(bs), _ip(hs), _ip(is_),
                           _dp(lse), _dp(o), _dp(delta), _dp(dq))
    return dict(lse=lse, o=o, delta=delta, dq=dq)


def sample_cols(pb: Problem, q, k, v, dout, bs, gs, js, sink=None):
    """Exact dK, dV at the listed key rows (b, kv head g, j)."""
    lib, keep = _load(), []
    q, k, v, dout = map(_f64, (q, k, v, dout))
    st = _mk(pb, sink, keep)
    bs, gs, js = (np.ascontiguousarray(x, dtype=np.int32) for x in (bs, gs, js))
    n = len(bs)
    dk = np.zeros((n, pb.Dqk))
    dv = np.zeros((n, pb.Dv))
    lib.oracle_sample_cols(ctypes.byref(st), _dp(q), _dp(k), _dp(v), _dp(dout), n, _ip(bs), _ip(gs), _ip(js),
                           _dp(dk), _dp(dv))
    return dict(dk=dk, dv=dv)


def row_stats(pb: Problem, q, k, v, dout, bs, hs, is_, sink=None):
    """Exact LSE and Delta at the listed query rows (b, h, i) (row-parallel; no dQ)."""
    lib, keep = _load(), []
    q, k, v, dout = map(_f64, (q, k, v, dout))
    st = _mk(pb, sink, keep)
    bs, hs, is_ = (np.ascontiguousarray(x, dtype=np.int32) for x in (bs, hs, is_))
    n = len(bs)
    lse = np.zeros(n)
    delta = np.zeros(n)
    lib.oracle_row_stats(ctypes.byref(st), _dp(q), _dp(k), _dp(v), _dp(dout), n, _ip(bs), _ip(hs), _ip(is_),
                         _dp(lse), _dp(delta))
    return dict(lse=lse, delta=delta)


def cols_with_stats(pb: Problem, q, k, v, dout, lse, delta, bs, gs, js, sink=None):
    """Exact dK, dV at the listed key rows (b, g, j), given LSE and Delta [B, Hq, S] of (at least)
    every query row that sees one of them."""
    lib, keep = _load(), []
    q, k, v, dout, lse, delta = map(_f64, (q, k, v, dout, lse, delta))
    st = _mk(pb, sink, keep)
    bs, gs, js = (np.ascontiguousarray(x, dtype=np.int32) for x in (bs, gs, js))
    n = len(bs)
    dk = np.zeros((n, pb.Dqk))
    dv = np.zeros((n, pb.Dv))
    lib.oracle_cols_with_stats(ctypes.byref(st), _dp(q), _dp(k), _dp(v), _dp(dout), _dp(lse), _dp(delta), n,
                               _ip(bs), _ip(gs), _ip(js), _dp(dk), _dp(dv))
    return dict(dk=dk, dv=dv)


def dsink(pb: Problem, lse, delta, sink):
    """dsink [Hq] from full LSE and Delta [B, Hq, S]."""
    lib, keep = _load(), []
    lse, delta = _f64(lse), _f64(delta)
    st = _mk(pb, sink, keep)
    out = np.zeros(pb.Hq)
    lib.oracle_dsink(ctypes.byref(st), _dp(lse), _dp(delta), _dp(out))
    return out
