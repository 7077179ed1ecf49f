"""ctypes binding of libgqa_attn.so (the C ABI in include/gqa_attn.h).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  Tensors are PyTorch tensors used as device buffers; their
``data_ptr()`` and the current CUDA stream are handed to the C entry points.
If the library has not been built the first call raises -- there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgqa_attn.so")

GQA_OK = 0
GQA_ERR_INVALID_ARG = -1
GQA_ERR_UNSUPPORTED = -2
GQA_ERR_WORKSPACE = -3
GQA_ERR_CUDA = -4
GQA_ERR_DEVICE_TIMEOUT = -5
GQA_ERR_DEVICE_INPUT = -6

GQA_F16, GQA_BF16 = 0, 1
GQA_GROUP_TMEM, GQA_GROUP_ATOMIC = 0, 1
GQA_RED_V4, GQA_RED_BULK, GQA_RED_SCALAR, GQA_RED_NONE = 0, 1, 2, 3

EXPORTS = (
    "gqa_attn_workspace_size", "gqa_attn_fwd", "gqa_attn_bwd_preprocess", "gqa_attn_bwd",
    "gqa_attn_bwd_postprocess", "gqa_attn_dsink", "gqa_attn_get_device_error", "gqa_attn_set_wait_limit",
    "gqa_attn_selftest_wait_timeout", "gqa_attn_strerror", "gqa_attn_bwd_noalloc", "gqa_attn_params_size",
    "gqa_attn_noalloc_get_device_error",
)


class GqaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} ({status})")


class Stride(ctypes.Structure):
    """gqa_stride: element strides along batch, head, sequence ({0,0,0} = contiguous BHSD)."""
    _fields_ = [("b", ctypes.c_int64), ("h", ctypes.c_int64), ("s", ctypes.c_int64)]


STRIDE_FIELDS = ("q_st", "k_st", "v_st", "o_st", "do_st", "dq_st", "dk_st", "dv_st")


class Params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("S", ctypes.c_int),
        ("Dqk", ctypes.c_int), ("Dv", ctypes.c_int), ("dtype", ctypes.c_int), ("causal", ctypes.c_int),
        ("window", ctypes.c_int), ("scale", ctypes.c_float), ("cu_seqlens", ctypes.c_void_p),
        ("nseq", ctypes.c_int), ("max_seqlen", ctypes.c_int), ("group_mode", ctypes.c_int),
        ("red_mode", ctypes.c_int), ("deterministic", ctypes.c_int),
    ] + [(n, Stride) for n in STRIDE_FIELDS] + [
        ("Sk", ctypes.c_int), ("cu_seqlens_k", ctypes.c_void_p), ("max_seqlen_k", ctypes.c_int),
        ("window_right", ctypes.c_int),
    ]


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load the shared library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing: build it with `python -m gqa_flashattention_backward_gb300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.POINTER(Params)
    vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    lib.gqa_attn_workspace_size.argtypes = [P]
    lib.gqa_attn_workspace_size.restype = sz
    lib.gqa_attn_params_size.argtypes = []
    lib.gqa_attn_params_size.restype = sz
    if lib.gqa_attn_params_size() != ctypes.sizeof(Params):
        raise ImportError(f"gqa_attn_params is {lib.gqa_attn_params_size()} bytes in {_LIB_PATH}, "
                          f"{ctypes.sizeof(Params)} in this binding: rebuild the library")
    lib.gqa_attn_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.gqa_attn_fwd.restype = st
    lib.gqa_attn_bwd_preprocess.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
    lib.gqa_attn_bwd_preprocess.restype = st
    lib.gqa_attn_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.gqa_attn_bwd.restype = st
    lib.gqa_attn_bwd_postprocess.argtypes = [P, vp, vp, vp, vp, sz, vp]
    lib.gqa_attn_bwd_postprocess.restype = st
    lib.gqa_attn_dsink.argtypes = [P, vp, vp, vp, vp, vp]
    lib.gqa_attn_dsink.restype = st
    lib.gqa_attn_get_device_error.argtypes = [vp, sz, vp, ctypes.POINTER(ctypes.c_int)]
    lib.gqa_attn_get_device_error.restype = st
    lib.gqa_attn_set_wait_limit.argtypes = [ctypes.c_longlong]
    lib.gqa_attn_set_wait_limit.restype = None
    lib.gqa_attn_selftest_wait_timeout.argtypes = [vp, sz, vp]
    lib.gqa_attn_selftest_wait_timeout.restype = st
    lib.gqa_attn_strerror.argtypes = [st]
    lib.gqa_attn_strerror.restype = ctypes.c_char_p
    _lib = lib
    return lib


def strerror(status: int) -> str:
    return load().gqa_attn_strerror(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, what: str):
    if status != GQA_OK:
        raise GqaError(status, what)


def make_params(B, Hq, Hkv, S, Dqk, Dv, dtype, causal=True, window=0, scale=None, cu_seqlens=None,
                max_seqlen=None, group_mode=GQA_GROUP_TMEM, red_mode=GQA_RED_V4, deterministic=False,
                strides=None, Sk=None, cu_seqlens_k=None, max_seqlen_k=None, window_right=0) -> Params:
    """Build the parameter struct.  `dtype` is a torch dtype (float16/bfloat16);
    `cu_seqlens` a device int32 tensor or None; `strides` maps some of "q", "k", "v", "o", "do",
    "dq", "dk", "dv" to (batch, head, sequence) element strides (missing: contiguous BHSD)."""
    p = Params()
    p.B, p.Hq, p.Hkv, p.S, p.Dqk, p.Dv = int(B), int(Hq), int(Hkv), int(S), int(Dqk), int(Dv)
    p.dtype = GQA_BF16 if dtype == torch.bfloat16 else (GQA_F16 if dtype == torch.float16 else -1)
    p.causal = int(bool(causal))
    p.window = int(window)
    p.scale = float(scale) if scale is not None else float(Dqk) ** -0.5
    if cu_seqlens is not None:
        p.cu_seqlens = cu_seqlens.data_ptr()
        p.nseq = cu_seqlens.numel() - 1
        p.max_seqlen = int(max_seqlen) if max_seqlen is not None else int(S)
    else:
        p.cu_seqlens = None
        p.nseq = 0
        p.max_seqlen = 0
    p.group_mode = int(group_mode)
    p.red_mode = int(red_mode)
    p.deterministic = int(bool(deterministic))
    p.Sk = int(Sk) if Sk is not None and int(Sk) != int(S) else 0
    p.cu_seqlens_k = cu_seqlens_k.data_ptr() if cu_seqlens_k is not None else None
    p.max_seqlen_k = int(max_seqlen_k) if max_seqlen_k is not None else 0
    p.window_right = int(window_right)
    for name, st in (strides or {}).items():
        s = getattr(p, name + "_st")
        s.b, s.h, s.s = (int(x) for x in st)
    return p


def tensor_strides(t: torch.Tensor):
    """(batch, head, sequence) element strides of a [B, H, S, D] tensor whose last dim is contiguous."""
    if t.dim() != 4 or (t.stride(3) != 1 and t.shape[3] > 1):
        raise ValueError("tensors must be [B, H, S, D] with a contiguous head dim")
    _, H, S, D = t.shape
    default = (H * S * D, S * D, D)
    # a dim of size 1 (or an empty tensor) may carry any stride: the kernels never step along it
    return tuple(default[i] if t.shape[i] <= 1 or t.numel() == 0 else t.stride(i) for i in range(3))


def workspace_size(p: Params) -> int:
    return int(load().gqa_attn_workspace_size(ctypes.byref(p)))


def alloc_workspace(p: Params, device="cuda") -> torch.Tensor:
    n = workspace_size(p)
    if n == 0:
        raise GqaError(GQA_ERR_INVALID_ARG, "workspace_size")
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    out = ws[off:off + n]
    out.zero_()
    return out


def fwd(p: Params, q, k, v, sink, o, lse, ws, stream=None):
    _check(load().gqa_attn_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(o), _ptr(lse),
                               _ptr(ws), ws.numel(), _stream(stream)), "gqa_attn_fwd")


def bwd_preprocess(p: Params, o, dout, lse, delta, ws, stream=None):
    _check(load().gqa_attn_bwd_preprocess(ctypes.byref(p), _ptr(o), _ptr(dout), _ptr(lse), _ptr(delta), _ptr(ws),
                                          ws.numel(), _stream(stream)), "gqa_attn_bwd_preprocess")


def bwd(p: Params, q, k, v, dout, dq, dk, dv, ws, stream=None):
    _check(load().gqa_attn_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                               _ptr(ws), ws.numel(), _stream(stream)), "gqa_attn_bwd")


def bwd_postprocess(p: Params, dq, dk, dv, ws, stream=None):
    _check(load().gqa_attn_bwd_postprocess(ctypes.byref(p), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(),
                                           _stream(stream)), "gqa_attn_bwd_postprocess")


def dsink(p: Params, sink, lse, delta, out, stream=None):
    _check(load().gqa_attn_dsink(ctypes.byref(p), _ptr(sink), _ptr(lse), _ptr(delta), _ptr(out), _stream(stream)),
           "gqa_attn_dsink")


def get_device_error(ws, stream=None):
    site = ctypes.c_int(0)
    st = load().gqa_attn_get_device_error(_ptr(ws), ws.numel(), _stream(stream), ctypes.byref(site))
    return int(st), int(site.value)


def set_wait_limit(cycles: int):
    load().gqa_attn_set_wait_limit(int(cycles))


def selftest_wait_timeout(ws, stream=None):
    _check(load().gqa_attn_selftest_wait_timeout(_ptr(ws), ws.numel(), _stream(stream)),
           "gqa_attn_selftest_wait_timeout")
