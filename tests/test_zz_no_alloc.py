"""The no-allocation backward entry point, called through the C ABI.

gqa_attn_bwd_noalloc exists for callers that cannot allocate device memory
(for example code running inside a CUDA graph capture that forbids cudaMalloc,
or a runtime whose device memory is fixed at start-up): it keeps its scratch in
a fixed device array inside the library instead of a caller workspace.  Its
device-side errors are read back with gqa_attn_noalloc_get_device_error.  This
file is named so pytest collects it last.
"""
import ctypes

import pytest
import torch

from gqa_flashattention_backward_gb300 import _native as nat
from gqa_flashattention_backward_gb300 import attention_backward, attention_forward
from gqa_flashattention_backward_gb300 import workloads as W
from tests._util import assert_close, f64

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    lib = nat.load()
    fn = lib.gqa_attn_bwd_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(nat.Params), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def _noalloc_error():
    fn = nat.load().gqa_attn_noalloc_get_device_error
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    fn.restype = ctypes.c_int
    site = ctypes.c_int(0)
    st = fn(torch.cuda.current_stream().cuda_stream, ctypes.byref(site))
    return st, site.value


@pytest.mark.parametrize("red_mode", [nat.GQA_RED_BULK, nat.GQA_RED_V4])
def test_noalloc_matches_workspace_path_twice(red_mode):
    """Both paths in the same dQ reduction mode (the bulk reduce is what attention_backward picks
    by default and what the benchmark times)."""
    fn = _noalloc_fn()
    dev = torch.device("cuda")
    w = W.Workload("noalloc", 20, B=1, Hq=4, Hkv=2, S=300, Dqk=64, Dv=64, dtype=torch.float16)
    q, k, v, do, _ = (t.to(dev) if t is not None else None for t in W.make_inputs(w))
    o, lse = attention_forward(q, k, v, causal=True, scale=w.resolved_scale)
    ref = attention_backward(q, k, v, o, lse, do, causal=True, scale=w.resolved_scale, red_mode=red_mode)
    p = nat.make_params(w.B, w.Hq, w.Hkv, w.S, w.Dqk, w.Dv, w.dtype, causal=True, scale=w.resolved_scale,
                        red_mode=red_mode)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        dq, dk, dv = torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))
        delta = torch.full_like(lse, float("nan"))
        st = fn(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                lse.data_ptr(), delta.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), stream)
        assert st == nat.GQA_OK, nat.strerror(st)
        torch.cuda.synchronize()
        for name, got in (("dq", dq), ("dk", dk), ("dv", dv), ("delta", delta)):
            assert_close(f"noalloc:{name}", f64(got), f64(ref[name]))
        assert _noalloc_error() == (nat.GQA_OK, 0)


def test_noalloc_reports_device_input_errors():
    """A packed sequence longer than max_seqlen is caught on the device; the caller reads the
    failure back from the library's scratch, and reading clears it."""
    fn = _noalloc_fn()
    dev = torch.device("cuda")
    S = 300
    q = torch.randn(1, 2, S, 64, device=dev, dtype=torch.float16)
    k = torch.randn(1, 1, S, 64, device=dev, dtype=torch.float16)
    v = torch.randn(1, 1, S, 64, device=dev, dtype=torch.float16)
    do = torch.randn(1, 2, S, 64, device=dev, dtype=torch.float16)
    o = torch.randn(1, 2, S, 64, device=dev, dtype=torch.float16)
    lse = torch.zeros(1, 2, S, device=dev)
    cu = torch.tensor([0, 100, 300], dtype=torch.int32, device=dev)
    p = nat.make_params(1, 2, 1, S, 64, 64, torch.float16, cu_seqlens=cu, max_seqlen=150, red_mode=nat.GQA_RED_BULK)
    dq, dk, dv, delta = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(lse)
    st = fn(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
            delta.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == nat.GQA_OK  # launched; the failure is found on the device
    status, site = _noalloc_error()
    assert status == nat.GQA_ERR_DEVICE_INPUT, (status, hex(site))
    assert _noalloc_error() == (nat.GQA_OK, 0)


def test_noalloc_rejects_problems_beyond_its_scratch():
    fn = _noalloc_fn()
    # fp32 dQ accumulator alone: 1 * 32 * 32768 * 64 * 4 bytes = 256 MiB > 16 MiB
    p = nat.make_params(1, 32, 8, 32768, 64, 64, torch.float16, causal=True)
    fake = 1 << 20
    st = fn(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, None)
    assert st == nat.GQA_ERR_WORKSPACE
