"""The no-allocation backward entry point, called through the C ABI.

gqa_attn_bwd_noalloc exists for callers that cannot allocate device memory
(for example code running inside a CUDA graph capture that forbids cudaMalloc,
or a runtime whose device memory is fixed at start-up): it keeps its scratch in
a fixed device array inside the library instead of a caller workspace.  This
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


def test_noalloc_matches_workspace_path_twice():
    fn = _noalloc_fn()
    dev = torch.device("cuda")
    w = W.Workload("noalloc", 20, B=1, Hq=4, Hkv=2, S=300, Dqk=64, Dv=64, dtype=torch.float16)
    q, k, v, do, _ = (t.to(dev) if t is not None else None for t in W.make_inputs(w))
    o, lse = attention_forward(q, k, v, causal=True, scale=w.resolved_scale)
    ref = attention_backward(q, k, v, o, lse, do, causal=True, scale=w.resolved_scale)
    p = nat.make_params(w.B, w.Hq, w.Hkv, w.S, w.Dqk, w.Dv, w.dtype, causal=True, scale=w.resolved_scale)
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


def test_noalloc_rejects_problems_beyond_its_scratch():
    fn = _noalloc_fn()
    # fp32 dQ accumulator alone: 1 * 32 * 32768 * 64 * 4 bytes = 256 MiB > 16 MiB
    p = nat.make_params(1, 32, 8, 32768, 64, 64, torch.float16, causal=True)
    fake = 1 << 20
    st = fn(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, None)
    assert st == nat.GQA_ERR_WORKSPACE
