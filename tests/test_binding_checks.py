"""The binding's checks of what the C ABI cannot see through raw pointers (dtype, shape, device and
contiguity of every tensor): a tensor of the wrong dtype would otherwise be read as the right one.
CPU tensors throughout; the checks run before any call into the library."""
import pytest
import torch

import gqa_flashattention_backward_gb300 as pkg

B, HQ, HKV, S, SK, DQK, DV = 2, 4, 2, 16, 24, 64, 32


def _good():
    f16, f32 = torch.float16, torch.float32
    q = torch.zeros(B, HQ, S, DQK, dtype=f16)
    k = torch.zeros(B, HKV, SK, DQK, dtype=f16)
    v = torch.zeros(B, HKV, SK, DV, dtype=f16)
    named = dict(o=torch.zeros(B, HQ, S, DV, dtype=f16), do=torch.zeros(B, HQ, S, DV, dtype=f16),
                 dq=torch.zeros(B, HQ, S, DQK, dtype=f16), dk=torch.zeros(B, HKV, SK, DQK, dtype=f16),
                 dv=torch.zeros(B, HKV, SK, DV, dtype=f16), lse=torch.zeros(B, HQ, S, dtype=f32),
                 delta=torch.zeros(B, HQ, S, dtype=f32), sink=torch.zeros(HQ, dtype=f32),
                 dsink=torch.zeros(HQ, dtype=f32))
    return q, k, v, named


def test_consistent_tensors_pass():
    q, k, v, named = _good()
    pkg._validate(q, k, v, **named)
    # layouts other than BHSD (a BSHD view) and packed offsets
    qs = torch.zeros(B, S, HQ, DQK, dtype=torch.float16).transpose(1, 2)
    pkg._validate(qs, k, v, o=torch.zeros(B, S, HQ, DV, dtype=torch.float16).transpose(1, 2))
    cu = torch.tensor([0, 5, 16], dtype=torch.int32)
    pkg._validate(q[:1], k[:1], v[:1], cu_seqlens=cu, cu_seqlens_k=torch.tensor([0, 9, 24], dtype=torch.int32))


@pytest.mark.parametrize("name, bad, match", [
    ("do", torch.zeros(B, HQ, S, DV, dtype=torch.float32), "do must be torch.float16"),
    ("o", torch.zeros(B, HQ, S, DV, dtype=torch.bfloat16), "o must be torch.float16"),
    ("o", torch.zeros(B, HQ, S, DQK, dtype=torch.float16), "o must have shape"),
    ("lse", torch.zeros(B, HQ, S, dtype=torch.float16), "lse must be torch.float32"),
    ("lse", torch.zeros(B, S, HQ, dtype=torch.float32).transpose(1, 2), "lse must be contiguous"),
    ("delta", torch.zeros(B, HQ, S + 1, dtype=torch.float32), "delta must have shape"),
    ("sink", torch.zeros(HQ, dtype=torch.float16), "sink must be torch.float32"),
    ("sink", torch.zeros(HKV, dtype=torch.float32), "sink must have shape"),
    ("dk", torch.zeros(B, HQ, SK, DQK, dtype=torch.float16), "dk must have shape"),
    ("dv", torch.zeros(B, HKV, S, DV, dtype=torch.float16), "dv must have shape"),
    ("cu_seqlens", torch.tensor([0, 5, 16], dtype=torch.int64), "cu_seqlens must be torch.int32"),
    ("cu_seqlens", torch.tensor([16], dtype=torch.int32), "at least two offsets"),
])
def test_mismatch_is_rejected(name, bad, match):
    q, k, v, named = _good()
    named[name] = bad
    with pytest.raises(ValueError, match=match):
        pkg._validate(q, k, v, **named)


def test_kv_shapes_and_offsets():
    q, k, v, _ = _good()
    with pytest.raises(ValueError, match="do not match q"):
        pkg._validate(q, k[..., :32], v)
    with pytest.raises(ValueError, match="do not match q"):
        pkg._validate(q, k, v[:, :, :SK - 1])
    cu = torch.tensor([0, 5, 16], dtype=torch.int32)
    with pytest.raises(ValueError, match="as many offsets"):
        pkg._validate(q[:1], k[:1], v[:1], cu_seqlens=cu, cu_seqlens_k=torch.tensor([0, 24], dtype=torch.int32))
