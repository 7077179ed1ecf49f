"""C ABI checks that need no GPU: the library loads, exports every function the
header declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

from gqa_flashattention_backward_gb300 import _native as nat

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "gqa_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_attn_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(nat.lib_path()):
        from gqa_flashattention_backward_gb300 import build
        build.build()
    return nat.load()


def test_exports_match_header(lib):
    declared = _header_functions()
    assert declared, "no declarations parsed"
    assert set(declared) == set(nat.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def _p(**kw):
    base = dict(B=2, Hq=8, Hkv=2, S=256, Dqk=64, Dv=64, dtype=None, causal=True, window=0, scale=0.125)
    base.update(kw)
    import torch
    dt = base.pop("dtype") or torch.float16
    return nat.make_params(dtype=dt, **base)


def test_workspace_size_valid_and_invalid(lib):
    assert nat.workspace_size(_p()) > 0
    assert nat.workspace_size(_p(Hq=7, Hkv=2)) == 0          # Hq % Hkv != 0
    assert nat.workspace_size(_p(Dqk=96, Dv=96)) == 0        # unsupported head dim
    assert nat.workspace_size(_p(window=16, causal=False)) == 0
    assert nat.workspace_size(_p(scale=0.0)) == 0
    assert nat.workspace_size(_p(scale=float("nan"))) == 0
    assert nat.workspace_size(_p(B=0)) == 0


def test_workspace_grows_with_accumulators(lib):
    det = nat.workspace_size(_p(deterministic=True))
    tmem = nat.workspace_size(_p())
    atomic = nat.workspace_size(_p(group_mode=nat.GQA_GROUP_ATOMIC))
    # fp32 dQ accumulator: B*Hq*S*Dqk*4 bytes; dK/dV accumulators: B*Hkv*S*(Dqk+Dv)*4
    assert tmem - det == 2 * 8 * 256 * 64 * 4
    assert atomic - tmem == 2 * 2 * 256 * (64 + 64) * 4


def test_entry_points_reject_bad_arguments(lib):
    p = _p()
    n = nat.workspace_size(p)
    fake = 1 << 20  # aligned, never dereferenced: validation fails first
    P = ctypes.byref
    # invalid params
    bad = _p(Hq=6, Hkv=4)
    assert lib.gqa_attn_fwd(P(bad), fake, fake, fake, None, fake, fake, fake, n, None) == nat.GQA_ERR_INVALID_ARG
    assert lib.gqa_attn_fwd(P(_p(Dqk=256, Dv=256)), fake, fake, fake, None, fake, fake, fake, n, None) == \
        nat.GQA_ERR_UNSUPPORTED
    # workspace problems
    assert lib.gqa_attn_fwd(P(p), fake, fake, fake, None, fake, fake, None, n, None) == nat.GQA_ERR_WORKSPACE
    assert lib.gqa_attn_fwd(P(p), fake, fake, fake, None, fake, fake, fake, n - 1, None) == nat.GQA_ERR_WORKSPACE
    assert lib.gqa_attn_fwd(P(p), fake, fake, fake, None, fake, fake, fake + 16, n, None) == nat.GQA_ERR_WORKSPACE
    # null / misaligned tensors
    assert lib.gqa_attn_fwd(P(p), None, fake, fake, None, fake, fake, fake, n, None) == nat.GQA_ERR_INVALID_ARG
    assert lib.gqa_attn_fwd(P(p), fake + 2, fake, fake, None, fake, fake, fake, n, None) == nat.GQA_ERR_INVALID_ARG
    assert lib.gqa_attn_bwd_preprocess(P(p), fake, None, fake, fake, fake, n, None) == nat.GQA_ERR_INVALID_ARG
    assert lib.gqa_attn_bwd(P(p), fake, fake, fake, fake, fake, None, fake, fake, n, None) == nat.GQA_ERR_INVALID_ARG
    pa = _p(group_mode=nat.GQA_GROUP_ATOMIC)
    na = nat.workspace_size(pa)
    assert lib.gqa_attn_bwd_postprocess(P(pa), fake, None, fake, fake, na, None) == nat.GQA_ERR_INVALID_ARG
    assert lib.gqa_attn_dsink(P(p), None, fake, fake, fake, None) == nat.GQA_ERR_INVALID_ARG
    assert lib.gqa_attn_get_device_error(None, 0, None, None) == nat.GQA_ERR_WORKSPACE
    assert lib.gqa_attn_selftest_wait_timeout(fake + 8, 4096, None) == nat.GQA_ERR_WORKSPACE


def test_packed_sequence_rules(lib):
    import torch
    cu = torch.zeros(3, dtype=torch.int32)  # CPU tensor: only its address is used by validation
    ok = nat.make_params(1, 4, 2, 300, 64, 64, torch.bfloat16, cu_seqlens=cu, max_seqlen=200)
    assert nat.workspace_size(ok) > 0
    assert nat.workspace_size(nat.make_params(2, 4, 2, 300, 64, 64, torch.bfloat16, cu_seqlens=cu,
                                              max_seqlen=200)) == 0          # needs B == 1
    assert nat.workspace_size(nat.make_params(1, 4, 2, 300, 64, 64, torch.bfloat16, cu_seqlens=cu,
                                              max_seqlen=301)) == 0          # max_seqlen > S
    assert nat.workspace_size(nat.make_params(1, 4, 2, 300, 64, 64, torch.bfloat16, cu_seqlens=cu,
                                              max_seqlen=0)) == 0


def test_bulk_reduce_support_matrix(lib):
    for dqk, dv in ((64, 64), (128, 128), (192, 128)):
        for det in (False, True):
            assert nat.workspace_size(_p(Dqk=dqk, Dv=dv, red_mode=nat.GQA_RED_BULK, deterministic=det)) > 0


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = nat.strerror(code)
        assert s and s != "unknown status"
    assert nat.strerror(-99) == "unknown status"


def test_params_struct_matches_library(lib):
    # the binding refuses to load a library whose struct differs; check the numbers directly too
    assert lib.gqa_attn_params_size() == ctypes.sizeof(nat.Params)


def test_layout_strides_validated(lib):
    B, H, S, D = 2, 8, 256, 64
    bshd = (S * H * D, D, H * D)
    assert nat.workspace_size(_p(strides={n: bshd for n in ("q", "o", "do", "dq")})) > 0
    kv_bshd = (S * 2 * D, D, 2 * D)  # Hkv = 2
    assert nat.workspace_size(_p(strides={"k": kv_bshd, "v": kv_bshd, "dk": kv_bshd, "dv": kv_bshd})) > 0
    assert nat.workspace_size(_p(strides={"q": (S * H * D, D, H * D + 4)})) == 0   # not a 16-byte multiple
    assert nat.workspace_size(_p(strides={"q": (S * H * D, 32, H * D)})) == 0      # rows closer than D
    assert nat.workspace_size(_p(strides={"dq": (0, D, H * D)})) == 0              # batch stride 0, B > 1
    assert nat.workspace_size(_p(B=1, strides={"dq": (0, D, H * D)})) > 0         # ... fine for B == 1
    assert nat.workspace_size(_p(strides={"v": (S * 2 * D, -D, 2 * D)})) == 0      # negative


def test_tensor_strides_of_common_layouts():
    import torch
    B, H, S, D = 2, 4, 10, 64
    x = torch.empty(B, S, H, D).transpose(1, 2)  # BSHD view
    assert nat.tensor_strides(x) == (S * H * D, D, H * D)
    thd = torch.empty(S, H, D).permute(1, 0, 2).unsqueeze(0)  # packed THD as [1, H, T, D]
    b, h, s = nat.tensor_strides(thd)
    assert (h, s) == (D, H * D)
    assert nat.tensor_strides(torch.empty(B, H, S, D)) == (H * S * D, S * D, D)
    with pytest.raises(ValueError):
        nat.tensor_strides(torch.empty(B, H, D, S).transpose(2, 3))  # head dim not contiguous


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No CPU fallback: without the compiled library loading raises, and CPU tensors are refused."""
    import torch

    import gqa_flashattention_backward_gb300 as pkg
    monkeypatch.setattr(nat, "_LIB_PATH", str(tmp_path / "libgqa_attn.so"))
    monkeypatch.setattr(nat, "_lib", None)
    with pytest.raises(ImportError):
        nat.load()
    q = torch.zeros(1, 2, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        pkg.attention_forward(q, q[:, :1], q[:, :1])
