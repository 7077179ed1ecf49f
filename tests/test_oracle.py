"""Pins for the fp64 CPU oracle (no GPU needed).

The oracle is checked against things other than itself:
  * central finite differences of the scalar loss L = sum(dO * O) through the
    oracle's forward (pins every gradient, where `scale` enters, the sink
    convention and the dsink sign);
  * an independent numpy implementation that materialises S x S and handles GQA
    by expanding K/V per query head and summing dK/dV over each group;
  * PyTorch fp64 autograd of plain masked softmax attention (a library routine),
    with the sink as an extra softmax column that has no value vector;
  * closed forms and invariants: sum_j P_ij + p_sink_i = 1,
    Delta_i = sum_j P_ij dP_ij, sum_j dV_j = sum_i (1 - p_sink_i) dO_i,
    sum_j dK_j = scale * sum_i p_sink_i Delta_i Q_i, dsink = -sum_ij dS_ij / scale,
    S = 1 and all-keys-equal special cases.
"""
import itertools

import numpy as np
import pytest
import torch

from oracle import brute
from oracle import oracle as orc

TINY = dict(B=1, Hq=4, Hkv=2, S=7, Dqk=5, Dv=3)


def _rand(shape, rng, std=1.0):
    return rng.standard_normal(shape) * std


def _inputs(pb, seed=0, with_sink=False):
    rng = np.random.default_rng(seed)
    q = _rand((pb.B, pb.Hq, pb.S, pb.Dqk), rng)
    k = _rand((pb.B, pb.Hkv, pb.key_len, pb.Dqk), rng)
    v = _rand((pb.B, pb.Hkv, pb.key_len, pb.Dv), rng)
    do = _rand((pb.B, pb.Hq, pb.S, pb.Dv), rng)
    sink = _rand((pb.Hq,), rng) if with_sink else None
    return q, k, v, do, sink


def _cases():
    out = []
    for causal, sink, window in itertools.product([False, True], [False, True], [0, 3]):
        if window and not causal:
            continue
        out.append(dict(causal=causal, sink=sink, window=window, cu=None))
    out.append(dict(causal=True, sink=False, window=0, cu=[0, 3, 7]))
    out.append(dict(causal=False, sink=True, window=0, cu=[0, 3, 7]))
    out.append(dict(causal=True, sink=True, window=2, cu=[0, 3, 7]))
    return out


def _pb(case, **shape):
    shp = dict(TINY)
    shp.update(shape)
    return orc.Problem(causal=case["causal"], window=case["window"], scale=0.7, cu_seqlens=case["cu"], **shp)


def _loss(pb, q, k, v, do, sink):
    o, _ = orc.forward(pb, q, k, v, sink)
    return float((o * do).sum())


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"c{int(c['causal'])}s{int(c['sink'])}w{c['window']}"
                         f"{'v' if c['cu'] else ''}")
def test_finite_differences(case):
    pb = _pb(case)
    q, k, v, do, sink = _inputs(pb, seed=11, with_sink=case["sink"])
    o, lse = orc.forward(pb, q, k, v, sink)
    g = orc.backward(pb, q, k, v, o, lse, do, sink)
    h = 1e-5

    def fd(x):
        num = np.zeros_like(x)
        flat, nflat = x.reshape(-1), num.reshape(-1)
        for t in range(flat.size):
            keep = flat[t]
            flat[t] = keep + h
            lp = _loss(pb, q, k, v, do, sink)
            flat[t] = keep - h
            lm = _loss(pb, q, k, v, do, sink)
            flat[t] = keep
            nflat[t] = (lp - lm) / (2 * h)
        return num

    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        num = fd(x)
        err = np.abs(num - g[name]).max()
        assert err <= 1e-7 * max(1.0, np.abs(num).max()), (name, err)
    if sink is not None:
        num = fd(sink)
        assert np.abs(num - g["dsink"]).max() <= 1e-7 * max(1.0, np.abs(num).max())


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"c{int(c['causal'])}s{int(c['sink'])}w{c['window']}"
                         f"{'v' if c['cu'] else ''}")
def test_against_bruteforce_group_loop(case):
    pb = _pb(case, S=7 if case["cu"] else 9)
    q, k, v, do, sink = _inputs(pb, seed=5, with_sink=case["sink"])
    o, lse = orc.forward(pb, q, k, v, sink)
    g = orc.backward(pb, q, k, v, o, lse, do, sink)
    r = brute.gqa(q, k, v, do, pb.resolved_scale(), causal=pb.causal, window=pb.window,
                  cu_seqlens=pb.cu_seqlens, sink=sink)
    np.testing.assert_allclose(o, r["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, r["lse"], rtol=0, atol=1e-12)
    for name in ("delta", "dq", "dk", "dv"):
        np.testing.assert_allclose(g[name], r[name], rtol=0, atol=1e-12, err_msg=name)
    if sink is not None:
        np.testing.assert_allclose(g["dsink"], r["dsink"], rtol=0, atol=1e-12)


def _torch_reference(pb, q, k, v, do, sink):
    """fp64 autograd of plain masked softmax attention (test-only library routine)."""
    G = pb.Hq // pb.Hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    ts = torch.tensor(sink, requires_grad=True) if sink is not None else None
    i = torch.arange(pb.S)[:, None]
    j = torch.arange(pb.S)[None, :]
    allowed = torch.ones(pb.S, pb.S, dtype=torch.bool)
    if pb.cu_seqlens is not None:
        sid = torch.zeros(pb.S, dtype=torch.long)
        for s in range(len(pb.cu_seqlens) - 1):
            sid[pb.cu_seqlens[s]:pb.cu_seqlens[s + 1]] = s
        allowed &= sid[:, None] == sid[None, :]
    if pb.causal:
        allowed &= j <= i
    if pb.window > 0:
        allowed &= (i - j) < pb.window
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    logits = torch.einsum("bhid,bhjd->bhij", tq, kk) * pb.resolved_scale()
    logits = logits.masked_fill(~allowed, float("-inf"))
    if ts is not None:
        col = ts.view(1, pb.Hq, 1, 1).expand(pb.B, pb.Hq, pb.S, 1)
        probs = torch.softmax(torch.cat([logits, col], dim=-1), dim=-1)[..., :pb.S]
    else:
        probs = torch.softmax(logits, dim=-1)
    o = probs @ vv
    (o * torch.tensor(do)).sum().backward()
    out = dict(o=o.detach().numpy(), dq=tq.grad.numpy(), dk=tk.grad.numpy(), dv=tv.grad.numpy())
    if ts is not None:
        out["dsink"] = ts.grad.numpy()
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"c{int(c['causal'])}s{int(c['sink'])}w{c['window']}"
                         f"{'v' if c['cu'] else ''}")
def test_against_torch_autograd(case):
    pb = _pb(case, S=7 if case["cu"] else 11, Dqk=6, Dv=4, Hq=6, Hkv=3)
    q, k, v, do, sink = _inputs(pb, seed=21, with_sink=case["sink"])
    o, lse = orc.forward(pb, q, k, v, sink)
    g = orc.backward(pb, q, k, v, o, lse, do, sink)
    t = _torch_reference(pb, q, k, v, do, sink)
    np.testing.assert_allclose(o, t["o"], rtol=0, atol=1e-12)
    for name in ("dq", "dk", "dv") + (("dsink",) if sink is not None else ()):
        np.testing.assert_allclose(g[name], t[name], rtol=0, atol=1e-11, err_msg=name)


@pytest.mark.parametrize("with_sink", [False, True])
@pytest.mark.parametrize("window", [0, 4])
def test_invariants(with_sink, window):
    pb = orc.Problem(B=2, Hq=4, Hkv=2, S=13, Dqk=8, Dv=6, causal=True, window=window, scale=0.4)
    q, k, v, do, sink = _inputs(pb, seed=3, with_sink=with_sink)
    o, lse = orc.forward(pb, q, k, v, sink)
    g = orc.backward(pb, q, k, v, o, lse, do, sink)
    r = brute.gqa(q, k, v, do, pb.resolved_scale(), causal=True, window=window, sink=sink)
    P, p_sink, dP, dS = r["P"], r["p_sink"], r["dP"], r["dS"]
    # probabilities over the keys plus the sink sum to one
    np.testing.assert_allclose(P.sum(-1) + p_sink, 1.0, atol=1e-13)
    # Delta_i = sum_j P_ij dP_ij
    np.testing.assert_allclose(g["delta"], (P * dP).sum(-1), atol=1e-12)
    G = pb.Hq // pb.Hkv
    for b in range(pb.B):
        for kvh in range(pb.Hkv):
            hs = range(kvh * G, (kvh + 1) * G)
            want_dv = sum(((1.0 - p_sink[b, h])[:, None] * do[b, h]).sum(0) for h in hs)
            np.testing.assert_allclose(g["dv"][b, kvh].sum(0), want_dv, atol=1e-11)
            want_dk = pb.resolved_scale() * sum(((p_sink[b, h] * g["delta"][b, h])[:, None] * q[b, h]).sum(0)
                                                for h in hs)
            np.testing.assert_allclose(g["dk"][b, kvh].sum(0), want_dk, atol=1e-11)
    if with_sink:
        want = -dS.sum(axis=(0, 2, 3)) / pb.resolved_scale()
        np.testing.assert_allclose(g["dsink"], want, atol=1e-11)
    else:
        # without a sink, shifting every key by a constant leaves the softmax unchanged
        np.testing.assert_allclose(g["dk"].sum(axis=2), 0.0, atol=1e-11)


def test_single_token():
    pb = orc.Problem(B=1, Hq=2, Hkv=1, S=1, Dqk=4, Dv=3, causal=True, scale=0.5)
    q, k, v, do, _ = _inputs(pb, seed=7)
    o, lse = orc.forward(pb, q, k, v)
    g = orc.backward(pb, q, k, v, o, lse, do)
    assert np.array_equal(o[0, 0], v[0, 0]) and np.array_equal(o[0, 1], v[0, 0])
    np.testing.assert_allclose(lse[0, :, 0], 0.5 * (q[0, :, 0] @ k[0, 0, 0]), atol=1e-15)
    assert np.all(g["dq"] == 0.0) and np.all(g["dk"] == 0.0)
    np.testing.assert_allclose(g["dv"][0, 0, 0], do[0, 0, 0] + do[0, 1, 0], atol=1e-15)


def test_equal_keys_closed_form():
    pb = orc.Problem(B=1, Hq=1, Hkv=1, S=10, Dqk=4, Dv=5, causal=True, scale=0.3)
    q, k, v, do, _ = _inputs(pb, seed=8)
    k[:] = k[:, :, :1, :]  # every key identical
    o, lse = orc.forward(pb, q, k, v)
    for i in range(pb.S):
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :i + 1].mean(0), atol=1e-13)
        s = 0.3 * q[0, 0, i] @ k[0, 0, 0]
        np.testing.assert_allclose(lse[0, 0, i], s + np.log(i + 1), atol=1e-13)


def test_sampled_matches_full():
    pb = orc.Problem(B=1, Hq=4, Hkv=2, S=23, Dqk=6, Dv=5, causal=True, window=9, scale=0.45,
                     cu_seqlens=[0, 10, 10, 23])
    q, k, v, do, sink = _inputs(pb, seed=9, with_sink=True)
    o, lse = orc.forward(pb, q, k, v, sink)
    g = orc.backward(pb, q, k, v, o, lse, do, sink)
    rows = [(0, h, i) for h in range(4) for i in (0, 5, 9, 10, 17, 22)]
    bs, hs, is_ = zip(*rows)
    sr = orc.sample_rows(pb, q, k, v, do, bs, hs, is_, sink)
    for t, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(sr["lse"][t], lse[b, h, i], atol=1e-13)
        np.testing.assert_allclose(sr["o"][t], o[b, h, i], atol=1e-13)
        np.testing.assert_allclose(sr["delta"][t], g["delta"][b, h, i], atol=1e-13)
        np.testing.assert_allclose(sr["dq"][t], g["dq"][b, h, i], atol=1e-13)
    cols = [(0, gg, j) for gg in range(2) for j in (0, 3, 9, 11, 20, 22)]
    bs, gs, js = zip(*cols)
    sc = orc.sample_cols(pb, q, k, v, do, bs, gs, js, sink)
    for t, (b, gg, j) in enumerate(cols):
        np.testing.assert_allclose(sc["dk"][t], g["dk"][b, gg, j], atol=1e-13)
        np.testing.assert_allclose(sc["dv"][t], g["dv"][b, gg, j], atol=1e-13)



@pytest.mark.parametrize("case", [
    dict(B=1, Hq=4, Hkv=2, S=23, Sk=None, causal=True, window=9, right=0, cu=[0, 10, 10, 23], sink=True),
    dict(B=2, Hq=6, Hkv=2, S=17, Sk=None, causal=True, window=0, right=0, cu=None, sink=False),
    dict(B=1, Hq=2, Hkv=1, S=9, Sk=14, causal=True, window=4, right=0, cu=None, sink=True),
    dict(B=1, Hq=4, Hkv=1, S=12, Sk=None, causal=False, window=3, right=2, cu=None, sink=True),
])
def test_row_stats_and_columns_match_full(case):
    """The row-statistics / column / dsink functions used at full size give exactly what the full
    passes give (which are pinned above by finite differences, brute force and autograd)."""
    pb = orc.Problem(B=case["B"], Hq=case["Hq"], Hkv=case["Hkv"], S=case["S"], Dqk=6, Dv=5, causal=case["causal"],
                     window=case["window"], window_right=case["right"], scale=0.41, cu_seqlens=case["cu"],
                     Sk=case["Sk"])
    q, k, v, do, sink = _inputs(pb, seed=21, with_sink=case["sink"])
    o, lse = orc.forward(pb, q, k, v, sink)
    g = orc.backward(pb, q, k, v, o, lse, do, sink)
    rows = [(b, h, i) for b in range(pb.B) for h in range(pb.Hq) for i in range(pb.S)]
    bs, hs, is_ = zip(*rows)
    st = orc.row_stats(pb, q, k, v, do, bs, hs, is_, sink)
    L = st["lse"].reshape(pb.B, pb.Hq, pb.S)
    D = st["delta"].reshape(pb.B, pb.Hq, pb.S)
    np.testing.assert_allclose(L, lse, atol=1e-13)
    np.testing.assert_allclose(D, g["delta"], atol=1e-13)
    cols = [(b, gg, j) for b in range(pb.B) for gg in range(pb.Hkv) for j in range(pb.key_len)]
    bs, gs, js = zip(*cols)
    sc = orc.cols_with_stats(pb, q, k, v, do, L, D, bs, gs, js, sink)
    np.testing.assert_allclose(sc["dk"].reshape(g["dk"].shape), g["dk"], atol=1e-13)
    np.testing.assert_allclose(sc["dv"].reshape(g["dv"].shape), g["dv"], atol=1e-13)
    if sink is not None:
        np.testing.assert_allclose(orc.dsink(pb, L, D, sink), g["dsink"], atol=1e-13)
    # the column pass reads only rows that see the key: unrelated rows may hold anything
    if case["causal"] and case["cu"] is None and case["Sk"] is None:
        Ln, Dn = L.copy(), D.copy()
        Ln[:, :, :3], Dn[:, :, :3] = np.nan, np.nan   # rows 0..2 never see key 5 under a causal mask
        c5 = orc.cols_with_stats(pb, q, k, v, do, Ln, Dn, [0], [0], [5], sink)
        np.testing.assert_allclose(c5["dk"][0], g["dk"][0, 0, 5], atol=1e-13)


def test_empty_sequence_rows_are_untouched():
    # an empty packed sequence contributes no rows; its neighbours are unaffected
    pb1 = orc.Problem(B=1, Hq=2, Hkv=1, S=9, Dqk=4, Dv=4, causal=True, scale=0.5, cu_seqlens=[0, 4, 4, 9])
    pb2 = orc.Problem(B=1, Hq=2, Hkv=1, S=9, Dqk=4, Dv=4, causal=True, scale=0.5, cu_seqlens=[0, 4, 9])
    q, k, v, do, _ = _inputs(pb1, seed=4)
    o1, l1 = orc.forward(pb1, q, k, v)
    o2, l2 = orc.forward(pb2, q, k, v)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---------------------------------------------------------------- Sq != Sk (bottom-right causal)
# query i of a sequence with Lq queries and Lk keys sees key j iff j <= i + (Lk - Lq) (causal) and
# i + (Lk - Lq) - j < W (window): the last query sees the last key.

def _cross_cases():
    return [
        dict(S=5, Sk=8, causal=True, window=0, sink=False, cu=None, cuk=None),   # chunked prefill
        dict(S=5, Sk=8, causal=True, window=3, sink=True, cu=None, cuk=None),
        dict(S=8, Sk=5, causal=True, window=0, sink=False, cu=None, cuk=None),   # 3 rows see nothing
        dict(S=8, Sk=5, causal=True, window=0, sink=True, cu=None, cuk=None),
        dict(S=4, Sk=7, causal=False, window=0, sink=True, cu=None, cuk=None),   # cross-attention
        dict(S=7, Sk=7, causal=True, window=0, sink=False, cu=[0, 3, 7], cuk=[0, 5, 7]),  # per-sequence offsets
    ]


def _cross_pb(c, **shape):
    shp = dict(TINY, S=c["S"])
    shp.update(shape)
    return orc.Problem(causal=c["causal"], window=c["window"], scale=0.7, cu_seqlens=c["cu"], Sk=c["Sk"],
                       cu_seqlens_k=c["cuk"], **shp)


def _cross_id(c):
    return f"q{c['S']}k{c['Sk']}c{int(c['causal'])}w{c['window']}s{int(c['sink'])}{'v' if c['cu'] else ''}"


@pytest.mark.parametrize("case", _cross_cases(), ids=_cross_id)
def test_cross_lengths_finite_differences(case):
    pb = _cross_pb(case)
    q, k, v, do, sink = _inputs(pb, seed=13, with_sink=case["sink"])
    o, lse = orc.forward(pb, q, k, v, sink)
    g = orc.backward(pb, q, k, v, o, lse, do, sink)
    h = 1e-5

    def fd(x):
        num = np.zeros_like(x)
        flat, nflat = x.reshape(-1), num.reshape(-1)
        for t in range(flat.size):
            keep = flat[t]
            flat[t] = keep + h
            lp = _loss(pb, q, k, v, do, sink)
            flat[t] = keep - h
            lm = _loss(pb, q, k, v, do, sink)
            flat[t] = keep
            nflat[t] = (lp - lm) / (2 * h)
        return num

    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        num = fd(x)
        assert np.abs(num - g[name]).max() <= 1e-7 * max(1.0, np.abs(num).max()), name
    if sink is not None:
        num = fd(sink)
        assert np.abs(num - g["dsink"]).max() <= 1e-7 * max(1.0, np.abs(num).max())


@pytest.mark.parametrize("case", _cross_cases(), ids=_cross_id)
def test_cross_lengths_against_bruteforce(case):
    pb = _cross_pb(case)
    q, k, v, do, sink = _inputs(pb, seed=17, with_sink=case["sink"])
    o, lse = orc.forward(pb, q, k, v, sink)
    g = orc.backward(pb, q, k, v, o, lse, do, sink)
    r = brute.gqa(q, k, v, do, pb.resolved_scale(), causal=pb.causal, window=pb.window, cu_seqlens=pb.cu_seqlens,
                  sink=sink, cu_seqlens_k=pb.cu_seqlens_k)
    np.testing.assert_allclose(o, r["o"], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(r["lse"]))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(lse[fin], r["lse"][fin], rtol=0, atol=1e-12)
    for name in ("delta", "dq", "dk", "dv"):
        np.testing.assert_allclose(g[name], r[name], rtol=0, atol=1e-12, err_msg=name)


@pytest.mark.parametrize("case", _cross_cases(), ids=_cross_id)
def test_cross_lengths_against_torch_autograd(case):
    pb = _cross_pb(case, Hq=6, Hkv=3, Dqk=6, Dv=4)
    q, k, v, do, sink = _inputs(pb, seed=23, with_sink=case["sink"])
    o, lse = orc.forward(pb, q, k, v, sink)
    g = orc.backward(pb, q, k, v, o, lse, do, sink)
    G = pb.Hq // pb.Hkv
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    ts = torch.tensor(sink, requires_grad=True) if sink is not None else None
    allowed = torch.tensor(brute.mask_matrix(pb.S, pb.causal, pb.window, pb.cu_seqlens, pb.key_len,
                                             pb.cu_seqlens_k))
    logits = torch.einsum("bhid,bhjd->bhij", tq, tk.repeat_interleave(G, dim=1)) * pb.resolved_scale()
    logits = logits.masked_fill(~allowed, float("-inf"))
    if ts is not None:
        logits = torch.cat([logits, ts.view(1, pb.Hq, 1, 1).expand(pb.B, pb.Hq, pb.S, 1)], dim=-1)
    probs = torch.nan_to_num(torch.softmax(logits, dim=-1))[..., :pb.key_len]  # rows that see nothing: 0
    out = probs @ tv.repeat_interleave(G, dim=1)
    (out * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(o, out.detach().numpy(), rtol=0, atol=1e-12)
    for name, t in (("dq", tq), ("dk", tk), ("dv", tv)) + ((("dsink", ts),) if ts is not None else ()):
        np.testing.assert_allclose(g[name], t.grad.numpy(), rtol=0, atol=1e-11, err_msg=name)


def test_decode_row_sees_every_key():
    """One query against Sk keys, causal bottom-right: it sees all of them, i.e. plain
    non-causal attention."""
    a = orc.Problem(B=1, Hq=4, Hkv=2, S=1, Dqk=5, Dv=3, causal=True, scale=0.7, Sk=9)
    b = orc.Problem(B=1, Hq=4, Hkv=2, S=1, Dqk=5, Dv=3, causal=False, scale=0.7, Sk=9)
    q, k, v, do, _ = _inputs(a, seed=3)
    oa, la = orc.forward(a, q, k, v)
    ob, lb = orc.forward(b, q, k, v)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(la, lb)
    ga, gb = orc.backward(a, q, k, v, oa, la, do), orc.backward(b, q, k, v, ob, lb, do)
    for n in ("dq", "dk", "dv"):
        np.testing.assert_array_equal(ga[n], gb[n])


def test_rows_without_keys():
    """More queries than keys, causal: the first S - Sk query rows see no key; without a sink
    their O and dQ are zero, LSE is -inf and they add nothing to dK / dV."""
    pb = orc.Problem(B=1, Hq=2, Hkv=1, S=8, Dqk=5, Dv=3, causal=True, scale=0.7, Sk=5)
    q, k, v, do, _ = _inputs(pb, seed=9)
    o, lse = orc.forward(pb, q, k, v)
    g = orc.backward(pb, q, k, v, o, lse, do)
    assert np.all(o[:, :, :3] == 0) and np.all(np.isneginf(lse[:, :, :3])) and np.all(np.isfinite(lse[:, :, 3:]))
    assert np.all(g["dq"][:, :, :3] == 0)
    do2 = do.copy()
    do2[:, :, :3] = 123.0  # the gradient of those rows cannot reach K or V
    g2 = orc.backward(pb, q, k, v, o, lse, do2)
    np.testing.assert_array_equal(g["dk"], g2["dk"])
    np.testing.assert_array_equal(g["dv"], g2["dv"])


# ---------------------------------------------------------------- right window (local attention)
# not causal, keys j with j - (i + Lk - Lq) < Wr (and, with a window W, i + Lk - Lq - j < W)

def _local_cases():
    return [
        dict(S=9, Sk=9, window=3, wr=2, sink=False, cu=None, cuk=None),    # two-sided, radius 2 / 1
        dict(S=9, Sk=9, window=0, wr=3, sink=True, cu=None, cuk=None),     # right side only
        dict(S=6, Sk=10, window=4, wr=4, sink=False, cu=None, cuk=None),   # with Sk != Sq
        dict(S=7, Sk=7, window=2, wr=3, sink=True, cu=[0, 3, 7], cuk=[0, 4, 7]),
    ]


def _local_pb(c, **shape):
    shp = dict(TINY, S=c["S"])
    shp.update(shape)
    return orc.Problem(causal=False, window=c["window"], window_right=c["wr"], scale=0.7, cu_seqlens=c["cu"],
                       Sk=c["Sk"], cu_seqlens_k=c["cuk"], **shp)


def _local_id(c):
    return f"q{c['S']}k{c['Sk']}w{c['window']}r{c['wr']}s{int(c['sink'])}{'v' if c['cu'] else ''}"


@pytest.mark.parametrize("case", _local_cases(), ids=_local_id)
def test_right_window_finite_differences(case):
    pb = _local_pb(case)
    q, k, v, do, sink = _inputs(pb, seed=29, with_sink=case["sink"])
    o, lse = orc.forward(pb, q, k, v, sink)
    g = orc.backward(pb, q, k, v, o, lse, do, sink)
    h = 1e-5

    def fd(x):
        num = np.zeros_like(x)
        flat, nflat = x.reshape(-1), num.reshape(-1)
        for t in range(flat.size):
            keep = flat[t]
            flat[t] = keep + h
            lp = _loss(pb, q, k, v, do, sink)
            flat[t] = keep - h
            lm = _loss(pb, q, k, v, do, sink)
            flat[t] = keep
            nflat[t] = (lp - lm) / (2 * h)
        return num

    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        num = fd(x)
        assert np.abs(num - g[name]).max() <= 1e-7 * max(1.0, np.abs(num).max()), name


@pytest.mark.parametrize("case", _local_cases(), ids=_local_id)
def test_right_window_against_bruteforce_and_torch(case):
    pb = _local_pb(case, Hq=6, Hkv=3, Dqk=6, Dv=4)
    q, k, v, do, sink = _inputs(pb, seed=31, with_sink=case["sink"])
    o, lse = orc.forward(pb, q, k, v, sink)
    g = orc.backward(pb, q, k, v, o, lse, do, sink)
    r = brute.gqa(q, k, v, do, pb.resolved_scale(), causal=False, window=pb.window, cu_seqlens=pb.cu_seqlens,
                  sink=sink, cu_seqlens_k=pb.cu_seqlens_k, window_right=pb.window_right)
    np.testing.assert_allclose(o, r["o"], rtol=0, atol=1e-12)
    for name in ("dq", "dk", "dv"):
        np.testing.assert_allclose(g[name], r[name], rtol=0, atol=1e-12, err_msg=name)
    # PyTorch autograd of softmax attention over the same explicit mask (a library routine)
    G = pb.Hq // pb.Hkv
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    allowed = torch.tensor(brute.mask_matrix(pb.S, False, pb.window, pb.cu_seqlens, pb.key_len, pb.cu_seqlens_k,
                                             pb.window_right))
    logits = torch.einsum("bhid,bhjd->bhij", tq, tk.repeat_interleave(G, dim=1)) * pb.resolved_scale()
    logits = logits.masked_fill(~allowed, float("-inf"))
    if sink is not None:
        logits = torch.cat([logits, torch.tensor(sink).view(1, pb.Hq, 1, 1).expand(pb.B, pb.Hq, pb.S, 1)], dim=-1)
    probs = torch.nan_to_num(torch.softmax(logits, dim=-1))[..., :pb.key_len]
    (probs @ tv.repeat_interleave(G, dim=1) * torch.tensor(do)).sum().backward()
    for name, t in (("dq", tq), ("dk", tk), ("dv", tv)):
        np.testing.assert_allclose(g[name], t.grad.numpy(), rtol=0, atol=1e-11, err_msg=name)


def test_right_window_closed_forms():
    """A right window of 1 with no left window is the causal mask; left and right windows wider
    than the sequence are plain non-causal attention."""
    base = dict(B=1, Hq=4, Hkv=2, S=8, Dqk=5, Dv=3, scale=0.7)
    a = orc.Problem(causal=False, window_right=1, **base)
    c = orc.Problem(causal=True, **base)
    q, k, v, do, _ = _inputs(a, seed=37)
    oa, la = orc.forward(a, q, k, v)
    oc, lc = orc.forward(c, q, k, v)
    np.testing.assert_array_equal(oa, oc)
    np.testing.assert_array_equal(la, lc)
    w = orc.Problem(causal=False, window=100, window_right=100, **base)
    n = orc.Problem(causal=False, **base)
    np.testing.assert_array_equal(orc.forward(w, q, k, v)[0], orc.forward(n, q, k, v)[0])
