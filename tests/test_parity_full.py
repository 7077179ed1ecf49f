"""Full-size parity: every workload at its real size, in the launch configuration the
benchmark times (dK/dV summed in TMEM, dQ added by the bulk tensor reduce that
attention_backward picks by default).

The fp64 oracle computes sampled outputs one by one:

* query rows: LSE, O, Delta and dQ at first / last / tile-edge rows of several heads
  and sequences;
* key rows: dK and dV at the rows that the fewest query tiles reach (the last rows of a
  causal sequence) and at the rows that the most reach (rows 0, 1, 127, 128 and the
  middle row: their dK/dV sum over every query tile of every head of the group, the
  longest accumulation chains of the main kernel -- 4096 iterations for key tile 0 of
  long_context); for long_context only the middle row of kv head 0 is taken among
  these, as each such row needs the statistics of 8 x 16384 query rows.  The oracle
  first forms LSE and Delta of every query row that sees a sampled key (row-parallel),
  then the column sums;
* dsink (sink_window): from the oracle's LSE and Delta of every query row.

Oracle cost (measured on 8 x86 cores; the time is the query-row statistics): mha_causal_n16384
8 s, varlen 2 s, sink_window 9 s (all 524,288 rows, for dsink), long_context 194 s (131,584 rows of
about 24,600 keys each).  A 16-core Arm host runs the whole GPU suite, these included, in under a
minute.
The tolerance is the suite's: max|gpu - ref| <= 2e-2 * max|ref over the sample| + 1e-3.
"""
import numpy as np
import pytest
import torch

from gqa_flashattention_backward_gb300 import workloads as W
from oracle import oracle as orc
from tests._util import assert_close, f64, gpu_run, problem_of

pytestmark = pytest.mark.gpu


def _seq_bounds(w):
    if w.cu_seqlens is None:
        return [(b, 0, w.S) for b in range(w.B)]
    cu = w.cu_seqlens
    return [(0, cu[s], cu[s + 1] - cu[s]) for s in range(len(cu) - 1) if cu[s + 1] > cu[s]]


def _row_samples(w, rng, per_seq=6):
    out = []
    for (b, start, n) in _seq_bounds(w)[:4]:
        cand = sorted({0, 1, 127, 128, n // 2, n - 129, n - 128, n - 1, int(rng.integers(0, n))})
        cand = [i for i in cand if 0 <= i < n]
        heads = sorted({0, w.Hq - 1, int(rng.integers(0, w.Hq))})
        for h in heads:
            for i in cand[:per_seq + 3]:
                out.append((b, h, start + i))
    return out


def _col_samples(w):
    """(b, kv head, absolute key row) triples, and for each the sequence (start, length) it lies in."""
    out = []
    for (b, start, n) in _seq_bounds(w)[:3]:
        if w.window > 0:  # under a window every key row is seen by about `window` query rows
            light, heavy = [0, 127, 128, n // 2, n - 1], []
        else:
            light = [n - 64, n - 17, n - 2, n - 1]        # seen by the fewest query tiles
            heavy = [n // 2] if w.name == "long_context" else [0, 1, 127, 128, n // 2]
        for g in sorted({0, w.Hkv - 1}):
            js = light + (heavy if (w.name != "long_context" or g == 0) else [])
            out += [(b, g, start + j, start, n) for j in sorted(set(js)) if 0 <= j < n]
    return out


def _rows_seeing(w, cols):
    """Linear indices (b*Hq + h)*S + i of every query row that sees one of the sampled keys
    (causal, Sq == Sk, optional left window: the full-size workloads)."""
    G = w.Hq // w.Hkv
    idx = []
    for (b, g, j, start, n) in cols:
        jl = j - start
        hi = n if w.window <= 0 else min(n, jl + w.window)
        i = start + np.arange(jl, hi, dtype=np.int64)
        for h in range(g * G, (g + 1) * G):
            idx.append((b * w.Hq + h) * w.S + i)
    return np.unique(np.concatenate(idx)) if idx else np.zeros(0, dtype=np.int64)


def _stats(w, pb, qf, kf, vf, dof, sink64, lin):
    """Full [B, Hq, S] LSE / Delta arrays holding the oracle's values at rows `lin`, NaN elsewhere
    (the column sums read only rows that see their key: a missed row shows up as NaN)."""
    L = np.full(w.B * w.Hq * w.S, np.nan)
    D = np.full(w.B * w.Hq * w.S, np.nan)
    bs = (lin // (w.Hq * w.S)).astype(np.int32)
    hs = ((lin // w.S) % w.Hq).astype(np.int32)
    is_ = (lin % w.S).astype(np.int32)
    st = orc.row_stats(pb, qf, kf, vf, dof, bs, hs, is_, sink64)
    L[lin], D[lin] = st["lse"], st["delta"]
    return L.reshape(w.B, w.Hq, w.S), D.reshape(w.B, w.Hq, w.S)


FULL = {
    "tiny": W.tiny,
    "mha_causal_n16384": lambda: W.mha_causal(16384),
    "varlen": W.varlen,
    "sink_window": W.sink_window,
    "long_context": W.long_context,
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled(name):
    w = FULL[name]()
    inputs = W.make_inputs(w)
    res = gpu_run(w, inputs)
    q, k, v, do, sink = inputs
    pb = problem_of(w)
    sink64 = f64(sink) if sink is not None else None
    qf, kf, vf, dof = f64(q), f64(k), f64(v), f64(do)
    rng = np.random.default_rng(7)

    rows = _row_samples(w, rng)
    bs, hs, is_ = (np.array(x, dtype=np.int32) for x in zip(*rows))
    ref = orc.sample_rows(pb, qf, kf, vf, dof, bs, hs, is_, sink64)
    got = {n: f64(res[n]) for n in ("o", "lse", "delta", "dq")}
    assert_close(f"{name}:lse", got["lse"][bs, hs, is_], ref["lse"], rtol=1e-3, atol=1e-3)
    assert_close(f"{name}:o", got["o"][bs, hs, is_], ref["o"])
    assert_close(f"{name}:delta", got["delta"][bs, hs, is_], ref["delta"])
    assert_close(f"{name}:dq", got["dq"][bs, hs, is_], ref["dq"])

    cols = _col_samples(w)
    if sink is not None:  # dsink needs every row's statistics, which also cover the sampled keys
        lin = np.arange(w.B * w.Hq * w.S, dtype=np.int64)
    else:
        lin = _rows_seeing(w, cols)
    L, D = _stats(w, pb, qf, kf, vf, dof, sink64, lin)
    cb, cg, cj = (np.array([c[i] for c in cols], dtype=np.int32) for i in range(3))
    refc = orc.cols_with_stats(pb, qf, kf, vf, dof, L, D, cb, cg, cj, sink64)
    assert_close(f"{name}:dk", f64(res["dk"])[cb, cg, cj], refc["dk"])
    assert_close(f"{name}:dv", f64(res["dv"])[cb, cg, cj], refc["dv"])

    if sink is not None:
        assert_close(f"{name}:dsink", f64(res["dsink"]), orc.dsink(pb, L, D, sink64))
    for n in ("dq", "dk", "dv"):
        assert torch.isfinite(res[n].float()).all(), n
