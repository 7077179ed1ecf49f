"""The tile ranges the kernels loop over (q_tiles_for_kv_tile, kv_tiles_for_q_tile and the forward's
fwd_pair_tiles in the CUDA path's common.cuh and fwd_tiles.cuh), compiled for the host and checked against brute-force visibility: every tile
holding a visible (query, key) pair lies in the range (a miss would silently drop gradient terms),
and the range is exactly the span of those tiles (no work on tiles that see nothing).  Covers
causal / non-causal, left and right windows, more or fewer keys than queries (bottom-right
diagonal), ragged lengths and both tile heights the kernels use."""
import os
import random
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gqa_flashattention_backward_gb300", "csrc")


@pytest.fixture(scope="module")
def ranges_bin(tmp_path_factory):
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("ranges") / "tile_ranges")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, "-o", out, os.path.join(ROOT, "tests", "tile_ranges_main.cu")],
                   check=True, capture_output=True)
    return out


def visible(lq, lk, right, window):
    """Query i sees key j iff d = i + (lk - lq) - j satisfies d > -right (right > 0) and d < window (window > 0)."""
    d = np.arange(lq)[:, None] + (lk - lq) - np.arange(lk)[None, :]
    m = np.ones((lq, lk), bool)
    if right > 0:
        m &= d > -right
    if window > 0:
        m &= d < window
    return m


def _cases(n, seed):
    rnd = random.Random(seed)
    lens = [1, 2, 63, 64, 65, 127, 128, 129, 200, 256, 300, 457, 513]
    out = []
    for _ in range(n):
        right = rnd.choice([0, 1, 1, 2, 17, 40, 128, 300])
        window = rnd.choice([0, 0, 1, 5, 64, 100, 129, 300])
        out.append((rnd.choice(lens), rnd.choice(lens), right, window))
    # the plain cases explicitly: causal and non-causal, equal and unequal lengths
    out += [(300, 300, 1, 0), (300, 300, 0, 0), (200, 456, 1, 0), (456, 200, 1, 0), (1, 300, 1, 0), (513, 513, 1, 128)]
    return out


def test_tile_ranges_exact(ranges_bin):
    lines, meta = [], []
    for lq, lk, right, window in _cases(500, 7):
        for rows in (64, 128):
            for kt in range((lk + 127) // 128):
                lines.append(f"q {kt} {lq} {lk} {rows} {right} {window}")
                meta.append(("q", kt, lq, lk, rows, right, window))
            for qt in range((lq + 127) // 128):
                lines.append(f"k {qt} {lq} {lk} {rows} {right} {window}")
                meta.append(("k", qt, lq, lk, rows, right, window))
    res = subprocess.run([ranges_bin], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True)
    got = [tuple(map(int, ln.split())) for ln in res.stdout.strip().split("\n")]
    assert len(got) == len(meta)
    masks = {}
    for (kind, t, lq, lk, rows, right, window), (a, b) in zip(meta, got):
        m = masks.setdefault((lq, lk, right, window), visible(lq, lk, right, window))
        if kind == "q":
            hit = np.nonzero(m[:, t * 128:(t + 1) * 128].any(axis=1))[0] // rows
        else:
            hit = np.nonzero(m[t * 128:(t + 1) * 128, :].any(axis=0))[0] // rows
        case = (kind, t, lq, lk, rows, right, window, (a, b))
        if hit.size:
            assert (a, b) == (int(hit.min()), int(hit.max()) + 1), case
        else:
            assert a == b, case  # nothing visible: an empty range


def test_forward_pair_tiles(ranges_bin):
    """The forward's CTA takes a pair of 128-row query tiles: it loads the union of their key tiles,
    and each query tile's warpgroup works on its own part only.  Each own part must be exactly the
    span of key tiles holding a key visible to that query tile's rows (empty if none, or if the
    sequence has no second tile), and the union exactly the span of the two parts."""
    lines, meta = [], []
    for lq, lk, right, window in _cases(500, 11):
        for bk in (64, 128):
            for tp in range((lq + 255) // 256):
                lines.append(f"f {tp} {lq} {lk} {bk} {right} {window}")
                meta.append((tp, lq, lk, bk, right, window))
    res = subprocess.run([ranges_bin], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True)
    got = [tuple(map(int, ln.split())) for ln in res.stdout.strip().split("\n")]
    assert len(got) == len(meta)
    masks = {}
    for (tp, lq, lk, bk, right, window), (k0, n, jlo0, jhi0, jlo1, jhi1) in zip(meta, got):
        m = masks.setdefault((lq, lk, right, window), visible(lq, lk, right, window))
        case = (tp, lq, lk, bk, right, window, (k0, n, jlo0, jhi0, jlo1, jhi1))
        spans = []
        for w, (jlo, jhi) in enumerate(((jlo0, jhi0), (jlo1, jhi1))):
            qt = 2 * tp + w
            hit = np.nonzero(m[qt * 128:(qt + 1) * 128, :].any(axis=0))[0] // bk if qt * 128 < lq else np.array([])
            assert 0 <= jlo <= jhi <= n, case
            if hit.size:
                assert (k0 + jlo, k0 + jhi) == (int(hit.min()), int(hit.max()) + 1), case
                spans.append((k0 + jlo, k0 + jhi))
            else:
                assert (jlo, jhi) == (0, 0), case
        if spans:
            assert (k0, k0 + n) == (min(a for a, _ in spans), max(b for _, b in spans)), case
        else:
            assert n == 0, case
