"""The main kernel's longest-first sequence order for packed batches (sched_fill in the CUDA path's
common.cuh), compiled for the host: the order is a permutation of the sequences (a missing slot would
leave a sequence's dK/dV unwritten and drop its dQ terms, a repeated one would add them twice), by
decreasing KV-tile count, ties in packing order."""
import os
import random
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gqa_flashattention_backward_gb300", "csrc")


@pytest.fixture(scope="module")
def sched_bin(tmp_path_factory):
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("sched") / "sched")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, "-o", out, os.path.join(ROOT, "tests", "sched_main.cu")],
                   check=True, capture_output=True)
    return out


def _cases():
    rng = random.Random(5)
    cases = [[30, 11, 26, 27, 14, 22, 24, 5],          # the varlen workload's KV tiles
             [32, 1, 1, 1, 24, 1, 0, 16],              # skewed: 4096, 64, 64, 64, 3000, 1, 0, 2048 tokens
             [0, 0, 0], [1], [5, 5, 5, 5], [0, 7]]
    for _ in range(20):
        n = rng.randint(1, 256)
        cases.append([rng.randint(0, 30) for _ in range(n)])
    return cases


def test_order_is_a_longest_first_permutation(sched_bin):
    cases = _cases()
    text = "".join(f"{len(k)} {' '.join(map(str, k))}\n" for k in cases)
    out = subprocess.run([sched_bin], input=text, capture_output=True, text=True, check=True).stdout.splitlines()
    assert len(out) == len(cases)
    for keys, line in zip(cases, out):
        perm = [int(x) for x in line.split()]
        assert sorted(perm) == list(range(len(keys))), keys      # every sequence once
        assert perm == sorted(range(len(keys)), key=lambda q: (-keys[q], q)), keys
