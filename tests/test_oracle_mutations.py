"""The oracle's pins must reject a wrong oracle.  Each case plants one plausible mistake in a copy of
oracle/gqa_oracle.c (a flipped sign, a dropped term, a wrong index or group map, an off-by-one
mask, the wrong causal alignment), builds it, and runs the pin suite (tests/test_oracle.py:
finite differences, the brute-force group loop, PyTorch autograd, invariants, closed forms)
against it: the suite must fail for every mutant and pass for the unmodified copy."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gqa_oracle.c")

# name -> [(text in gqa_oracle.c, replacement, expected occurrences)]
MUTANTS = {
    "dsink_sign": [("dsink[h] = -acc;", "dsink[h] = acc;", 2)],
    "scale_dropped_in_dS": [("return pij * (dpij - D_i) * p->scale;", "return pij * (dpij - D_i);", 1)],
    "group_map_modulo": [("h / (p->Hq / p->Hkv)", "h % p->Hkv", 2), ("h / G", "h % p->Hkv", 4)],
    "window_one_key_wider": [("il + off - p->window + 1 > a) a = il + off - p->window + 1;",
                              "il + off - p->window > a) a = il + off - p->window;", 1)],
    "sink_left_out_of_denominator": [("double z = p->sink ? exp(p->sink[h] - m) : 0.0;", "double z = 0.0;", 2)],
    "dV_from_dS": [("dvj[d] += pij * doi[d];", "dvj[d] += ds * doi[d];", 3)],
    "causal_excludes_diagonal": [("if (p->causal && il + off + 1 < b) b = il + off + 1;",
                                  "if (p->causal && il + off < b) b = il + off;", 1)],
    "causal_top_left_when_lengths_differ": [("off = kl - ql;", "off = 0;", 1)],
    "right_window_one_key_wider": [("b = il + off + p->window_right;", "b = il + off + p->window_right + 1;", 1)],
    "delta_halved": [("p->Dv);\n}\n\n/* dS_ij", "p->Dv) * 0.5;\n}\n\n/* dS_ij", 1)],
}


def _build(tmp, name, edits):
    src = open(SRC).read()
    for old, new, count in edits:
        assert src.count(old) == count, (name, old, src.count(old))
        src = src.replace(old, new)
    c = os.path.join(tmp, f"{name}.c")
    so = os.path.join(tmp, f"lib{name}.so")
    with open(c, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", so, c, "-lm"], check=True, capture_output=True)
    return so


def _pins(so):
    env = dict(os.environ, GQA_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True)
    return r.returncode, r.stdout[-600:]


@pytest.fixture(scope="module")
def tmpdir_mut(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    return str(tmp_path_factory.mktemp("oracle_mutants"))


def test_unmodified_copy_passes(tmpdir_mut):
    rc, out = _pins(_build(tmpdir_mut, "unmodified", []))
    assert rc == 0, out


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mutant_is_rejected(tmpdir_mut, name):
    rc, out = _pins(_build(tmpdir_mut, name, MUTANTS[name]))
    assert rc == 1, f"{name}: the pins did not fail (exit {rc})\n{out}"
