"""Pins for the CPU oracle (CPU only)."""
import json
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest

import oracle
from oracle import exact
from tests import oracle_pins
from workloads import WORKLOADS, matrix, sample_entries

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("check", oracle_pins.ALL, ids=lambda c: c.__name__)
def test_oracle_pin(orc, check):
    assert check(orc) == []


def test_golden_tiny_gemms(orc):
    with open(os.path.join(GOLDEN, "tiny_gemm.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        A = np.array(c["A"], dtype=np.float32)
        B = np.array(c["B"], dtype=np.float32)
        C0 = np.array(c["C0"], dtype=np.float32)
        want = np.array(c["C"], dtype=np.float32)
        got = orc.gemm(A, B, c["alpha"], c["beta"], C0)
        assert np.array_equal(got, want), c["seed"]


def test_round_to_f32_matches_numpy_on_doubles():
    # For a value that is already a double, numpy's float64->float32 cast is
    # correctly rounded (ties to even): an independent check of round_to_f32.
    from fractions import Fraction
    rng = np.random.default_rng(5)
    xs = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-5, 5, 2000),
                         [1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, -(1.0 + 2.0 ** -24), 0.0]])
    for x in xs:
        assert exact.round_to_f32(Fraction(float(x))) == np.float32(x)


def test_flop_count_matches_page():
    # 2 * 4096^3 = 137,438,953,472, about 137.4 GFLOP ("Project - tiled
    # matrix multiply", section "Numerical background").
    with open(os.path.join(GOLDEN, "page_facts.json")) as f:
        facts = json.load(f)["flops_4096"]
    w = WORKLOADS["sq4096"]
    assert w.flops == 2 * facts["n_cubed"] == 137_438_953_472
    assert round(w.flops / 1e9, 1) == facts["gflop_rounded_1dp"]


def test_sampled_positions_cover_edges():
    rows, cols = sample_entries(65536, 64)
    assert rows.size == 4096 and cols.size == 4096
    pairs = set(zip(rows.tolist(), cols.tolist()))
    for p in [(0, 0), (0, 63), (65535, 0), (65535, 63)]:
        assert p in pairs
    assert rows.min() >= 0 and rows.max() < 65536 and cols.max() < 64
    r2, c2 = sample_entries(65536, 64)
    assert np.array_equal(rows, r2) and np.array_equal(cols, c2)


def test_generators_are_exact_and_in_range():
    u = matrix(64, 64, None, 1, "u11")
    assert u.min() >= -1.0 and u.max() < 1.0
    # 24-bit dyadic values: 2^24 * (u+1)/2 is an integer
    assert np.all(((u.astype(np.float64) + 1.0) * 2.0 ** 23) % 1.0 == 0.0)
    i = matrix(64, 64, None, 2, "int2")
    assert set(np.unique(i).tolist()) <= {-2.0, -1.0, 0.0, 1.0, 2.0}
    assert len(np.unique(i)) == 5
    n = matrix(256, 256, None, 3, "normal", 0.02)
    assert abs(float(n.std()) - 0.02) < 0.001 and abs(float(n.mean())) < 0.001
    p = matrix(3, 4, 7, 4, "u11")
    assert p.shape == (3, 7) and np.all(np.isnan(p[:, 4:]))


def test_error_metrics():
    ref = np.array([[1.0, 2.0], [0.0, -3.0]], dtype=np.float32)
    got = np.array([[1.0, 2.5], [0.0, -3.0]], dtype=np.float32)
    D = np.array([[2.0, 5.0], [0.0, 3.0]])
    assert oracle.err_normalised(got, ref, D) == pytest.approx(0.1)
    assert oracle.mismatches(got, ref) == 1
    assert oracle.err_pages(got, ref) == pytest.approx(0.25)
    nan = got.copy()
    nan[0, 0] = np.nan
    assert oracle.err_normalised(nan, ref, D) == float("inf")
    assert oracle.mismatches(nan, ref) == 2


# Each mutation is a plausible mistake in the oracle's source.  The pin suite
# must reject every one of them.
MUTANTS = {
    "drop_last_k": ("k < K; ++k", "k < K - 1; ++k"),
    "transpose_B": ("B[k * ldb + j]", "B[j * ldb + k]"),
    "beta_sign": ("r += beta * c;", "r -= beta * c;"),
    "alpha_ignored": ("double r = alpha * s;", "double r = s;"),
    "lda_ignored": ("A + i * lda", "A + i * K"),
    "float_accumulator": ("double s = 0.0, sa = 0.0;", "float s = 0.0f; double sa = 0.0;"),
    "bound_without_beta": ("d += fabs(beta) * fabs(c);", "(void)d;"),
    "reads_c_when_beta_zero": ("if (beta != 0.0) {", "if (Cin) {"),
    "reads_ab_when_alpha_zero": ("if (alpha == 0.0) K = 0;", ";"),
}

_RUNNER = r"""
import sys
sys.path.insert(0, {root!r})
import oracle
from tests import oracle_pins
fails = oracle_pins.run_all(oracle.Oracle({lib!r}))
print("FAILS", len(fails))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "oracle", "gemm_oracle.c")) as f:
        src = f.read()
    old, new = MUTANTS[name]
    assert old in src, f"mutation anchor for {name} no longer in the oracle source"
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "mut.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.compile_source(path, os.path.join(d, "libmut.so"))
        # run in a child: a broken oracle may read out of bounds
        r = subprocess.run([sys.executable, "-c", _RUNNER.format(root=root, lib=lib)],
                           capture_output=True, text=True, timeout=300)
    caught = r.returncode != 0 or ("FAILS 0" not in r.stdout)
    assert caught, f"mutant {name} passed every pin:\n{r.stdout}\n{r.stderr}"
