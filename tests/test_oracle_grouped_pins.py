"""Pins for the grouped (Mixture-of-Experts) oracle.

``oracle.grouped_gemm_f64`` composes the plain oracle per expert.  These
tests tie it to things other than itself: exact rational brute force per
expert on tiny shapes (``oracle.exact_gemm``, independent of the C code),
the masked rows keeping the output's prior contents, and invariants a slip
would break (an expert's result depends on neither its padding rows nor
any other expert's data).  ``test_grouped_pins_catch_planted_mistakes``
plants typical mistakes in a small copy and checks that a pin rejects each.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

from test_oracle_pins import rand_f16


def _case(rng, E, M, N, K, rows):
    A = rand_f16(rng, (E, M, K))
    B = rand_f16(rng, (E, K, N))
    return A, B, np.asarray(rows, dtype=np.int32)


def _exact_grouped_ok(C, A, B, rows, E, M, N, K, sentinel):
    """Rows below each count within fp64 rounding of the exact sum; the rest
    equal to the sentinel they started with."""
    ok = True
    for e in range(E):
        m = int(rows[e])
        if m:
            X = oracle.exact_gemm(A[e, :m], B[e], m, N, K)
            bound = (np.abs(A[e, :m].astype(np.float64)) @ np.abs(B[e].astype(np.float64))
                     * (K * 2.0 ** -53))
            for i in range(m):
                for j in range(N):
                    ok &= abs(Fraction(float(C[e, i, j])) - X[i][j]) <= Fraction(float(bound[i, j]))
        ok &= bool(np.all(C[e, m:] == sentinel))
    return bool(ok)


@pytest.mark.parametrize("E,M,N,K,rows", [
    (3, 5, 3, 4, [0, 2, 5]),
    (4, 7, 2, 3, [7, 1, 0, 6]),
    (1, 3, 4, 5, [3]),
    (2, 1, 5, 2, [1, 0]),
])
def test_grouped_matches_exact_rationals(E, M, N, K, rows):
    rng = np.random.default_rng(100 + E * M)
    A, B, r = _case(rng, E, M, N, K, rows)
    C0 = np.full((E, M, N), -7.0)
    C = oracle.grouped_gemm_f64(A, B, r, E, M, N, K, C=C0)
    assert _exact_grouped_ok(C, A, B, r, E, M, N, K, -7.0)


def test_masked_rows_keep_prior_contents_and_default_is_nan():
    rng = np.random.default_rng(5)
    A, B, r = _case(rng, 3, 6, 4, 5, [2, 0, 6])
    C = oracle.grouped_gemm_f64(A, B, r, 3, 6, 4, 5)
    assert np.all(np.isnan(C[0, 2:])) and np.all(np.isnan(C[1]))
    assert np.all(np.isfinite(C[0, :2])) and np.all(np.isfinite(C[2]))


def test_padding_rows_and_other_experts_do_not_matter():
    rng = np.random.default_rng(6)
    E, M, N, K = 4, 9, 5, 6
    A, B, r = _case(rng, E, M, N, K, [3, 9, 0, 4])
    C = oracle.grouped_gemm_f64(A, B, r, E, M, N, K)
    A2 = A.copy()
    for e in range(E):
        A2[e, r[e]:] = np.float16(np.nan)   # rows past the count
    B2 = B.copy()
    B2[2] = np.float16(np.inf)             # the expert with no tokens
    C2 = oracle.grouped_gemm_f64(A2, B2, r, E, M, N, K)
    np.testing.assert_array_equal(C, C2)
    # Expert 1 alone gives the same rows as inside the group.
    C1 = oracle.grouped_gemm_f64(A[1:2], B[1:2], r[1:2], 1, M, N, K)
    np.testing.assert_array_equal(C1[0], C[1])


def test_full_counts_and_ones_closed_form():
    E, M, N, K = 3, 4, 5, 6
    A = np.ones((E, M, K), np.float16)
    B = np.ones((E, K, N), np.float16)
    C = oracle.grouped_gemm_f64(A, B, [4, 4, 4], E, M, N, K)
    assert np.all(C == K)
    C = oracle.grouped_gemm_f64(A, B, [1, 0, 3], E, M, N, K, C=np.zeros((E, M, N)))
    expect = np.zeros((E, M, N))
    expect[0, :1] = K
    expect[2, :3] = K
    np.testing.assert_array_equal(C, expect)


def test_rejects_counts_outside_range():
    A = np.ones((2, 3, 2), np.float16)
    B = np.ones((2, 2, 2), np.float16)
    with pytest.raises(ValueError):
        oracle.grouped_gemm_f64(A, B, [1, 4], 2, 3, 2, 2)
    with pytest.raises(ValueError):
        oracle.grouped_gemm_f64(A, B, [-1, 1], 2, 3, 2, 2)


# ---------------------------------------------------------------- planted mistakes

def _grouped_like(A, B, rows, E, M, N, K, C, mistake=None):
    """A small copy of the definition with an optional planted mistake."""
    out = np.array(C, dtype=np.float64, copy=True)
    for e in range(E):
        m = int(rows[e])
        if mistake == "all_rows":
            m = M
        elif mistake == "one_row_short":
            m = max(m - 1, 0)
        elif mistake == "counts_shifted":
            m = int(rows[(e + 1) % E])
        be = 0 if mistake == "first_expert_weights" else e
        for i in range(m):
            for j in range(N):
                out[e, i, j] = float(np.dot(A[e, i].astype(np.float64), B[be][:, j].astype(np.float64)))
        if mistake == "zero_masked_rows":
            out[e, m:] = 0.0
    return out


def _grouped_pins_pass(fn):
    rng = np.random.default_rng(77)
    ok = True
    for (E, M, N, K, rows) in [(3, 5, 3, 4, [0, 2, 5]), (4, 7, 2, 3, [7, 1, 0, 6])]:
        A, B, r = _case(rng, E, M, N, K, rows)
        C = fn(A, B, r, E, M, N, K, np.full((E, M, N), -7.0))
        ok &= _exact_grouped_ok(C, A, B, r, E, M, N, K, -7.0)
    return bool(ok)


def test_grouped_pins_catch_planted_mistakes():
    assert _grouped_pins_pass(lambda *a: _grouped_like(*a))
    assert _grouped_pins_pass(lambda A, B, r, E, M, N, K, C: oracle.grouped_gemm_f64(A, B, r, E, M, N, K, C=C))
    for mistake in ("all_rows", "one_row_short", "counts_shifted", "first_expert_weights",
                    "zero_masked_rows"):
        assert not _grouped_pins_pass(lambda *a, m=mistake: _grouped_like(*a, mistake=m)), mistake
