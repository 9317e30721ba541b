"""Pins for the oracle: each checks it against something other than itself.

* numpy's own float16 conversion (all 65536 bit patterns of the decoder),
* exact rational brute force on tiny shapes (``fractions.Fraction``),
* closed forms (all-ones -> K in every cell, identity -> copy, the pages'
  row-sum worked values),
* numpy's integer matmul on small-integer inputs (exact),
* invariants that a plausible slip would break (the transpose identity,
  zero padding of K, cells against the full product).

``test_pins_catch_planted_mistakes`` plants typical mistakes in small
Python copies of the definition and checks that some pin rejects each one.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_f16(rng, shape, with_subnormals=True):
    """Random finite f16 values over several magnitudes, some subnormal."""
    mant = rng.uniform(-1.0, 1.0, size=shape)
    expo = rng.integers(-6, 3, size=shape)
    x = (mant * np.exp2(expo)).astype(np.float16)
    if with_subnormals:
        sub = rng.random(shape) < 0.15
        bits = rng.integers(1, 1024, size=shape).astype(np.uint16)
        bits |= (rng.random(shape) < 0.5).astype(np.uint16) << 15
        x = np.where(sub, bits.view(np.float16), x)
    return x


def padded(x, ld):
    """Copy a 2-D array into a wider row-major buffer (row stride ``ld``)."""
    rows, cols = x.shape
    buf = np.full((rows, ld), np.float16(np.nan), dtype=np.float16)
    buf[:, :cols] = x
    return buf


# ---------------------------------------------------------------- decoder

def test_decoder_matches_numpy_on_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    ours = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # the sign of zero is kept too
    assert math.copysign(1.0, oracle.f16_to_f64(0x8000)) == -1.0


# ---------------------------------------------------------------- brute force

SHAPES = [(M, N, K) for M in (1, 2, 3, 5, 8) for N in (1, 3, 7, 17) for K in (1, 2, 5, 8, 17)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_matches_exact_rationals(M, N, K):
    rng = np.random.default_rng(M * 10000 + N * 100 + K)
    A = rand_f16(rng, (M, K))
    B = rand_f16(rng, (K, N))
    C = oracle.gemm_f64(A, B, M, N, K)
    E = oracle.exact_gemm(A, B, M, N, K)
    a = A.astype(np.float64)
    b = B.astype(np.float64)
    # recursive summation of K exact products: |error| <= (K-1) u sum|a b|, u = 2^-53
    bound = np.abs(a) @ np.abs(b) * (K * 2.0 ** -53)
    for i in range(M):
        for j in range(N):
            err = abs(Fraction(C[i, j]) - E[i][j])
            assert err <= Fraction(bound[i, j]), (i, j, float(err), bound[i, j])


@pytest.mark.parametrize("lda_pad,ldb_pad", [(1, 0), (0, 3), (5, 8)])
def test_strides_in_elements(lda_pad, ldb_pad):
    """Row strides larger than the row: padding (NaN here) is never read."""
    M, N, K = 5, 7, 9
    rng = np.random.default_rng(7)
    A = rand_f16(rng, (M, K))
    B = rand_f16(rng, (K, N))
    lda, ldb = K + lda_pad, N + ldb_pad
    C = oracle.gemm_f64(padded(A, lda), padded(B, ldb), M, N, K, lda=lda, ldb=ldb)
    E = oracle.exact_gemm(A, B, M, N, K)
    assert np.all(np.isfinite(C))
    for i in range(M):
        for j in range(N):
            assert abs(Fraction(C[i, j]) - E[i][j]) <= Fraction(2.0 ** -40)


def test_integer_inputs_are_exact():
    rng = np.random.default_rng(11)
    M, N, K = 37, 29, 300
    A = rng.integers(-4, 5, size=(M, K))
    B = rng.integers(-4, 5, size=(K, N))
    C = oracle.gemm_f64(A.astype(np.float16), B.astype(np.float16), M, N, K)
    assert np.array_equal(C, (A @ B).astype(np.float64))


def test_random_inputs_agree_with_numpy_float64():
    rng = np.random.default_rng(12)
    M, N, K = 64, 48, 1000
    A = rng.standard_normal((M, K)).astype(np.float16)
    B = rng.standard_normal((K, N)).astype(np.float16)
    C = oracle.gemm_f64(A, B, M, N, K)
    R = A.astype(np.float64) @ B.astype(np.float64)
    assert np.max(np.abs(C - R)) <= 1e-12 * np.max(np.abs(R))


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("M,N,K", [(64, 128, 128), (3, 5, 1), (17, 9, 1000)])
def test_all_ones_give_K(M, N, K):
    C = oracle.gemm_f64(np.ones((M, K), np.float16), np.ones((K, N), np.float16), M, N, K)
    assert np.all(C == K)


def test_all_ones_long_K_cells():
    """The 256 x 256 x 65536 shape: every sampled cell is exactly 65536."""
    M, N, K = 256, 256, 65536
    rows = np.array([0, 255, 17, 128, 200])
    cols = np.array([0, 255, 250, 3, 129])
    out = oracle.gemm_cells(np.ones((M, K), np.float16), np.ones((K, N), np.float16),
                            M, N, K, rows, cols)
    assert np.all(out == K)


def test_identity_copies_B():
    rng = np.random.default_rng(3)
    K, N = 33, 21
    B = rand_f16(rng, (K, N))
    C = oracle.gemm_f64(np.eye(K, dtype=np.float16), B, K, N, K)
    assert np.array_equal(C, B.astype(np.float64))


def test_identity_on_the_right_copies_A():
    rng = np.random.default_rng(4)
    M, K = 19, 40
    A = rand_f16(rng, (M, K))
    C = oracle.gemm_f64(A, np.eye(K, dtype=np.float16), M, K, K)
    assert np.array_equal(C, A.astype(np.float64))


def test_row_sum_worked_values_from_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "row_sum_worked_examples.json")))
    for case in g["row_sums"]:
        x = np.array(case["x"], dtype=np.float16)
        R, Kc = x.shape
        C = oracle.gemm_f64(x, np.ones((Kc, 1), np.float16), R, 1, Kc)
        assert C[:, 0].tolist() == case["expected"], case["cite"]


def test_masked_tiles_equal_zero_padding():
    """The pages' masked tile loads read 0 past the edge.  Zero-padding K up
    to whole tiles therefore must not change the result: the oracle with K
    rounded up and the pad zeroed equals the oracle on the true K."""
    g = json.load(open(os.path.join(GOLDEN, "row_sum_worked_examples.json")))
    rng = np.random.default_rng(5)
    for case in g["masked_tiles"]:
        n, blk = case["n_cols"], case["block"]
        tiles = -(-n // blk)
        masks = [[t * blk + l < n for l in range(blk)] for t in range(tiles)]
        assert masks == case["masks"], case["cite"]
        x = rand_f16(rng, (4, n))
        xpad = np.zeros((4, tiles * blk), np.float16)
        xpad[:, :n] = x
        ones = np.ones((tiles * blk, 1), np.float16)
        r_true = oracle.gemm_f64(x, ones[:n], 4, 1, n)
        r_pad = oracle.gemm_f64(xpad, ones, 4, 1, tiles * blk)
        assert np.array_equal(r_true, r_pad)
        ones_row = oracle.gemm_f64(np.ones((1, n), np.float16), ones[:n], 1, 1, n)
        assert ones_row[0, 0] == n
        if "acc_after_last_tile" in case:
            chunk = [1.0 if m else 0.0 for m in masks[-1]]
            assert chunk == case["acc_after_last_tile"]


def test_K_zero_is_the_empty_sum():
    C = oracle.gemm_f64(np.zeros((0,), np.float16), np.zeros((0,), np.float16), 3, 4, 0)
    assert np.all(C == 0.0)


# ---------------------------------------------------------------- invariants

def test_transpose_identity_is_bitwise():
    """(A.B)^T == B^T.A^T, cell for cell: the same products, summed in the same
    ascending k, so even random inputs agree bit for bit."""
    rng = np.random.default_rng(9)
    M, N, K = 23, 31, 77
    A = rand_f16(rng, (M, K))
    B = rand_f16(rng, (K, N))
    C = oracle.gemm_f64(A, B, M, N, K)
    Ct = oracle.gemm_f64(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T), N, M, K)
    assert np.array_equal(C, Ct.T)


def test_cells_equal_full_product():
    rng = np.random.default_rng(10)
    M, N, K = 40, 50, 123
    A = rand_f16(rng, (M, K))
    B = rand_f16(rng, (K, N))
    C = oracle.gemm_f64(A, B, M, N, K)
    rows = rng.integers(0, M, 200)
    cols = rng.integers(0, N, 200)
    assert np.array_equal(oracle.gemm_cells(A, B, M, N, K, rows, cols), C[rows, cols])


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(13)
    M, N, K = 57, 33, 500
    A = rand_f16(rng, (M, K))
    B = rand_f16(rng, (K, N))
    C1 = oracle.gemm_f64(A, B, M, N, K, nthreads=1)
    C3 = oracle.gemm_f64(A, B, M, N, K, nthreads=3)
    assert np.array_equal(C1, C3)


def special_values_case():
    """A small case with one NaN row and one +Inf entry in A (seeded, int4
    elsewhere, so the finite cells are exact), and what IEEE arithmetic
    makes of it: row 3 of C is all NaN; cell (5, j) is +Inf, -Inf or NaN as
    B[7, j] is positive, negative or zero (one infinite term per cell, so
    the summation order does not matter); every other cell is finite."""
    rng = np.random.default_rng(77)
    M, N, K = 16, 40, 24
    A = rng.integers(-4, 5, size=(M, K)).astype(np.float16)
    B = rng.integers(-4, 5, size=(K, N)).astype(np.float16)
    A[3, 10] = np.float16(np.nan)
    A[5, 7] = np.float16(np.inf)
    nan_cells = np.zeros((M, N), dtype=bool)
    nan_cells[3, :] = True
    nan_cells[5, :] = B[7, :] == 0
    pos_inf = np.zeros((M, N), dtype=bool)
    neg_inf = np.zeros((M, N), dtype=bool)
    pos_inf[5, :] = B[7, :] > 0
    neg_inf[5, :] = B[7, :] < 0
    return A, B, nan_cells, pos_inf, neg_inf


def test_nan_and_inf_propagate_as_ieee():
    A, B, nan_cells, pos_inf, neg_inf = special_values_case()
    M, K = A.shape
    N = B.shape[1]
    C = oracle.gemm_f64(A, B, M, N, K)
    assert np.array_equal(np.isnan(C), nan_cells)
    assert np.array_equal(np.isposinf(C), pos_inf)
    assert np.array_equal(np.isneginf(C), neg_inf)
    finite = ~(nan_cells | pos_inf | neg_inf)
    exact = np.where(np.isfinite(A), A, 0).astype(np.int64) @ B.astype(np.int64)
    assert np.array_equal(C[finite], exact[finite].astype(np.float64))


def test_rejects_bad_arguments():
    with pytest.raises(RuntimeError):
        oracle.gemm_cells(np.ones(4, np.float16), np.ones(4, np.float16), 2, 2, 2,
                          [2], [0])


# ---------------------------------------------------------------- planted mistakes

def _oracle_like(A, B, M, N, K, mistake=None):
    """A small copy of the definition with an optional planted mistake."""
    a = A.astype(np.float64)
    b = B.astype(np.float64)
    C = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                if mistake == "drop_last_k" and k == K - 1:
                    continue
                if mistake == "transposed_B":
                    s += a[i, k] * b.reshape(-1)[j * K + k] if j * K + k < b.size else 0.0
                elif mistake == "wrong_sign" and k % 2:
                    s -= a[i, k] * b[k, j]
                elif mistake == "swap_ij":
                    s += a[j % M, k] * b[k, i % N]
                else:
                    s += a[i, k] * b[k, j]
            if mistake == "f16_rounding":
                s = float(np.float16(s))
            C[i, j] = s
    return C


def _pins_pass(fn):
    rng = np.random.default_rng(21)
    ok = True
    for (M, N, K) in [(3, 5, 7), (2, 2, 2), (4, 1, 3)]:
        A = rand_f16(rng, (M, K))
        B = rand_f16(rng, (K, N))
        C = fn(A, B, M, N, K)
        E = oracle.exact_gemm(A, B, M, N, K)
        bound = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)) * (K * 2.0 ** -53)
        for i in range(M):
            for j in range(N):
                ok &= abs(Fraction(C[i, j]) - E[i][j]) <= Fraction(bound[i, j])
    C = fn(np.ones((2, 6), np.float16), np.ones((6, 3), np.float16), 2, 3, 6)
    ok &= bool(np.all(C == 6))
    return bool(ok)


def test_pins_catch_planted_mistakes():
    assert _pins_pass(lambda A, B, M, N, K: _oracle_like(A, B, M, N, K))
    assert _pins_pass(lambda A, B, M, N, K: oracle.gemm_f64(A, B, M, N, K))
    for mistake in ("drop_last_k", "transposed_B", "wrong_sign", "swap_ij", "f16_rounding"):
        assert not _pins_pass(lambda A, B, M, N, K, m=mistake: _oracle_like(A, B, M, N, K, m)), mistake
