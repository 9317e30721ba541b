"""Pins for the row-sum and GEMV oracles.

``oracle.rowsum_f64`` is checked against the worked values the row-sum page
prints, against the page's own tiled algorithm (masks, zero-padded lanes)
re-expressed in small Python, against exact rational brute force over
strided views for all three element types, and against the GEMM oracle with
a column of ones (two independent codes).  ``oracle.gemv_f64`` is checked
by brute force with strided x.  Planted mistakes (the -inf padding trap the
page describes, a dropped last tile, swapped strides, summing in f16) must
each fail a pin."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

from test_oracle_pins import rand_f16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "row_sum_worked_examples.json")


def _golden():
    return json.load(open(GOLDEN))


def test_worked_values_from_the_page():
    for case in _golden()["row_sums"]:
        x = np.array(case["x"], dtype=np.float32)
        R, C = x.shape
        for elem, buf in (("f32", x), ("f16", x.astype(np.float16)),
                          ("bf16", (x.view(np.uint32) >> 16).astype(np.uint16))):
            got = oracle.rowsum_f64(buf.reshape(-1), R, C, C, 1, elem)
            assert got.tolist() == case["expected"], (case["cite"], elem)


def _tiled_row_sum(x, C, block, pad=0.0, drop_last=False, f16_acc=False):
    """The page's kernel for one row, in Python: a BLOCK-wide accumulator,
    masked tile loads that read `pad` past the row, one tree sum at the end.
    Returns (sum, masks)."""
    acc = np.zeros(block, dtype=np.float16 if f16_acc else np.float64)
    masks = []
    starts = list(range(0, C, block))
    if drop_last:
        starts = starts[:-1]
    for off in starts:
        idx = off + np.arange(block)
        mask = idx < C
        masks.append(mask.tolist())
        chunk = np.where(mask, x[np.minimum(idx, C - 1)], pad)
        acc = acc + chunk.astype(acc.dtype)
    return float(np.sum(acc.astype(np.float64))), masks


def test_the_pages_masks_and_tiled_sum():
    g = _golden()
    for case in g["masked_tiles"]:
        C, block = case["n_cols"], case["block"]
        x = np.ones(C)
        s, masks = _tiled_row_sum(x, C, block)
        assert masks == case["masks"], case["cite"]
        assert s == oracle.rowsum_f64(np.ones(C, np.float32), 1, C, C, 1, "f32")[0] == C
    rng = np.random.default_rng(4)
    for C in (1, 3, 5, 16, 33, 100):
        x = rand_f16(rng, (C,)).astype(np.float64)
        for block in (4, 8, 32):
            s, _ = _tiled_row_sum(x, C, block)
            ref = oracle.rowsum_f64(x.astype(np.float16), 1, C, C, 1, "f16")[0]
            assert abs(s - ref) <= C * 2.0 ** -52 * np.sum(np.abs(x))


@pytest.mark.parametrize("elem", ["f32", "f16", "bf16"])
def test_strided_views_against_exact_rationals(elem):
    rng = np.random.default_rng(5)
    for (R, C, rs, cs) in [(3, 5, 11, 2), (4, 1, 1, 1), (2, 7, 7, 1), (5, 3, 2, 5), (1, 9, 0, 3)]:
        size = (R - 1) * rs + (C - 1) * cs + 1
        vals = rng.normal(size=size) * 10.0 ** rng.integers(-3, 4, size=size)
        if elem == "f32":
            buf = vals.astype(np.float32)
            exact = [Fraction(float(v)) for v in buf]
        elif elem == "f16":
            buf = vals.astype(np.float16)
            exact = [Fraction(float(v)) for v in buf]
        else:
            f = vals.astype(np.float32)
            buf = (f.view(np.uint32) >> 16).astype(np.uint16)   # truncated: any bf16 pattern will do
            exact = [Fraction(float((np.array([b], np.uint32) << 16).view(np.float32)[0])) for b in buf]
        got = oracle.rowsum_f64(buf, R, C, rs, cs, elem)
        for r in range(R):
            s = sum((exact[r * rs + c * cs] for c in range(C)), Fraction(0))
            assert abs(Fraction(got[r]) - s) <= abs(s) * Fraction(2) ** -52 + Fraction(2) ** -1074


def test_row_sum_equals_the_gemm_with_ones():
    rng = np.random.default_rng(6)
    R, C = 37, 203
    X = rand_f16(rng, (R, C))
    a = oracle.rowsum_f64(X, R, C, C, 1, "f16")
    b = oracle.gemm_f64(X, np.ones((C, 1), np.float16), R, 1, C)[:, 0]
    bound = C * 2.0 ** -52 * np.abs(X.astype(np.float64)).sum(axis=1)
    assert np.all(np.abs(a - b) <= bound)


def test_gemv_against_exact_rationals():
    rng = np.random.default_rng(7)
    M, K, lda, incx = 6, 9, 11, 3
    A = rand_f16(rng, (M * lda,))
    x = rand_f16(rng, ((K - 1) * incx + 1,))
    y = oracle.gemv_f64(A, x, M, K, lda, incx)
    fa = [Fraction(float(v)) for v in A]
    fx = [Fraction(float(v)) for v in x]
    for i in range(M):
        s = sum((fa[i * lda + k] * fx[k * incx] for k in range(K)), Fraction(0))
        bound = sum((abs(fa[i * lda + k] * fx[k * incx]) for k in range(K)), Fraction(0)) * K * Fraction(2) ** -53
        assert abs(Fraction(y[i]) - s) <= bound


def test_row_sum_pins_catch_planted_mistakes():
    g = _golden()

    def passes(fn):
        ok = True
        for case in g["row_sums"]:
            x = np.array(case["x"], dtype=np.float64)
            ok &= [fn(row) for row in x] == case["expected"]
        rng = np.random.default_rng(8)
        x = rand_f16(rng, (70,)).astype(np.float64)
        ref = oracle.rowsum_f64(x.astype(np.float16), 1, 70, 70, 1, "f16")[0]
        ok &= abs(fn(x) - ref) <= 70 * 2.0 ** -52 * np.sum(np.abs(x))
        return bool(ok)

    assert passes(lambda row: _tiled_row_sum(row, row.size, 4)[0])
    assert not passes(lambda row: _tiled_row_sum(row, row.size, 4, pad=-math.inf)[0])   # the -inf trap
    assert not passes(lambda row: _tiled_row_sum(row, row.size, 4, drop_last=True)[0])
    assert not passes(lambda row: _tiled_row_sum(row, row.size, 4, f16_acc=True)[0])
