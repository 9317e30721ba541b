"""Pins for the fused-epilogue oracle (activation, scale and bias, output
rounding).

Each ties ``oracle.activation_f64`` / ``epilogue_f64`` / ``round_to_out`` to
something other than itself: table values of the standard normal CDF and of
the logistic function, odd-symmetry identities that a wrong constant or sign
breaks, limits, PyTorch's own float64 GELU (exact and tanh form) and SiLU,
a brute-force bfloat16 rounding that decodes candidate bit patterns
independently, and numpy's float16 on exact tie cases.
``test_epilogue_pins_catch_planted_mistakes`` plants typical slips in a
small copy and checks that some pin rejects each."""
import importlib.util
import math

import numpy as np
import pytest

import oracle

PHI_1 = 0.8413447460685429    # standard normal CDF at 1 (table value)
SIGMA_1 = 0.7310585786300049  # logistic function at 1, 1 / (1 + e^-1)


def test_table_values():
    f = oracle.activation_f64
    assert abs(f(np.array([1.0]), "gelu")[0] - PHI_1) < 1e-15
    assert abs(f(np.array([-1.0]), "gelu")[0] + (1 - PHI_1)) < 1e-15
    assert abs(f(np.array([1.0]), "silu")[0] - SIGMA_1) < 1e-15
    assert abs(f(np.array([-1.0]), "silu")[0] + (1 - SIGMA_1)) < 1e-15
    x = np.array([-3.0, -0.5, 0.0, 0.25, 7.0])
    np.testing.assert_array_equal(f(x, "relu"), [0, 0, 0, 0.25, 7])
    np.testing.assert_array_equal(f(x, "leaky_relu", 0.25), [-0.75, -0.125, 0, 0.25, 7])
    np.testing.assert_array_equal(f(x, "none"), x)


@pytest.mark.parametrize("name", ["gelu", "gelu_tanh", "silu", "relu"])
def test_odd_symmetry_identity(name):
    # f(x) - f(-x) = x: erf, tanh and (sigma(x) + sigma(-x) = 1) make every
    # one of these x * (an S-curve symmetric about 1/2)
    x = np.linspace(-6, 6, 241)
    d = oracle.activation_f64(x, name) - oracle.activation_f64(-x, name)
    np.testing.assert_allclose(d, x, rtol=0, atol=1e-14)


def test_leaky_relu_identity():
    x = np.linspace(0.1, 5, 50)
    f = oracle.activation_f64
    np.testing.assert_allclose(f(x, "leaky_relu", 0.1) - f(-x, "leaky_relu", 0.1), 1.1 * x,
                               rtol=1e-15)


def test_limits_and_the_tanh_approximation():
    f = oracle.activation_f64
    big = np.array([12.0, 30.0])
    np.testing.assert_allclose(f(big, "gelu"), big, rtol=1e-15)
    np.testing.assert_allclose(f(-big, "gelu"), 0.0, atol=1e-30)
    np.testing.assert_allclose(f(big, "silu"), big, rtol=1e-5)
    x = np.linspace(-4, 4, 801)
    # the tanh form approximates the erf form to within 5e-4 on [-4, 4]
    assert np.max(np.abs(f(x, "gelu_tanh") - f(x, "gelu"))) < 5e-4
    assert np.max(np.abs(f(x, "gelu_tanh") - f(x, "gelu"))) > 1e-5  # and is not the same function


def test_activations_match_the_library_routines():
    # PyTorch's own CPU implementations in float64 (independent code): the
    # exact GELU, the tanh form (its 0.044715 and sqrt(2/pi) constants
    # included, which the symmetry and band pins above cannot fix) and SiLU
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    x = np.linspace(-8, 8, 1601)
    t = torch.tensor(x, dtype=torch.float64)
    f = oracle.activation_f64
    np.testing.assert_allclose(f(x, "gelu"), F.gelu(t).numpy(), rtol=0, atol=1e-15)
    np.testing.assert_allclose(f(x, "gelu_tanh"), F.gelu(t, approximate="tanh").numpy(), rtol=0, atol=1e-14)
    np.testing.assert_allclose(f(x, "silu"), F.silu(t).numpy(), rtol=0, atol=1e-14)


def _bf16_brute(v: float) -> float:
    """Nearest bfloat16 to v, ties to the even bit pattern, by decoding the
    candidate patterns (the upper 16 bits of a binary32)."""
    if v == 0 or math.isnan(v):
        return v
    f32 = np.array([v], dtype=np.float64).astype(np.float32)  # only to find the neighbourhood
    bits = int(f32.view(np.uint32)[0]) >> 16
    cands = []
    for b in range(max(bits - 2, 0), min(bits + 3, 0xFFFF + 1)):
        val = float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0])
        if math.isnan(val):
            continue
        cands.append((abs(val - v), b & 1, val))
    cands.sort()
    best = [c for c in cands if c[0] == cands[0][0]]
    if len(best) > 1:
        best = [c for c in best if c[1] == 0]
    return best[0][2]


def test_bf16_rounding_against_brute_force():
    rng = np.random.default_rng(3)
    vals = np.concatenate([
        rng.normal(size=400) * 10.0 ** rng.integers(-6, 6, size=400),
        1 + np.arange(-8, 9) * 2.0 ** -9,               # ties and their neighbours near 1
        [3.0, -2.5, 1e-39, -3e-39, 2.0 ** -133, 1.5 * 2.0 ** -133],
    ])
    got = oracle.round_to_bf16(vals)
    want = np.array([_bf16_brute(float(v)) for v in vals])
    np.testing.assert_array_equal(got, want)
    assert oracle.round_to_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0           # tie -> even
    assert oracle.round_to_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert math.isinf(oracle.round_to_bf16(np.array([3.4e38 * 1.01]))[0])


def _bf16_exact_rational(v: float) -> float:
    """The same rounding element by element in exact rational arithmetic:
    |v| / 2^q rounded to the nearest integer (Python rounds exact halves to
    even), times 2^q, with q = max(e - 8, -133) for |v| = m 2^e."""
    from fractions import Fraction
    if v == 0.0 or math.isnan(v) or math.isinf(v):
        return v
    _, e = math.frexp(abs(v))
    q = max(e - 8, -133)
    y = float(round(Fraction(abs(v)) / Fraction(2) ** q) * Fraction(2) ** q)
    if y > (2.0 - 2.0 ** -7) * 2.0 ** 127:
        y = math.inf
    return math.copysign(y, v)


def test_bf16_rounding_vectorised_equals_exact_rational():
    """Ties and near-ties at every binade from the subnormal range to the
    overflow boundary, both signs, plus random values: the vectorised
    rounding must equal the element-by-element exact-rational one."""
    rng = np.random.default_rng(5)
    vals = [0.0, -0.0, math.inf, -math.inf]
    for e in range(-140, 129, 3):
        base = 2.0 ** e
        for k in (1, 2, 3, 255, 256, 257, 511):
            for d in (-1, 0, 1):
                vals.append((k + 0.5) * 2.0 ** (e - 8) + d * 2.0 ** (e - 40) if e - 40 > -1074 else (k + 0.5) * 2.0 ** (e - 8))
        vals.append(base * 1.5)
    vals += list(rng.normal(size=2000) * 10.0 ** rng.integers(-40, 38, size=2000))
    vals += [(2.0 - 2.0 ** -8) * 2.0 ** 127, (2.0 - 2.0 ** -9) * 2.0 ** 127, 3.4e38, 1.5 * 2.0 ** -133,
             2.5 * 2.0 ** -133, 0.5 * 2.0 ** -133, 0.75 * 2.0 ** -133]
    v = np.array(vals + [-x for x in vals], dtype=np.float64)
    got = oracle.round_to_bf16(v)
    want = np.array([_bf16_exact_rational(float(x)) for x in v])
    np.testing.assert_array_equal(got, want)


def test_f16_and_f32_rounding_tie_cases():
    r = oracle.round_to_out
    assert r(np.array([1 + 2.0 ** -11]), "f16")[0] == 1.0
    assert r(np.array([1 + 3 * 2.0 ** -11]), "f16")[0] == 1 + 2.0 ** -9
    assert math.isinf(r(np.array([65520.0]), "f16")[0])
    assert r(np.array([65519.0]), "f16")[0] == 65504.0
    assert r(np.array([1 + 2.0 ** -24]), "f32")[0] == 1.0
    assert r(np.array([1 + 3 * 2.0 ** -24]), "f32")[0] == 1 + 2.0 ** -22


def test_composition_order():
    e = oracle.epilogue_f64
    # bias before the activation: relu(-1 + 3) = 2 (after it would give 3)
    assert e(np.array([[-1.0]]), 1.0, [3.0], "relu")[0, 0] == 2.0
    # alpha scales the product only: 2 * 1 + 1 = 3 (scaling the bias would give 4)
    assert e(np.array([[1.0]]), 2.0, [1.0], "none")[0, 0] == 3.0
    # one bias per column, and per batch when given one per batch
    acc = np.zeros((2, 2, 3))
    out = e(acc, 1.0, np.array([[1.0, 2, 3], [4, 5, 6]]), "none")
    np.testing.assert_array_equal(out[1, 1], [4, 5, 6])
    np.testing.assert_array_equal(out[0, 0], [1, 2, 3])


# ---------------------------------------------------------------- planted mistakes

def _epi_like(acc, alpha, bias, name, slope=0.01, mistake=None):
    v = alpha * acc if mistake != "alpha_on_bias" else alpha * (acc + bias)
    if mistake not in ("alpha_on_bias", "bias_after"):
        v = v + bias
    if name == "gelu":
        arg = v if mistake == "erf_no_sqrt2" else v / math.sqrt(2.0)
        v = 0.5 * v * (1 + np.vectorize(math.erf)(arg))
    elif name == "gelu_tanh":
        k = 0.04715 if mistake == "tanh_cubic" else 0.044715
        c = math.sqrt(2.0 * math.pi) if mistake == "tanh_sqrt" else math.sqrt(2.0 / math.pi)
        v = 0.5 * v * (1 + np.tanh(c * (v + k * v ** 3)))
    elif name == "silu":
        v = v / (1 + np.exp(v if mistake == "silu_sign" else -v))
    elif name == "leaky_relu":
        v = np.where(v > 0, v, (-slope if mistake == "slope_sign" else slope) * v)
    elif name == "relu":
        v = np.maximum(v, 0)
    if mistake == "bias_after":
        v = v + bias
    return v


def _epi_pins_pass(fn):
    ok = True
    ok &= abs(fn(np.array([1.0]), 1.0, 0.0, "gelu")[0] - PHI_1) < 1e-15
    ok &= abs(fn(np.array([1.0]), 1.0, 0.0, "silu")[0] - SIGMA_1) < 1e-15
    ok &= fn(np.array([-1.0]), 1.0, 3.0, "relu")[0] == 2.0
    ok &= fn(np.array([1.0]), 2.0, 1.0, "relu")[0] == 3.0
    ok &= fn(np.array([-2.0]), 1.0, 0.0, "leaky_relu", 0.25)[0] == -0.5
    try:
        import torch
        x = np.array([-3.0, -1.0, 0.5, 2.0])
        ref = torch.nn.functional.gelu(torch.tensor(x, dtype=torch.float64), approximate="tanh").numpy()
        ok &= bool(np.all(np.abs(fn(x, 1.0, 0.0, "gelu_tanh") - ref) < 1e-14))
    except ImportError:
        pass
    return bool(ok)


def test_epilogue_pins_catch_planted_mistakes():
    assert _epi_pins_pass(lambda *a: _epi_like(*a))
    assert _epi_pins_pass(lambda acc, alpha, bias, name, slope=0.01: oracle.epilogue_f64(
        acc, alpha, np.array([bias]) if np.ndim(bias) == 0 else bias, name, slope))
    mistakes = ["alpha_on_bias", "bias_after", "erf_no_sqrt2", "silu_sign", "slope_sign"]
    if importlib.util.find_spec("torch") is not None:
        mistakes += ["tanh_cubic", "tanh_sqrt"]
    for m in mistakes:
        assert not _epi_pins_pass(lambda *a, m=m: _epi_like(*a, mistake=m)), m
