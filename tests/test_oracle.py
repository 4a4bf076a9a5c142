"""Pins for the fp64 CPU oracle: worked examples, closed forms, invariants,
special cases, exact brute force on tiny inputs, and the format conversions
checked against numpy / torch / exact rational arithmetic.  CPU only."""
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from rmsnorm_fwd_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(vals):
    return np.asarray(vals, dtype=np.float32)


# --------------------------------------------------------------- worked examples

def _read_hand():
    d = {}
    with open(os.path.join(GOLDEN, "hand_example.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            d[k] = v
    return d


def test_hand_example_matches_closed_form():
    d = _read_hand()
    x = f32([float(v) for v in d["x"]])[None, :]
    w = f32([float(v) for v in d["w"]])
    y = oracle.rmsnorm_f64(x, w, float(d["eps"][0]), "f32")[0]
    want = [float(v) for v in d["y"]]
    assert y == pytest.approx(want, rel=1e-15, abs=0)
    # The closed form written in the fixture: [3, 4] * sqrt(2) / 5.
    assert y == pytest.approx([3 * math.sqrt(2) / 5, 4 * math.sqrt(2) / 5], rel=1e-15)
    # The divisor is the row length, not the row length minus one.
    assert not np.allclose(y, [0.6, 0.8])


def test_row_examples():
    n = 0
    with open(os.path.join(GOLDEN, "row_examples.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            eps_s, xs, ws, ys = (p.split() for p in line.split("|"))
            x = f32([float(v) for v in xs])[None, :]
            w = f32([float(v) for v in ws])
            y = oracle.rmsnorm_f64(x, w, float(eps_s[0]), "f32")[0]
            assert y == pytest.approx([float(v) for v in ys], rel=1e-15, abs=1e-300)
            n += 1
    assert n == 6


# --------------------------------------------------------------- invariants

def test_unit_weight_rms_closed_form():
    """With w = 1 the output row's RMS is exactly sqrt(S / (S + hidden*eps))."""
    rng = np.random.default_rng(1)
    for hidden, eps in ((7, 1e-5), (128, 1e-6), (333, 0.5), (1, 2.0)):
        x = f32(rng.standard_normal((5, hidden)) * rng.uniform(0.01, 10, (5, 1)))
        w = np.ones(hidden, np.float32)
        y = oracle.rmsnorm_f64(x, w, eps, "f32")
        xd = x.astype(np.float64)
        S = (xd * xd).sum(1)
        rms = np.sqrt((y * y).mean(1))
        e = float(np.float32(eps))
        assert rms == pytest.approx(np.sqrt(S / (S + hidden * e)), rel=1e-13)


def test_scale_invariance_eps_zero_powers_of_two_exact():
    """eps = 0: y(2^k x) == y(x) bit for bit (power-of-two scaling is exact)."""
    rng = np.random.default_rng(2)
    x = f32(rng.standard_normal((4, 50)))
    w = f32(rng.uniform(0, 2, 50))
    y0 = oracle.rmsnorm_f64(x, w, 0.0, "f32")
    for k in (-20, -3, 1, 7, 30):
        yk = oracle.rmsnorm_f64(f32(x * np.float32(2.0 ** k)), w, 0.0, "f32")
        assert np.array_equal(y0, yk)


def test_scale_invariance_general_c():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 40)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, 40).astype(np.float32)
    y0 = oracle.rmsnorm_f64(x, w, 0.0, "f32")
    for c in (0.37, 3.3, 1234.5):
        xc = (x.astype(np.float64) * c)
        # Build xc exactly representable: use the binary32 rounding of c*x and
        # compare against the oracle on that same input (invariance up to the
        # input rounding, which is relative 2^-24 per element).
        yc = oracle.rmsnorm_f64(xc.astype(np.float32), w, 0.0, "f32")
        assert yc == pytest.approx(y0, rel=2e-7, abs=1e-7)


def test_scale_with_eps_closed_form():
    """eps > 0: y(c x) / y(x) = c * sqrt((S/h + eps) / (c^2 S/h + eps))."""
    x = f32([[1.0, -2.0, 0.5, 4.0]])
    w = f32([1.0, 1.0, 1.0, 1.0])
    eps = 0.25
    S = 1 + 4 + 0.25 + 16
    for c in (0.5, 2.0, 8.0):
        y1 = oracle.rmsnorm_f64(x, w, eps, "f32")
        yc = oracle.rmsnorm_f64(f32(x * c), w, eps, "f32")
        ratio = c * math.sqrt((S / 4 + eps) / (c * c * S / 4 + eps))
        assert yc == pytest.approx(y1 * ratio, rel=1e-14)


# --------------------------------------------------------------- special cases

def test_hidden_one():
    """hidden = 1: y = x / sqrt(x^2 + eps) * w; with eps = 0 it is sign(x) * w."""
    x = f32([[3.0], [-0.5], [1e-3]])
    w = f32([2.0])
    y = oracle.rmsnorm_f64(x, w, 0.0, "f32")[:, 0]
    assert list(y) == [2.0, -2.0, 2.0]
    y = oracle.rmsnorm_f64(x, w, 1.0, "f32")[:, 0]
    xd = x[:, 0].astype(np.float64)
    assert y == pytest.approx(xd / np.sqrt(xd * xd + 1.0) * 2.0, rel=1e-15)


def test_constant_row():
    a, eps, h = 0.75, 0.0625, 9
    x = np.full((1, h), a, np.float32)
    w = np.arange(1, h + 1, dtype=np.float32)
    y = oracle.rmsnorm_f64(x, w, eps, "f32")[0]
    assert y == pytest.approx(a / math.sqrt(a * a + eps) * np.arange(1, h + 1), rel=1e-15)


def test_weight_indexed_by_column():
    """Each output column j takes weight j (not the row index)."""
    x = np.ones((3, 5), np.float32)
    w = f32([10, 20, 30, 40, 50])
    y = oracle.rmsnorm_f64(x, w, 0.0, "f32")
    for i in range(3):
        assert list(y[i]) == [10, 20, 30, 40, 50]


def test_zero_weight_gives_zero():
    rng = np.random.default_rng(4)
    x = f32(rng.standard_normal((2, 17)))
    y = oracle.rmsnorm_f64(x, np.zeros(17, np.float32), 1e-6, "f32")
    assert np.all(y == 0)


def test_zero_row():
    x = np.zeros((2, 8), np.float32)
    w = np.ones(8, np.float32)
    assert np.all(oracle.rmsnorm_f64(x, w, 1e-5, "f32") == 0)
    assert np.all(np.isnan(oracle.rmsnorm_f64(x, w, 0.0, "f32")))


def test_rows_are_independent_and_not_transposed():
    """Normalisation is per row: each row alone gives the same result, and
    with w = 1 every row (not every column) has RMS ~ 1."""
    rng = np.random.default_rng(5)
    x = f32(rng.standard_normal((6, 11)) * np.array([[0.01], [1], [100], [3], [0.5], [7]]))
    w = np.ones(11, np.float32)
    y = oracle.rmsnorm_f64(x, w, 0.0, "f32")
    for i in range(6):
        assert np.array_equal(y[i], oracle.rmsnorm_f64(x[i:i + 1], w, 0.0, "f32")[0])
    assert np.sqrt((y * y).mean(1)) == pytest.approx(np.ones(6), rel=1e-14)
    assert not np.allclose(np.sqrt((y * y).mean(0)), 1.0, rtol=1e-3)


def test_nonfinite_propagates():
    x = f32([[1.0, np.inf, 2.0], [1.0, np.nan, 0.0]])
    w = np.ones(3, np.float32)
    y = oracle.rmsnorm_f64(x, w, 1e-6, "f32")
    assert np.isnan(y[1]).all()
    assert np.isnan(y[0, 1])  # inf * (1/inf) = inf * 0 = nan


def test_bad_arguments_rejected():
    with pytest.raises(ValueError):
        oracle.rmsnorm_f64(np.zeros((2, 3), np.float32), np.zeros(4, np.float32), 0.0, "f32")
    with pytest.raises(TypeError):
        oracle.rmsnorm_f64(np.zeros((2, 3), np.float64), np.zeros(3, np.float64), 0.0, "f32")


# --------------------------------------------------------------- exact brute force

def _exact_row(xs, ws, eps, digits=60):
    """High-precision restatement: exact rational sum of squares, then a
    60-digit decimal square root."""
    getcontext().prec = digits
    S = sum((Fraction(v) * Fraction(v) for v in xs), Fraction(0))
    m = S / len(xs) + Fraction(eps)
    r = 1 / (Decimal(m.numerator) / Decimal(m.denominator)).sqrt()
    return [Decimal(float(v)) * r * Decimal(float(wv)) for v, wv in zip(xs, ws)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_bruteforce_tiny(dtype):
    rng = np.random.default_rng(6)
    for trial in range(25):
        rows = int(rng.integers(1, 6))
        hidden = int(rng.integers(1, 18))
        eps = float(np.float32(rng.choice([0.0, 1e-6, 1e-2, 1.5])))
        xf = rng.standard_normal((rows, hidden)).astype(np.float32) * np.float32(rng.uniform(0.1, 4))
        wf = rng.uniform(-2, 2, hidden).astype(np.float32)
        x = inputs.to_storage(xf, dtype)
        w = inputs.to_storage(wf, dtype)
        xd, wd = oracle.widen(x, dtype), oracle.widen(w, dtype)
        y = oracle.rmsnorm_f64(x, w, eps, dtype)
        for i in range(rows):
            if eps == 0.0 and not np.any(xd[i]):
                continue
            want = _exact_row(list(xd[i]), list(wd), eps)
            for j in range(hidden):
                assert y[i, j] == pytest.approx(float(want[j]), rel=4e-16, abs=1e-300)
        # Rounded output equals exact nearest-even rounding of the fp64 value.
        yr = oracle.rmsnorm(x, w, eps, dtype)
        assert np.array_equal(yr.view(np.uint8), oracle.round_to(y, dtype).view(np.uint8))


# --------------------------------------------------------------- formats

def _exact_rne(v: float, p: int, emin: int, emax: int) -> float:
    """Nearest-even rounding via exact rationals (brute force)."""
    if v == 0 or not math.isfinite(v):
        return v
    a = Fraction(abs(v))
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    q = Fraction(2) ** (e - p + 1)
    n = a / q
    fl = math.floor(n)
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * q
    maxf = (2 ** p - 1) * Fraction(2) ** (emax - p + 1)
    out = math.inf if r > maxf else float(r)
    return out if v > 0 else -out


def test_widen_all_f16_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_widen_all_bf16_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.widen(bits, "bf16")
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def _probe_values(rng, n=20000):
    mags = np.exp2(rng.uniform(-150, 130, n)) * rng.choice([-1, 1], n)
    return mags


def test_round_f16_matches_numpy():
    rng = np.random.default_rng(7)
    v = np.concatenate([_probe_values(rng),
                        # exact ties and near-ties around 1, subnormals and overflow
                        [1 + 2 ** -11, 1 + 3 * 2 ** -11, 1 + 2 ** -11 + 2 ** -40, 2 ** -25,
                         3 * 2 ** -25, 2 ** -26, 65504.0, 65519.99, 65520.0, 1e6, -65520.0,
                         6.1e-5, 5.96e-8, 2.98e-8]])
    got = oracle.round_to(v, "f16")
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_round_f32_matches_numpy():
    rng = np.random.default_rng(8)
    v = np.concatenate([_probe_values(rng), [1 + 2 ** -24, 1 + 3 * 2 ** -24, 2 ** -150,
                                             3 * 2 ** -150, 3.5e38, 3.4028235677973366e38]])
    got = oracle.round_to(v, "f32")
    with np.errstate(over="ignore"):
        want = v.astype(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_round_bf16_matches_torch_on_binary32_values():
    rng = np.random.default_rng(9)
    with np.errstate(over="ignore"):             # magnitudes beyond binary32 become inf
        v32 = _probe_values(rng).astype(np.float32)
    v32 = v32[np.isfinite(v32)]
    got = oracle.round_to(v32.astype(np.float64), "bf16")
    want = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_round_bf16_exact_from_binary64():
    """Values with bits beyond binary32 (where rounding through binary32 first
    would round twice) against exact rational nearest-even."""
    rng = np.random.default_rng(10)
    vals = [1 + 2 ** -8 + 2 ** -40, 1 + 2 ** -8 - 2 ** -40, 1 + 2 ** -8, 1 + 3 * 2 ** -8,
            2 ** -133, 1.5 * 2 ** -133, 2 ** -134, 2 ** -134 + 2 ** -170, 3.3e38, 3.4e38]
    vals += list(_probe_values(rng, 3000))
    for v in vals:
        got = oracle.round_to(np.array([v]), "bf16")
        g = oracle.widen(got, "bf16")[0]
        assert g == _exact_rne(v, 8, -126, 127) or (math.isinf(g) and math.isinf(
            _exact_rne(v, 8, -126, 127))), v


def test_rounded_output_consistent_with_f64():
    x, w = inputs.make_inputs("f32_64x128")
    for dt in ("bf16", "f16"):
        xs = inputs.to_storage(x, dt)
        ws = inputs.to_storage(w, dt)
        y64 = oracle.rmsnorm_f64(xs, ws, 1e-6, dt)
        yr = oracle.rmsnorm(xs, ws, 1e-6, dt)
        assert np.array_equal(yr, oracle.round_to(y64, dt))
        # rounding error at most half an ulp of the format: relative 2^-8 / 2^-11
        rel = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}[dt]
        back = oracle.widen(yr, dt)
        big = np.abs(y64) > 1e-3
        assert np.all(np.abs(back - y64)[big] <= rel * np.abs(y64)[big])
