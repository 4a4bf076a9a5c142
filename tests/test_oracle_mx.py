"""Pins for the oracle's weight-bias rows and its MXFP8 quantiser: a block
worked by hand, every E4M3 code against torch's float8_e4m3fn, the rounding
against a brute-force nearest search over the finite codes, the scale's
defining invariant, the quantisation error bound and the special blocks.
CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from rmsnorm_fwd_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

FINITE = [c for c in range(256) if (c & 0x7F) != 0x7F]


def _golden():
    d = {}
    with open(os.path.join(GOLDEN, "mxfp8_hand_example.txt")) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                k, *v = line.split()
                d[k] = [float(t) for t in v]
    return d


def _decode(codes):
    return np.array([oracle.e4m3_value(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))


# ------------------------------------------------------------------ E4M3

def test_e4m3_decode_every_code_matches_torch():
    t = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    want = t.to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))
    assert max(got[ok]) == 448.0 and min(v for v in got[ok] if v > 0) == 2.0 ** -9


def test_e4m3_encode_round_trips_every_finite_code():
    for c in FINITE:
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c


def _brute_nearest(v):
    """Nearest finite E4M3 value by exhaustive search; ties go to the code
    whose fraction field is even; beyond the range the nearest is +-448."""
    best = None
    for c in FINITE:
        d = abs(oracle.e4m3_value(c) - v)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0 and (best[1] & 1)):
            best = (d, c)
    return best[1]


def test_e4m3_encode_matches_brute_force_nearest():
    rng = np.random.default_rng(5)
    vals = list(rng.choice([-1, 1], 400) * np.exp2(rng.uniform(-12, 10, 400)))
    pos = sorted({oracle.e4m3_value(c) for c in FINITE if oracle.e4m3_value(c) >= 0})
    mids = [(a + b) / 2 for a, b in zip(pos, pos[1:])]          # exact ties
    vals += mids + [m * (1 + 2 ** -40) for m in mids] + [m * (1 - 2 ** -40) for m in mids]
    vals += [-m for m in mids[::7]] + [448.0, 460.0, 464.0, 470.0, 1e6, -1e6, 2 ** -10, 2 ** -11]
    for v in vals:
        got = oracle.e4m3_encode(v)
        want = _brute_nearest(v)
        assert oracle.e4m3_value(got) == oracle.e4m3_value(want), (v, got, want)


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(6)
    v = (rng.choice([-1, 1], 5000) * np.exp2(rng.uniform(-11, 8.7, 5000))).astype(np.float32)
    v = v[np.abs(v) <= 448]
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(t)) for t in v], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_e4m3_saturates_and_keeps_nan():
    assert oracle.e4m3_value(oracle.e4m3_encode(1e30)) == 448.0
    assert oracle.e4m3_value(oracle.e4m3_encode(-math.inf)) == -448.0
    assert oracle.e4m3_encode(math.nan) & 0x7F == 0x7F
    assert oracle.e4m3_encode(-0.0) == 0x80


# ------------------------------------------------------------------ MX blocks

def test_mx_hand_example():
    g = _golden()
    v = np.array([g["v1"], [t * 2.0 ** -20 for t in g["v1"]],
                  [0.001] + [0.0] * 30 + [300.0]])
    codes, scales = oracle.mxfp8_quantize(v)
    assert scales[:, 0].tolist() == [g["s1"][0], g["s2"][0], g["s3"][0]]
    assert _decode(codes[0]).tolist() == g["q1"]
    assert _decode(codes[1]).tolist() == g["q1"]
    assert _decode(codes[2, :1]).tolist() == g["q3_first"]
    assert _decode(codes[2, -1:]).tolist() == g["q3_last"]


def _blocks(rng, n, lo=-140, hi=127):
    """n blocks of 32 with a random magnitude each and mixed signs."""
    mag = np.exp2(rng.uniform(lo, hi, n))[:, None]
    return rng.standard_normal((n, 32)) * mag


def test_mx_scale_invariant_and_error_bound():
    rng = np.random.default_rng(7)
    v = _blocks(rng, 3000)
    v[::97, :] = 0.0                                       # zero blocks
    codes, scales = oracle.mxfp8_quantize(v.reshape(-1, 64))
    codes = codes.reshape(-1, 32)
    scales = scales.reshape(-1)
    for b in range(v.shape[0]):
        amax = np.max(np.abs(v[b]))
        s = int(scales[b]) - 127
        X = 2.0 ** s
        if amax == 0:
            assert scales[b] == 0 and all(c in (0, 0x80) for c in codes[b])
            continue
        # the defining property of the shared exponent: max |v| / X in
        # [256, 512), unless the exponent sits at the bottom of the E8M0 range
        if s > -127:
            assert 256.0 <= amax / X < 512.0, (b, amax, s)
        else:
            assert amax / X < 512.0
        rec = _decode(codes[b]) * X
        t = v[b] / X
        for i in range(32):
            a = abs(t[i])
            if a >= 448:
                assert abs(rec[i]) == 448 * X and np.sign(rec[i]) == np.sign(t[i])
            elif a >= 2.0 ** -6:
                e = math.floor(math.log2(a))
                assert abs(rec[i] - v[b, i]) <= 2.0 ** (e - 4) * X   # half of 2^(e-3)
            else:
                assert abs(rec[i] - v[b, i]) <= 2.0 ** -10 * X        # half of 2^-9


def test_mx_special_blocks():
    v = np.zeros((4, 32))
    v[0, 3] = math.nan
    v[1, 5] = -math.inf
    v[2, :] = 2.0 ** -125                                  # scale clamps at 2^-127
    v[3, :] = 3.0e38                                       # floor(log2) = 127 -> s = 119
    codes, scales = oracle.mxfp8_quantize(v)
    assert scales[0, 0] == 0xFF and scales[1, 0] == 0xFF
    assert scales[2, 0] == 0
    assert set(_decode(codes[2]).tolist()) == {4.0}        # 2^-125 / 2^-127
    assert scales[3, 0] == 119 + 127
    with pytest.raises(ValueError):
        oracle.mxfp8_quantize(np.zeros((1, 48)))


# ------------------------------------------------------------------ weight bias

def test_bias_hand_example():
    # x = [3, 4] with w = 0 and bias 1 is the hand example with unit weights.
    x = np.asarray([[3, 4]], dtype=np.float32)
    y = oracle.rmsnorm_bias_f64(x, np.zeros(2, np.float32), 1.0, 0.0, "f32")[0]
    assert y == pytest.approx([3 * math.sqrt(2) / 5, 4 * math.sqrt(2) / 5], rel=1e-15)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_bias_against_plain_rows(dtype):
    x, w = inputs.random_case(5, 96, dtype, seed=3)
    # negative zero is the additive identity: the plain rows, bit for bit
    assert np.array_equal(oracle.rmsnorm_bias(x, w, -0.0, 1e-6, dtype),
                          oracle.rmsnorm(x, w, 1e-6, dtype))
    # a zero weight plus a bias b is the plain norm with every weight b
    b = 1.5
    wb = inputs.to_storage(np.full(96, b, np.float32), dtype)
    z = inputs.to_storage(np.zeros(96, np.float32), dtype)
    assert np.array_equal(oracle.rmsnorm_bias_f64(x, z, b, 1e-6, dtype),
                          oracle.rmsnorm_f64(x, wb, 1e-6, dtype))
    # linear in the bias: y(b) - y(0) = b * x * r = y(w = 0, b)
    d = oracle.rmsnorm_bias_f64(x, w, b, 1e-6, dtype) - oracle.rmsnorm_bias_f64(x, w, 0.0, 1e-6,
                                                                                dtype)
    ref = oracle.rmsnorm_bias_f64(x, z, b, 1e-6, dtype)
    assert np.allclose(d, ref, rtol=1e-12, atol=1e-14)


def test_bias_rows_match_single_head_qk_norm():
    # One head per token over the whole row: the QK oracle's arithmetic on the
    # same numbers (a separate loop nest in the oracle).
    x, w = inputs.random_case(6, 128, "bf16", seed=4)
    q, _ = oracle.qk_norm(x.ravel(), np.zeros(0, np.uint16), w, w, 6, 1, 0, 128, 128, 0, 0.25,
                          1e-6, "bf16")
    assert np.array_equal(q.reshape(6, 128), oracle.rmsnorm_bias(x, w, 0.25, 1e-6, "bf16"))


def test_rmsnorm_mxfp8_reconstructs_rows():
    x, w = inputs.random_case(4, 256, "bf16", seed=8)
    codes, scales = oracle.rmsnorm_mxfp8(x, w, 0.0, 1e-6, "bf16")
    y = oracle.rmsnorm_f64(x, w, 1e-6, "bf16")
    X = np.exp2(scales.astype(np.float64) - 127).repeat(32, axis=1)
    rec = _decode(codes) * X
    # E4M3 keeps 4 significant bits: relative error <= 2^-4 above the
    # subnormal range of each block
    big = np.abs(y) / X >= 2.0 ** -6
    assert np.all(np.abs(rec - y)[big] <= 2.0 ** -4 * np.abs(y)[big] * (1 + 1e-6))
    lo, _ = oracle.rmsnorm_mxfp8(x, w, 0.0, 1e-6, "bf16", rel=-1e-5)
    hi, _ = oracle.rmsnorm_mxfp8(x, w, 0.0, 1e-6, "bf16", rel=1e-5)
    # the bracket moves only codes near a rounding boundary
    assert np.mean(lo != hi) < 0.01
