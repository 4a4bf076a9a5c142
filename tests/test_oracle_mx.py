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


# ------------------------------------------------------------------ E2M1, MXFP4, NVFP4

E2M1_CODES = list(range(16))


def _golden_fp4():
    d = {}
    with open(os.path.join(GOLDEN, "fp4_hand_example.txt")) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                k, *v = line.split()
                d[k] = [float(t) for t in v]
    return d


def _unpack(codes, cols):
    """[rows, cols / 2] packed bytes -> [rows, cols] 4-bit codes (even element low)."""
    lo = codes & 0xF
    hi = codes >> 4
    out = np.empty((codes.shape[0], cols), dtype=np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def _e2m1(codes):
    return np.array([oracle.e2m1_value(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))


def test_e2m1_values_and_brute_force_rounding():
    mags = [oracle.e2m1_value(c) for c in range(8)]
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [oracle.e2m1_value(c + 8) for c in range(8)] == [-m for m in mags]
    pos = sorted(set(mags))
    mids = [(a + b) / 2 for a, b in zip(pos, pos[1:])]
    rng = np.random.default_rng(9)
    vals = list(rng.uniform(-8, 8, 500)) + mids + [-m for m in mids] + \
        [m * (1 + 1e-9) for m in mids] + [m * (1 - 1e-9) for m in mids] + [7.0, -100.0, 1e30]
    from fractions import Fraction
    for v in vals:
        best = None
        for c in E2M1_CODES:
            dd = abs(Fraction(oracle.e2m1_value(c)) - Fraction(v))   # exact distances
            if best is None or dd < best[0] or (dd == best[0] and (c & 1) == 0 and (best[1] & 1)):
                best = (dd, c)
        got = oracle.e2m1_encode(v)
        assert oracle.e2m1_value(got) == oracle.e2m1_value(best[1]), (v, got, best)
    for c in E2M1_CODES:
        if c != 8:   # -0 encodes as 8, +0 as 0
            assert oracle.e2m1_encode(oracle.e2m1_value(c)) == c


def test_fp4_hand_examples():
    g = _golden_fp4()
    v = np.arange(1, 33, dtype=np.float64)[None, :]
    codes, scales = oracle.mxfp4_quantize(v)
    assert scales[0, 0] == g["mx4_scale"][0]
    assert codes[0, :4].tolist() == g["mx4_bytes0_3"]          # the nibble order
    q = _e2m1(_unpack(codes, 32))[0]
    assert q[:8].tolist() == g["mx4_first8"] and q[-2:].tolist() == g["mx4_last2"]
    codes, scales = oracle.nvfp4_quantize(v, 1.0)
    assert scales[0].tolist() == g["nv4_scales"]
    q = _e2m1(_unpack(codes, 32))[0]
    assert q[:4].tolist() == g["nv4_first4"] and q[15] == g["nv4_last_of_block0"][0]
    assert [q[16], q[31]] == g["nv4_block1_first_last"]


def test_mxfp4_invariant_and_error_bound():
    rng = np.random.default_rng(10)
    v = _blocks(rng, 2000, lo=-130, hi=120)
    v[::89] = 0.0
    codes, scales = oracle.mxfp4_quantize(v.reshape(-1, 64))
    q = _e2m1(_unpack(codes, 64)).reshape(-1, 32)
    scales = scales.reshape(-1)
    for b in range(v.shape[0]):
        amax = np.max(np.abs(v[b]))
        s = int(scales[b]) - 127
        X = 2.0 ** s
        if amax == 0:
            assert scales[b] == 0 and not q[b].any()
            continue
        if s > -127:
            assert 4.0 <= amax / X < 8.0, (b, amax, s)   # the shared exponent's definition
        t = np.abs(v[b]) / X
        rec = q[b] * X
        for i in range(32):
            if t[i] >= 6:
                assert abs(q[b, i]) == 6
            else:
                step = 0.5 if t[i] < 2 else 2.0 ** (np.floor(np.log2(t[i])) - 1)
                assert abs(rec[i] - v[b, i]) <= step / 2 * X


def test_nvfp4_scale_and_error_bound():
    rng = np.random.default_rng(11)
    for g in (1.0, 3.7e-3, 250.0):
        v = _blocks(rng, 1500, lo=-20, hi=20) * g
        v[::97] = 0.0
        codes, scales = oracle.nvfp4_quantize(v.reshape(-1, 64), g)
        q = _e2m1(_unpack(codes, 64)).reshape(-1, 16)
        s = np.array([oracle.e4m3_value(c) for c in scales.reshape(-1)])
        vb = v.reshape(-1, 16)
        for b in range(vb.shape[0]):
            amax = np.max(np.abs(vb[b]))
            t = amax / (6 * g)
            # the scale is E4M3's rounding of max / (6 g): within half a step
            if 2.0 ** -6 <= t <= 448:
                assert abs(s[b] - t) <= 2.0 ** (np.floor(np.log2(t)) - 4) * (1 + 1e-12)
            if s[b] == 0:
                assert not q[b].any()
                continue
            d = s[b] * g
            tt = np.abs(vb[b]) / d
            for i in range(16):
                if tt[i] >= 6:
                    assert abs(q[b, i]) == 6
                else:
                    step = 0.5 if tt[i] < 2 else 2.0 ** (np.floor(np.log2(tt[i])) - 1)
                    assert abs(q[b, i] * d - vb[b, i]) <= step / 2 * d * (1 + 1e-12)
    # special blocks and argument checks
    v = np.zeros((3, 16))
    v[1, 4] = np.nan
    v[2, :] = 1e-30
    codes, scales = oracle.nvfp4_quantize(v, 1.0)
    assert scales[0, 0] == 0 and not codes[0].any()
    assert scales[1, 0] == 0x7F
    assert scales[2, 0] == 0 and not (codes[2] & 0x77).any()   # signed zeros only
    with pytest.raises(ValueError):
        oracle.nvfp4_quantize(np.zeros((1, 24)), 1.0)
    with pytest.raises(ValueError):
        oracle.nvfp4_quantize(np.zeros((1, 16)), 0.0)


def test_nvfp4_extreme_global_scales_saturate_or_vanish():
    """Closed forms at the per-tensor scales the GPU tests use outside the
    flush-to-zero range: with g = 1e-37 every nonzero block's max / (6 g) is
    far above 448, so the scale saturates to 448 (code 0x7E) and each element
    becomes E2M1(v / (448 g)): +-6 for |v / (448 g)| >= 5, the rest follow the
    E2M1 grid; with g = 1e31 max / (6 g) is far below E4M3's smallest
    subnormal half-step (2^-10), so the scale is 0 and every code is a zero of
    the element's sign."""
    rng = np.random.default_rng(21)
    v = rng.standard_normal((8, 64))
    v[3, 16:32] = 0.0
    codes, scales = oracle.nvfp4_quantize(v, 1e-37)
    q = _e2m1(_unpack(codes, 64)).reshape(8, 64)
    for r in range(8):
        for b in range(4):
            blk = v[r, 16 * b:16 * (b + 1)]
            if not blk.any():
                assert scales[r, b] == 0 and not q[r, 16 * b:16 * (b + 1)].any()
                continue
            assert scales[r, b] == 0x7E                     # 448
            t = np.abs(blk) / (448 * 1e-37)
            assert (np.abs(q[r, 16 * b:16 * (b + 1)])[t >= 5] == 6).all()
            assert np.array_equal(np.sign(q[r, 16 * b:16 * (b + 1)])[t >= 5],
                                  np.sign(blk)[t >= 5])
    codes, scales = oracle.nvfp4_quantize(v, 1e31)
    assert not scales.any()
    q = _e2m1(_unpack(codes, 64)).reshape(8, 64)
    assert not q.any()
    nz = v != 0
    assert np.array_equal(np.signbit(q)[nz], np.signbit(v)[nz])


def test_zero_weight_codes_carry_the_ieee_sign_of_the_product():
    """(x * r) * (w + offset) with w = -0: offset -0 keeps w = -0, so the
    zero code's sign is the opposite of x's; offset +0 makes w + 0 = +0, so
    it is x's own sign (MXFP8 bytes 0x80 / 0x00, E2M1 nibbles 0x8 / 0x0)."""
    x, w = inputs.random_case(4, 64, "bf16", seed=8)
    w = w.copy()
    w[:32] = 0x8000                                     # bf16 -0.0
    xs = np.signbit(oracle.widen(x, "bf16"))[:, :32]
    for bias, flip in ((-0.0, True), (0.0, False)):
        c8, _ = oracle.rmsnorm_mxfp8(x, w, bias, 1e-6, "bf16")
        assert np.array_equal(c8[:, :32] == 0x80, xs != flip)
        assert np.isin(c8[:, :32], (0x00, 0x80)).all()
        c4, _ = oracle.rmsnorm_fp4(x, w, bias, 1e-6, "bf16", "nvfp4", global_scale=0.01)
        nib = _unpack(c4, 64)[:, :32]
        assert np.isin(nib, (0x0, 0x8)).all()
        assert np.array_equal(nib == 0x8, xs != flip)
