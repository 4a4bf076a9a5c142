"""The GPU tests' comparison helpers, exercised on the CPU with results the
oracle itself produced (must pass) and with planted mistakes (must fail)."""
import numpy as np
import pytest

import oracle
from rmsnorm_fwd_gb300 import inputs

from _parity import compare, compare_mx, compare_quant


def test_compare_accepts_oracle_and_rejects_one_ulp_plus():
    x, w = inputs.random_case(8, 256, "bf16", seed=2)
    y = oracle.rmsnorm_bias(x, w, 0.75, 1e-6, "bf16")
    compare(y, x, w, 1e-6, "bf16", bias=0.75)
    bad = y.copy()
    bad[2, 9] += 2                       # two units in the last place
    with pytest.raises(AssertionError):
        compare(bad, x, w, 1e-6, "bf16", bias=0.75)
    with pytest.raises(AssertionError):  # the plain norm is not the biased one
        compare(oracle.rmsnorm(x, w, 1e-6, "bf16"), x, w, 1e-6, "bf16", bias=0.75)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_compare_mx_accepts_band_and_rejects_planted(dtype):
    x, w = inputs.random_case(64, 512, dtype, seed=1)
    c, s = oracle.rmsnorm_mxfp8(x, w, 0.5, 1e-6, dtype)
    assert compare_mx(c, s, x, w, 0.5, 1e-6, dtype)["exact_codes"] == 1.0
    # results within the band (a 3e-6 relative change of every value) pass
    c3, s3 = oracle.rmsnorm_mxfp8(x, w, 0.5, 1e-6, dtype, rel=3e-6)
    compare_mx(c3, s3, x, w, 0.5, 1e-6, dtype)
    # a code one step off, a scale one binade off, a 1e-3 relative error: fail
    c2 = c.copy()
    c2[3, 17] ^= 1
    with pytest.raises(AssertionError):
        compare_mx(c2, s, x, w, 0.5, 1e-6, dtype)
    s2 = s.copy()
    s2[5, 2] += 1
    with pytest.raises(AssertionError):
        compare_mx(c, s2, x, w, 0.5, 1e-6, dtype)
    c4, s4 = oracle.rmsnorm_mxfp8(x, w, 0.5, 1e-6, dtype, rel=1e-3)
    with pytest.raises(AssertionError):
        compare_mx(c4, s4, x, w, 0.5, 1e-6, dtype)


def test_compare_mx_band_scale_block():
    # A block whose maximum sits just below a power of two: a 1e-6 relative
    # change moves its scale; both choices (with their own codes) pass.
    x = np.zeros((1, 32), np.float32)
    x[0, :] = 1.0
    x[0, 0] = np.float32(np.sqrt(32.0))  # sets the row's RMS
    w = np.ones(32, np.float32)
    y = oracle.rmsnorm_bias_f64(x, w, 0.0, 0.0, "f32")
    # scale the weight so the maximum lands at 2^3 * (1 - 2e-6)
    k = (8.0 * (1 - 2e-6)) / y.max()
    w = (w * np.float32(k)).astype(np.float32)
    c, s = oracle.rmsnorm_mxfp8(x, w, 0.0, 0.0, "f32")
    chi, shi = oracle.rmsnorm_mxfp8(x, w, 0.0, 0.0, "f32", rel=1e-5)
    assert shi[0, 0] == s[0, 0] + 1
    assert compare_mx(c, s, x, w, 0.0, 0.0, "f32")["band_blocks"] == 1
    compare_mx(chi, shi, x, w, 0.0, 0.0, "f32")


@pytest.mark.parametrize("fmt,g", [("mxfp4", 1.0), ("nvfp4", 1.0), ("nvfp4", 0.004)])
def test_compare_quant_fp4_accepts_band_and_rejects_planted(fmt, g):
    x, w = inputs.random_case(48, 256, "bf16", seed=3)
    c, s = oracle.rmsnorm_fp4(x, w, 0.5, 1e-6, "bf16", fmt, global_scale=g)
    assert compare_quant(c, s, x, w, 0.5, 1e-6, "bf16", fmt, g)["exact_codes"] == 1.0
    c3, s3 = oracle.rmsnorm_fp4(x, w, 0.5, 1e-6, "bf16", fmt, global_scale=g, rel=3e-6)
    compare_quant(c3, s3, x, w, 0.5, 1e-6, "bf16", fmt, g)
    c2 = c.copy()
    nz = np.argwhere((c2 & 0x7) > 1)[0]      # a code with room to move down one step
    c2[tuple(nz)] -= 1
    with pytest.raises(AssertionError):
        compare_quant(c2, s, x, w, 0.5, 1e-6, "bf16", fmt, g)
    c2 = c.copy()
    c2[0, 0] ^= 0x88                          # both signs of the first byte flipped
    if (c[0, 0] & 0x77) != 0:
        with pytest.raises(AssertionError):
            compare_quant(c2, s, x, w, 0.5, 1e-6, "bf16", fmt, g)
    s2 = s.copy()
    s2[5, 2] += 1
    with pytest.raises(AssertionError):
        compare_quant(c, s2, x, w, 0.5, 1e-6, "bf16", fmt, g)
    with pytest.raises(AssertionError):     # the nibble order swapped
        compare_quant(((c & 0xF) << 4) | (c >> 4), s, x, w, 0.5, 1e-6, "bf16", fmt, g)


@pytest.mark.parametrize("fmt,g", [("mxfp8", 1.0), ("mxfp4", 1.0), ("nvfp4", 0.004)])
def test_compare_quant_checks_the_sign_of_zero_codes(fmt, g):
    """A zero weight with a -0 or +0 offset: the zero codes' signs follow the
    IEEE signs of (x * r) * (w + offset); a flipped zero sign is rejected."""
    x, w = inputs.random_case(8, 256, "bf16", seed=4)
    w = w.copy()
    w[:64] = 0x8000                             # -0.0 weights (bf16 bits)
    w[64:96] = 0x0000                           # +0.0 weights
    for bias in (-0.0, 0.0):
        if fmt == "mxfp8":
            c, s = oracle.rmsnorm_mxfp8(x, w, bias, 1e-6, "bf16")
        else:
            c, s = oracle.rmsnorm_fp4(x, w, bias, 1e-6, "bf16", fmt, global_scale=g)
        compare_quant(c, s, x, w, bias, 1e-6, "bf16", fmt, g)
        c2 = c.copy()
        if fmt == "mxfp8":
            c2[0, 0] ^= 0x80                    # column 0: a zero code, its sign flipped
        else:
            c2[0, 0] ^= 0x08
        with pytest.raises(AssertionError):
            compare_quant(c2, s, x, w, bias, 1e-6, "bf16", fmt, g)
    # the two offsets give different signs where x > 0 and w = -0
    c_m, _ = (oracle.rmsnorm_mxfp8(x, w, -0.0, 1e-6, "bf16") if fmt == "mxfp8" else
              oracle.rmsnorm_fp4(x, w, -0.0, 1e-6, "bf16", fmt, global_scale=g))
    c_p, _ = (oracle.rmsnorm_mxfp8(x, w, 0.0, 1e-6, "bf16") if fmt == "mxfp8" else
              oracle.rmsnorm_fp4(x, w, 0.0, 1e-6, "bf16", fmt, global_scale=g))
    assert (c_m != c_p).any()


def test_compare_quant_subnormal_results_band():
    """Row results in binary32's subnormal range (f32 rows of subnormal
    numbers, eps 1e-6: y about 2^-133) carry fewer than 24 bits, so a kernel
    that rounds twice can land a unit of 2^-149 away from the oracle's single
    rounding; the bar's absolute term (four such units) accepts that and
    still rejects a code one step off."""
    rng = np.random.default_rng(4)
    f = (rng.standard_normal((4, 64)) * 2.0 ** -143).astype(np.float32)
    x, w = f, np.ones(64, np.float32) * np.float32(1.5)
    for fmt, g in (("mxfp8", 1.0), ("nvfp4", 1.0)):
        c, s = (oracle.rmsnorm_mxfp8(x, w, 0.0, 1e-6, "f32") if fmt == "mxfp8"
                else oracle.rmsnorm_fp4(x, w, 0.0, 1e-6, "f32", fmt, global_scale=g))
        compare_quant(c, s, x, w, 0.0, 1e-6, "f32", fmt, g)
        # every result one unit of 2^-149 further from zero, and nearer to it
        for sgn in (1.0, -1.0):
            y = oracle.rmsnorm_bias_f64(x, w, 0.0, 1e-6, "f32")
            y32 = oracle.round_to(y, "f32").astype(np.float64)
            moved = np.copysign(np.maximum(np.abs(y32) + sgn * 2.0 ** -149, 0.0), y32)
            cm, sm = (oracle.mxfp8_quantize(moved) if fmt == "mxfp8"
                      else oracle.nvfp4_quantize(moved, g))
            compare_quant(cm, sm, x, w, 0.0, 1e-6, "f32", fmt, g)
    # a code one step off in a block the band leaves alone
    c, s = oracle.rmsnorm_mxfp8(x, w, 0.0, 1e-6, "f32")
    lo, _ = oracle.rmsnorm_mxfp8(x, w, 0.0, 1e-6, "f32", rel=-1e-5, absolute=2.0 ** -147)
    hi, _ = oracle.rmsnorm_mxfp8(x, w, 0.0, 1e-6, "f32", rel=1e-5, absolute=2.0 ** -147)
    i, j = np.argwhere((lo == c) & (hi == c) & (c != 0))[0]
    bad = c.copy()
    bad[i, j] ^= 1
    with pytest.raises(AssertionError):
        compare_quant(bad, s, x, w, 0.0, 1e-6, "f32", "mxfp8", 1.0)
