"""GPU parity at the ends of the element types' range.

The squares are summed in fp32 ("CuTeDSL at Perplexity", section "QK
Norm"), but bf16 and f32 elements reach fp32's whole exponent range: rows
scaled by 2^64 and more overflow that sum, rows scaled by 2^-63 and less lose
their squares to underflow.  The definition (mean of the squares, plus eps,
reciprocal square root, times x and the weight -- "Build a GPU compiler from
scratch ... (Emmy)", section "Tensor IR") has no such limit, and the oracle
computes it in binary64.  Every variant and element type must match the
oracle at the usual bar on:

* rows scaled by powers of two from 2^-145 (f32 subnormals) to 2^126, each
  row its own scale, so rows that need the range guard's redo sit beside
  rows that do not in one warp, block or launch; eps = 0 and eps = 1e-6;
* rows of subnormal numbers with eps = 0 (the factor exceeds the float range
  and x is scaled up before the scaling pass);
* rows mixing one huge element with ordinary ones, and halves of a row at
  opposite ends of the range (the cluster and grid variants' per-block
  partial sums at different scales);
* the weight-offset and block-scaled outputs, the per-head QK norm;
* NaN, +-Inf and subnormal elements in x and in the weight, -0 and +0
  weights, through the plain and weight-offset outputs of every variant
  (non-finite values propagate by IEEE arithmetic, as in the oracle).
"""
import numpy as np
import pytest

import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import compare, compare_quant, from_device, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rn.ensure_context(0)
    yield
    torch.cuda.synchronize()
    assert rn.rmsnorm_get_device_status() == rn.OK


VARIANTS = [rn.VARIANT_AUTO, rn.VARIANT_WARP_PER_ROW, rn.VARIANT_CTA_PER_ROW,
            rn.VARIANT_STAGED, rn.VARIANT_PERSISTENT, rn.VARIANT_GENERIC, rn.VARIANT_CLUSTER,
            rn.VARIANT_GRID]

# Row scale exponents: both ends of fp32's range and the band around the
# guard's thresholds (sums near 2^-100 and 2^128), plus ordinary rows.
EXPS = {
    "bf16": [-133, -130, -126, -120, -110, -100, -90, -80, -70, -64, -60, -50, 0, 50, 60, 63,
             64, 70, 80, 90, 100, 110, 120, 126],
    "f32": [-145, -140, -133, -126, -120, -110, -100, -90, -80, -70, -64, -60, -50, 0, 50, 60,
            63, 64, 70, 80, 90, 100, 110, 120, 126],
    # f16 squares stay inside fp32's range; its own range ends instead (2^14 is
    # the top binade that 3.9 * 2^e keeps below f16's largest value, 65504;
    # Inf entries are the non-finite test's)
    "f16": [-24, -20, -14, -10, 0, 5, 10, 13, 14],
}


def accepts(rows, hidden, dtype, variant):
    if rows == 0:
        return True
    sms, optin = rn.rmsnorm_device_limits()
    base = 1 << 30
    rc, _ = rn.rmsnorm_plan_status(base, 3 * base, 5 * base, rows, hidden, rn.DTYPE_CODES[dtype],
                                   sms, optin, variant)
    return rc == rn.OK


def scaled_rows(hidden, dtype, exps, seed, reps=1):
    """One row per exponent (repeated `reps` times): N(0,1) draws times 2^e,
    clipped to |z| < 3.9 so 2^126 rows stay finite, in binary32, then rounded
    to the element type."""
    rng = np.random.default_rng(seed)
    e = np.repeat(np.asarray(exps, dtype=np.float64), reps)
    z = np.clip(rng.standard_normal((len(e), hidden)), -3.9, 3.9)
    f = (z * np.exp2(e)[:, None]).astype(np.float32)
    return inputs.to_storage(f, dtype)


def weight(hidden, dtype, seed=7):
    _, w = inputs.random_case(1, hidden, dtype, seed=seed)
    return w


def run(x_np, w_np, eps, dtype, variant=rn.VARIANT_AUTO):
    x = to_device(x_np, dtype)
    w = to_device(w_np, dtype)
    y = rn.rms_norm(x, w, eps, variant=variant)
    torch.cuda.synchronize()
    return from_device(y, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("hidden", [64, 128, 1000, 1023, 4096, 7168, 16384, 32768])
def test_scaled_rows_every_variant(dtype, hidden):
    x = scaled_rows(hidden, dtype, EXPS[dtype], seed=hidden, reps=2)
    w = weight(hidden, dtype)
    checked = 0
    for eps in (0.0, 1e-6):
        for v in VARIANTS:
            if not accepts(x.shape[0], hidden, dtype, v):
                continue
            compare(run(x, w, eps, dtype, v), x, w, eps, dtype)
            checked += 1
    assert checked >= 4


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_scaled_rows_in_place(dtype):
    hidden = 4096
    x_np = scaled_rows(hidden, dtype, EXPS[dtype], seed=3)
    w_np = weight(hidden, dtype)
    for v in (rn.VARIANT_AUTO, rn.VARIANT_STAGED, rn.VARIANT_GENERIC, rn.VARIANT_WARP_PER_ROW):
        if not accepts(x_np.shape[0], hidden, dtype, v):
            continue
        x = to_device(x_np, dtype)
        rn.rms_norm(x, to_device(w_np, dtype), 0.0, out=x, variant=v)
        torch.cuda.synchronize()
        compare(from_device(x, dtype), x_np, w_np, 0.0, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows,hidden", [(4, 65536), (3, 131072), (2, 300000), (1, 1 << 20)])
def test_scaled_long_rows(dtype, rows, hidden):
    """Long decode rows (thread-block clusters, the grid variant, the looped
    body): whole rows at the range's ends, and rows whose halves sit at
    opposite ends, so the blocks' partial sums need different treatment."""
    if dtype == "f32":
        hidden //= 2
    rng = np.random.default_rng(rows + hidden)
    z = np.clip(rng.standard_normal((4 * rows, hidden)), -3.9, 3.9)
    e = np.zeros((4 * rows, hidden))
    for i in range(rows):
        e[4 * i] = 110 - 7 * i
        e[4 * i + 1] = -110 - 7 * i if dtype == "f32" else -110 + 5 * i
        e[4 * i + 2, : hidden // 2] = 100           # huge half, ordinary half
        e[4 * i + 3, : hidden // 3] = -100          # tiny third, zero rest
        z[4 * i + 3, hidden // 3:] = 0.0
    x = inputs.to_storage((z * np.exp2(e)).astype(np.float32), dtype)
    w = weight(hidden, dtype)
    for eps in (0.0, 1e-6):
        for v in (rn.VARIANT_AUTO, rn.VARIANT_CLUSTER, rn.VARIANT_GRID, rn.VARIANT_CTA_PER_ROW,
                  rn.VARIANT_GENERIC):
            if not accepts(x.shape[0], hidden, dtype, v):
                continue
            compare(run(x, w, eps, dtype, v), x, w, eps, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_subnormal_rows_eps_zero(dtype):
    """Rows made only of subnormal numbers with eps = 0: 1 / RMS is beyond
    the float range, so x is scaled up by 2^100 (exactly) before scaling."""
    lo = -133 if dtype == "bf16" else -149
    rng = np.random.default_rng(5)
    for hidden in (64, 4096, 65536):
        rows = 6
        k = rng.integers(0, 8, (rows, hidden))
        sign = np.where(rng.random((rows, hidden)) < 0.5, -1.0, 1.0)
        f = (sign * k * np.exp2(lo)).astype(np.float32)  # small multiples of the least subnormal
        f[0, :] = np.float32(np.exp2(lo))                 # a constant row: y = w
        f[1, 0] = np.float32(3 * np.exp2(lo))
        f[1, 1:] = 0.0                                    # one nonzero element: y = sqrt(n) w
        x = inputs.to_storage(f, dtype)
        w = weight(hidden, dtype)
        for v in VARIANTS:
            if not accepts(rows, hidden, dtype, v):
                continue
            compare(run(x, w, 0.0, dtype, v), x, w, 0.0, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_one_huge_element(dtype):
    """One element of 2^100 (its square overflows fp32) among ordinary ones:
    the others' outputs are about 2^-94, still normal numbers, and must match."""
    hidden = 4096
    rng = np.random.default_rng(9)
    f = rng.standard_normal((8, hidden)).astype(np.float32)
    for i in range(8):
        f[i, (i * 517) % hidden] = np.float32(np.exp2(100 + 3 * i))
    x = inputs.to_storage(f, dtype)
    w = weight(hidden, dtype)
    for v in VARIANTS:
        if accepts(8, hidden, dtype, v):
            compare(run(x, w, 1e-6, dtype, v), x, w, 1e-6, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_scaled_rows_weight_bias(dtype):
    hidden = 4096
    x_np = scaled_rows(hidden, dtype, EXPS[dtype], seed=21)
    w_np = weight(hidden, dtype)
    for eps in (0.0, 1e-6):
        for v in (rn.VARIANT_AUTO, rn.VARIANT_STAGED, rn.VARIANT_GENERIC, rn.VARIANT_WARP_PER_ROW):
            if not accepts(x_np.shape[0], hidden, dtype, v):
                continue
            y = rn.rms_norm_bias(to_device(x_np, dtype), to_device(w_np, dtype), 0.5, eps,
                                 variant=v)
            torch.cuda.synchronize()
            compare(from_device(y, dtype), x_np, w_np, eps, dtype, bias=0.5)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("fmt,g", [("mxfp8", 1.0), ("mxfp4", 1.0), ("nvfp4", 0.05)])
@pytest.mark.parametrize("bias", [-0.0, 1.0])
def test_scaled_rows_block_scaled(dtype, fmt, g, bias):
    """Block-scaled outputs of rows at the range's ends (with an offset of -0
    the 16-bit elements take the exact-product form), in the automatic plan,
    the staged ring and the looped body (64 KiB rows)."""
    for hidden in (1024, 4096, 32768 if dtype == "bf16" else 16384):
        x_np = scaled_rows(hidden, dtype, EXPS[dtype], seed=hidden + 1)
        w_np = weight(hidden, dtype)
        for eps in (0.0, 1e-6):
            for v in (rn.VARIANT_AUTO, rn.VARIANT_STAGED, rn.VARIANT_CTA_PER_ROW):
                sms, optin = rn.rmsnorm_device_limits()
                rc, _ = rn.rmsnorm_plan_epilogue_status(
                    1 << 30, 3 << 30, 5 << 30, x_np.shape[0], hidden, rn.DTYPE_CODES[dtype],
                    rn.EPI_CODES[fmt], sms, optin, variant=v)
                if rc != rn.OK:
                    continue
                q, s = rn.rms_norm_quant(to_device(x_np, dtype), to_device(w_np, dtype), eps,
                                         fmt=fmt, weight_bias=bias, global_scale=g, variant=v)
                torch.cuda.synchronize()
                compare_quant(q.cpu().numpy(), s.cpu().numpy(), x_np, w_np, bias, eps, dtype,
                              fmt, g)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_scaled_heads_qk_norm(dtype):
    """Per-head QK norm with every head at its own scale (q and k views of a
    fused [q | k | v] buffer), eps = 0 and 1e-6."""
    import oracle
    from _parity import monotone
    tokens, qh, kh, hd = 12, 4, 2, 128
    exps = EXPS[dtype]
    rng = np.random.default_rng(17)
    nh = qh + 2 * kh
    width = nh * hd
    z = np.clip(rng.standard_normal((tokens, nh, hd)), -3.9, 3.9)
    e = np.array([exps[i % len(exps)] for i in range(tokens * nh)], dtype=np.float64)
    f = (z * np.exp2(e).reshape(tokens, nh, 1)).astype(np.float32)
    buf_np = inputs.to_storage(f.reshape(tokens, width), dtype)
    flat = buf_np.ravel()
    qw = weight(hd, dtype, seed=1)
    kw = weight(hd, dtype, seed=2)
    k_off = qh * hd
    for eps in (0.0, 1e-6):
        ref, _ = oracle.qk_norm(flat, np.zeros(1, flat.dtype), qw, kw, tokens, qh, 0, hd, width,
                                0, 0.0, eps, dtype)
        _, ref_k = oracle.qk_norm(np.zeros(1, flat.dtype), ref[k_off:], qw, kw, tokens, 0, kh,
                                  hd, 0, width, 0.0, eps, dtype)
        want = np.concatenate([ref[:k_off], ref_k]).reshape(tokens, width)
        buf = to_device(buf_np, dtype)
        q = buf[:, :k_off]
        k = buf[:, k_off:(qh + kh) * hd]
        rn.qk_norm(q, k, to_device(qw, dtype), to_device(kw, dtype), hd, eps, weight_bias=0.0)
        torch.cuda.synchronize()
        got = from_device(buf, dtype)
        if dtype == "f32":
            g, r = got.astype(np.float64), want.astype(np.float64)
            d = np.abs(g - r)
            ok = (d <= 1e-5) | (d <= 1e-5 * np.abs(r)) | (np.isnan(r) & np.isnan(g))
            assert ok.all(), np.argwhere(~ok)[:3]
        else:
            dist = np.abs(monotone(got) - monotone(want))
            dist[np.isnan(oracle.widen(want, dtype)) & np.isnan(oracle.widen(got, dtype))] = 0
            assert dist.max() <= 1, np.argwhere(dist > 1)[:3]
        assert np.array_equal(got[:, (qh + kh) * hd:], buf_np[:, (qh + kh) * hd:])  # v untouched


def special_rows(hidden, dtype, seed):
    """Rows with NaN, +-Inf and subnormal elements beside ordinary rows."""
    rng = np.random.default_rng(seed)
    f = rng.standard_normal((10, hidden)).astype(np.float32)
    tiny = {"bf16": np.exp2(-130.0), "f32": np.exp2(-147.0), "f16": np.exp2(-23.0)}[dtype]
    j = lambda i: (i * 37 + 5) % hidden
    f[0, j(0)] = np.nan
    f[1, j(1)] = np.inf
    f[2, j(2)] = -np.inf
    f[3, j(3)] = np.inf
    f[3, j(4)] = -np.inf
    f[4, ::3] = np.float32(tiny) * (np.arange(1, hidden + 1, dtype=np.float32)[::3] % 7)
    f[5] = np.float32(tiny) * (1 + rng.integers(0, 5, hidden))          # all subnormal
    f[6, :] = 0.0
    f[6, j(6)] = np.float32(tiny)                                       # one subnormal
    f[7, 1::2] = 0.0
    return inputs.to_storage(f, dtype)


def special_weight(hidden, dtype):
    """The usual weight with NaN, +-Inf, a subnormal, -0 and +0 in it."""
    _, w = inputs.random_case(1, hidden, dtype, seed=31)
    wf = oracle_widen(w, dtype).astype(np.float32)
    tiny = {"bf16": np.exp2(-130.0), "f32": np.exp2(-147.0), "f16": np.exp2(-23.0)}[dtype]
    wf[1:7] = [np.nan, np.inf, -np.inf, tiny, -0.0, 0.0]
    return inputs.to_storage(wf, dtype)


def oracle_widen(a, dtype):
    import oracle
    return oracle.widen(a, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("hidden", [64, 1000, 1023, 4096, 40000, 65536])
def test_nonfinite_and_subnormal_every_variant(dtype, hidden):
    x = special_rows(hidden, dtype, seed=hidden)
    w_plain = weight(hidden, dtype)
    w_special = special_weight(hidden, dtype)
    checked = 0
    for w in (w_plain, w_special):
        for eps in (0.0, 1e-6):
            for v in VARIANTS:
                if not accepts(x.shape[0], hidden, dtype, v):
                    continue
                compare(run(x, w, eps, dtype, v), x, w, eps, dtype)
                checked += 1
                if v in (rn.VARIANT_CLUSTER, rn.VARIANT_GRID):
                    continue  # plain output only
                for bias in (0.25, -0.0):
                    y = rn.rms_norm_bias(to_device(x, dtype), to_device(w, dtype), bias, eps,
                                         variant=v)
                    torch.cuda.synchronize()
                    compare(from_device(y, dtype), x, w, eps, dtype, bias=bias)
    assert checked >= 8
