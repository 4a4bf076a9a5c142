"""GPU parity of the epilogues against the fp64 oracle: the weight offset
(w + WEIGHT_BIAS of "CuTeDSL at Perplexity", section "QK Norm") and the
fused block-scaled outputs MXFP8, MXFP4 (the OCP MX v1.0 definitions) and
NVFP4 (NVIDIA's description) named in the same page's section "Blackwell
support".

* every workload shape (full compare where the oracle is quick, sampled rows
  at the 65536-row shapes), in the selector's automatic plan;
* every shape class the selector distinguishes (decode, short, mid, wide,
  staged-range, looped) for f32 / bf16 / f16;
* bias -0 reproduces the plain kernel bit for bit; in place; ragged rows;
* MXFP8 special blocks (zero rows, NaN / Inf inputs, extreme row scales),
  argument errors, guard bytes around the codes and the scales.
"""
import numpy as np
import pytest

import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import compare, compare_mx, compare_quant, from_device, sample_rows, to_device

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


def run_bias(x_np, w_np, bias, eps, dtype, out_is_x=False):
    x = to_device(x_np, dtype)
    w = to_device(w_np, dtype)
    y = rn.rms_norm_bias(x, w, bias, eps, out=x if out_is_x else None)
    torch.cuda.synchronize()
    return from_device(y, dtype)


def run_mx(x_np, w_np, bias, eps, dtype, variant=rn.VARIANT_AUTO):
    x = to_device(x_np, dtype)
    w = to_device(w_np, dtype)
    q, s = rn.rms_norm_mxfp8(x, w, eps, weight_bias=bias, variant=variant)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


SMALL = ["f32_64x128", "embed_bf16_8192x1024", "decode_bf16_1x4096", "decode_bf16_8x4096",
         "decode_bf16_32x4096", "prefill_bf16_16384x4096"]
WIDE = [n for n in inputs.WORKLOADS if n.startswith("wide_")]
# (rows, hidden): decode warp / block bodies, short and mid prefill rows,
# 16-32 KiB persistent rows, the 32-72 KiB range (staged for the plain
# output, looped here), and rows longer than the register bodies hold.
SHAPES = [(1, 256), (7, 1024), (100, 4096), (152, 8192), (3, 65536), (513, 64), (2049, 512),
          (1000, 1536), (333, 2048), (97, 5120), (160, 8192), (64, 12288), (40, 20480),
          (33, 36864), (9, 65536), (5, 131072)]


@pytest.mark.parametrize("name", SMALL)
def test_bias_workloads(name):
    wl = inputs.WORKLOADS[name]
    x, w = inputs.make_inputs(wl)
    y = run_bias(x, w, 1.0, wl.eps, wl.dtype)
    compare(y, x, w, wl.eps, wl.dtype, bias=1.0)


@pytest.mark.parametrize("name", SMALL)
def test_mx_workloads(name):
    wl = inputs.WORKLOADS[name]
    x, w = inputs.make_inputs(wl)
    q, s = run_mx(x, w, 0.0, wl.eps, wl.dtype)
    r = compare_mx(q, s, x, w, 0.0, wl.eps, wl.dtype)
    assert r["rows"] == wl.rows and r["exact_codes"] > 0.999


@pytest.mark.parametrize("name", WIDE)
def test_epilogues_wide_workloads_sampled(name):
    wl = inputs.WORKLOADS[name]
    x, w = inputs.make_inputs(wl)
    idx = sample_rows(wl.rows, 48, seed=wl.key)
    compare(run_bias(x, w, 0.5, wl.eps, wl.dtype), x, w, wl.eps, wl.dtype, rows_idx=idx,
            bias=0.5)
    q, s = run_mx(x, w, 0.5, wl.eps, wl.dtype)
    compare_mx(q, s, x, w, 0.5, wl.eps, wl.dtype, rows_idx=idx)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,hidden", SHAPES)
def test_epilogue_shape_classes(dtype, rows, hidden):
    if dtype == "f32" and hidden > 65536:
        hidden //= 2
    x, w = inputs.random_case(rows, hidden, dtype, seed=rows + hidden)
    idx = sample_rows(rows, 64, seed=hidden) if rows * hidden > (1 << 22) else None
    compare(run_bias(x, w, -0.25, 1e-6, dtype), x, w, 1e-6, dtype, rows_idx=idx, bias=-0.25)
    q, s = run_mx(x, w, 1.0, 1e-6, dtype)
    compare_mx(q, s, x, w, 1.0, 1e-6, dtype, rows_idx=idx)


def test_bias_minus_zero_is_the_plain_kernel_bit_for_bit():
    for name in ("embed_bf16_8192x1024", "f32_64x128", "decode_bf16_8x4096"):
        wl = inputs.WORKLOADS[name]
        x_np, w_np = inputs.make_inputs(wl)
        x = to_device(x_np, wl.dtype)
        w = to_device(w_np, wl.dtype)
        y0 = rn.rms_norm(x, w, wl.eps)
        y1 = rn.rms_norm_bias(x, w, -0.0, wl.eps)
        torch.cuda.synchronize()
        assert np.array_equal(from_device(y0, wl.dtype), from_device(y1, wl.dtype))


def test_bias_in_place_and_ragged():
    wl = inputs.WORKLOADS["embed_bf16_8192x1024"]
    x, w = inputs.make_inputs(wl)
    compare(run_bias(x, w, 1.0, wl.eps, wl.dtype, out_is_x=True), x, w, wl.eps, wl.dtype,
            bias=1.0)
    for dtype, hidden in (("bf16", 1001), ("f16", 4097), ("f32", 33)):
        x, w = inputs.random_case(65, hidden, dtype, seed=hidden)
        y = run_bias(x, w, 0.75, 1e-6, dtype)
        assert rn.rmsnorm_last_variant() == rn.VARIANT_GENERIC
        compare(y, x, w, 1e-6, dtype, bias=0.75)


def test_bias_every_forced_variant():
    x, w = inputs.random_case(300, 4096, "bf16", seed=9)
    xd, wd = to_device(x, "bf16"), to_device(w, "bf16")
    for v in (rn.VARIANT_WARP_PER_ROW, rn.VARIANT_CTA_PER_ROW, rn.VARIANT_PERSISTENT,
              rn.VARIANT_GENERIC, rn.VARIANT_STAGED):
        try:
            y = rn.rms_norm_bias(xd, wd, 2.0, 1e-6, variant=v)
        except rn.RmsnormError as e:
            assert e.status == rn.ERR_VARIANT and v == rn.VARIANT_WARP_PER_ROW
            continue
        torch.cuda.synchronize()
        compare(from_device(y, "bf16"), x, w, 1e-6, "bf16", bias=2.0)
    for v in (rn.VARIANT_CLUSTER, rn.VARIANT_GRID):   # plain output only
        with pytest.raises(rn.RmsnormError) as e:
            rn.rms_norm_bias(xd, wd, 2.0, 1e-6, variant=v)
        assert e.value.status == rn.ERR_VARIANT


def test_mx_special_blocks():
    rows, hidden = 12, 1024
    for dtype in ("bf16", "f16", "f32"):
        z = np.random.default_rng(3).standard_normal((rows, hidden)).astype(np.float32)
        z[0] = 0.0                                   # all-zero row: scale 2^-127, zero codes
        z[1, 5] = np.nan                             # NaN: the sum and so the whole row is NaN
        z[2, 700] = np.inf                           # Inf: r = 0, one NaN element (Inf * 0)
        z[3, :32] = 0.0                              # one zero block in a live row
        # tiny and huge rows, normalised anyway (squares stay inside the fp32
        # range the pages' fp32 accumulator has)
        z[4] *= 1e-15 if dtype == "f32" else 1e-3
        z[5] *= 1e15 if dtype == "f32" else (1e4 if dtype == "f16" else 3e4)
        z[6, ::2] = 0.0
        z[6, 1] = 1e4 if dtype != "f16" else 6e4     # one outlier: others go subnormal in E4M3
        x = inputs.to_storage(z, dtype)
        _, w = inputs.random_case(1, hidden, dtype, seed=2)
        for eps in (1e-6, 0.0):
            q, s = run_mx(x, w, 0.0, eps, dtype)
            compare_mx(q, s, x, w, 0.0, eps, dtype)
            if eps == 0.0:                           # 0 * inf: NaN row, NaN scales
                assert (s[0] == 0xFF).all()
            else:
                assert (s[0] == 0).all() and np.isin(q[0], (0x00, 0x80)).all()
            assert (s[1] == 0xFF).all()
            assert s[2, 700 // 32] == 0xFF and (np.delete(s[2], 700 // 32) == 0).all()


def test_mx_every_forced_variant_and_guard_bytes():
    rows, hidden = 161, 4096
    x, w = inputs.random_case(rows, hidden, "bf16", seed=12)
    xd, wd = to_device(x, "bf16"), to_device(w, "bf16")
    pad = 4096
    for v in (rn.VARIANT_AUTO, rn.VARIANT_CTA_PER_ROW, rn.VARIANT_PERSISTENT,
              rn.VARIANT_STAGED):
        qb = torch.full((rows * hidden + 2 * pad,), 0x5A, dtype=torch.uint8, device="cuda")
        sb = torch.full((rows * hidden // 32 + 2 * pad,), 0x5A, dtype=torch.uint8, device="cuda")
        q = qb[pad:pad + rows * hidden].view(rows, hidden)
        s = sb[pad:pad + rows * hidden // 32].view(rows, hidden // 32)
        rn.rms_norm_mxfp8(xd, wd, 1e-6, weight_bias=0.0, out=q, scales=s, variant=v)
        torch.cuda.synchronize()
        for b in (qb, sb):
            assert (b[:pad] == 0x5A).all() and (b[-pad:] == 0x5A).all()
        compare_mx(q.cpu().numpy(), s.cpu().numpy(), x, w, 0.0, 1e-6, "bf16")
    for v, st in ((rn.VARIANT_CLUSTER, rn.ERR_VARIANT), (rn.VARIANT_GENERIC, rn.ERR_VARIANT)):
        with pytest.raises(rn.RmsnormError) as e:
            rn.rms_norm_mxfp8(xd, wd, 1e-6, variant=v)
        assert e.value.status == st


def test_mx_argument_errors():
    x, w = inputs.random_case(8, 4096, "bf16", seed=13)
    xd, wd = to_device(x, "bf16"), to_device(w, "bf16")
    xfull = to_device(np.concatenate([np.zeros(8, np.uint16), x.ravel()]), "bf16")
    lib = rn._load()
    q = torch.empty(8, 4096, dtype=torch.uint8, device="cuda")
    s = torch.empty(8, 128, dtype=torch.uint8, device="cuda")
    # misaligned x (one element in): no scalar MX body
    assert lib.rmsnorm_fwd_mxfp8(xfull.data_ptr() + 2, wd.data_ptr(), q.data_ptr(), s.data_ptr(),
                                 8, 4096, 0.0, 1e-6, rn.BF16, None) == rn.ERR_MISALIGNED
    # hidden not a multiple of 32 (4080 = 127.5 blocks)
    assert lib.rmsnorm_fwd_mxfp8(xd.data_ptr(), wd.data_ptr(), q.data_ptr(), s.data_ptr(), 8, 4080,
                                 0.0, 1e-6, rn.BF16, None) == rn.ERR_INVALID_ARG
    # scales inside the codes, codes inside x
    assert lib.rmsnorm_fwd_mxfp8(xd.data_ptr(), wd.data_ptr(), q.data_ptr(),
                                 q.data_ptr() + 1024, 8, 4096, 0.0, 1e-6, rn.BF16,
                                 None) == rn.ERR_ALIASING
    assert lib.rmsnorm_fwd_mxfp8(xd.data_ptr(), wd.data_ptr(), xd.data_ptr(), s.data_ptr(), 8,
                                 4096, 0.0, 1e-6, rn.BF16, None) == rn.ERR_ALIASING
    # the zero-row call launches nothing and succeeds
    assert lib.rmsnorm_fwd_mxfp8(xd.data_ptr(), wd.data_ptr(), q.data_ptr(), s.data_ptr(), 0,
                                 4096, 0.0, 1e-6, rn.BF16, None) == rn.OK
    torch.cuda.synchronize()



# ------------------------------------------------------------------ MXFP4 / NVFP4

FP4 = [("mxfp4", 1.0), ("nvfp4", 1.0), ("nvfp4", 0.0021)]


def run_q(x_np, w_np, bias, eps, dtype, fmt, g, variant=rn.VARIANT_AUTO):
    x = to_device(x_np, dtype)
    w = to_device(w_np, dtype)
    q, s = rn.rms_norm_quant(x, w, eps, fmt, weight_bias=bias, global_scale=g, variant=variant)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("fmt,g", FP4)
@pytest.mark.parametrize("name", SMALL)
def test_fp4_workloads(name, fmt, g):
    wl = inputs.WORKLOADS[name]
    x, w = inputs.make_inputs(wl)
    q, s = run_q(x, w, 0.0, wl.eps, wl.dtype, fmt, g)
    r = compare_quant(q, s, x, w, 0.0, wl.eps, wl.dtype, fmt, g)
    assert r["rows"] == wl.rows and r["exact_codes"] > 0.999


@pytest.mark.parametrize("fmt,g", FP4[:2])
@pytest.mark.parametrize("name", WIDE)
def test_fp4_wide_workloads_sampled(name, fmt, g):
    wl = inputs.WORKLOADS[name]
    x, w = inputs.make_inputs(wl)
    idx = sample_rows(wl.rows, 32, seed=wl.key)
    q, s = run_q(x, w, 0.5, wl.eps, wl.dtype, fmt, g)
    compare_quant(q, s, x, w, 0.5, wl.eps, wl.dtype, fmt, g, rows_idx=idx)


@pytest.mark.parametrize("fmt,g", FP4)
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,hidden", SHAPES + [(77, 48), (9, 16), (300, 2064)])
def test_fp4_shape_classes(dtype, rows, hidden, fmt, g):
    if dtype == "f32" and hidden > 65536:
        hidden //= 2
    if fmt == "mxfp4" and hidden % 32:
        return
    x, w = inputs.random_case(rows, hidden, dtype, seed=rows + 3 * hidden)
    idx = sample_rows(rows, 64, seed=hidden) if rows * hidden > (1 << 22) else None
    q, s = run_q(x, w, 1.0, 1e-6, dtype, fmt, g)
    compare_quant(q, s, x, w, 1.0, 1e-6, dtype, fmt, g, rows_idx=idx)


@pytest.mark.parametrize("fmt,g", FP4)
def test_fp4_special_blocks(fmt, g):
    rows, hidden = 10, 512
    for dtype in ("bf16", "f16", "f32"):
        z = np.random.default_rng(5).standard_normal((rows, hidden)).astype(np.float32)
        z[0] = 0.0
        z[1, 5] = np.nan
        z[2, 300] = np.inf
        z[3, :32] = 0.0
        z[4] *= 1e-15 if dtype == "f32" else 1e-3
        z[5] *= 1e15 if dtype == "f32" else (1e4 if dtype == "f16" else 3e4)
        z[6, ::2] = 0.0
        z[6, 1] = 1e4 if dtype != "f16" else 6e4
        x = inputs.to_storage(z, dtype)
        _, w = inputs.random_case(1, hidden, dtype, seed=7)
        for eps in (1e-6, 0.0):
            q, s = run_q(x, w, 0.0, eps, dtype, fmt, g)
            compare_quant(q, s, x, w, 0.0, eps, dtype, fmt, g)
            nan_code = 0x7F if fmt == "nvfp4" else 0xFF
            assert (s[1] == nan_code).all()
            if eps > 0:
                assert (s[0] == 0).all() and not (q[0] & 0x77).any()


QFMTS = [("mxfp8", 1.0), ("mxfp4", 1.0), ("nvfp4", 1.0), ("nvfp4", 0.0021)]


@pytest.mark.parametrize("fmt,g", QFMTS)
@pytest.mark.parametrize("name", SMALL)
def test_quant_workloads_without_offset(name, fmt, g):
    """Weight offset -0 (no offset, the binding's default): 16-bit inputs take
    the exact-product path (x * w by the mixed-precision fma, then r)."""
    wl = inputs.WORKLOADS[name]
    x, w = inputs.make_inputs(wl)
    q, s = run_q(x, w, -0.0, wl.eps, wl.dtype, fmt, g)
    r = compare_quant(q, s, x, w, -0.0, wl.eps, wl.dtype, fmt, g)
    assert r["rows"] == wl.rows and r["exact_codes"] > 0.999


@pytest.mark.parametrize("fmt,g", QFMTS + [("nvfp4", 1e-37), ("nvfp4", 1e31)])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_quant_exact_products_special_and_extreme_blocks(dtype, fmt, g):
    """Blocks the exact-product path hands back to the (x * r) * w order --
    zero, NaN and Inf blocks, products below 2^-100 or above 2^100 -- next to
    blocks it keeps, in the same warps; zero weights of both signs (zero
    codes keep the IEEE sign of x * w); NVFP4 global scales outside the
    flush-to-zero range (1e-37, 1e31) take the order above throughout."""
    rows, hidden = 12, 1024
    rng = np.random.default_rng(11)
    z = rng.standard_normal((rows, hidden)).astype(np.float32)
    z[0] = 0.0
    z[1, 5] = np.nan
    z[2, 700] = np.inf
    z[3, :32] = 0.0
    z[3, 64:96] = 0.0
    wz = np.abs(np.random.default_rng(12).normal(1.0, 0.1, hidden)).astype(np.float32)
    if dtype == "f16":                           # f16 products never leave fp32's range
        z[4, 32:64] *= 1e-3
        z[5] *= 1e-2
        z[6, 96:128] *= 300.0
        wz[96:128] *= 100.0
    else:
        # one block of products below 2^-100 beside normal blocks; a row of
        # tiny x whose sum of squares stays a normal fp32 number, meeting
        # tiny weights in one block; products above 2^100 from large weights
        z[4, 32:64] *= 1e-32
        z[5] *= 1e-18 if dtype == "bf16" else 1e-15
        wz[232:264] *= 1e-14
        z[6, 96:128] *= 1e9
        wz[96:128] *= 1e25
    z[7, ::2] = 0.0
    z[7, 1] = 1e4 if dtype != "f16" else 6e4
    z[8] = -np.abs(z[8])
    x = inputs.to_storage(z, dtype)
    wz[200:216] = -0.0
    wz[216:232] = 0.0
    w = inputs.to_storage(wz[None, :], dtype)[0]
    if dtype == "f32":
        assert w[200] == 0 and np.signbit(w[200])
    else:
        assert int(w[200]) == 0x8000 and int(w[216]) == 0
    for eps in (1e-6, 0.0):
        for bias in (-0.0, 0.0):
            q, s = run_q(x, w, bias, eps, dtype, fmt, g)
            compare_quant(q, s, x, w, bias, eps, dtype, fmt, g)


@pytest.mark.parametrize("fmt,g", QFMTS)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_quant_exact_products_fallback_in_every_prefill_body(dtype, fmt, g):
    """Prefill batches (more rows than SMs) at widths that reach every
    block-scaled prefill body (16-bit elements) -- a warp per row (2 KiB
    rows), the one-warp block (3 KiB), the 64-thread two-vector body (4 KiB),
    the compile-time 64 / 96 / 128-thread four-vector blocks (5.6, 8, 10, 14
    and 16 KiB rows, some with idle lanes) and the 24 KiB persistent body --
    with blocks the
    exact-product form hands back (zero, NaN, Inf, products below 2^-100) at
    the start, middle and end of rows, so that the warp's one vote per row
    fires for each vector slot of a thread; the other rows of the batch keep
    the fast form.  Every row is compared with the oracle."""
    rows = 160
    for hidden in (1024, 1536, 2048, 2880, 4096, 5120, 7168, 8192, 12288):
        rng = np.random.default_rng(hidden)
        z = rng.standard_normal((rows, hidden)).astype(np.float32)
        h32 = hidden // 32
        at = lambda i: 32 * i
        for r, blk in enumerate((0, h32 // 4, h32 // 2, 3 * h32 // 4, h32 - 1), start=1):
            z[r, at(blk):at(blk) + 32] = 0.0              # one zero block per row
        z[6, [at(b) for b in (0, h32 // 3, 2 * h32 // 3, h32 - 1)]] = np.nan
        z[7, hidden - 1] = np.inf
        z[8, :] = 0.0
        for k in range(4):                               # a zero block per quarter
            z[9, at(k * h32 // 4):at(k * h32 // 4) + 32] = 0.0
        if dtype == "bf16":                              # products below 2^-100
            z[10, at(h32 // 2):at(h32 // 2) + 32] *= 1e-32
            z[11, hidden - 32:] *= 1e-32
        x = inputs.to_storage(z, dtype)
        w = inputs.to_storage(np.abs(rng.normal(1.0, 0.1, (1, hidden))).astype(np.float32),
                              dtype)[0]
        q, s = run_q(x, w, -0.0, 1e-6, dtype, fmt, g)
        compare_quant(q, s, x, w, -0.0, 1e-6, dtype, fmt, g)


@pytest.mark.parametrize("fmt,g", QFMTS)
def test_quant_without_offset_every_forced_variant(fmt, g):
    """The exact-product path in every body that writes block-scaled rows:
    warp-per-row (short rows), block-per-row, persistent, looped (long rows)
    and the shared-memory ring (x read back from its slot on a fallback)."""
    cases = [(700, 1024, (rn.VARIANT_AUTO, rn.VARIANT_WARP_PER_ROW, rn.VARIANT_CTA_PER_ROW)),
             (161, 4096, (rn.VARIANT_AUTO, rn.VARIANT_CTA_PER_ROW, rn.VARIANT_PERSISTENT,
                          rn.VARIANT_STAGED)),
             (40, 36864, (rn.VARIANT_AUTO, rn.VARIANT_CTA_PER_ROW, rn.VARIANT_STAGED))]
    for rows, hidden, variants in cases:
        for dtype in ("bf16", "f16"):
            x, w = inputs.random_case(rows, hidden, dtype, seed=rows + hidden)
            x = x.copy()
            x[1, 32:96] = 0                      # fallback blocks inside a live row
            x[2, :] = 0                          # and a zero row
            xd, wd = to_device(x, dtype), to_device(w, dtype)
            idx = sample_rows(rows, 48, seed=hidden) if rows * hidden > (1 << 22) else None
            if idx is not None:
                idx = np.union1d(idx, [1, 2])
            for v in variants:
                q, s = rn.rms_norm_quant(xd, wd, 1e-6, fmt, weight_bias=-0.0, global_scale=g,
                                         variant=v)
                torch.cuda.synchronize()
                compare_quant(q.cpu().numpy(), s.cpu().numpy(), x, w, -0.0, 1e-6, dtype, fmt,
                              g, rows_idx=idx)


def test_fp4_argument_errors():
    lib = rn._load()
    x, w = inputs.random_case(8, 4096, "bf16", seed=13)
    xd, wd = to_device(x, "bf16"), to_device(w, "bf16")
    q = torch.empty(8, 2048, dtype=torch.uint8, device="cuda")
    s = torch.empty(8, 256, dtype=torch.uint8, device="cuda")
    P = (xd.data_ptr(), wd.data_ptr(), q.data_ptr(), s.data_ptr())
    assert lib.rmsnorm_fwd_mxfp4(*P, 8, 4080, 0.0, 1e-6, rn.BF16, None) == rn.ERR_INVALID_ARG
    assert lib.rmsnorm_fwd_nvfp4(*P, 8, 4088, 1.0, 0.0, 1e-6, rn.BF16, None) == \
        rn.ERR_INVALID_ARG
    for gbad in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.rmsnorm_fwd_nvfp4(*P, 8, 4096, gbad, 0.0, 1e-6, rn.BF16, None) == \
            rn.ERR_INVALID_ARG
    assert lib.rmsnorm_fwd_nvfp4(xd.data_ptr(), wd.data_ptr(), q.data_ptr(), q.data_ptr() + 64,
                                 8, 4096, 1.0, 0.0, 1e-6, rn.BF16, None) == rn.ERR_ALIASING
    assert lib.rmsnorm_fwd_mxfp4(*P, 8, 4096, 0.0, 1e-6, rn.BF16, None) == rn.OK
    assert lib.rmsnorm_fwd_nvfp4(*P, 8, 4096, 1.0, 0.0, 1e-6, rn.BF16, None) == rn.OK
    torch.cuda.synchronize()
    compare_quant(q.cpu().numpy(), s.cpu().numpy(), x, w, 0.0, 1e-6, "bf16", "nvfp4", 1.0)



@pytest.mark.parametrize("epi", ["bias", "mxfp8", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("rows,hidden,dtype", [(2048, 20480, "bf16"), (1024, 32768, "f16"),
                                               (600, 9000, "f32"), (160, 36864, "bf16")])
def test_epilogues_on_the_staged_ring(epi, rows, hidden, dtype):
    """32-72 KiB rows: the weight-bias output runs on the shared-memory ring
    above 40 KiB (one block per row with 32-byte vectors on 32-40 KiB rows),
    and on the ring when forced; the block-scaled outputs on the looped body,
    and on the ring when forced."""
    x, w = inputs.random_case(rows, hidden, dtype, seed=hidden + 7)
    idx = sample_rows(rows, 48, seed=rows)
    xd, wd = to_device(x, dtype), to_device(w, dtype)
    if epi == "bias":
        row_bytes = hidden * (4 if dtype == "f32" else 2)
        for v in (rn.VARIANT_AUTO, rn.VARIANT_STAGED):
            y = rn.rms_norm_bias(xd, wd, 0.5, 1e-6, variant=v)
            torch.cuda.synchronize()
            if v == rn.VARIANT_STAGED or row_bytes > 40960:
                assert rn.rmsnorm_last_variant() == rn.VARIANT_STAGED
            elif row_bytes > 32768:
                assert rn.rmsnorm_last_variant() == rn.VARIANT_CTA_PER_ROW
            compare(from_device(y, dtype), x, w, 1e-6, dtype, rows_idx=idx, bias=0.5)
        return
    if hidden % 32:
        return
    # the automatic plan (the looped body) and the ring, forced
    for v in (rn.VARIANT_AUTO, rn.VARIANT_STAGED):
        q, s = rn.rms_norm_quant(xd, wd, 1e-6, epi, weight_bias=0.5, global_scale=0.004,
                                 variant=v)
        torch.cuda.synchronize()
        compare_quant(q.cpu().numpy(), s.cpu().numpy(), x, w, 0.5, 1e-6, dtype, epi, 0.004,
                      rows_idx=idx)
