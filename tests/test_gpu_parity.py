"""GPU parity: the CUDA library (through the C ABI) against the fp64 CPU
oracle on the same seeded inputs.

* every workload shape, in the launch configuration the benchmark uses
  (the selector's automatic plan), compared in full where the oracle is quick
  and on sampled rows for the 65536-row wide-hidden shapes;
* every variant forced on every shape it accepts, over a grid of hidden
  sizes (powers of two, ragged, non-power-of-two LLM sizes) and row counts
  (0, 1, 2, 31, 160, 161);
* in place (y == x), guard bytes around y, misaligned pointers, zero rows,
  eps = 0, a non-default stream.
"""
import numpy as np
import pytest

import oracle
import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import compare, compare_quant, from_device, sample_rows, to_device

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


def run(x_np, w_np, eps, dtype, variant=rn.VARIANT_AUTO, plan=None):
    x = to_device(x_np, dtype)
    w = to_device(w_np, dtype)
    y = rn.rms_norm(x, w, eps, variant=variant, plan=plan)
    torch.cuda.synchronize()
    return from_device(y, dtype)


# ------------------------------------------------------------------ workloads

SMALL = ["f32_64x128", "embed_bf16_8192x1024", "decode_bf16_1x4096", "decode_bf16_8x4096",
         "decode_bf16_32x4096", "prefill_bf16_16384x4096"]
WIDE = [n for n in inputs.WORKLOADS if n.startswith("wide_")]


@pytest.mark.parametrize("name", SMALL)
def test_workload_full_compare(name):
    wl = inputs.WORKLOADS[name]
    x, w = inputs.make_inputs(wl)
    y = run(x, w, wl.eps, wl.dtype)
    s = compare(y, x, w, wl.eps, wl.dtype)
    assert s["rows"] == wl.rows


@pytest.mark.slow
@pytest.mark.parametrize("name", WIDE)
def test_wide_workload_sampled(name):
    """65536 rows at 7168/5120/2880: full GPU run, 384 sampled rows checked."""
    wl = inputs.WORKLOADS[name]
    x, w = inputs.make_inputs(wl)
    y = run(x, w, wl.eps, wl.dtype)
    compare(y, x, w, wl.eps, wl.dtype, rows_idx=sample_rows(wl.rows, 384, seed=wl.key))
    # every row is finite (weights U(0,2), eps > 0)
    assert np.isfinite(oracle.widen(y[::97], wl.dtype)).all()


@pytest.mark.parametrize("variant", [rn.VARIANT_WARP_PER_ROW, rn.VARIANT_CTA_PER_ROW,
                                     rn.VARIANT_STAGED, rn.VARIANT_PERSISTENT,
                                     rn.VARIANT_GENERIC, rn.VARIANT_CLUSTER, rn.VARIANT_GRID])
def test_headline_shape_every_variant(variant):
    wl = inputs.WORKLOADS["prefill_bf16_16384x4096"]
    x, w = inputs.make_inputs(wl)
    if not accepts(wl.rows, wl.hidden, wl.dtype, variant):
        with pytest.raises(rn.RmsnormError) as e:
            run(x, w, wl.eps, wl.dtype, variant=variant)
        assert e.value.status == rn.ERR_VARIANT
        return
    y = run(x, w, wl.eps, wl.dtype, variant=variant)
    compare(y, x, w, wl.eps, wl.dtype)


# ------------------------------------------------------------------ edge grid

HIDDEN = [1, 2, 3, 7, 8, 9, 31, 33, 127, 128, 129, 1000, 1023, 1024, 1025, 2880, 4096, 5120,
          7168, 8191, 16384, 32768]
ROWS = [0, 1, 2, 31, 160, 161]
VARIANTS = [rn.VARIANT_AUTO, rn.VARIANT_WARP_PER_ROW, rn.VARIANT_CTA_PER_ROW,
            rn.VARIANT_STAGED, rn.VARIANT_PERSISTENT, rn.VARIANT_GENERIC, rn.VARIANT_CLUSTER,
            rn.VARIANT_GRID]


def accepts(rows, hidden, dtype, variant):
    """Whether the selector takes this forced variant (host-only query)."""
    if rows == 0:
        return True
    sms, optin = rn.rmsnorm_device_limits()
    base = 1 << 30
    rc, _ = rn.rmsnorm_plan_status(base, 3 * base, 5 * base, rows, hidden, rn.DTYPE_CODES[dtype],
                                   sms, optin, variant)
    return rc == rn.OK


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("hidden", HIDDEN)
def test_edge_grid(dtype, hidden):
    checked = 0
    for rows in ROWS:
        x, w = inputs.random_case(rows, hidden, dtype, seed=rows)
        for v in VARIANTS:
            if not accepts(rows, hidden, dtype, v):
                continue
            y = run(x, w, 1e-6, dtype, variant=v)
            compare(y, x, w, 1e-6, dtype)
            checked += 1
    assert checked > 0


# ------------------------------------------------------------------ properties

def test_in_place():
    for name in ("embed_bf16_8192x1024", "decode_bf16_32x4096", "f32_64x128"):
        wl = inputs.WORKLOADS[name]
        x_np, w_np = inputs.make_inputs(wl)
        for v in (rn.VARIANT_AUTO, rn.VARIANT_GENERIC, rn.VARIANT_STAGED, rn.VARIANT_CTA_PER_ROW):
            if not accepts(wl.rows, wl.hidden, wl.dtype, v):
                continue
            x = to_device(x_np, wl.dtype)
            w = to_device(w_np, wl.dtype)
            rn.rms_norm(x, w, wl.eps, out=x, variant=v)
            torch.cuda.synchronize()
            compare(from_device(x, wl.dtype), x_np, w_np, wl.eps, wl.dtype)


def test_guard_bytes_untouched():
    for dtype, hidden in (("bf16", 4096), ("f16", 7168), ("f32", 128), ("bf16", 1025)):
        rows = 161
        x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=3)
        x = to_device(x_np, dtype)
        w = to_device(w_np, dtype)
        pad = 4096
        buf = torch.full((rows * hidden + 2 * pad,), 77.0, dtype=x.dtype, device="cuda")
        y = buf[pad:pad + rows * hidden].view(rows, hidden)
        for v in (rn.VARIANT_AUTO, rn.VARIANT_STAGED, rn.VARIANT_GENERIC):
            if not accepts(rows, hidden, dtype, v):
                continue
            rn.rms_norm(x, w, 1e-6, out=y, variant=v)
            torch.cuda.synchronize()
            assert (buf[:pad] == 77.0).all() and (buf[pad + rows * hidden:] == 77.0).all()
            compare(from_device(y, dtype), x_np, w_np, 1e-6, dtype)


def test_misaligned_pointers_use_generic_and_match():
    dtype, rows, hidden = "bf16", 33, 4096
    x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=4)
    x_full = to_device(np.concatenate([np.zeros(1, np.uint16), x_np.ravel()]), dtype)
    x = x_full[1:].view(rows, hidden)  # 2-byte offset
    w = to_device(w_np, dtype)
    y = rn.rms_norm(x, w, 1e-6)
    assert rn.rmsnorm_last_variant() == rn.VARIANT_GENERIC
    torch.cuda.synchronize()
    compare(from_device(y, dtype), x_np, w_np, 1e-6, dtype)
    with pytest.raises(rn.RmsnormError) as e:
        rn.rms_norm(x, w, 1e-6, variant=rn.VARIANT_CTA_PER_ROW)
    assert e.value.status == rn.ERR_MISALIGNED


def test_zero_rows_and_eps_zero():
    dtype = "bf16"
    x_np = np.zeros((4, 256), np.uint16)
    _, w_np = inputs.random_case(4, 256, dtype, seed=5)
    for v in (rn.VARIANT_AUTO, rn.VARIANT_GENERIC, rn.VARIANT_STAGED):
        y = run(x_np, w_np, 0.0, dtype, variant=v)  # 0 * inf -> NaN, as in the oracle
        compare(y, x_np, w_np, 0.0, dtype)
        y = run(x_np, w_np, 1e-5, dtype, variant=v)
        assert (oracle.widen(y, dtype) == 0).all()


def test_dynamic_range_rows():
    """Rows scaled from 1e-3 to 1e3 (log-uniform), f16 and bf16."""
    for dtype in ("f16", "bf16"):
        rng = np.random.default_rng(11)
        z = rng.standard_normal((256, 5120)).astype(np.float32)
        z *= (10.0 ** rng.uniform(-3, 3, (256, 1))).astype(np.float32)
        x_np = inputs.to_storage(z, dtype)
        _, w_np = inputs.random_case(1, 5120, dtype, seed=6, w_dist="u0_2")
        for v in (rn.VARIANT_AUTO, rn.VARIANT_STAGED, rn.VARIANT_CTA_PER_ROW):
            compare(run(x_np, w_np, 1e-5, dtype, variant=v), x_np, w_np, 1e-5, dtype)


def test_non_default_stream():
    wl = inputs.WORKLOADS["embed_bf16_8192x1024"]
    x_np, w_np = inputs.make_inputs(wl)
    x = to_device(x_np, wl.dtype)
    w = to_device(w_np, wl.dtype)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        y = rn.rms_norm(x, w, wl.eps)
    s.synchronize()
    compare(from_device(y, wl.dtype), x_np, w_np, wl.eps, wl.dtype)


def test_raw_c_abi_call():
    """rmsnorm_fwd called with raw pointers and a raw stream handle."""
    wl = inputs.WORKLOADS["decode_bf16_8x4096"]
    x_np, w_np = inputs.make_inputs(wl)
    x = to_device(x_np, wl.dtype)
    w = to_device(w_np, wl.dtype)
    y = torch.empty_like(x)
    rn.rmsnorm_fwd(x.data_ptr(), w.data_ptr(), y.data_ptr(), wl.rows, wl.hidden, wl.eps, rn.BF16,
                   torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    compare(from_device(y, wl.dtype), x_np, w_np, wl.eps, wl.dtype)


def test_plan_written_back_and_replayed():
    wl = inputs.WORKLOADS["prefill_bf16_16384x4096"]
    x_np, w_np = inputs.make_inputs(wl)
    p = rn.Plan()
    y1 = run(x_np, w_np, wl.eps, wl.dtype, plan=p)
    assert p.variant != rn.VARIANT_AUTO and p.grid > 0
    y2 = run(x_np, w_np, wl.eps, wl.dtype, plan=p)  # explicit plan path
    assert np.array_equal(y1, y2)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,hidden", [(1, 65536), (8, 65536), (1, 131072), (20, 32768),
                                         (32, 32768), (76, 32768), (3, 40000), (77, 65536),
                                         (48, 131072), (24, 24576), (96, 40960), (128, 65536),
                                         (128, 131072)])
def test_long_decode_rows(dtype, rows, hidden):
    """Decode rows of 64 KiB and more: the automatic plan splits each row over
    a thread-block cluster, in one wave or, for up to 128 rows of 64-256 KiB,
    several (f32 rows twice as long in bytes)."""
    x, w = inputs.random_case(rows, hidden, dtype, seed=hidden + rows)
    y = run(x, w, 1e-6, dtype)
    es = 4 if dtype == "f32" else 2
    if hidden * es >= 65536 and hidden * es <= 256 * 1024 and rows <= 128:
        assert rn.rmsnorm_last_variant() == rn.VARIANT_CLUSTER
    compare(y, x, w, 1e-6, dtype, rows_idx=sample_rows(rows, 16, seed=rows))



@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,hidden", [(1, 1 << 20), (4, 300000), (2, 262152), (64, 140000),
                                         (1, 2 * 1024 * 1024 + 8)])
def test_huge_decode_rows_grid(dtype, rows, hidden):
    """Decode rows longer than a cluster holds (above 512 KiB): the automatic
    plan spreads them over every SM with one grid barrier."""
    if dtype == "f32" and hidden > (1 << 20):
        hidden //= 2
    x, w = inputs.random_case(rows, hidden, dtype, seed=hidden % 1000 + rows)
    y = run(x, w, 1e-6, dtype)
    es = 4 if dtype == "f32" else 2
    if hidden * es > 512 * 1024 and hidden * es % 16 == 0:
        assert rn.rmsnorm_last_variant() == rn.VARIANT_GRID
    compare(y, x, w, 1e-6, dtype, rows_idx=sample_rows(rows, 8, seed=rows))
    # in place
    xd = to_device(x, dtype)
    rn.rms_norm(xd, to_device(w, dtype), 1e-6, out=xd, variant=rn.VARIANT_GRID)
    torch.cuda.synchronize()
    compare(from_device(xd, dtype), x, w, 1e-6, dtype, rows_idx=sample_rows(rows, 8, seed=rows))



def test_maximum_row_length():
    """The longest row the library takes (2^26 elements, a 128 MiB bf16 row):
    the grid variant, and the scalar body forced; one element more is refused."""
    hidden = 1 << 26
    x, w = inputs.random_case(1, hidden, "bf16", seed=26)
    for v in (rn.VARIANT_AUTO, rn.VARIANT_GENERIC):
        y = run(x, w, 1e-6, "bf16", variant=v)
        compare(y, x, w, 1e-6, "bf16")
    sms, optin = rn.rmsnorm_device_limits()
    base = 1 << 30
    rc, _ = rn.rmsnorm_plan_status(base, 3 * base, 5 * base, 1, hidden + 8, rn.BF16, sms, optin)
    assert rc == rn.ERR_INVALID_ARG



@pytest.mark.parametrize("hidden,dtype", [(10240, "bf16"), (12288, "f16"), (20480, "bf16"),
                                          (5120, "f32"), (10000, "bf16")])
def test_prefill_20_to_40_kib_rows(hidden, dtype):
    """Prefill rows of 20-40 KiB (32-byte vectors, one block per row), in the
    automatic plan, sampled rows against the oracle."""
    rows = 3000
    x, w = inputs.random_case(rows, hidden, dtype, seed=hidden)
    y = run(x, w, 1e-6, dtype)
    compare(y, x, w, 1e-6, dtype, rows_idx=sample_rows(rows, 64, seed=hidden))


# ------------------------------------------------------------------ 64-bit offsets

def _accepts_far(rows, hidden, dtype, variant, epi=rn.EPI_PLAIN):
    """accepts() with fake pointers far enough apart for tensors of several GiB."""
    sms, optin = rn.rmsnorm_device_limits()
    base = 1 << 40
    p = rn.Plan()
    rc = rn._load().rmsnorm_plan_epilogue(base, 3 * base, 5 * base, rows, hidden,
                                          rn.DTYPE_CODES[dtype], epi, sms, optin, variant,
                                          rn.ctypes.byref(p))
    return rc == rn.OK


@pytest.mark.parametrize("dtype,hidden", [("bf16", 4096), ("f32", 1000), ("f16", 2880)])
def test_offsets_beyond_4_gib(dtype, hidden):
    """Tensors of more than 2^32 bytes (and, for 16-bit types, 2^31 elements):
    rows around and past those offsets, on every body that takes the shape (plain output), and the
    weight-offset and MXFP8 outputs on the automatic plan, against the oracle.
    The rows repeat a block of 64 seeded rows (rows are independent), so the
    oracle runs on that block only."""
    es = 4 if dtype == "f32" else 2
    rows = (1 << 32) // (hidden * es) + 97        # the last 97 rows start beyond 4 GiB
    assert rows * hidden * es > (1 << 32)
    blk = 64
    xs, w_np = inputs.random_case(blk, hidden, dtype, seed=hidden)
    reps = -(-rows // blk)
    x = to_device(xs, dtype).repeat(reps, 1)[:rows]
    w = to_device(w_np, dtype)
    # first rows, rows around 2^31 elements and 2^32 bytes, the last rows
    marks = [0, (1 << 31) // hidden, (1 << 32) // (hidden * es)]
    idx = np.unique(np.clip(np.concatenate(
        [np.arange(m - 3, m + 4) for m in marks] + [np.arange(rows - 8, rows)]), 0, rows - 1))
    sel = torch.from_numpy(idx).cuda()
    x_sel = xs[idx % blk]
    y = torch.empty_like(x)
    ran = 0
    for v in VARIANTS:
        if not _accepts_far(rows, hidden, dtype, v):
            continue
        y.zero_()
        rn.rms_norm(x, w, 1e-6, out=y, variant=v)
        torch.cuda.synchronize()
        compare(from_device(y.index_select(0, sel), dtype), x_sel, w_np, 1e-6, dtype)
        ran += 1
    assert ran >= 3
    y.zero_()
    rn.rms_norm_bias(x, w, 0.5, 1e-6, out=y)
    torch.cuda.synchronize()
    compare(from_device(y.index_select(0, sel), dtype), x_sel, w_np, 1e-6, dtype, bias=0.5)
    del y
    if hidden % 32 == 0:
        q, s = rn.rms_norm_quant(x, w, 1e-6, "mxfp8")
        torch.cuda.synchronize()
        compare_quant(q.index_select(0, sel).cpu().numpy(), s.index_select(0, sel).cpu().numpy(),
                      x_sel, w_np, -0.0, 1e-6, dtype, "mxfp8")


def test_more_rows_than_a_grid_holds_blocks_of():
    """2^31 + 5 rows of 16 bytes (x and y 34 GB each): more rows than the
    launch grid has blocks, so every body that takes the shape walks its rows
    with a 64-bit grid-stride loop; the first rows, rows around 2^31 and the
    last rows against the oracle.  The rows repeat a block of 64 seeded rows."""
    dtype, hidden, blk = "bf16", 8, 64
    rows = (1 << 31) + 5
    xs, w_np = inputs.random_case(blk, hidden, dtype, seed=31)
    x = to_device(xs, dtype).repeat(-(-rows // blk), 1)[:rows]
    w = to_device(w_np, dtype)
    idx = np.unique(np.concatenate([np.arange(0, 4), np.arange((1 << 31) - 4, rows)]))
    sel = torch.from_numpy(idx).cuda()
    y = torch.empty_like(x)
    ran = []
    for v in VARIANTS:
        if not _accepts_far(rows, hidden, dtype, v):
            continue
        y.fill_(0)
        p = rn.Plan()
        rn.rms_norm(x, w, 1e-6, out=y, variant=v, plan=p)
        torch.cuda.synchronize()
        assert 0 < p.grid < rows
        compare(from_device(y.index_select(0, sel), dtype), xs[idx % blk], w_np, 1e-6, dtype)
        ran.append(p.variant)
    assert len(set(ran)) >= 4, ran
