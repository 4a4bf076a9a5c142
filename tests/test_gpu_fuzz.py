"""Seeded random cases through the C ABI against the oracle: row counts and
row lengths drawn log-uniformly, the three element types, every variant the
selector accepts for the shape (or the automatic plan), the plain,
weight-offset and block-scaled outputs, in-place calls, pointers one element
off a 16-byte boundary, eps of zero, and rows scaled over many decades.  Each
case draws its own inputs; up to 24 rows of each output are compared.  The
cases complement the fixed grids of the other tests with shapes nobody
picked by hand."""
import numpy as np
import pytest

import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import compare, compare_quant, from_device, sample_rows, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

VARIANTS = [rn.VARIANT_AUTO, rn.VARIANT_WARP_PER_ROW, rn.VARIANT_CTA_PER_ROW,
            rn.VARIANT_STAGED, rn.VARIANT_PERSISTENT, rn.VARIANT_GENERIC, rn.VARIANT_CLUSTER,
            rn.VARIANT_GRID]
EPIS = ["plain", "bias", "mxfp8", "mxfp4", "nvfp4"]
BLOCK = {"mxfp8": 32, "mxfp4": 32, "nvfp4": 16}
N_CASES = 600


@pytest.fixture(scope="module", autouse=True)
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rn.ensure_context(0)
    yield
    torch.cuda.synchronize()
    assert rn.rmsnorm_get_device_status() == rn.OK


def accepts(rows, hidden, dtype, variant, epi, x_off, y_off):
    """The selector's answer for this forced variant (host-only query, with
    fake pointers that keep the call's alignment)."""
    sms, optin = rn.rmsnorm_device_limits()
    base = 1 << 40
    p = rn.Plan()
    return rn._load().rmsnorm_plan_epilogue(base + x_off, 3 * base, 5 * base + y_off, rows,
                                            hidden, rn.DTYPE_CODES[dtype], epi, sms, optin,
                                            variant, rn.ctypes.byref(p))


def draw_case(i):
    rng = np.random.default_rng(1000 + i)
    dtype = ["bf16", "f16", "f32"][rng.integers(3)]
    hidden = int(np.exp(rng.uniform(0, np.log(70000))))
    epi = EPIS[rng.integers(len(EPIS))]
    if epi in BLOCK:
        blk = BLOCK[epi]
        hidden = max(blk, hidden // blk * blk)
    cap = (1 << 24) // hidden                    # at most 2^24 elements per case
    rows = int(np.exp(rng.uniform(0, np.log(max(2, min(5000, cap))))))
    variant = VARIANTS[rng.integers(len(VARIANTS))]
    in_place = epi in ("plain", "bias") and rng.random() < 0.3
    misaligned = epi in ("plain", "bias") and dtype != "f32" and rng.random() < 0.15
    eps = [1e-6, 1e-5, 0.0][rng.integers(3)]
    bias = float([0.0, 1.0, -0.0, 0.5][rng.integers(4)]) if epi != "plain" else None
    g = float(np.exp(rng.uniform(np.log(1e-3), np.log(1.0)))) if epi == "nvfp4" else 1.0
    scaled = rng.random() < 0.3
    return dict(dtype=dtype, hidden=hidden, rows=rows, epi=epi, variant=variant,
                in_place=in_place, misaligned=misaligned, eps=eps, bias=bias, g=g,
                scaled=scaled, seed=int(rng.integers(1 << 30)))


def make_x(c):
    x, w = inputs.random_case(c["rows"], c["hidden"], c["dtype"], seed=c["seed"])
    if c["scaled"]:
        # rows scaled by powers of two over many decades (exact in every type
        # while the values stay in range): f16 keeps to 2^-8..2^8
        rng = np.random.default_rng(c["seed"])
        span = 8 if c["dtype"] == "f16" else 60
        k = rng.integers(-span, span + 1, size=(c["rows"], 1)).astype(np.float64)
        z = oracle_widen(x, c["dtype"]) * np.exp2(k)
        x = inputs.to_storage(z.astype(np.float32), c["dtype"])
    return x, w


def oracle_widen(a, dtype):
    import oracle
    return oracle.widen(a, dtype)


def device_x(x_np, dtype, misaligned):
    if not misaligned:
        return to_device(x_np, dtype)
    flat = np.concatenate([np.zeros(1, x_np.dtype), x_np.ravel()])
    return to_device(flat, dtype)[1:].view(x_np.shape)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(i):
    c = draw_case(i)
    epi = {"plain": rn.EPI_PLAIN, "bias": rn.EPI_BIAS, "mxfp8": rn.EPI_MXFP8,
           "mxfp4": rn.EPI_MXFP4, "nvfp4": rn.EPI_NVFP4}[c["epi"]]
    x_off = 2 if c["misaligned"] else 0
    rc = accepts(c["rows"], c["hidden"], c["dtype"], c["variant"], epi, x_off,
                 x_off if c["in_place"] else 0)
    x_np, w_np = make_x(c)
    x = device_x(x_np, c["dtype"], c["misaligned"])
    w = to_device(w_np, c["dtype"])
    idx = sample_rows(c["rows"], 24, seed=i)
    out = x if c["in_place"] else None
    if rc != rn.OK:
        # the library refuses the same forced variant with the planner's status
        with pytest.raises(rn.RmsnormError) as e:
            if c["epi"] in BLOCK:
                rn.rms_norm_quant(x, w, c["eps"], c["epi"], weight_bias=c["bias"],
                                  global_scale=c["g"], variant=c["variant"])
            elif c["epi"] == "bias":
                rn.rms_norm_bias(x, w, c["bias"], c["eps"], out=out, variant=c["variant"])
            else:
                rn.rms_norm(x, w, c["eps"], out=out, variant=c["variant"])
        assert e.value.status == rc, c
        return
    if c["epi"] in BLOCK:
        q, s = rn.rms_norm_quant(x, w, c["eps"], c["epi"], weight_bias=c["bias"],
                                 global_scale=c["g"], variant=c["variant"])
        torch.cuda.synchronize()
        compare_quant(q.cpu().numpy(), s.cpu().numpy(), x_np, w_np, c["bias"], c["eps"],
                      c["dtype"], c["epi"], c["g"], rows_idx=idx)
        return
    if c["epi"] == "bias":
        y = rn.rms_norm_bias(x, w, c["bias"], c["eps"], out=out, variant=c["variant"])
    else:
        y = rn.rms_norm(x, w, c["eps"], out=out, variant=c["variant"])
    torch.cuda.synchronize()
    compare(from_device(y, c["dtype"]), x_np, w_np, c["eps"], c["dtype"], rows_idx=idx,
            bias=c["bias"])


def test_cases_cover_the_space():
    """The drawn cases reach every element type, epilogue and variant, and
    in-place, misaligned, eps = 0 and scaled calls."""
    cs = [draw_case(i) for i in range(N_CASES)]
    assert {c["dtype"] for c in cs} == {"bf16", "f16", "f32"}
    assert {c["epi"] for c in cs} == set(EPIS)
    assert {c["variant"] for c in cs} == set(VARIANTS)
    for key in ("in_place", "misaligned", "scaled"):
        assert any(c[key] for c in cs), key
    assert any(c["eps"] == 0.0 for c in cs)
