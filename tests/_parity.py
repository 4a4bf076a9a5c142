"""Parity helpers shared by the GPU tests: move seeded inputs to the device,
run the library, and compare with the oracle.

Tolerance (stated for the method's outputs):
* f32: |gpu - oracle_f64| <= 1e-5 or <= 1e-5 * |oracle_f64| (element-wise OR);
* bf16 / f16: at most 1 unit in the last place between the GPU's output and
  the oracle's binary64 result rounded to the format with nearest-even
  (distance measured on the monotone integer line of the bit patterns, so it
  is exact across binades and signs); NaN must meet NaN.
* Block-scaled codes (MXFP8, MXFP4, NVFP4): the scale and every code the
  oracle gives for the row result in binary32 (a code is an integer that
  floating point decides, so both sides decide on values of the kernel's
  precision), unless moving that result by MX_REL relative (the f32 bar)
  plus MX_ABS absolute changes the decision -- then the GPU's choice must
  lie within the codes the oracle gives at both ends of that band (the band
  is where the device's rounding order may decide it either way; MX_ABS,
  four units of binary32's smallest subnormal, covers results in binary32's
  subnormal range, which carry fewer than 24 bits).
"""
from __future__ import annotations

import numpy as np

import oracle

F32_TOL = 1e-5
ULP_TOL = 1


def to_device(a: np.ndarray, dtype: str):
    import torch
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).cuda()


def from_device(t, dtype: str) -> np.ndarray:
    import torch
    c = t.detach().cpu().contiguous()
    if dtype == "f32":
        return c.numpy()
    return c.view(torch.int16).numpy().view(np.uint16)


def monotone(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def compare(gpu: np.ndarray, x: np.ndarray, w: np.ndarray, eps: float, dtype: str,
            rows_idx: np.ndarray | None = None, bias: float | None = None) -> dict:
    """Compare GPU output rows with the oracle on the same inputs.

    ``rows_idx`` selects the rows to check (the oracle runs on just those);
    None checks every row.  Returns a summary; raises AssertionError on a
    violation, naming the first bad element."""
    if rows_idx is None:
        xs, gs = x, gpu
    else:
        xs, gs = x[rows_idx], gpu[rows_idx]
    if xs.shape[0] == 0:
        return {"rows": 0}
    if dtype == "f32":
        ref = (oracle.rmsnorm_f64(xs, w, eps, dtype) if bias is None
               else oracle.rmsnorm_bias_f64(xs, w, bias, eps, dtype))
        g = gs.astype(np.float64)
        nan_ref = np.isnan(ref)
        assert np.array_equal(nan_ref, np.isnan(g)), "NaN pattern differs"
        with np.errstate(invalid="ignore"):       # inf - inf where both are inf
            d = np.abs(g - ref)
        ok = (d <= F32_TOL) | (d <= F32_TOL * np.abs(ref)) | nan_ref | (g == ref)
        if not ok.all():
            i, j = np.argwhere(~ok)[0]
            raise AssertionError(f"f32 mismatch at row {i} col {j}: gpu {g[i, j]!r} oracle "
                                 f"{ref[i, j]!r}")
        fin = ~nan_ref
        return {"rows": xs.shape[0], "max_abs": float(d[fin].max(initial=0.0)),
                "max_rel": float((d[fin] / np.maximum(np.abs(ref[fin]), 1e-30)).max(initial=0.0))}
    ref_bits = (oracle.rmsnorm(xs, w, eps, dtype) if bias is None
                else oracle.rmsnorm_bias(xs, w, bias, eps, dtype))
    ref_w = oracle.widen(ref_bits, dtype)
    g_w = oracle.widen(gs, dtype)
    nan_ref = np.isnan(ref_w)
    assert np.array_equal(nan_ref, np.isnan(g_w)), "NaN pattern differs"
    dist = np.abs(monotone(gs) - monotone(ref_bits))
    dist[nan_ref] = 0
    if (dist > ULP_TOL).any():
        i, j = np.argwhere(dist > ULP_TOL)[0]
        raise AssertionError(f"{dtype} mismatch at row {i} col {j}: gpu {g_w[i, j]!r} oracle "
                             f"{ref_w[i, j]!r} ({dist[i, j]} ulp)")
    return {"rows": xs.shape[0], "max_ulp": int(dist.max(initial=0)),
            "frac_off_by_one": float((dist == 1).mean())}


def sample_rows(rows: int, n: int, seed: int = 0) -> np.ndarray:
    """First, last and n-2 seeded rows in between (sorted, unique)."""
    if rows <= n:
        return np.arange(rows)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, rows - 1), size=n - 2, replace=False)
    return np.unique(np.concatenate([[0, rows - 1], mid]))


MX_REL = 1e-5
MX_ABS = 2.0 ** -147
_TABLES = {}


def e4m3_table() -> np.ndarray:
    """Value of every E4M3 code (the oracle's decoder)."""
    if "e4m3" not in _TABLES:
        _TABLES["e4m3"] = np.array([oracle.e4m3_value(c) for c in range(256)])
    return _TABLES["e4m3"]


def e2m1_table() -> np.ndarray:
    if "e2m1" not in _TABLES:
        _TABLES["e2m1"] = np.array([oracle.e2m1_value(c) for c in range(16)])
    return _TABLES["e2m1"]


# fmt -> (elements per block, bits per code, NaN scale code)
QFMT = {"mxfp8": (32, 8, 0xFF), "mxfp4": (32, 4, 0xFF), "nvfp4": (16, 4, 0x7F)}


def _oracle_q(x, w, bias, eps, dtype, fmt, gscale, rel=0.0):
    a = MX_ABS if rel else 0.0
    if fmt == "mxfp8":
        return oracle.rmsnorm_mxfp8(x, w, bias, eps, dtype, rel=rel, absolute=a)
    return oracle.rmsnorm_fp4(x, w, bias, eps, dtype, fmt, global_scale=gscale, rel=rel,
                              absolute=a)


def _decode(codes, fmt, hidden):
    """Element values of stored codes [rows, hidden * bits / 8] -> [rows, hidden]."""
    if QFMT[fmt][1] == 8:
        return e4m3_table()[codes]
    un = np.empty((codes.shape[0], hidden), dtype=np.uint8)
    un[:, 0::2] = codes & 0xF
    un[:, 1::2] = codes >> 4
    return e2m1_table()[un]


def _scale_values(scales, fmt, gscale):
    if fmt == "nvfp4":
        return e4m3_table()[scales] * gscale
    return np.exp2(scales.astype(np.float64) - 127.0)


def _half_step(t, fmt):
    """Half the spacing of the element grid at magnitude t (scaled units)."""
    if QFMT[fmt][1] == 8:
        return np.where(t >= 2.0 ** -6,
                        np.exp2(np.floor(np.log2(np.maximum(t, 2.0 ** -6))) - 4), 2.0 ** -10)
    return np.where(t < 2, 0.25, np.where(t < 4, 0.5, 1.0))


def compare_quant(codes: np.ndarray, scales: np.ndarray, x: np.ndarray, w: np.ndarray,
                  bias: float, eps: float, dtype: str, fmt: str = "mxfp8", gscale: float = 1.0,
                  rows_idx: np.ndarray | None = None) -> dict:
    """Compare GPU block-scaled rows (codes as stored, scales [rows, hidden /
    block]) with the oracle; raises AssertionError on a violation."""
    if rows_idx is not None:
        x, codes, scales = x[rows_idx], codes[rows_idx], scales[rows_idx]
    if x.shape[0] == 0:
        return {"rows": 0}
    block, bits, nan_code = QFMT[fmt]
    rows, hidden = x.shape
    nb = hidden // block
    c0, s0 = _oracle_q(x, w, bias, eps, dtype, fmt, gscale)
    clo, slo = _oracle_q(x, w, bias, eps, dtype, fmt, gscale, rel=-MX_REL)
    chi, shi = _oracle_q(x, w, bias, eps, dtype, fmt, gscale, rel=MX_REL)
    band = (slo != shi) | (slo != s0) | (shi != s0)
    ok_s = (scales == s0) | (band & ((scales == slo) | (scales == shi)))
    if not ok_s.all():
        i, b = np.argwhere(~ok_s)[0]
        raise AssertionError(f"{fmt} scale mismatch row {i} block {b}: gpu {scales[i, b]} "
                             f"oracle {s0[i, b]} (band {slo[i, b]}..{shi[i, b]})")
    g = _decode(codes, fmt, hidden).reshape(rows, nb, block)
    lo = _decode(clo, fmt, hidden).reshape(rows, nb, block)
    hi = _decode(chi, fmt, hidden).reshape(rows, nb, block)
    ref = _decode(c0, fmt, hidden).reshape(rows, nb, block)
    special = s0 == nan_code                   # a NaN in the block: the scale says it all
    same = (scales == s0) & ~band & ~special
    lo_v, hi_v = np.minimum(lo, hi), np.maximum(lo, hi)
    inside = (g >= lo_v) & (g <= hi_v)
    bad = same[:, :, None] & ~inside
    if bad.any():
        i, b, j = np.argwhere(bad)[0]
        raise AssertionError(f"{fmt} code mismatch row {i} col {b * block + j}: gpu "
                             f"{g[i, b, j]!r} oracle {ref[i, b, j]!r} "
                             f"(band {lo[i, b, j]!r}..{hi[i, b, j]!r})")
    # A zero code carries the sign of the value it stands for (IEEE signs of
    # zero products included), which the comparison of values above ignores.
    zsign = same[:, :, None] & (ref == 0) & (np.signbit(g) != np.signbit(ref))
    if zsign.any():
        i, b, j = np.argwhere(zsign)[0]
        raise AssertionError(f"{fmt} zero-code sign mismatch row {i} col {b * block + j}: gpu "
                             f"{g[i, b, j]!r} oracle {ref[i, b, j]!r}")
    # Blocks whose scale sits in the band: every element within the error
    # bound of the element grid at the GPU's scale.
    amb = band & ~special
    if amb.any():
        y = oracle.rmsnorm_bias_f64(x, w, bias, eps, dtype).reshape(rows, nb, block)
        X = _scale_values(scales, fmt, gscale)[:, :, None]
        with np.errstate(divide="ignore", invalid="ignore"):
            t = np.where(X > 0, np.abs(y) / X, 0.0)
        err = np.abs(g * X - y)
        maxmag = 448.0 if bits == 8 else 6.0
        sat = t >= maxmag
        tol = (_half_step(t, fmt) * (1 + MX_REL) + MX_REL * t) * X + MX_ABS
        good = np.where(X == 0, g == 0, np.where(sat, np.abs(g) == maxmag, err <= tol))
        good &= (g != 0) | np.isnan(y) | (np.signbit(g) == np.signbit(y))
        badb = amb[:, :, None] & ~good
        if badb.any():
            i, b, j = np.argwhere(badb)[0]
            raise AssertionError(f"{fmt} band-scale block row {i} block {b} elem {j}: gpu "
                                 f"{g[i, b, j]!r} x {X[i, b, 0]!r} vs {y[i, b, j]!r}")
    same_e = np.repeat(same, block, axis=1)
    return {"rows": rows, "blocks": rows * nb, "band_blocks": int(band.sum()),
            "exact_codes": float((g.reshape(rows, hidden) == ref.reshape(rows, hidden))[same_e]
                                 .mean()) if same.any() else 1.0}


def compare_mx(codes: np.ndarray, scales: np.ndarray, x: np.ndarray, w: np.ndarray, bias: float,
               eps: float, dtype: str, rows_idx: np.ndarray | None = None) -> dict:
    """compare_quant for MXFP8."""
    return compare_quant(codes, scales, x, w, bias, eps, dtype, "mxfp8", 1.0, rows_idx)
