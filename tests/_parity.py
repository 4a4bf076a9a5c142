"""Parity helpers shared by the GPU tests: move seeded inputs to the device,
run the library, and compare with the oracle.

Tolerance (stated for the method's outputs):
* f32: |gpu - oracle_f64| <= 1e-5 or <= 1e-5 * |oracle_f64| (element-wise OR);
* bf16 / f16: at most 1 unit in the last place between the GPU's output and
  the oracle's binary64 result rounded to the format with nearest-even
  (distance measured on the monotone integer line of the bit patterns, so it
  is exact across binades and signs); NaN must meet NaN.
* MXFP8 codes: the scale and every code the oracle gives for the row result
  in binary32, unless a relative change of at most MX_REL (the f32 bar) in
  that result moves the decision -- then the GPU's choice must lie within the
  codes the oracle gives at both ends of that band (a code is an integer that
  floating point decides; the band is where fp32 rounding order may decide
  it either way).
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
_E4M3 = None


def e4m3_table() -> np.ndarray:
    """Value of every E4M3 code (the oracle's decoder)."""
    global _E4M3
    if _E4M3 is None:
        _E4M3 = np.array([oracle.e4m3_value(c) for c in range(256)])
    return _E4M3


def compare_mx(codes: np.ndarray, scales: np.ndarray, x: np.ndarray, w: np.ndarray, bias: float,
               eps: float, dtype: str, rows_idx: np.ndarray | None = None) -> dict:
    """Compare GPU MXFP8 rows (uint8 codes [rows, hidden], uint8 scales
    [rows, hidden / 32]) with the oracle; raises AssertionError on a
    violation.  Returns counts of exact and band-decided results."""
    if rows_idx is not None:
        x, codes, scales = x[rows_idx], codes[rows_idx], scales[rows_idx]
    if x.shape[0] == 0:
        return {"rows": 0}
    rows, hidden = x.shape
    nb = hidden // 32
    c0, s0 = oracle.rmsnorm_mxfp8(x, w, bias, eps, dtype)
    clo, slo = oracle.rmsnorm_mxfp8(x, w, bias, eps, dtype, rel=-MX_REL)
    chi, shi = oracle.rmsnorm_mxfp8(x, w, bias, eps, dtype, rel=MX_REL)
    band = (slo != shi) | (slo != s0) | (shi != s0)
    ok_s = (scales == s0) | (band & ((scales == slo) | (scales == shi)))
    if not ok_s.all():
        i, b = np.argwhere(~ok_s)[0]
        raise AssertionError(f"scale mismatch row {i} block {b}: gpu {scales[i, b]} oracle "
                             f"{s0[i, b]} (band {slo[i, b]}..{shi[i, b]})")
    tab = e4m3_table()
    g = tab[codes].reshape(rows, nb, 32)
    lo = tab[clo].reshape(rows, nb, 32)
    hi = tab[chi].reshape(rows, nb, 32)
    ref = tab[c0].reshape(rows, nb, 32)
    special = s0 == 0xFF                       # NaN / Inf in the block: the scale says it all
    same = (scales == s0) & ~band & ~special   # the scale is the oracle's, not in the band
    lo_v, hi_v = np.minimum(lo, hi), np.maximum(lo, hi)
    inside = (g >= lo_v) & (g <= hi_v)
    bad = same[:, :, None] & ~inside
    if bad.any():
        i, b, j = np.argwhere(bad)[0]
        raise AssertionError(f"code mismatch row {i} col {b * 32 + j}: gpu {g[i, b, j]!r} "
                             f"oracle {ref[i, b, j]!r} (band {lo[i, b, j]!r}..{hi[i, b, j]!r})")
    # Blocks whose scale sits in the band: every element within the MX
    # error bound of the binary64 result at the GPU's scale.
    amb = band & ~special
    if amb.any():
        y = oracle.rmsnorm_bias_f64(x, w, bias, eps, dtype).reshape(rows, nb, 32)
        X = np.exp2(scales.astype(np.float64) - 127.0)[:, :, None]
        t = np.abs(y) / X
        step = np.where(t >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(t, 2.0 ** -6))) - 3),
                        2.0 ** -9)
        err = np.abs(g * X - y)
        sat = t >= 448
        tol = (step / 2 * (1 + MX_REL) + MX_REL * t) * X
        good = np.where(sat, np.abs(g) == 448, err <= tol)
        badb = amb[:, :, None] & ~good
        if badb.any():
            i, b, j = np.argwhere(badb)[0]
            raise AssertionError(f"band-scale block row {i} block {b} elem {j}: gpu "
                                 f"{g[i, b, j]!r} * 2^{int(scales[i, b]) - 127} vs {y[i, b, j]!r}")
    return {"rows": rows, "blocks": rows * nb, "band_blocks": int(band.sum()),
            "exact_codes": float((codes == c0)[np.repeat(same, 32, axis=1)].mean())
            if same.any() else 1.0}
