"""Parity helpers shared by the GPU tests: move seeded inputs to the device,
run the library, and compare with the oracle.

Tolerance (stated for the method's outputs):
* f32: |gpu - oracle_f64| <= 1e-5 or <= 1e-5 * |oracle_f64| (element-wise OR);
* bf16 / f16: at most 1 unit in the last place between the GPU's output and
  the oracle's binary64 result rounded to the format with nearest-even
  (distance measured on the monotone integer line of the bit patterns, so it
  is exact across binades and signs); NaN must meet NaN.
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
            rows_idx: np.ndarray | None = None) -> dict:
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
        ref = oracle.rmsnorm_f64(xs, w, eps, dtype)
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
    ref_bits = oracle.rmsnorm(xs, w, eps, dtype)
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
