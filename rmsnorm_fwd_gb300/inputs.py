"""Seeded synthetic inputs for the RMSNorm forward workloads.

This module draws inputs only; it holds none of the normalisation's
arithmetic.  Both sides of every parity check (the CUDA library and the CPU
oracle) consume exactly the bytes it returns.

Recipe (one ``numpy.random.PCG64`` stream per tensor, seeded from
``SeedSequence(seed, spawn_key=(workload key, tensor index))``):

* values are drawn in binary32 (``standard_normal`` / ``random`` with
  ``dtype=float32``) in fixed blocks of rows, then rounded to the element
  format with round-to-nearest-even (binary16 via numpy's own conversion,
  bfloat16 by the usual carry-into-bit-16 rule on the binary32 pattern);
* x is drawn before the weight; the per-row scale and the outlier mask come
  from a third stream so that the x values do not depend on them.

Workloads (shapes of the pages' norm use: small embedding-model batches,
decode rows and prefill token blocks at LLM hidden sizes):

============================  ======  =====  =====  =====  ==========================  ============
name                          dtype   rows   hidden eps    x                           weight
============================  ======  =====  =====  =====  ==========================  ============
f32_64x128                    f32     64     128    1e-6   N(0,1)                      U(0.5,1.5)
embed_bf16_8192x1024          bf16    8192   1024   1e-6   N(0,1), 1% entries x20      N(1,0.1)
decode_bf16_{1,8,32}x4096     bf16    1/8/32 4096   1e-6   N(0,2) (std 2)              N(1,0.1)
prefill_bf16_16384x4096       bf16    16384  4096   1e-6   N(0,1)                      N(1,0.1)
wide_{f16,bf16}_65536x{H}     f16/bf16 65536 7168/5120/2880 1e-5  N(0,1) x row scale U(1e-3,1e3)  U(0,2)
============================  ======  =====  =====  =====  ==========================  ============
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

DTYPES = ("f32", "bf16", "f16")
STORAGE = {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16}
ITEMSIZE = {"f32": 4, "bf16": 2, "f16": 2}

_BLOCK_ROWS = 1024  # rows drawn per block; fixed so the stream order is fixed


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str
    rows: int
    hidden: int
    eps: float
    x_dist: str     # "normal", "normal_outliers", "normal_std2", "normal_rowscale"
    w_dist: str     # "u0.5_1.5", "n1_0.1", "u0_2"
    key: int        # seeding key (distinct per workload)

    @property
    def bytes_per_call(self) -> int:
        """Algorithmic bytes: read x, read the weight once, write y."""
        s = ITEMSIZE[self.dtype]
        return 2 * self.rows * self.hidden * s + self.hidden * s

    def with_shape(self, rows: int, hidden: int | None = None) -> "Workload":
        return replace(self, rows=rows, hidden=self.hidden if hidden is None else hidden,
                       name=f"{self.name}@{rows}x{self.hidden if hidden is None else hidden}")


def _mk() -> dict[str, Workload]:
    w = {}
    w["f32_64x128"] = Workload("f32_64x128", "f32", 64, 128, 1e-6, "normal", "u0.5_1.5", 1)
    w["embed_bf16_8192x1024"] = Workload("embed_bf16_8192x1024", "bf16", 8192, 1024, 1e-6,
                                         "normal_outliers", "n1_0.1", 2)
    for i, r in enumerate((1, 8, 32)):
        n = f"decode_bf16_{r}x4096"
        w[n] = Workload(n, "bf16", r, 4096, 1e-6, "normal_std2", "n1_0.1", 30 + i)
    w["prefill_bf16_16384x4096"] = Workload("prefill_bf16_16384x4096", "bf16", 16384, 4096,
                                            1e-6, "normal", "n1_0.1", 4)
    k = 50
    for dt in ("f16", "bf16"):
        for h in (7168, 5120, 2880):
            n = f"wide_{dt}_65536x{h}"
            w[n] = Workload(n, dt, 65536, h, 1e-5, "normal_rowscale", "u0_2", k)
            k += 1
    return w


WORKLOADS: dict[str, Workload] = _mk()
HEADLINE = "prefill_bf16_16384x4096"


def _rng(seed: int, key: int, tensor: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(key, tensor))))


def to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 bit patterns, round-to-nearest-even (finite inputs)."""
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def to_storage(f32: np.ndarray, dtype: str) -> np.ndarray:
    """Round binary32 draws to the element format's storage."""
    if dtype == "f32":
        return np.ascontiguousarray(f32, dtype=np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(f32.astype(np.float16)).view(np.uint16)
    if dtype == "bf16":
        return to_bf16_bits(f32)
    raise ValueError(dtype)


def _draw_weight(wl: Workload, rng: np.random.Generator) -> np.ndarray:
    h = wl.hidden
    if wl.w_dist == "u0.5_1.5":
        v = 0.5 + rng.random(h, dtype=np.float32)
    elif wl.w_dist == "n1_0.1":
        v = np.float32(1.0) + np.float32(0.1) * rng.standard_normal(h, dtype=np.float32)
    elif wl.w_dist == "u0_2":
        v = np.float32(2.0) * rng.random(h, dtype=np.float32)
    else:
        raise ValueError(wl.w_dist)
    return to_storage(v, wl.dtype)


def make_weight(wl: Workload, seed: int = 0) -> np.ndarray:
    return _draw_weight(wl, _rng(seed, wl.key, 1))


def make_x(wl: Workload, seed: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """x as [rows, hidden] storage, drawn block by block."""
    rows, h = wl.rows, wl.hidden
    if out is None:
        out = np.empty((rows, h), dtype=STORAGE[wl.dtype])
    zr = _rng(seed, wl.key, 0)
    ar = _rng(seed, wl.key, 2)
    for r0 in range(0, rows, _BLOCK_ROWS):
        r1 = min(rows, r0 + _BLOCK_ROWS)
        z = zr.standard_normal((r1 - r0, h), dtype=np.float32)
        if wl.x_dist == "normal":
            pass
        elif wl.x_dist == "normal_std2":
            z *= np.float32(2.0)
        elif wl.x_dist == "normal_outliers":
            mask = ar.random((r1 - r0, h), dtype=np.float32) < np.float32(0.01)
            z[mask] *= np.float32(20.0)
        elif wl.x_dist == "normal_rowscale":
            u = ar.random(r1 - r0, dtype=np.float64)
            scale = (1e-3 + (1e3 - 1e-3) * u).astype(np.float32)
            z *= scale[:, None]
        else:
            raise ValueError(wl.x_dist)
        out[r0:r1] = to_storage(z, wl.dtype)
    return out


def make_inputs(wl: Workload | str, seed: int = 0):
    """(x, weight) storage arrays for a workload (or its name)."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    return make_x(wl, seed), make_weight(wl, seed)


def random_case(rows: int, hidden: int, dtype: str, seed: int, scale: float = 1.0,
                w_dist: str = "n1_0.1"):
    """Small ad-hoc case (edge-case tests): x ~ N(0, scale^2), weight per w_dist."""
    wl = Workload(f"case_{rows}x{hidden}_{dtype}", dtype, rows, hidden, 1e-6, "normal", w_dist,
                  key=100000 + hidden)
    zr = _rng(seed, wl.key, rows)
    z = zr.standard_normal((rows, hidden), dtype=np.float32) * np.float32(scale)
    return to_storage(z, dtype), _draw_weight(wl, _rng(seed, wl.key, 10**6 + rows))


@dataclass(frozen=True)
class QkWorkload:
    """Per-head QK norm shapes: q and k heads of a fused [q | k | v] buffer per
    token (v as wide as k), x ~ N(0,1), weights ~ N(1,0.1)."""
    name: str
    dtype: str
    tokens: int
    q_heads: int
    k_heads: int
    head_dim: int
    eps: float
    key: int

    @property
    def width(self) -> int:
        return (self.q_heads + 2 * self.k_heads) * self.head_dim

    @property
    def bytes_per_call(self) -> int:
        s = ITEMSIZE[self.dtype]
        return 2 * self.tokens * (self.q_heads + self.k_heads) * self.head_dim * s \
            + 2 * self.head_dim * s


QK_WORKLOADS: dict[str, QkWorkload] = {
    w.name: w for w in (
        QkWorkload("qk_bf16_16384tok_32q8k_128", "bf16", 16384, 32, 8, 128, 1e-6, 70),
        QkWorkload("qk_bf16_32tok_32q8k_128", "bf16", 32, 32, 8, 128, 1e-6, 71),
        QkWorkload("qk_bf16_16384tok_64q4k_128", "bf16", 16384, 64, 4, 128, 1e-6, 72),
        QkWorkload("qk_bf16_8192tok_16q8k_256", "bf16", 8192, 16, 8, 256, 1e-6, 73),
    )
}


def make_qk_inputs(wl: QkWorkload, seed: int = 0):
    """(qkv [tokens * width] storage, q weight [head_dim], k weight [head_dim])."""
    zr = _rng(seed, wl.key, 0)
    buf = np.empty(wl.tokens * wl.width, dtype=STORAGE[wl.dtype])
    step = _BLOCK_ROWS * wl.width
    for o in range(0, buf.size, step):
        n = min(step, buf.size - o)
        buf[o:o + n] = to_storage(zr.standard_normal(n, dtype=np.float32), wl.dtype)
    wr = _rng(seed, wl.key, 1)
    qw = to_storage(np.float32(1) + np.float32(0.1) * wr.standard_normal(wl.head_dim,
                                                                           dtype=np.float32),
                    wl.dtype)
    kw = to_storage(np.float32(1) + np.float32(0.1) * wr.standard_normal(wl.head_dim,
                                                                           dtype=np.float32),
                    wl.dtype)
    return buf, qw, kw
