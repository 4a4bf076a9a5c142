"""fp64 CPU oracle for the row-wise RMSNorm forward.

TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
benchmark's CPU baseline (and its ``--impl reference`` arm) may import this
module; the CUDA library and its Python binding never do.  It shares no code
with the CUDA path: the arithmetic lives in ``oracle.c`` (plain C, binary64),
built here with gcc into ``oracle/_build/liboracle.so``.

What it computes is the RMSNorm of "Build a GPU compiler from scratch: from
PyTorch to CUDA via multi-level IR (Emmy)" (introduction and section "Tensor
IR": square, sum, divide by the count, add epsilon, rsqrt, two multiplies)
and "CuTeDSL at Perplexity", section "QK Norm" (rsqrt of the mean square plus
EPS, times the element, times the weight plus WEIGHT_BIAS, cast back to the
element type), with the MXFP8 output the same page's section "Blackwell
support" names, in the OCP Microscaling v1.0 definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

F32, BF16, F16 = 0, 1, 2
_FMT = {"f32": F32, "bf16": BF16, "f16": F16}
_STORAGE = {F32: np.float32, BF16: np.uint16, F16: np.uint16}

_lib = None


def fmt_code(dtype) -> int:
    """Accept 'f32' / 'bf16' / 'f16' or an integer code."""
    if isinstance(dtype, str):
        return _FMT[dtype]
    return int(dtype)


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (plain C11, -O2, no SIMD intrinsics)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(os.path.join(_HERE, "oracle.h")))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        l = ctypes.CDLL(build())
        vp, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
        for name in ("oracle_rmsnorm_f64", "oracle_rmsnorm"):
            getattr(l, name).argtypes = [vp, vp, vp, i64, i64, f32, i32]
            getattr(l, name).restype = i32
        for name in ("oracle_widen_array", "oracle_round_array"):
            getattr(l, name).argtypes = [vp, vp, i64, i32]
            getattr(l, name).restype = i32
        for name in ("oracle_rmsnorm_bias_f64", "oracle_rmsnorm_bias"):
            getattr(l, name).argtypes = [vp, vp, vp, i64, i64, f32, f32, i32]
            getattr(l, name).restype = i32
        l.oracle_mxfp8_quantize.argtypes = [vp, i64, i64, vp, vp]
        l.oracle_mxfp8_quantize.restype = i32
        l.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        l.oracle_e4m3_value.restype = ctypes.c_double
        l.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        l.oracle_e4m3_encode.restype = ctypes.c_uint8
        l.oracle_mxfp4_quantize.argtypes = [vp, i64, i64, vp, vp]
        l.oracle_mxfp4_quantize.restype = i32
        l.oracle_nvfp4_quantize.argtypes = [vp, i64, i64, ctypes.c_double, vp, vp]
        l.oracle_nvfp4_quantize.restype = i32
        l.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        l.oracle_e2m1_value.restype = ctypes.c_double
        l.oracle_e2m1_encode.argtypes = [ctypes.c_double]
        l.oracle_e2m1_encode.restype = ctypes.c_uint8
        l.oracle_qk_norm.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, f32, i32]
        l.oracle_qk_norm.restype = i32
        l.oracle_round_value.argtypes = [ctypes.c_double, i32]
        l.oracle_round_value.restype = ctypes.c_double
        _lib = l
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check_storage(a: np.ndarray, fmt: int) -> np.ndarray:
    want = _STORAGE[fmt]
    if a.dtype != want:
        raise TypeError(f"format {fmt} wants storage {np.dtype(want)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def rmsnorm_f64(x: np.ndarray, w: np.ndarray, eps: float, dtype) -> np.ndarray:
    """y = x * rsqrt(mean(x^2) + eps) * w per row, in binary64 (unrounded).

    ``x`` is [rows, hidden] storage (float32, or uint16 bit patterns for
    bf16/f16); ``w`` is [hidden] of the same storage."""
    fmt = fmt_code(dtype)
    x = _check_storage(x, fmt)
    w = _check_storage(w, fmt)
    rows, hidden = x.shape
    if w.shape != (hidden,):
        raise ValueError("weight must have shape [hidden]")
    y = np.empty((rows, hidden), dtype=np.float64)
    rc = lib().oracle_rmsnorm_f64(_ptr(x), _ptr(w), _ptr(y), rows, hidden, float(eps), fmt)
    if rc != 0:
        raise ValueError("oracle_rmsnorm_f64 rejected its arguments")
    return y


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float, dtype) -> np.ndarray:
    """The oracle's result rounded (nearest-even, from binary64) to the
    element format; returned in the same storage as ``x``."""
    fmt = fmt_code(dtype)
    x = _check_storage(x, fmt)
    w = _check_storage(w, fmt)
    rows, hidden = x.shape
    if w.shape != (hidden,):
        raise ValueError("weight must have shape [hidden]")
    y = np.empty((rows, hidden), dtype=_STORAGE[fmt])
    rc = lib().oracle_rmsnorm(_ptr(x), _ptr(w), _ptr(y), rows, hidden, float(eps), fmt)
    if rc != 0:
        raise ValueError("oracle_rmsnorm rejected its arguments")
    return y


def rmsnorm_bias_f64(x: np.ndarray, w: np.ndarray, weight_bias: float, eps: float,
                     dtype) -> np.ndarray:
    """y = x * rsqrt(mean(x^2) + eps) * (w + weight_bias) per row, binary64."""
    fmt = fmt_code(dtype)
    x = _check_storage(x, fmt)
    w = _check_storage(w, fmt)
    rows, hidden = x.shape
    if w.shape != (hidden,):
        raise ValueError("weight must have shape [hidden]")
    y = np.empty((rows, hidden), dtype=np.float64)
    rc = lib().oracle_rmsnorm_bias_f64(_ptr(x), _ptr(w), _ptr(y), rows, hidden,
                                       float(weight_bias), float(eps), fmt)
    if rc != 0:
        raise ValueError("oracle_rmsnorm_bias_f64 rejected its arguments")
    return y


def rmsnorm_bias(x: np.ndarray, w: np.ndarray, weight_bias: float, eps: float,
                 dtype) -> np.ndarray:
    """rmsnorm_bias_f64 rounded nearest-even to the element format."""
    fmt = fmt_code(dtype)
    x = _check_storage(x, fmt)
    w = _check_storage(w, fmt)
    rows, hidden = x.shape
    if w.shape != (hidden,):
        raise ValueError("weight must have shape [hidden]")
    y = np.empty((rows, hidden), dtype=_STORAGE[fmt])
    rc = lib().oracle_rmsnorm_bias(_ptr(x), _ptr(w), _ptr(y), rows, hidden, float(weight_bias),
                                   float(eps), fmt)
    if rc != 0:
        raise ValueError("oracle_rmsnorm_bias rejected its arguments")
    return y


def mxfp8_quantize(v: np.ndarray) -> tuple:
    """MXFP8 of a [rows, cols] array of values (cols a multiple of 32):
    (E4M3 codes uint8 [rows, cols], E8M0 scales uint8 [rows, cols / 32])."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    rows, cols = v.shape
    codes = np.empty((rows, cols), dtype=np.uint8)
    scales = np.empty((rows, max(cols // 32, 0)), dtype=np.uint8)
    rc = lib().oracle_mxfp8_quantize(_ptr(v), rows, cols, _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("oracle_mxfp8_quantize rejected its arguments")
    return codes, scales


def _decision_values(y: np.ndarray, rel: float, absolute: float) -> np.ndarray:
    """The row results in binary32, the precision a kernel holding fp32 values
    takes its decisions in (nearest-even from the binary64 results); with
    ``rel`` != 0 their magnitudes moved by |y| * rel and by ``absolute`` in
    the same direction (away from zero for rel > 0, towards it, never across
    it, for rel < 0), which brackets the codes any binary32 result within that
    distance may take."""
    y32 = round_to(y, "f32").astype(np.float64)
    if not rel:
        return y32
    with np.errstate(invalid="ignore"):
        mag = np.abs(y32) * (1.0 + rel) + np.copysign(absolute, rel)
        return np.copysign(np.maximum(mag, 0.0), y32)


def rmsnorm_mxfp8(x: np.ndarray, w: np.ndarray, weight_bias: float, eps: float, dtype,
                  rel: float = 0.0, absolute: float = 0.0) -> tuple:
    """The normalised rows quantised to MXFP8 (OCP MX v1.0).

    The value that decides each code is the row result in binary32 (the
    binary64 result rounded nearest-even to binary32), as a kernel holding
    fp32 values decides it; ``rel`` and ``absolute`` move those values first
    (_decision_values), which brackets the codes any result within that
    distance may take."""
    y = rmsnorm_bias_f64(x, w, weight_bias, eps, dtype)
    return mxfp8_quantize(_decision_values(y, rel, absolute))


def mxfp4_quantize(v: np.ndarray) -> tuple:
    """MXFP4 of a [rows, cols] array (cols a multiple of 32): (packed E2M1
    codes uint8 [rows, cols / 2], even element in the low nibble; E8M0 scales
    uint8 [rows, cols / 32])."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    rows, cols = v.shape
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    scales = np.empty((rows, max(cols // 32, 0)), dtype=np.uint8)
    if lib().oracle_mxfp4_quantize(_ptr(v), rows, cols, _ptr(codes), _ptr(scales)) != 0:
        raise ValueError("oracle_mxfp4_quantize rejected its arguments")
    return codes, scales


def nvfp4_quantize(v: np.ndarray, global_scale: float) -> tuple:
    """NVFP4 of a [rows, cols] array (cols a multiple of 16) against the
    per-tensor scale: (packed E2M1 codes uint8 [rows, cols / 2]; E4M3 scales
    uint8 [rows, cols / 16])."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    rows, cols = v.shape
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    scales = np.empty((rows, max(cols // 16, 0)), dtype=np.uint8)
    if lib().oracle_nvfp4_quantize(_ptr(v), rows, cols, float(global_scale), _ptr(codes),
                                   _ptr(scales)) != 0:
        raise ValueError("oracle_nvfp4_quantize rejected its arguments")
    return codes, scales


def rmsnorm_fp4(x: np.ndarray, w: np.ndarray, weight_bias: float, eps: float, dtype, fmt: str,
                global_scale: float = 1.0, rel: float = 0.0, absolute: float = 0.0) -> tuple:
    """The normalised rows quantised to "mxfp4" or "nvfp4"; the deciding
    values are the binary32 row results, moved by ``rel`` and ``absolute``,
    as for rmsnorm_mxfp8."""
    y = _decision_values(rmsnorm_bias_f64(x, w, weight_bias, eps, dtype), rel, absolute)
    if fmt == "mxfp4":
        return mxfp4_quantize(y)
    if fmt == "nvfp4":
        return nvfp4_quantize(y, global_scale)
    raise ValueError(fmt)


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e2m1_encode(v: float) -> int:
    return int(lib().oracle_e2m1_encode(float(v)))


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(int(code))


def e4m3_encode(v: float) -> int:
    return int(lib().oracle_e4m3_encode(float(v)))


def widen(a: np.ndarray, dtype) -> np.ndarray:
    """Exact binary64 values of stored elements."""
    fmt = fmt_code(dtype)
    a = _check_storage(a, fmt)
    out = np.empty(a.shape, dtype=np.float64)
    lib().oracle_widen_array(_ptr(a), _ptr(out), a.size, fmt)
    return out


def round_to(v: np.ndarray, dtype) -> np.ndarray:
    """Round binary64 values to the format, nearest-even, in its storage."""
    fmt = fmt_code(dtype)
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=_STORAGE[fmt])
    lib().oracle_round_array(_ptr(v), _ptr(out), v.size, fmt)
    return out


def qk_norm(q: np.ndarray, k: np.ndarray, q_weight: np.ndarray, k_weight: np.ndarray,
            tokens: int, q_heads: int, k_heads: int, head_dim: int, q_token_stride: int,
            k_token_stride: int, weight_bias: float, eps: float, dtype) -> tuple:
    """Per-head QK norm ("CuTeDSL at Perplexity", section "QK Norm") on copies
    of q and k (flat storage arrays); returns the normalised copies."""
    fmt = fmt_code(dtype)
    qo = np.array(_check_storage(q, fmt), copy=True)
    ko = np.array(_check_storage(k, fmt), copy=True)
    qw = _check_storage(q_weight, fmt)
    kw = _check_storage(k_weight, fmt)
    if qw.size < head_dim or kw.size < head_dim:
        raise ValueError("weights need head_dim elements")
    if tokens > 0 and (qo.size < (tokens - 1) * q_token_stride + q_heads * head_dim
                       or ko.size < (tokens - 1) * k_token_stride + k_heads * head_dim):
        raise ValueError("q/k storage too small for tokens x stride")
    rc = lib().oracle_qk_norm(_ptr(qo), _ptr(ko), _ptr(qw), _ptr(kw), tokens, q_heads, k_heads,
                              head_dim, q_token_stride, k_token_stride, float(weight_bias),
                              float(eps), fmt)
    if rc != 0:
        raise ValueError("oracle_qk_norm rejected its arguments")
    return qo, ko
