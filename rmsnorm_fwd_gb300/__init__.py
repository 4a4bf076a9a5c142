"""Row-wise RMSNorm forward for GB300 (sm_103a): hand-written CUDA kernels
behind the C ABI of ``include/rmsnorm.h`` (``librmsnorm.so``).

This module is the thin Python binding: the functions below have the C
names and only marshal arguments (pointers, sizes, the stream handle) into
the library.  Every step of the computation runs in the library's kernels;
there is no Python, PyTorch or CPU fallback.  If the library cannot be built
or loaded, the first call raises.

PyTorch is used only for device memory and streams (``rms_norm`` takes
tensors, reads their data pointers and the current stream, and calls
``rmsnorm_fwd``).
"""
from __future__ import annotations

import ctypes
import threading

# element types (rmsnorm_dtype_t)
F32, BF16, F16 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", BF16: "bf16", F16: "f16"}
DTYPE_CODES = {"f32": F32, "bf16": BF16, "f16": F16}

# status codes (rmsnorm_status_t)
OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED_DTYPE = 2
ERR_NOT_INITIALIZED = 3
ERR_ALIASING = 4
ERR_CUDA = 5
ERR_DEVICE_TIMEOUT = 6
ERR_MISALIGNED = 7
ERR_UNSUPPORTED_DEVICE = 8
ERR_VARIANT = 9
ERR_TOO_LARGE = 10

# variants (rmsnorm_variant_t)
VARIANT_AUTO = 0
VARIANT_WARP_PER_ROW = 1
VARIANT_CTA_PER_ROW = 2
VARIANT_STAGED = 3
VARIANT_PERSISTENT = 4
VARIANT_GENERIC = 5
VARIANT_CLUSTER = 6
VARIANT_GRID = 7
VARIANT_NAMES = {0: "auto", 1: "warp_per_row", 2: "cta_per_row", 3: "staged", 4: "persistent",
                 5: "generic", 6: "cluster", 7: "grid"}

# epilogues (rmsnorm_epilogue_t)
EPI_PLAIN, EPI_BIAS, EPI_MXFP8, EPI_MXFP4, EPI_NVFP4 = 0, 1, 2, 3, 4
EPI_NAMES = {EPI_PLAIN: "plain", EPI_BIAS: "bias", EPI_MXFP8: "mxfp8", EPI_MXFP4: "mxfp4",
             EPI_NVFP4: "nvfp4"}
EPI_CODES = {v: k for k, v in EPI_NAMES.items()}
# block-scaled outputs: (elements per scale block, bits per element code)
QUANT_FORMATS = {EPI_MXFP8: (32, 8), EPI_MXFP4: (32, 4), EPI_NVFP4: (16, 4)}


class RmsnormError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({rmsnorm_status_string(status)})")


class Plan(ctypes.Structure):
    """rmsnorm_plan_t."""
    _fields_ = [(name, ctypes.c_int32) for name in (
        "variant", "vec_bytes", "threads_per_row", "vecs_per_thread", "block_threads",
        "rows_per_block", "stages", "grid", "smem_bytes", "kernel_index")]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class QkPlan(ctypes.Structure):
    """rmsnorm_qk_plan_t."""
    _fields_ = [(name, ctypes.c_int32) for name in (
        "lanes_per_head", "vecs_per_lane", "heads_per_group", "grid")]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class KernelInfo(ctypes.Structure):
    """rmsnorm_kernel_info_t."""
    _fields_ = [(name, ctypes.c_int32) for name in (
        "variant", "dtype", "vec_bytes", "tpr", "nv", "block", "min_blocks", "cache_policy",
        "epilogue")]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    from . import _build
    return _build.LIB


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import _build
        path = _build.build()  # compiles in-tree if stale; raises if nvcc is missing
        lib = ctypes.CDLL(path, mode=ctypes.RTLD_GLOBAL)
        vp, i64, i32, f32, u64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                  ctypes.c_uint64)
        pp = ctypes.POINTER(Plan)
        sig = {
            "rmsnorm_create": ([], i32),
            "rmsnorm_destroy": ([], i32),
            "rmsnorm_fwd": ([vp, vp, vp, i64, i64, f32, i32, vp], i32),
            "rmsnorm_fwd_ex": ([vp, vp, vp, i64, i64, f32, i32, vp, i32, pp], i32),
            "rmsnorm_plan": ([vp, vp, vp, i64, i64, i32, i32, i32, i32, pp], i32),
            "rmsnorm_plan_host_mapped": ([vp, vp, vp, i64, i64, i32, i32, i32, pp], i32),
            "rmsnorm_fwd_host": ([vp, vp, vp, i64, i64, f32, i32, vp, ctypes.c_size_t, i64, vp],
                                 i32),
            "rmsnorm_qk_norm": ([vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, f32, i32, vp],
                                i32),
            "rmsnorm_qk_norm_ex": ([vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, f32, i32, vp,
                                    ctypes.POINTER(QkPlan)], i32),
            "rmsnorm_fwd_bias": ([vp, vp, vp, i64, i64, f32, f32, i32, vp], i32),
            "rmsnorm_fwd_mxfp8": ([vp, vp, vp, vp, i64, i64, f32, f32, i32, vp], i32),
            "rmsnorm_fwd_mxfp4": ([vp, vp, vp, vp, i64, i64, f32, f32, i32, vp], i32),
            "rmsnorm_fwd_nvfp4": ([vp, vp, vp, vp, i64, i64, f32, f32, f32, i32, vp], i32),
            "rmsnorm_fwd_epilogue_ex": ([vp, vp, vp, vp, i64, i64, i32, f32, f32, f32, i32, vp,
                                         i32, pp], i32),
            "rmsnorm_plan_epilogue": ([vp, vp, vp, i64, i64, i32, i32, i32, i32, i32, pp], i32),
            "rmsnorm_validate_plan_epilogue": ([pp, vp, vp, vp, i64, i64, i32, i32, i32, i32],
                                               i32),
            "rmsnorm_last_variant": ([], i32),
            "rmsnorm_kernel_count": ([], i32),
            "rmsnorm_validate_plan": ([pp, vp, vp, vp, i64, i64, i32, i32, i32], i32),
            "rmsnorm_device_limits": ([ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)],
                                      i32),
            "rmsnorm_kernel_info": ([i32, ctypes.POINTER(KernelInfo)], i32),
            "rmsnorm_get_device_status": ([ctypes.POINTER(ctypes.c_int)], i32),
            "rmsnorm_set_wait_limit_ns": ([u64], i32),
            "rmsnorm_set_pdl": ([i32], i32),
            "rmsnorm_get_pdl": ([], i32),
            "rmsnorm_test_staged_timeout": ([vp, vp, vp, i64, i64, i32, u64, vp], i32),
            "rmsnorm_test_grid_timeout": ([vp, vp, vp, i64, i64, i32, u64, vp], i32),
            "rmsnorm_fwd_staged_noalloc": ([vp, vp, vp, i64, i64, f32, i32, vp], i32),
            "rmsnorm_test_staged_noalloc_timeout": ([vp, vp, vp, i64, i64, i32, u64, vp], i32),
            "rmsnorm_noalloc_block_status": ([ctypes.POINTER(ctypes.c_int), i32], i32),
            "rmsnorm_status_string": ([i32], ctypes.c_char_p),
            "rmsnorm_version": ([], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(rc: int, where: str) -> None:
    if rc != OK:
        raise RmsnormError(rc, where)


# ------------------------------------------------------------------ C names

def rmsnorm_create() -> None:
    _check(_load().rmsnorm_create(), "rmsnorm_create")


def rmsnorm_destroy() -> None:
    _check(_load().rmsnorm_destroy(), "rmsnorm_destroy")


def rmsnorm_fwd(x: int, weight: int, y: int, rows: int, hidden: int, eps: float, dtype: int,
                stream: int | None) -> None:
    """Raw call: device pointers as integers, stream as a cudaStream_t integer."""
    _check(_load().rmsnorm_fwd(x, weight, y, rows, hidden, eps, dtype, stream or None),
           "rmsnorm_fwd")


def rmsnorm_fwd_ex(x: int, weight: int, y: int, rows: int, hidden: int, eps: float, dtype: int,
                   stream: int | None, variant: int = VARIANT_AUTO,
                   plan: Plan | None = None) -> Plan | None:
    ref = ctypes.byref(plan) if plan is not None else None
    _check(_load().rmsnorm_fwd_ex(x, weight, y, rows, hidden, eps, dtype, stream or None,
                                  variant, ref), "rmsnorm_fwd_ex")
    return plan


def rmsnorm_fwd_host(x_host: int, weight: int, y_host: int, rows: int, hidden: int, eps: float,
                     dtype: int, workspace: int, workspace_bytes: int, chunk_rows: int,
                     stream: int | None) -> None:
    """Host-buffer call: host x/y (pinned for overlap), device weight and
    workspace, chunked upload / kernel / download pipeline."""
    _check(_load().rmsnorm_fwd_host(x_host, weight, y_host, rows, hidden, eps, dtype, workspace,
                                    workspace_bytes, chunk_rows, stream or None),
           "rmsnorm_fwd_host")


def rmsnorm_qk_norm(q: int, k: int, q_weight: int, k_weight: int, tokens: int, q_heads: int,
                    k_heads: int, head_dim: int, q_token_stride: int, k_token_stride: int,
                    weight_bias: float, eps: float, dtype: int, stream: int | None) -> None:
    """Per-head QK norm in place (device pointers as integers)."""
    _check(_load().rmsnorm_qk_norm(q or None, k or None, q_weight or None, k_weight or None,
                                   tokens, q_heads, k_heads, head_dim, q_token_stride,
                                   k_token_stride, weight_bias, eps, dtype, stream or None),
           "rmsnorm_qk_norm")


def rmsnorm_qk_norm_ex(q: int, k: int, q_weight: int, k_weight: int, tokens: int, q_heads: int,
                       k_heads: int, head_dim: int, q_token_stride: int, k_token_stride: int,
                       weight_bias: float, eps: float, dtype: int, stream: int | None,
                       plan: QkPlan | None = None) -> QkPlan | None:
    _check(_load().rmsnorm_qk_norm_ex(q or None, k or None, q_weight or None, k_weight or None,
                                      tokens, q_heads, k_heads, head_dim, q_token_stride,
                                      k_token_stride, weight_bias, eps, dtype, stream or None,
                                      ctypes.byref(plan) if plan is not None else None),
           "rmsnorm_qk_norm_ex")
    return plan


def qk_norm(q, k, q_weight, k_weight, head_dim: int, eps: float, weight_bias: float = 0.0,
            stream=None) -> None:
    """In-place per-head norm of PyTorch CUDA tensors q [..., q_heads * head_dim]
    and k [..., k_heads * head_dim] (the last dimension holds a token's heads;
    the token dimension may be strided, e.g. views into a fused QKV tensor)."""
    import torch
    for t in (q, k):
        if not t.is_cuda or t.stride(-1) != 1:
            raise ValueError("q and k must be CUDA tensors with a contiguous last dimension")
    tokens = q.numel() // q.shape[-1]
    if k.numel() // k.shape[-1] != tokens:
        raise ValueError("q and k must hold the same number of tokens")
    qs = q.stride(-2) if q.dim() > 1 else q.shape[-1]
    ks = k.stride(-2) if k.dim() > 1 else k.shape[-1]
    ensure_context(q.device.index)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device.index):
        rmsnorm_qk_norm(q.data_ptr(), k.data_ptr(), q_weight.data_ptr(), k_weight.data_ptr(),
                        tokens, q.shape[-1] // head_dim, k.shape[-1] // head_dim, head_dim, qs, ks,
                        float(weight_bias), float(eps), torch_dtype_code(q.dtype), s.cuda_stream)


def rmsnorm_fwd_bias(x: int, weight: int, y: int, rows: int, hidden: int, weight_bias: float,
                     eps: float, dtype: int, stream: int | None) -> None:
    _check(_load().rmsnorm_fwd_bias(x, weight, y, rows, hidden, weight_bias, eps, dtype,
                                    stream or None), "rmsnorm_fwd_bias")


def rmsnorm_fwd_mxfp8(x: int, weight: int, q: int, scales: int, rows: int, hidden: int,
                      weight_bias: float, eps: float, dtype: int, stream: int | None) -> None:
    _check(_load().rmsnorm_fwd_mxfp8(x, weight, q, scales, rows, hidden, weight_bias, eps, dtype,
                                     stream or None), "rmsnorm_fwd_mxfp8")


def rmsnorm_fwd_mxfp4(x: int, weight: int, q: int, scales: int, rows: int, hidden: int,
                      weight_bias: float, eps: float, dtype: int, stream: int | None) -> None:
    _check(_load().rmsnorm_fwd_mxfp4(x, weight, q, scales, rows, hidden, weight_bias, eps, dtype,
                                     stream or None), "rmsnorm_fwd_mxfp4")


def rmsnorm_fwd_nvfp4(x: int, weight: int, q: int, scales: int, rows: int, hidden: int,
                      global_scale: float, weight_bias: float, eps: float, dtype: int,
                      stream: int | None) -> None:
    _check(_load().rmsnorm_fwd_nvfp4(x, weight, q, scales, rows, hidden, global_scale,
                                     weight_bias, eps, dtype, stream or None), "rmsnorm_fwd_nvfp4")


def rmsnorm_fwd_epilogue_ex(x: int, weight: int, y: int, scales: int | None, rows: int,
                            hidden: int, epilogue: int, weight_bias: float, eps: float,
                            dtype: int, stream: int | None, variant: int = VARIANT_AUTO,
                            plan: Plan | None = None, global_scale: float = 1.0) -> None:
    _check(_load().rmsnorm_fwd_epilogue_ex(x, weight, y, scales or None, rows, hidden, epilogue,
                                           weight_bias, global_scale, eps, dtype, stream or None,
                                           variant,
                                           ctypes.byref(plan) if plan is not None else None),
           "rmsnorm_fwd_epilogue_ex")


def rmsnorm_plan_epilogue_status(x: int, weight: int, y: int, rows: int, hidden: int, dtype: int,
                                 epilogue: int, sm_count: int, smem_optin: int,
                                 variant: int = VARIANT_AUTO):
    """(status, plan) of the selector for an epilogue, without raising."""
    p = Plan()
    rc = _load().rmsnorm_plan_epilogue(x, weight, y, rows, hidden, dtype, epilogue, sm_count,
                                       smem_optin, variant, ctypes.byref(p))
    return rc, p


def rmsnorm_validate_plan_epilogue(plan: Plan, x: int, weight: int, y: int, rows: int,
                                   hidden: int, dtype: int, epilogue: int, sm_count: int,
                                   smem_optin: int) -> int:
    return _load().rmsnorm_validate_plan_epilogue(ctypes.byref(plan), x, weight, y, rows, hidden,
                                                  dtype, epilogue, sm_count, smem_optin)


def rmsnorm_plan(x: int, weight: int, y: int, rows: int, hidden: int, dtype: int, sm_count: int,
                 smem_optin: int, variant: int = VARIANT_AUTO) -> Plan:
    p = Plan()
    _check(_load().rmsnorm_plan(x, weight, y, rows, hidden, dtype, sm_count, smem_optin, variant,
                                ctypes.byref(p)), "rmsnorm_plan")
    return p


def rmsnorm_plan_status(x: int, weight: int, y: int, rows: int, hidden: int, dtype: int,
                        sm_count: int, smem_optin: int, variant: int = VARIANT_AUTO):
    """(status, plan) without raising."""
    p = Plan()
    rc = _load().rmsnorm_plan(x, weight, y, rows, hidden, dtype, sm_count, smem_optin, variant,
                              ctypes.byref(p))
    return rc, p


def rmsnorm_plan_host_mapped_status(x_host: int, weight: int, y_host: int, rows: int,
                                    hidden: int, dtype: int, sm_count: int, smem_optin: int):
    """(status, plan) of rmsnorm_fwd_host's page-locked path, without raising."""
    p = Plan()
    rc = _load().rmsnorm_plan_host_mapped(x_host, weight, y_host, rows, hidden, dtype, sm_count,
                                          smem_optin, ctypes.byref(p))
    return rc, p


def rmsnorm_device_limits() -> tuple[int, int]:
    """(SM count, opt-in shared memory per block) of the current device."""
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    _check(_load().rmsnorm_device_limits(ctypes.byref(a), ctypes.byref(b)),
           "rmsnorm_device_limits")
    return a.value, b.value


def rmsnorm_validate_plan(plan: Plan, x: int, weight: int, y: int, rows: int, hidden: int,
                          dtype: int, sm_count: int, smem_optin: int) -> int:
    """Status rmsnorm_fwd_ex would give this explicit plan (host only)."""
    return _load().rmsnorm_validate_plan(ctypes.byref(plan), x, weight, y, rows, hidden, dtype,
                                         sm_count, smem_optin)


def rmsnorm_kernel_count() -> int:
    return _load().rmsnorm_kernel_count()


def rmsnorm_kernel_info(index: int) -> KernelInfo:
    k = KernelInfo()
    _check(_load().rmsnorm_kernel_info(index, ctypes.byref(k)), "rmsnorm_kernel_info")
    return k


def kernels() -> list[dict]:
    """Every compiled instantiation, with its index."""
    return [dict(index=i, **rmsnorm_kernel_info(i).as_dict()) for i in range(rmsnorm_kernel_count())]


def rmsnorm_last_variant() -> int:
    return _load().rmsnorm_last_variant()


def rmsnorm_get_device_status() -> int:
    v = ctypes.c_int(0)
    _check(_load().rmsnorm_get_device_status(ctypes.byref(v)), "rmsnorm_get_device_status")
    return v.value


def rmsnorm_set_wait_limit_ns(limit_ns: int) -> None:
    _check(_load().rmsnorm_set_wait_limit_ns(limit_ns), "rmsnorm_set_wait_limit_ns")


def rmsnorm_set_pdl(enable: bool) -> None:
    _check(_load().rmsnorm_set_pdl(1 if enable else 0), "rmsnorm_set_pdl")


def rmsnorm_get_pdl() -> bool:
    return bool(_load().rmsnorm_get_pdl())


def rmsnorm_test_staged_timeout(x: int, weight: int, y: int, rows: int, hidden: int, dtype: int,
                                limit_ns: int, stream: int | None) -> None:
    _check(_load().rmsnorm_test_staged_timeout(x, weight, y, rows, hidden, dtype, limit_ns,
                                               stream or None), "rmsnorm_test_staged_timeout")


def rmsnorm_test_grid_timeout(x: int, weight: int, y: int, rows: int, hidden: int, dtype: int,
                              limit_ns: int, stream: int | None) -> None:
    _check(_load().rmsnorm_test_grid_timeout(x, weight, y, rows, hidden, dtype, limit_ns,
                                             stream or None), "rmsnorm_test_grid_timeout")


def rmsnorm_fwd_staged_noalloc(x: int, weight: int, y: int, rows: int, hidden: int, eps: float,
                               dtype: int, stream: int | None) -> None:
    """The allocation-free entry point (no context, no device allocation):
    device pointers as integers, stream as a cudaStream_t integer."""
    _check(_load().rmsnorm_fwd_staged_noalloc(x, weight, y, rows, hidden, eps, dtype,
                                              stream or None), "rmsnorm_fwd_staged_noalloc")


def rmsnorm_test_staged_noalloc_timeout(x: int, weight: int, y: int, rows: int, hidden: int,
                                        dtype: int, limit_ns: int, stream: int | None) -> None:
    _check(_load().rmsnorm_test_staged_noalloc_timeout(x, weight, y, rows, hidden, dtype,
                                                       limit_ns, stream or None),
           "rmsnorm_test_staged_noalloc_timeout")


def rmsnorm_noalloc_block_status(n: int) -> list[int]:
    """The first n words of the allocation-free entry point's static status
    array (one per block of its last launch)."""
    buf = (ctypes.c_int * max(n, 1))()
    _check(_load().rmsnorm_noalloc_block_status(buf, n), "rmsnorm_noalloc_block_status")
    return list(buf[:n])


def rmsnorm_status_string(status: int) -> str:
    return _load().rmsnorm_status_string(status).decode()


def rmsnorm_version() -> int:
    return _load().rmsnorm_version()


# ------------------------------------------------------------------ tensors

_created = set()


def ensure_context(device_index: int) -> None:
    """rmsnorm_create on `device_index` once per process."""
    if device_index in _created:
        return
    import torch
    with torch.cuda.device(device_index):
        rmsnorm_create()
    _created.add(device_index)


def torch_dtype_code(dt) -> int:
    import torch
    table = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}
    if dt not in table:
        raise TypeError(f"unsupported dtype {dt}")
    return table[dt]


def rms_norm(x, weight, eps: float, out=None, variant: int = VARIANT_AUTO, plan: Plan | None = None,
             stream=None):
    """y = x * rsqrt(mean(x^2, -1) + eps) * weight through rmsnorm_fwd_ex.

    ``x``: CUDA tensor [..., hidden], contiguous; ``weight``: [hidden], same
    dtype and device; ``out``: optional preallocated output (may be ``x``).
    Runs on ``stream`` (default: PyTorch's current stream)."""
    import torch
    if not (x.is_cuda and weight.is_cuda):
        raise ValueError("rms_norm takes CUDA tensors (there is no CPU path)")
    if x.dtype != weight.dtype:
        raise TypeError("x and weight must share a dtype")
    if not x.is_contiguous() or not weight.is_contiguous():
        raise ValueError("x and weight must be contiguous")
    hidden = x.shape[-1]
    if weight.numel() != hidden:
        raise ValueError("weight must have hidden elements")
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must match x (shape, dtype, contiguous)")
    ensure_context(x.device.index)
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    rows = x.numel() // hidden if hidden else 0
    with torch.cuda.device(x.device.index):
        rmsnorm_fwd_ex(x.data_ptr(), weight.data_ptr(), out.data_ptr(), rows, hidden, float(eps),
                       torch_dtype_code(x.dtype), s.cuda_stream, variant, plan)
    return out


def rms_norm_bias(x, weight, weight_bias: float, eps: float, out=None, variant: int = VARIANT_AUTO,
                  plan: Plan | None = None, stream=None):
    """y = x * rsqrt(mean(x^2, -1) + eps) * (weight + weight_bias) through
    rmsnorm_fwd_epilogue_ex (tensors as for ``rms_norm``)."""
    import torch
    _check_rows(x, weight)
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must match x (shape, dtype, contiguous)")
    ensure_context(x.device.index)
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    with torch.cuda.device(x.device.index):
        rmsnorm_fwd_epilogue_ex(x.data_ptr(), weight.data_ptr(), out.data_ptr(), None, rows, hidden,
                                EPI_BIAS, float(weight_bias), float(eps),
                                torch_dtype_code(x.dtype), s.cuda_stream, variant, plan, 1.0)
    return out


def rms_norm_quant(x, weight, eps: float, fmt: str = "mxfp8", weight_bias: float = -0.0,
                   global_scale: float = 1.0, out=None, scales=None,
                   variant: int = VARIANT_AUTO, plan: Plan | None = None, stream=None):
    """RMSNorm with a block-scaled output, fmt "mxfp8" | "mxfp4" | "nvfp4":
    (codes uint8 [..., hidden * bits / 8] -- E4M3 bytes, or two E2M1 codes per
    byte with the even element in the low nibble -- and scales uint8
    [..., hidden / block] -- E8M0 exponents, or E4M3 values for NVFP4, which
    stand for code * scale * global_scale)."""
    import torch
    _check_rows(x, weight)
    epi = EPI_CODES[fmt]
    block, bits = QUANT_FORMATS[epi]
    hidden = x.shape[-1]
    if hidden % block:
        raise ValueError(f"hidden must be a multiple of {block} for {fmt}")
    lead = tuple(x.shape[:-1])
    if out is None:
        out = torch.empty(lead + (hidden * bits // 8,), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(lead + (hidden // block,), dtype=torch.uint8, device=x.device)
    if out.dtype != torch.uint8 or out.numel() * 8 != x.numel() * bits or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous uint8 tensor of x.numel() * {bits} / 8 bytes")
    if scales.dtype != torch.uint8 or scales.numel() * block != x.numel() or \
            not scales.is_contiguous():
        raise ValueError(f"scales must be a contiguous uint8 tensor of x.numel() / {block} bytes")
    ensure_context(x.device.index)
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    rows = x.numel() // hidden if hidden else 0
    with torch.cuda.device(x.device.index):
        rmsnorm_fwd_epilogue_ex(x.data_ptr(), weight.data_ptr(), out.data_ptr(), scales.data_ptr(),
                                rows, hidden, epi, float(weight_bias), float(eps),
                                torch_dtype_code(x.dtype), s.cuda_stream, variant, plan,
                                float(global_scale))
    return out, scales


def rms_norm_mxfp8(x, weight, eps: float, weight_bias: float = -0.0, out=None, scales=None,
                   variant: int = VARIANT_AUTO, plan: Plan | None = None, stream=None):
    """RMSNorm with an MXFP8 output: (codes uint8 [..., hidden] holding E4M3
    bit patterns, scales uint8 [..., hidden / 32] holding E8M0 exponents)."""
    return rms_norm_quant(x, weight, eps, "mxfp8", weight_bias, 1.0, out, scales, variant, plan,
                          stream)


def _check_rows(x, weight):
    if not (x.is_cuda and weight.is_cuda):
        raise ValueError("CUDA tensors required (there is no CPU path)")
    if x.dtype != weight.dtype:
        raise TypeError("x and weight must share a dtype")
    if not x.is_contiguous() or not weight.is_contiguous():
        raise ValueError("x and weight must be contiguous")
    if weight.numel() != x.shape[-1]:
        raise ValueError("weight must have hidden elements")
