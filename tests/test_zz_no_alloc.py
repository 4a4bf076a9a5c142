"""The allocation-free entry point, rmsnorm_fwd_staged_noalloc.

It exists for callers that may not allocate device memory themselves (a
caller-owned memory pool or arena, a fixed memory budget, an embedding
process whose allocator policy forbids allocation): they cannot call
rmsnorm_create, which allocates the device status word and the grid
variant's scratch.  This entry point keeps its kernel's status words in a
static device array instead.

The tests call it through the C ABI, two calls in a row per shape with fresh
inputs each time, and check each output element by element against the fp64
oracle at the parity bar every other test uses (1 unit in the last place for
bf16/f16, 1e-5 absolute or relative for f32), and against the regular entry
point (rmsnorm_fwd) on the same inputs.  Its failure path is exercised
without a fault: the row copies withheld, a 1 ms limit on the bounded waits,
NaN rows and a DEVICE_TIMEOUT word per block, and a correct call right
after.  The file is named so that pytest collects it last."""
import numpy as np
import pytest

import oracle
import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import F32_TOL, ULP_TOL, compare, from_device, monotone, sample_rows, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CASES = [("bf16", 16384, 4096), ("f16", 4096, 7168), ("bf16", 777, 2880), ("f32", 300, 2048),
         ("bf16", 5, 24576)]


def close(a: np.ndarray, b: np.ndarray, dtype: str) -> None:
    if dtype == "f32":
        a64, b64 = a.astype(np.float64), b.astype(np.float64)
        d = np.abs(a64 - b64)
        assert np.all((d <= F32_TOL) | (d <= F32_TOL * np.abs(b64)))
    else:
        assert np.abs(monotone(a) - monotone(b)).max() <= ULP_TOL


def staged_grid(rows: int, hidden: int, dtype: str) -> int:
    """Blocks of the staged launch the entry point makes (the host-only
    selector, with the device limits a regular context reads)."""
    rn.ensure_context(0)
    sms, optin = rn.rmsnorm_device_limits()
    base = 1 << 30
    rc, p = rn.rmsnorm_plan_status(base, 3 * base, 5 * base, rows, hidden, rn.DTYPE_CODES[dtype],
                                   sms, optin, rn.VARIANT_STAGED)
    assert rc == rn.OK
    return p.grid


def test_noalloc_matches_oracle_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rn.ensure_context(0)  # for the regular entry point only
    stream = torch.cuda.current_stream().cuda_stream
    for dtype, rows, hidden in CASES:
        code = rn.DTYPE_CODES[dtype]
        for call in range(2):
            x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=10 + call)
            x = to_device(x_np, dtype)
            w = to_device(w_np, dtype)
            y_ref = torch.empty_like(x)
            y_new = torch.full_like(x, 7.0)
            rn.rmsnorm_fwd_staged_noalloc(x.data_ptr(), w.data_ptr(), y_new.data_ptr(), rows,
                                          hidden, 1e-6, code, stream)
            rn.rmsnorm_fwd(x.data_ptr(), w.data_ptr(), y_ref.data_ptr(), rows, hidden, 1e-6, code,
                           stream)
            torch.cuda.synchronize()
            a = from_device(y_new, dtype)
            assert not np.isnan(oracle.widen(a, dtype)).any(), (dtype, rows, hidden, call)
            idx = sample_rows(rows, 512, seed=call) if rows > 2048 else None
            compare(a, x_np, w_np, 1e-6, dtype, rows_idx=idx)       # the definition
            close(a, from_device(y_ref, dtype), dtype)             # the regular entry point
            assert rn.rmsnorm_noalloc_block_status(staged_grid(rows, hidden, dtype)) == \
                [0] * staged_grid(rows, hidden, dtype)


def test_noalloc_timeout_writes_nan_rows_and_block_words():
    """Copies withheld (nothing ever completes the slots' barriers) with a
    1 ms limit: every block gives up, records DEVICE_TIMEOUT in its word and
    writes its rows as NaN; the next call is correct and clears the words."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    stream = torch.cuda.current_stream().cuda_stream
    for dtype, rows, hidden in (("bf16", 300, 24576), ("f32", 64, 12288)):
        code = rn.DTYPE_CODES[dtype]
        grid = staged_grid(rows, hidden, dtype)
        x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=4)
        x, w = to_device(x_np, dtype), to_device(w_np, dtype)
        y = torch.zeros_like(x)
        rn.rmsnorm_test_staged_noalloc_timeout(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows,
                                               hidden, code, 1_000_000, stream)
        torch.cuda.synchronize()
        assert np.isnan(oracle.widen(from_device(y, dtype), dtype)).all()
        assert rn.rmsnorm_noalloc_block_status(grid) == [rn.ERR_DEVICE_TIMEOUT] * grid
        rn.rmsnorm_fwd_staged_noalloc(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, hidden,
                                      1e-6, code, stream)
        torch.cuda.synchronize()
        compare(from_device(y, dtype), x_np, w_np, 1e-6, dtype)
        assert rn.rmsnorm_noalloc_block_status(grid) == [0] * grid


def test_noalloc_rejects_misaligned_rows_and_pointers():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    stream = torch.cuda.current_stream().cuda_stream
    x = torch.zeros(4, 2881, dtype=torch.bfloat16, device="cuda")  # 5762-byte rows
    w = torch.ones(2881, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(rn.RmsnormError) as e:
        rn.rmsnorm_fwd_staged_noalloc(x.data_ptr(), w.data_ptr(), y.data_ptr(), 4, 2881, 1e-6,
                                      rn.BF16, stream)
    assert e.value.status == rn.ERR_MISALIGNED
    xb = torch.zeros(4 * 4096 + 1, dtype=torch.bfloat16, device="cuda")
    wb = torch.ones(4096, dtype=torch.bfloat16, device="cuda")
    yb = torch.empty(4 * 4096, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rn.RmsnormError) as e:  # x two bytes off a 16-byte boundary
        rn.rmsnorm_fwd_staged_noalloc(xb.data_ptr() + 2, wb.data_ptr(), yb.data_ptr(), 4, 4096,
                                      1e-6, rn.BF16, stream)
    assert e.value.status == rn.ERR_MISALIGNED


def test_noalloc_rejects_rows_beyond_its_scratch_and_shared_memory():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x = torch.empty(2, 1 << 17, dtype=torch.bfloat16, device="cuda")
    w = torch.empty(1 << 17, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(rn.RmsnormError) as e:  # a 256 KiB row cannot be staged
        rn.rmsnorm_fwd_staged_noalloc(x.data_ptr(), w.data_ptr(), y.data_ptr(), 2, 1 << 17, 1e-6,
                                      rn.BF16, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == rn.ERR_TOO_LARGE
