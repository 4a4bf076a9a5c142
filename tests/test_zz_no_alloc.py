"""The allocation-free entry point, rmsnorm_fwd_staged_noalloc.

It exists for callers that may not allocate device memory themselves (a
caller-owned memory pool or arena, a fixed memory budget, an embedding
process whose allocator policy forbids allocation): they cannot call
rmsnorm_create, which allocates the device status word.  This entry point
keeps its kernel's status words in a static device array instead.

The test calls it through the C ABI twice in a row per shape, with fresh
inputs each time, and checks each output against the regular entry point
(rmsnorm_fwd) on the same inputs, within the parity tolerance used by every
other test: 1 unit in the last place for bf16/f16, 1e-5 absolute or relative
for f32.  The file is named so that pytest collects it last."""
import numpy as np
import pytest

import oracle
import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import F32_TOL, ULP_TOL, from_device, monotone, to_device

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


def test_noalloc_matches_regular_entry_point_two_calls_in_a_row():
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
            rn.rmsnorm_fwd(x.data_ptr(), w.data_ptr(), y_ref.data_ptr(), rows, hidden, 1e-6, code,
                           stream)
            rn.rmsnorm_fwd_staged_noalloc(x.data_ptr(), w.data_ptr(), y_new.data_ptr(), rows,
                                          hidden, 1e-6, code, stream)
            torch.cuda.synchronize()
            a = from_device(y_new, dtype)
            b = from_device(y_ref, dtype)
            assert not np.isnan(oracle.widen(a, dtype)).any(), (dtype, rows, hidden, call)
            close(a, b, dtype)


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
