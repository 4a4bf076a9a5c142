"""Failure detection on the GPU without a fault: the bounded waits of the
staged kernel (the row copies withheld, a flag nothing sets) and of the
grid variant's barrier (one block's arrival withheld).  Every wait runs out
after a short limit; the kernel must record RMSNORM_ERR_DEVICE_TIMEOUT in
the status word, leave y untouched, and leave the context usable."""
import pytest

import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import compare, from_device, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rn.ensure_context(0)


def test_staged_wait_timeout_is_reported_and_context_survives():
    dtype, rows, hidden = "bf16", 64, 4096
    x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=9)
    x = to_device(x_np, dtype)
    w = to_device(w_np, dtype)
    y = torch.full_like(x, 5.0)
    assert rn.rmsnorm_get_device_status() == rn.OK
    rn.rmsnorm_test_staged_timeout(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, hidden,
                                   rn.BF16, 20_000_000, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rn.rmsnorm_get_device_status() == rn.ERR_DEVICE_TIMEOUT
    assert rn.rmsnorm_get_device_status() == rn.OK  # read clears it
    assert (y == 5.0).all()
    # the context still works, on the same kernel
    out = rn.rms_norm(x, w, 1e-6, variant=rn.VARIANT_STAGED)
    torch.cuda.synchronize()
    compare(from_device(out, dtype), x_np, w_np, 1e-6, dtype)
    assert rn.rmsnorm_get_device_status() == rn.OK


def test_wait_limit_setting_round_trips():
    rn.rmsnorm_set_wait_limit_ns(50_000_000)
    wl = inputs.WORKLOADS["wide_bf16_65536x2880"].with_shape(2048)
    x_np, w_np = inputs.make_inputs(wl)
    x = to_device(x_np, wl.dtype)
    w = to_device(w_np, wl.dtype)
    out = rn.rms_norm(x, w, wl.eps, variant=rn.VARIANT_STAGED)
    torch.cuda.synchronize()
    rn.rmsnorm_set_wait_limit_ns(0)  # back to the default
    assert rn.rmsnorm_get_device_status() == rn.OK
    compare(from_device(out, wl.dtype), x_np, w_np, wl.eps, wl.dtype)


def test_grid_barrier_timeout_is_reported_and_context_survives():
    dtype, rows, hidden = "bf16", 3, 1 << 19   # 1 MiB rows: the grid variant's shapes
    x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=10)
    x = to_device(x_np, dtype)
    w = to_device(w_np, dtype)
    y = torch.full_like(x, 5.0)
    assert rn.rmsnorm_get_device_status() == rn.OK
    rn.rmsnorm_test_grid_timeout(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, hidden,
                                 rn.BF16, 20_000_000, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rn.rmsnorm_get_device_status() == rn.ERR_DEVICE_TIMEOUT
    assert rn.rmsnorm_get_device_status() == rn.OK
    assert (y == 5.0).all()
    # the context still works, on the same kernel, twice in a row (the
    # barrier counters start from zero again)
    for _ in range(2):
        out = rn.rms_norm(x, w, 1e-6, variant=rn.VARIANT_GRID)
        torch.cuda.synchronize()
        compare(from_device(out, dtype), x_np, w_np, 1e-6, dtype)
    assert rn.rmsnorm_get_device_status() == rn.OK
