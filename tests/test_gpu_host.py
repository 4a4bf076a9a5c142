"""rmsnorm_fwd_host: host x / y.  Pinned (device-mapped) buffers are read and
written by the kernel directly; pageable ones go through the chunked
upload / kernel / download pipeline over a caller-provided device workspace.
Checked against the oracle for both paths, chunk sizes that leave ragged
last chunks, one to three buffers, one pinned and one pageable buffer (the
pipeline), in place, and zero rows."""
import numpy as np
import pytest

import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import compare, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rn.ensure_context(0)
    yield
    torch.cuda.synchronize()
    assert rn.rmsnorm_get_device_status() == rn.OK


def host_tensor(a: np.ndarray, dtype: str, pinned: bool):
    t = torch.from_numpy(np.ascontiguousarray(a).copy())
    if dtype != "f32":
        t = t.view(torch.int16).view(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.pin_memory() if pinned else t


def to_numpy(t, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype,rows,hidden,chunk,ws_rows,pinned", [
    ("bf16", 1000, 4096, 0, 300, True),     # default chunking, three buffers
    ("bf16", 1000, 4096, 7, 3, True),       # ragged chunks, one row per buffer
    ("f16", 513, 2880, 64, 200, True),
    ("f32", 77, 1000, 10, 20, True),        # two buffers
    ("bf16", 50, 7168, 16, 1, True),        # a single buffer of one row
    ("bf16", 333, 1025, 0, 50, True),       # ragged hidden (scalar kernel)
    ("bf16", 200, 4096, 32, 100, False),    # pageable host memory
    ("f16", 1000, 5120, 0, 100, False),
    ("bf16", 77, 1025, 8, 10, False),       # pageable, ragged hidden
])
def test_host_pipeline_matches_oracle(dtype, rows, hidden, chunk, ws_rows, pinned):
    es = 4 if dtype == "f32" else 2
    x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=rows)
    xh = host_tensor(x_np, dtype, pinned)
    yh = host_tensor(np.zeros_like(x_np), dtype, pinned)
    w = to_device(w_np, dtype)
    ws_bytes = ws_rows * hidden * es + 1024
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    rn.rmsnorm_fwd_host(xh.data_ptr(), w.data_ptr(), yh.data_ptr(), rows, hidden, 1e-6,
                        rn.DTYPE_CODES[dtype], ws.data_ptr(), ws_bytes, chunk, s.cuda_stream)
    s.synchronize()
    compare(to_numpy(yh, dtype), x_np, w_np, 1e-6, dtype)


def test_host_mixed_pinned_and_pageable_uses_the_pipeline():
    dtype, rows, hidden = "bf16", 300, 2880
    x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=3)
    xh = host_tensor(x_np, dtype, True)
    yh = host_tensor(np.zeros_like(x_np), dtype, False)
    w = to_device(w_np, dtype)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    rn.rmsnorm_fwd_host(xh.data_ptr(), w.data_ptr(), yh.data_ptr(), rows, hidden, 1e-6, rn.BF16,
                        ws.data_ptr(), 1 << 20, 16, s.cuda_stream)
    s.synchronize()
    compare(to_numpy(yh, dtype), x_np, w_np, 1e-6, dtype)


def test_host_pipeline_in_place_and_repeated():
    dtype, rows, hidden = "bf16", 600, 4096
    x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=1)
    w = to_device(w_np, dtype)
    ws_bytes = 64 << 20
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    for pinned in (True, False, False):  # direct, then the pipeline twice (reused streams)
        xh = host_tensor(x_np, dtype, pinned)
        rn.rmsnorm_fwd_host(xh.data_ptr(), w.data_ptr(), xh.data_ptr(), rows, hidden, 1e-6,
                            rn.BF16, ws.data_ptr(), ws_bytes, 0, s.cuda_stream)
        s.synchronize()
        compare(to_numpy(xh, dtype), x_np, w_np, 1e-6, dtype)


def test_host_pipeline_rejects_small_workspace_and_handles_zero_rows():
    w = torch.ones(4096, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    xh = torch.zeros(4, 4096, dtype=torch.bfloat16)  # pageable: needs the workspace
    with pytest.raises(rn.RmsnormError) as e:
        rn.rmsnorm_fwd_host(xh.data_ptr(), w.data_ptr(), xh.data_ptr(), 4, 4096, 1e-6, rn.BF16,
                            ws.data_ptr(), 1024, 0, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == rn.ERR_INVALID_ARG
    rn.rmsnorm_fwd_host(xh.data_ptr(), w.data_ptr(), xh.data_ptr(), 0, 4096, 1e-6, rn.BF16,
                        ws.data_ptr(), 1024, 0, torch.cuda.current_stream().cuda_stream)


def test_host_mapped_path_launches_the_host_link_plan():
    """Page-locked buffers: the kernel runs the plan rmsnorm_plan_host_mapped
    gives (a persistent grid of two blocks per SM for many rows)."""
    dtype, rows, hidden = "bf16", 4096, 4096
    x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=21)
    xh = host_tensor(x_np, dtype, True)
    yh = host_tensor(np.zeros_like(x_np), dtype, True)
    w = to_device(w_np, dtype)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    sms, optin = rn.rmsnorm_device_limits()
    rc, p = rn.rmsnorm_plan_host_mapped_status(xh.data_ptr(), w.data_ptr(), yh.data_ptr(), rows,
                                               hidden, rn.BF16, sms, optin)
    assert rc == rn.OK and p.variant == rn.VARIANT_PERSISTENT and p.grid == 2 * sms
    rn.rmsnorm_fwd_host(xh.data_ptr(), w.data_ptr(), yh.data_ptr(), rows, hidden, 1e-6, rn.BF16,
                        ws.data_ptr(), 1 << 20, 0, s.cuda_stream)
    s.synchronize()
    assert rn.rmsnorm_last_variant() == rn.VARIANT_PERSISTENT
    compare(to_numpy(yh, dtype), x_np, w_np, 1e-6, dtype)
