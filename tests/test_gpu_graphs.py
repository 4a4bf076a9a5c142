"""Calls captured into CUDA graphs and replayed (the way decode loops run
them), and calls from several host threads on their own streams at once:
every body, including the cluster split and the grid barrier variant with
the context's scratch (allocated once at create), against the oracle."""
import threading

import pytest

import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import compare, compare_quant, from_device, sample_rows, to_device

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


# (rows, hidden, dtype): warp, block, persistent, staged, looped, cluster and grid bodies
SHAPES = [(64, 128, "f32"), (8192, 1024, "bf16"), (8, 4096, "bf16"), (1024, 20480, "bf16"),
          (64, 131072, "f16"), (8, 65536, "bf16"), (2, 1 << 20, "bf16"), (300, 4097, "bf16")]


@pytest.mark.parametrize("rows,hidden,dtype", SHAPES)
def test_graph_capture_and_replay(rows, hidden, dtype):
    x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=rows + hidden)
    x, w = to_device(x_np, dtype), to_device(w_np, dtype)
    y = torch.zeros_like(x)
    s = torch.cuda.Stream()
    rn.rms_norm(x, w, 1e-6, out=y, stream=s)   # plan and first call outside the capture
    torch.cuda.synchronize()
    y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            rn.rms_norm(x, w, 1e-6, out=y, stream=s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    idx = sample_rows(rows, 64, seed=rows) if rows * hidden > (1 << 22) else None
    compare(from_device(y, dtype), x_np, w_np, 1e-6, dtype, rows_idx=idx)


def test_graph_capture_block_scaled_and_qk():
    x_np, w_np = inputs.random_case(512, 4096, "bf16", seed=1)
    x, w = to_device(x_np, "bf16"), to_device(w_np, "bf16")
    q = torch.zeros(512, 2048, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(512, 256, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    rn.rms_norm_quant(x, w, 1e-6, "nvfp4", 0.0, 0.01, out=q, scales=sc, stream=s)
    torch.cuda.synchronize()
    q.zero_(), sc.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rn.rms_norm_quant(x, w, 1e-6, "nvfp4", 0.0, 0.01, out=q, scales=sc, stream=s)
    g.replay()
    torch.cuda.synchronize()
    compare_quant(q.cpu().numpy(), sc.cpu().numpy(), x_np, w_np, 0.0, 1e-6, "bf16", "nvfp4", 0.01)


def test_concurrent_host_threads_on_own_streams():
    cases = [(rows, hidden, dtype, seed) for seed, (rows, hidden, dtype) in enumerate(SHAPES)]
    data = []
    for rows, hidden, dtype, seed in cases:
        x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=100 + seed)
        data.append((x_np, w_np, to_device(x_np, dtype), to_device(w_np, dtype)))
    outs = [None] * len(cases)
    errors = []

    def work(i):
        try:
            rows, hidden, dtype, _ = cases[i]
            _, _, x, w = data[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                y = torch.empty_like(x)
                for _ in range(5):
                    rn.rms_norm(x, w, 1e-6, out=y, stream=s)
            s.synchronize()
            outs[i] = y
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for i, (rows, hidden, dtype, _) in enumerate(cases):
        x_np, w_np, _, _ = data[i]
        idx = sample_rows(rows, 32, seed=i) if rows * hidden > (1 << 22) else None
        compare(from_device(outs[i], dtype), x_np, w_np, 1e-6, dtype, rows_idx=idx)
