"""Programmatic dependent launch, tested as a feature.

"CuTeDSL at Perplexity", sections "Grid synchronization" and "Prefill and
decode specialization", name programmatic dependent launch as the way to
hide launch latency between dependent kernels.  Every kernel of the library
waits for the grid it depends on (griddepcontrol.wait) before its first
global access and then lets the next launch on the stream be scheduled
(griddepcontrol.launch_dependents), and its launches carry the
programmatic-stream-serialization attribute; so the next norm on a stream is
already resident while the previous one's last blocks run.  If a wait sat
after a read, that next norm would read x before the previous kernel had
finished writing it.

These tests chain launches that each read what the one before wrote, on one
stream: a PyTorch kernel writes x, then several in-place norms run back to
back (each reading the previous one's output), a PyTorch kernel rescales x
in the middle of the chain, and a block-scaled or weight-offset norm reads
the last output.  After every step a copy kernel takes a snapshot; each
step's output is compared with the oracle applied to that step's own input
(the previous snapshot), at the usual bar, with the attribute on and off.
The bodies covered: warp-per-row, block-per-row, persistent, staged,
looped, generic, cluster and grid.
"""
import numpy as np
import pytest

import oracle
import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import compare, compare_quant, from_device, monotone, sample_rows, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rn.ensure_context(0)
    was = rn.rmsnorm_get_pdl()
    yield
    rn.rmsnorm_set_pdl(was)
    torch.cuda.synchronize()
    assert rn.rmsnorm_get_device_status() == rn.OK


# (rows, hidden, dtype): the headline (many waves of blocks), warp, decode,
# staged, looped, generic, cluster and grid bodies
SHAPES = [(16384, 4096, "bf16"), (8192, 1024, "bf16"), (64, 128, "f32"), (32, 4096, "bf16"),
          (4000, 24576, "bf16"), (600, 40960, "f16"), (3000, 4097, "bf16"), (8, 65536, "bf16"),
          (2, 1 << 20, "bf16")]
STEPS = 4


def doubled(a: np.ndarray, dtype: str) -> np.ndarray:
    """2 * x in storage (exact: no element is near overflow)."""
    return inputs.to_storage((oracle.widen(a, dtype) * 2.0).astype(np.float32), dtype)


def check(got, x_in, w, eps, dtype, rows):
    idx = sample_rows(rows, 256, seed=rows) if rows > 4096 else None
    compare(got, x_in, w, eps, dtype, rows_idx=idx)


@pytest.mark.parametrize("pdl", [True, False])
@pytest.mark.parametrize("rows,hidden,dtype", SHAPES)
def test_dependent_chain_in_place(pdl, rows, hidden, dtype):
    rn.rmsnorm_set_pdl(pdl)
    x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=rows + hidden)
    src = to_device(x_np, dtype)
    w = to_device(w_np, dtype)
    x = torch.zeros_like(src)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    snaps = []
    with torch.cuda.stream(s):
        x.copy_(src)                                  # a PyTorch kernel writes x ...
        for k in range(STEPS):                        # ... and each norm reads the last write
            rn.rms_norm(x, w, 1e-6, out=x, stream=s)
            snaps.append(x.clone())
            if k == 1:
                x.mul_(2.0)                           # a PyTorch kernel in mid-chain
    s.synchronize()
    assert rn.rmsnorm_get_pdl() == pdl
    prev = x_np
    for k in range(STEPS):
        got = from_device(snaps[k], dtype)
        check(got, prev, w_np, 1e-6, dtype, rows)
        prev = doubled(got, dtype) if k == 1 else got


@pytest.mark.parametrize("pdl", [True, False])
def test_chain_into_epilogues_and_qk(pdl):
    """A plain norm writes x; a weight-offset norm, an NVFP4 norm and the
    per-head QK norm read it next, each launched right behind its writer."""
    rn.rmsnorm_set_pdl(pdl)
    rows, hidden, dtype = 8192, 4096, "bf16"
    x_np, w_np = inputs.random_case(rows, hidden, dtype, seed=77)
    x = to_device(x_np, dtype)
    w = to_device(w_np, dtype)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        rn.rms_norm(x, w, 1e-6, out=x, stream=s)
        snap1 = x.clone()
        y_bias = rn.rms_norm_bias(x, w, 0.5, 1e-6, stream=s)
        rn.rms_norm(x, w, 1e-6, out=x, stream=s)
        snap2 = x.clone()
        q, sc = rn.rms_norm_quant(x, w, 1e-6, "nvfp4", -0.0, 0.02, stream=s)
        # QK norm in place on views of x: 24 q heads and 8 k heads of 128 per row
        rn.qk_norm(x[:, : 24 * 128], x[:, 24 * 128:], w[:128], w[128:256], 128, 1e-6, stream=s)
    s.synchronize()
    a = from_device(snap1, dtype)
    check(a, x_np, w_np, 1e-6, dtype, rows)
    idx = sample_rows(rows, 256, seed=1)
    compare(from_device(y_bias, dtype), a, w_np, 1e-6, dtype, rows_idx=idx, bias=0.5)
    b = from_device(snap2, dtype)
    check(b, a, w_np, 1e-6, dtype, rows)
    compare_quant(q.cpu().numpy(), sc.cpu().numpy(), b, w_np, -0.0, 1e-6, dtype, "nvfp4", 0.02,
                  rows_idx=idx)
    got = from_device(x, dtype)[idx].reshape(-1)
    bb = b[idx].reshape(-1).copy()
    ref_q, _ = oracle.qk_norm(bb, np.zeros(1, bb.dtype), w_np[:128], w_np[128:256], len(idx),
                              24, 0, 128, hidden, 0, 0.0, 1e-6, dtype)
    _, ref_k = oracle.qk_norm(np.zeros(1, bb.dtype), ref_q[24 * 128:], w_np[:128],
                              w_np[128:256], len(idx), 0, 8, 128, 0, hidden, 0.0, 1e-6, dtype)
    ref = np.concatenate([ref_q[: 24 * 128], ref_k])
    assert np.abs(monotone(got) - monotone(ref)).max() <= 1
