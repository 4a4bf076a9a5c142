"""GPU parity of the per-head QK norm (rmsnorm_qk_norm) against the oracle:
head sizes 64..512 and unaligned ones, q-only / k-only, shared weights, weight
bias 0 and 1, contiguous q/k and views into a fused QKV buffer (V and
everything outside the heads untouched), 1..4000 tokens, three element
types."""
import numpy as np
import pytest

import oracle
import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import from_device, to_device

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


def rand(n, dtype, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return inputs.to_storage((rng.standard_normal(n) * scale).astype(np.float32), dtype)


def check_equal_within(gpu, ref, dtype):
    """Element-wise tolerance of the parity tests on flat arrays."""
    compare_flat = lambda a: a.reshape(1, -1)
    if dtype == "f32":
        g, r = gpu.astype(np.float64), ref.astype(np.float64)
        d = np.abs(g - r)
        assert np.all((d <= 1e-5) | (d <= 1e-5 * np.abs(r)))
    else:
        from _parity import monotone
        assert np.abs(monotone(gpu) - monotone(ref)).max(initial=0) <= 1


CASES = [
    # dtype, tokens, q_heads, k_heads, head_dim, bias, fused
    ("bf16", 1000, 8, 2, 128, 0.0, False),
    ("bf16", 1000, 8, 2, 128, 1.0, True),
    ("bf16", 7, 32, 8, 128, 0.0, True),
    ("bf16", 1, 64, 8, 128, 0.0, True),
    ("f16", 300, 16, 4, 64, 0.0, False),
    ("f16", 300, 16, 4, 256, 1.0, True),
    ("f32", 200, 4, 4, 128, 0.0, True),
    ("f32", 50, 2, 1, 512, 0.0, False),
    ("bf16", 100, 4, 0, 128, 0.0, False),     # q only
    ("bf16", 100, 0, 4, 64, 0.0, True),       # k only
    ("bf16", 64, 6, 2, 80, 0.0, True),        # 160-byte heads (vector body, idle lanes)
    ("bf16", 64, 6, 2, 72, 0.0, True),        # 144-byte heads: the scalar body
    ("f32", 33, 3, 3, 7, 0.5, False),         # tiny odd heads: scalar body
    ("bf16", 4000, 32, 8, 128, 0.0, True),
    ("bf16", 20, 4, 2, 1024, 0.0, False),     # longer than the vector bodies: scalar
]


@pytest.mark.parametrize("dtype,T,hq,hk,d,bias,fused", CASES)
def test_qk_norm_matches_oracle(dtype, T, hq, hk, d, bias, fused):
    if fused:  # [q | k | v] per token, v as wide as k
        width = (hq + 2 * hk) * d
        buf = rand(T * width, dtype, 1)
        q_off, k_off, qs, ks = 0, hq * d, width, width
        qh, kh = buf, buf
    else:
        qh = rand(T * hq * d, dtype, 2)
        kh = rand(T * hk * d, dtype, 3, scale=3.0)
        q_off = k_off = 0
        qs, ks = hq * d, hk * d
    qw = rand(d, dtype, 4)
    kw = rand(d, dtype, 5) if hq % 2 == 0 else qw  # sometimes one shared weight
    # oracle on host copies
    if fused:
        ref, _ = oracle.qk_norm(buf, np.zeros(1, buf.dtype), qw, kw, T, hq, 0, d, qs, 0, bias,
                                1e-6, dtype)
        _, ref_k = oracle.qk_norm(np.zeros(1, buf.dtype), ref[k_off:], qw, kw, T, 0, hk, d, 0,
                                  ks, bias, 1e-6, dtype)
        ref = np.concatenate([ref[:k_off], ref_k])
    else:
        ref_q, ref_k = oracle.qk_norm(qh, kh, qw, kw, T, hq, hk, d, qs, ks, bias, 1e-6, dtype)
    # device
    if fused:
        dbuf = to_device(buf, dtype)
        qp = dbuf.data_ptr()
        kp = qp + k_off * dbuf.element_size()
    else:
        dq, dk = to_device(qh, dtype), to_device(kh, dtype)
        qp, kp = dq.data_ptr(), dk.data_ptr()
    dqw, dkw = to_device(qw, dtype), to_device(kw, dtype)
    rn.rmsnorm_qk_norm(qp if hq else 0, kp if hk else 0, dqw.data_ptr(), dkw.data_ptr(), T, hq,
                       hk, d, qs, ks, bias, 1e-6, rn.DTYPE_CODES[dtype],
                       torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    if fused:
        got = from_device(dbuf, dtype)
        check_equal_within(got, ref, dtype)
        # everything outside the q and k heads (the v slot) is bit-identical
        v = got.reshape(T, -1)[:, (hq + hk) * d:]
        assert np.array_equal(v, buf.reshape(T, -1)[:, (hq + hk) * d:])
    else:
        check_equal_within(from_device(dq, dtype), ref_q, dtype)
        check_equal_within(from_device(dk, dtype), ref_k, dtype)


def test_qk_norm_tensor_helper_on_fused_views():
    T, hq, hk, d = 257, 16, 4, 128
    qkv = torch.randn(T, (hq + 2 * hk) * d, device="cuda").to(torch.bfloat16)
    before = qkv.clone()
    q = qkv[:, : hq * d]
    k = qkv[:, hq * d:(hq + hk) * d]
    qw = (1 + 0.1 * torch.randn(d, device="cuda")).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.randn(d, device="cuda")).to(torch.bfloat16)
    rn.qk_norm(q, k, qw, kw, d, 1e-6)
    torch.cuda.synchronize()
    host = before.cpu().view(torch.int16).numpy().view(np.uint16).ravel()
    width = (hq + 2 * hk) * d
    ref, _ = oracle.qk_norm(host, np.zeros(1, np.uint16),
                            qw.cpu().view(torch.int16).numpy().view(np.uint16),
                            kw.cpu().view(torch.int16).numpy().view(np.uint16), T, hq, 0, d, width,
                            0, 0.0, 1e-6, "bf16")
    got = qkv.cpu().view(torch.int16).numpy().view(np.uint16).reshape(T, width)
    check_equal_within(got[:, : hq * d].ravel(), ref.reshape(T, width)[:, : hq * d].ravel(),
                       "bf16")
    assert torch.equal(qkv[:, (hq + hk) * d:], before[:, (hq + hk) * d:])


@pytest.mark.parametrize("name", sorted(inputs.QK_WORKLOADS))
def test_qk_workloads_sampled_tokens(name):
    """The benchmark's QK workloads at full size (fused layout, the launch the
    benchmark times); 64 sampled tokens (first and last included) checked."""
    wl = inputs.QK_WORKLOADS[name]
    buf, qw, kw = inputs.make_qk_inputs(wl)
    d, hq, hk, T, width = wl.head_dim, wl.q_heads, wl.k_heads, wl.tokens, wl.width
    dbuf = to_device(buf, wl.dtype)
    es = dbuf.element_size()
    dqw, dkw = to_device(qw, wl.dtype), to_device(kw, wl.dtype)  # kept alive over the launch
    rn.rmsnorm_qk_norm(dbuf.data_ptr(), dbuf.data_ptr() + hq * d * es, dqw.data_ptr(),
                       dkw.data_ptr(), T, hq, hk, d, width, width, 0.0, wl.eps,
                       rn.DTYPE_CODES[wl.dtype], torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    got = from_device(dbuf, wl.dtype).reshape(T, width)
    rows = buf.reshape(T, width)
    rng = np.random.default_rng(wl.key)
    toks = np.unique(np.concatenate([[0, T - 1], rng.choice(T, size=min(T, 62), replace=False)]))
    for t in toks:
        tok = rows[t].copy()
        ref, _ = oracle.qk_norm(tok, np.zeros(1, tok.dtype), qw, kw, 1, hq, 0, d, width, 0, 0.0,
                                wl.eps, wl.dtype)
        _, ref_k = oracle.qk_norm(np.zeros(1, tok.dtype), ref[hq * d:], qw, kw, 1, 0, hk, d, 0,
                                  width - hq * d, 0.0, wl.eps, wl.dtype)
        ref = np.concatenate([ref[:hq * d], ref_k])
        check_equal_within(got[t], ref, wl.dtype)


def test_qk_norm_fused_buffer_beyond_4_gib():
    """A fused QKV buffer of more than 2^32 bytes (32 q + 8 k + 8 v heads of
    128 bf16 per token): tokens around and past the 4 GiB offset against the
    oracle, v untouched.  The tokens repeat a block of 64 seeded tokens
    (heads are independent), so the oracle runs on that block only."""
    dtype, hq, hk, d, blk = "bf16", 32, 8, 128, 64
    width = (hq + 2 * hk) * d
    T = (1 << 32) // (width * 2) + 40
    small = rand(blk * width, dtype, 11)
    qw, kw = rand(d, dtype, 12), rand(d, dtype, 13)
    ref, _ = oracle.qk_norm(small, np.zeros(1, small.dtype), qw, kw, blk, hq, 0, d, width, 0,
                            0.0, 1e-6, dtype)
    _, ref_k = oracle.qk_norm(np.zeros(1, small.dtype), ref[hq * d:], qw, kw, blk, 0, hk, d, 0,
                              width, 0.0, 1e-6, dtype)
    ref = np.concatenate([ref[:hq * d], ref_k]).reshape(blk, width)
    dbuf = to_device(small.reshape(blk, width), dtype).repeat(-(-T // blk), 1)[:T]
    dqw, dkw = to_device(qw, dtype), to_device(kw, dtype)
    qp = dbuf.data_ptr()
    kp = qp + hq * d * dbuf.element_size()
    rn.rmsnorm_qk_norm(qp, kp, dqw.data_ptr(), dkw.data_ptr(), T, hq, hk, d, width, width, 0.0,
                       1e-6, rn.DTYPE_CODES[dtype], torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    mark = (1 << 32) // (width * 2)
    idx = np.unique(np.concatenate([np.arange(0, 4), np.arange(mark - 4, mark + 4),
                                    np.arange(T - 8, T)]))
    got = from_device(dbuf.index_select(0, torch.from_numpy(idx).cuda()), dtype)
    want = ref[idx % blk]
    check_equal_within(got[:, :(hq + hk) * d].ravel(), want[:, :(hq + hk) * d].ravel(), dtype)
    assert np.array_equal(got[:, (hq + hk) * d:],
                          small.reshape(blk, width)[idx % blk][:, (hq + hk) * d:])


def _draw_qk(i):
    rng = np.random.default_rng(7000 + i)
    dtype = ["bf16", "f16", "f32"][rng.integers(3)]
    d = int(rng.choice([64, 128, 256, 512, 80, 96, 192])) if rng.random() < 0.7 else \
        int(rng.integers(1, 600))
    hq = int(rng.integers(0, 40))
    hk = int(rng.integers(0 if hq else 1, 12))
    T = int(np.exp(rng.uniform(0, np.log(max(2, min(3000, (1 << 21) // ((hq + 2 * hk) * d)))))))
    bias = float([0.0, 1.0, 0.5][rng.integers(3)])
    fused = hk > 0 and rng.random() < 0.6
    return dtype, T, hq, hk, d, bias, fused


@pytest.mark.parametrize("i", range(200))
def test_qk_norm_random_cases(i):
    """Seeded random head counts (q-only and k-only included), head sizes
    (the vector bodies' sizes and arbitrary ones for the scalar body), token
    counts, offsets, element types and layouts (separate q / k, or views into
    one fused [q | k | v] buffer), every token against the oracle."""
    test_qk_norm_matches_oracle(*_draw_qk(i))
