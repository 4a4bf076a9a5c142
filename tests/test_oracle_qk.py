"""Pins for the oracle's per-head QK norm ("CuTeDSL at Perplexity", section
"QK Norm"): against the already-pinned row oracle on flattened heads, a
hand-worked head with WEIGHT_BIAS, weight bias folded into exactly
representable weights, strided heads inside a fused QKV buffer (V untouched),
q-only / k-only and zero tokens.  CPU only."""
import math

import numpy as np
import pytest

import oracle
from rmsnorm_fwd_gb300 import inputs


def rand(shape, dtype, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return inputs.to_storage((rng.standard_normal(shape) * scale).astype(np.float32), dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_contiguous_heads_equal_row_oracle(dtype):
    T, hq, hk, d = 5, 4, 2, 64
    q = rand((T * hq * d,), dtype, 1)
    k = rand((T * hk * d,), dtype, 2)
    qw = rand((d,), dtype, 3)
    kw = rand((d,), dtype, 4)
    qo, ko = oracle.qk_norm(q, k, qw, kw, T, hq, hk, d, hq * d, hk * d, 0.0, 1e-6, dtype)
    assert np.array_equal(qo.reshape(T * hq, d), oracle.rmsnorm(q.reshape(T * hq, d), qw, 1e-6,
                                                                 dtype))
    assert np.array_equal(ko.reshape(T * hk, d), oracle.rmsnorm(k.reshape(T * hk, d), kw, 1e-6,
                                                                 dtype))


def test_hand_worked_head_with_weight_bias():
    # head x = [3, 4], weight 0, WEIGHT_BIAS 1, eps 0 -> [3, 4] * sqrt(2) / 5
    q = np.array([3, 4, 30, 40], np.float32)  # two heads of 2; the second is 10x the first
    k = np.array([1, -1], np.float32)
    w = np.zeros(2, np.float32)
    qo, ko = oracle.qk_norm(q, k, w, w, 1, 2, 1, 2, 4, 2, 1.0, 0.0, "f32")
    r = math.sqrt(2) / 5
    assert qo == pytest.approx(np.float32([3 * r, 4 * r, 3 * r, 4 * r]), rel=1e-7)
    assert list(ko) == [1.0, -1.0]  # mean square 1 -> r = 1


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_weight_bias_equals_shifted_weight(dtype):
    T, hq, hk, d = 3, 2, 1, 128
    q = rand((T * hq * d,), dtype, 5)
    k = rand((T * hk * d,), dtype, 6)
    rng = np.random.default_rng(7)
    wf = (rng.integers(-4, 4, d) * 0.25).astype(np.float32)  # exact in bf16 and f16, and w + 1
    w = inputs.to_storage(wf, dtype)
    w1 = inputs.to_storage(wf + 1.0, dtype)
    qo, ko = oracle.qk_norm(q, k, w, w, T, hq, hk, d, hq * d, hk * d, 1.0, 1e-6, dtype)
    q1, k1 = oracle.qk_norm(q, k, w1, w1, T, hq, hk, d, hq * d, hk * d, 0.0, 1e-6, dtype)
    assert np.array_equal(qo, q1) and np.array_equal(ko, k1)


def test_strided_heads_in_a_fused_qkv_buffer():
    dtype, T, hq, hk, d = "bf16", 4, 3, 2, 64
    width = (hq + 2 * hk) * d  # [q | k | v] per token
    qkv = rand((T * width,), dtype, 8)
    qw = rand((d,), dtype, 9)
    kw = rand((d,), dtype, 10)
    q_view = qkv  # q starts at element 0 of each token
    k_off = hq * d
    qo, _ = oracle.qk_norm(q_view, np.zeros(1, np.uint16), qw, kw, T, hq, 0, d, width, 0, 0.0,
                           1e-6, dtype)
    _, ko = oracle.qk_norm(np.zeros(1, np.uint16), qkv[k_off:], qw, kw, T, 0, hk, d, 0, width,
                           0.0, 1e-6, dtype)
    rows = qkv.reshape(T, width)
    q_ref = oracle.rmsnorm(rows[:, :hq * d].reshape(T * hq, d).copy(), qw, 1e-6, dtype)
    k_ref = oracle.rmsnorm(rows[:, k_off:k_off + hk * d].reshape(T * hk, d).copy(), kw, 1e-6,
                           dtype)
    qo_rows = qo.reshape(T, width)
    assert np.array_equal(qo_rows[:, :hq * d].reshape(T * hq, d), q_ref)
    assert np.array_equal(qo_rows[:, hq * d:], rows[:, hq * d:])  # k and v untouched by q pass
    ko_rows = np.concatenate([qkv[:k_off], ko]).reshape(T, width)
    assert np.array_equal(ko_rows[:, k_off:k_off + hk * d].reshape(T * hk, d), k_ref)
    assert np.array_equal(ko_rows[:, k_off + hk * d:], rows[:, k_off + hk * d:])  # v untouched


def test_zero_tokens_and_bad_strides():
    q = rand((128,), "bf16", 11)
    w = rand((64,), "bf16", 12)
    qo, ko = oracle.qk_norm(q, q, w, w, 0, 2, 0, 64, 128, 0, 0.0, 1e-6, "bf16")
    assert np.array_equal(qo, q)
    with pytest.raises(ValueError):
        oracle.qk_norm(q, q, w, w, 1, 2, 0, 64, 64, 0, 0.0, 1e-6, "bf16")  # stride < heads * d
