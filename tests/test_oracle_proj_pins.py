"""Pins of the oracle's q/w projection (CPU only): exact bf16 widening, a
brute-force loop on tiny shapes, one-hot inputs that select a weight column,
and the head/dim layout of q (feature h * 64 + e).  A transposed weight or a
swapped head/dim reshape must fail one of them."""
import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I


def _bits(rng, shape, scale=1.0):
    return I.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def test_brute_force_small(oracle):
    rng = np.random.default_rng(0)
    B, d = 3, 64
    x, wq, ww = _bits(rng, (B, d)), _bits(rng, (2048, d)), _bits(rng, (32, d))
    q, w = oracle.qw_proj(x, wq, ww)
    xf, wqf, wwf = (I.bf16_bits_to_f32(a).astype(np.float64) for a in (x, wq, ww))
    for b in range(B):
        for h in (0, 5, 31):
            for e in (0, 17, 63):
                ref = sum(xf[b, t] * wqf[h * 64 + e, t] for t in range(d))
                assert abs(q[b, h, e] - ref) <= 1e-12 * max(1.0, abs(ref))
            assert abs(w[b, h] - sum(xf[b, t] * wwf[h, t] for t in range(d))) <= 1e-12 * max(1.0, abs(w[b, h]))


def test_one_hot_hidden_state_selects_a_weight_column(oracle):
    rng = np.random.default_rng(1)
    d = 128
    x = np.zeros((2, d), dtype=np.uint16)
    x[0, 7] = I.f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    x[1, 100] = I.f32_to_bf16_bits(np.array([-2.0], np.float32))[0]
    wq, ww = _bits(rng, (2048, d)), _bits(rng, (32, d))
    q, w = oracle.qw_proj(x, wq, ww)
    wqf, wwf = I.bf16_bits_to_f32(wq).astype(np.float64), I.bf16_bits_to_f32(ww).astype(np.float64)
    np.testing.assert_array_equal(q[0].reshape(-1), wqf[:, 7])
    np.testing.assert_array_equal(q[1].reshape(-1), -2.0 * wqf[:, 100])
    np.testing.assert_array_equal(w[0], wwf[:, 7])
    np.testing.assert_array_equal(w[1], -2.0 * wwf[:, 100])


def test_head_dim_layout(oracle):
    """Weight row h * 64 + e feeds q[:, h, e]: a row of ones at feature 2 * 64 + 3 lands at head 2, dim 3."""
    d = 64
    x = I.f32_to_bf16_bits(np.arange(1, d + 1, dtype=np.float32)[None, :] / 64.0)
    wq = np.zeros((2048, d), dtype=np.uint16)
    wq[2 * 64 + 3] = I.f32_to_bf16_bits(np.ones(d, np.float32))
    q, _ = oracle.qw_proj(x, wq, np.zeros((32, d), np.uint16))
    expect = np.zeros((1, 32, 64))
    expect[0, 2, 3] = np.sum(I.bf16_bits_to_f32(x).astype(np.float64))
    np.testing.assert_array_equal(q, expect)


@pytest.mark.parametrize("slip", ["transpose", "reshape"])
def test_planted_slips_fail_a_pin(oracle, monkeypatch, slip):
    from oracle import oracle as o
    real = o.qw_proj

    def bad(x_bits, wq_bits, ww_bits):
        q, w = real(x_bits, wq_bits, ww_bits)
        if slip == "transpose":  # head and dim axes swapped
            return q.reshape(q.shape[0], 64, 32).transpose(0, 2, 1), w
        return q.reshape(q.shape[0], -1).reshape(q.shape[0], 64, 32).reshape(q.shape[0], 32, 64)[:, ::-1], w
    monkeypatch.setattr(o, "qw_proj", bad)
    with pytest.raises(AssertionError):
        test_head_dim_layout(o)
