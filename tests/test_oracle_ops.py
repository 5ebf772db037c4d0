"""Pins for the oracle's pointwise/attention ops (CPU only): invariants,
hand-worked values and special cases with a known answer."""
import math

import numpy as np
import pytest

import oracle


# --- RMSNorm --------------------------------------------------------------
def test_rmsnorm_unit_rms_and_gain():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(4096) * 1e4
    y = oracle.rmsnorm(x, np.ones(4096, np.float32), 0.0)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-12
    g = (1 + 0.1 * rng.standard_normal(4096)).astype(np.float32)
    yg = oracle.rmsnorm(x, g, 0.0)
    assert np.allclose(yg, y * g.astype(np.float64), rtol=1e-14)


def test_rmsnorm_scale_invariant_and_eps():
    x = np.array([3.0, 4.0])            # mean square 12.5
    y = oracle.rmsnorm(x, np.ones(2, np.float32), 0.0)
    assert np.allclose(y, x / math.sqrt(12.5))
    assert np.allclose(oracle.rmsnorm(7 * x, np.ones(2, np.float32), 0.0), y)
    # eps enters under the square root: mean square 12.5 + eps 12.5 -> divide by 5
    assert np.allclose(oracle.rmsnorm(x, np.ones(2, np.float32), 12.5), x / 5.0)


# --- RoPE -----------------------------------------------------------------
def test_rope_identity_at_pos0():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(4 * 128)
    assert np.array_equal(oracle.rope(v, 4, 128, 0, 500000.0), v)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(2 * 128)
    r = oracle.rope(v, 2, 128, 1234, 500000.0)
    n0 = np.hypot(v[0::2], v[1::2])
    n1 = np.hypot(r[0::2], r[1::2])
    assert np.allclose(n0, n1, rtol=1e-13)


def test_rope_hand_worked_angles():
    # head_dim 4, theta 10000: pair 0 turns by pos rad, pair 1 by pos * 10000^(-1/2) = pos/100 rad
    v = np.array([1.0, 0.0, 1.0, 0.0])
    r = oracle.rope(v, 1, 4, 100, 10000.0)
    assert np.allclose(r[:2], [math.cos(100.0), math.sin(100.0)], atol=1e-12)
    assert np.allclose(r[2:], [math.cos(1.0), math.sin(1.0)], atol=1e-12)
    # rotation direction: (0, 1) turned by 1 rad -> (-sin 1, cos 1)
    r2 = oracle.rope(np.array([0.0, 1.0]), 1, 2, 1, 10000.0)
    assert np.allclose(r2, [-math.sin(1.0), math.cos(1.0)], atol=1e-14)


def test_rope_relative_position_property():
    """<rope(q, m), rope(k, n)> depends only on m - n (the point of rotary embeddings)."""
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    a = oracle.rope(q, 1, 128, 50, 500000.0) @ oracle.rope(k, 1, 128, 20, 500000.0)
    b = oracle.rope(q, 1, 128, 1030, 500000.0) @ oracle.rope(k, 1, 128, 1000, 500000.0)
    assert abs(a - b) < 1e-9 * abs(a)


def test_rope_composes():
    rng = np.random.default_rng(5)
    v = rng.standard_normal(3 * 128)
    a = oracle.rope(oracle.rope(v, 3, 128, 17, 500000.0), 3, 128, 25, 500000.0)
    b = oracle.rope(v, 3, 128, 42, 500000.0)
    assert np.allclose(a, b, atol=1e-11)


# --- softmax / attention --------------------------------------------------
def test_softmax_sum_shift_and_value():
    rng = np.random.default_rng(6)
    s = rng.standard_normal(1000) * 50
    p = oracle.softmax(s)
    assert abs(p.sum() - 1.0) < 1e-12
    assert np.allclose(oracle.softmax(s + 1e4), p, rtol=1e-10)
    assert np.allclose(oracle.softmax([0.0, math.log(3.0)]), [0.25, 0.75])


def _kv(n_kvh, stride, hd, rng):
    K = rng.standard_normal((n_kvh, stride, hd)).astype(np.float16)
    V = rng.standard_normal((n_kvh, stride, hd)).astype(np.float16)
    return K, V


def test_attention_single_position_returns_v():
    rng = np.random.default_rng(7)
    K, V = _kv(2, 8, 128, rng)
    q = rng.standard_normal(4 * 128) * 30
    o = oracle.attn_decode(q, K, V, 4, 2, 128, 1, 8).reshape(4, 128)
    for h in range(4):
        assert np.array_equal(o[h], V[h // 2, 0].astype(np.float64))


def test_attention_identical_keys_give_mean_v():
    rng = np.random.default_rng(8)
    K, V = _kv(1, 16, 128, rng)
    K[0, :] = K[0, 0]
    q = rng.standard_normal(128)
    o = oracle.attn_decode(q, K, V, 1, 1, 128, 11, 16)
    assert np.allclose(o, V[0, :11].astype(np.float64).mean(axis=0), atol=1e-12)


def test_attention_scale_and_gqa_mapping():
    hd = 128
    # two positions, scores differ by ln 3 after the 1/sqrt(128) scale -> weights 1/4, 3/4
    K = np.zeros((2, 4, hd), np.float16)
    V = np.zeros((2, 4, hd), np.float16)
    K[:, 1, 0] = 1.0
    for g in range(2):
        V[g, 0, :] = 10 * g + 1
        V[g, 1, :] = 10 * g + 5
    q = np.zeros((4, hd))
    q[:, 0] = math.log(3.0) * math.sqrt(hd)
    o = oracle.attn_decode(q.ravel(), K, V, 4, 2, hd, 2, 4).reshape(4, hd)
    for h in range(4):
        g = h // 2                                   # consecutive q heads share a KV head
        assert np.allclose(o[h], 0.25 * (10 * g + 1) + 0.75 * (10 * g + 5))


def test_attention_rejects_bad_args():
    K = np.zeros((2, 4, 128), np.float16)
    with pytest.raises(ValueError):
        oracle.attn_decode(np.zeros(3 * 128), K, K, 3, 2, 128, 2, 4)
    with pytest.raises(ValueError):
        oracle.attn_decode(np.zeros(4 * 128), K, K, 4, 2, 128, 5, 4)


# --- SwiGLU / argmax / cosine / skip --------------------------------------
def test_silu_values():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - 0.7310585786300049) < 1e-15       # 1 / (1 + e^-1)
    assert oracle.silu(1000.0) == 1000.0
    v = oracle.silu(-1000.0)
    assert v == 0.0 and not math.isnan(v)


def test_swiglu_elementwise():
    g = np.array([0.0, 1.0, -1.0, 2.0])
    u = np.array([5.0, 2.0, 3.0, -1.0])
    h = oracle.swiglu(g, u)
    assert np.allclose(h, [oracle.silu(x) * y for x, y in zip(g, u)], rtol=0, atol=0)
    assert h[0] == 0.0


def test_argmax_lowest_index_on_ties():
    assert oracle.argmax([1.0, 3.0, 2.0, 3.0]) == 1
    assert oracle.argmax([-5.0]) == 0
    assert oracle.argmax([7.0, 7.0, 7.0]) == 0


def test_cos_sim():
    rng = np.random.default_rng(9)
    a = rng.standard_normal(100)
    assert abs(oracle.cos_sim(a, a) - 1.0) < 1e-14
    assert abs(oracle.cos_sim(a, -3 * a) + 1.0) < 1e-14
    assert abs(oracle.cos_sim([1.0, 0.0], [0.0, 2.0])) == 0.0


def test_layer_skip_select():
    cos = [0.1, 0.9, 0.5, 0.9, 0.95, 0.2]
    assert list(oracle.layer_skip_select(cos, 3)) == [0, 1, 0, 1, 1, 0]
    assert list(oracle.layer_skip_select(cos, 0)) == [0] * 6
    assert list(oracle.layer_skip_select([0.3, 0.3, 0.3], 2)) == [1, 1, 0]
