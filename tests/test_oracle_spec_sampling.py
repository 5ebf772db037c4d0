"""Pins for the oracle's speculative sampling with sampled drafts (CPU only).

The pages name self-speculative decoding ("ntransformer - moteur d'inférence
NVMe-to-GPU…", "Fonctionnalités principales") and a sampler ("Architecture et
structure du code": inference/); the acceptance rule for sampled drafts is the
published speculative sampling rule (Leviathan, Kalman & Matias 2023, section
2.3).  Each check ties the oracle to something other than itself: the
theorem that the output follows the target distribution, the closed-form
acceptance threshold min(1, p/q), exact big-integer arithmetic in Python, and
the special cases q == p (always accept) and disjoint supports (the residual
is the target itself)."""
from fractions import Fraction

import numpy as np
import pytest

import oracle

Z_DRAFT = np.array([1.5, 0.2, -0.4, 0.9, -2.0, 0.0], dtype=np.float32)
Z_TARGET = np.array([0.1, 1.1, 0.3, -0.2, 0.6, -1.0], dtype=np.float32)


def _dist(w):
    w = np.asarray(w, dtype=np.float64)
    return w / w.sum()


@pytest.mark.parametrize("T,P", [(1.0, 1.0), (0.8, 0.85), (1.7, 0.6)])
def test_weights_are_the_nucleus_softmax(T, P):
    """w / W is softmax(z / T) restricted to the nucleus and renormalised, and
    the sampler's pick is the inverse CDF of those weights."""
    rng = np.random.default_rng(5)
    z = (rng.standard_normal(300) * 2).astype(np.float32)
    w, W = oracle.sample_weights(z, T, P)
    assert W == int(w.astype(object).sum())
    soft = np.exp((z.astype(np.float64) - z.max()) / T)
    soft /= soft.sum()
    order = np.argsort(-z, kind="stable")
    keep = order[:np.searchsorted(np.cumsum(soft[order]), P - 1e-12) + 1]
    assert set(np.flatnonzero(w)) == set(keep.tolist())
    ref = np.zeros_like(soft)
    ref[keep] = soft[keep] / soft[keep].sum()
    assert np.allclose(_dist(w), ref, rtol=1e-9, atol=1e-12)
    cum = np.cumsum(w.astype(object))
    for u in (0.0, 0.25, 0.5, 0.999):
        r = int(np.floor(u * float(W)))
        assert oracle.sample(z, T, P, u)[0] == int(np.argmax(cum > r))


@pytest.mark.parametrize("wq_d,Wq,wp_d,Wp", [(2, 4, 1, 4), (7, 10, 3, 10), (5, 9, 2, 13),
                                             (2**40, 3 * 2**40 + 17, 2**39 + 5, 2**56 + 3)])
def test_accept_threshold_is_p_over_q(wq_d, Wq, wp_d, Wp):
    """Accept exactly when k / 2^24 < p(d) / q(d): probed at and around the
    threshold k* = ceil(2^24 p / q)."""
    ratio = Fraction(wp_d, Wp) / Fraction(wq_d, Wq)
    assert ratio < 1
    kstar = -((-ratio.numerator * 2**24) // ratio.denominator)   # ceil(2^24 * ratio)
    for k in (0, kstar - 2, kstar - 1, kstar, kstar + 1, 2**24 - 1):
        if 0 <= k < 2**24:
            assert oracle.spec_accept(wq_d, Wq, wp_d, Wp, k) == (Fraction(k, 2**24) < ratio), k


def test_accept_limits():
    assert all(oracle.spec_accept(3, 10, 3, 10, k) for k in (0, 2**23, 2**24 - 1))      # p == q
    assert all(oracle.spec_accept(3, 10, 5, 10, k) for k in (0, 2**24 - 1))             # p > q
    assert not any(oracle.spec_accept(3, 10, 0, 10, k) for k in (0, 1, 2**24 - 1))      # p(d) = 0


@pytest.mark.parametrize("k_res", [0, 1, 2**23, 12345678, 2**24 - 1])
def test_residual_exact_big_integers(k_res):
    """8192 tokens with weights near 2^40: the residual sums reach ~2^105, so
    a product that lost its top bits would pick another token.  Python's
    exact integers give the expected pick."""
    rng = np.random.default_rng(k_res)
    n = 8192
    wp = rng.integers(2**39, 2**40, n, dtype=np.uint64)
    wq = rng.integers(2**39, 2**40, n, dtype=np.uint64)
    wp[rng.random(n) < 0.1] = 0
    Wp, Wq = int(wp.astype(object).sum()), int(wq.astype(object).sum())
    R = [max(0, int(a) * Wq - int(b) * Wp) for a, b in zip(wp, wq)]
    total = sum(R)
    assert total > 2**100
    r = k_res * total // 2**24
    acc, want = 0, -1
    for t, x in enumerate(R):
        acc += x
        if acc > r:
            want = t
            break
    assert oracle.spec_residual(wp, Wp, wq, Wq, k_res) == want


def test_residual_empty_when_equal():
    w = np.array([5, 0, 7, 1], dtype=np.uint64)
    assert oracle.spec_residual(w, 13, w, 13, 100) == -1


def test_residual_frequencies():
    """Over many uniforms the residual follows max(0, p - q) renormalised."""
    wq, Wq = oracle.sample_weights(Z_DRAFT, 1.0, 1.0)
    wp, Wp = oracle.sample_weights(Z_TARGET, 1.0, 1.0)
    res = np.maximum(0.0, _dist(wp) - _dist(wq))
    res /= res.sum()
    n = 20000
    counts = np.zeros(len(res))
    for c in range(n):
        counts[oracle.spec_residual(wp, Wp, wq, Wq, oracle.spec_uniforms(3, c)[1])] += 1
    assert np.all(counts[res == 0] == 0)
    m = res > 0
    assert np.sum((counts[m] - n * res[m]) ** 2 / (n * res[m])) < 25.0


def test_uniform_pair():
    ka, kr = np.array([oracle.spec_uniforms(77, c) for c in range(4000)]).T
    assert ka.min() >= 0 and ka.max() < 2**24 and kr.min() >= 0 and kr.max() < 2**24
    assert abs(np.corrcoef(ka, kr)[0, 1]) < 0.06
    # the odd counters: disjoint from the sampler's uniform at the same counter
    assert sum(int(a) == int(oracle.sample_uniform(77, c) * 2**24) for c, a in enumerate(ka)) < 3
    grid = np.histogram2d(ka / 2**24, kr / 2**24, bins=4, range=[[0, 1], [0, 1]])[0]
    assert np.sum((grid - 250) ** 2 / 250) < 40.0   # 15 degrees of freedom


@pytest.mark.parametrize("T,P", [(1.0, 1.0), (0.8, 0.9)])
def test_output_follows_target_distribution(T, P):
    """The speculative sampling theorem: whatever the draft, the first token
    of a step is distributed as the target's sampler distribution p.  The
    draft's own distribution q is far from p here, so a wrong acceptance
    test or residual (max(0, q - p), no max, p and q swapped) fails."""
    wp, _ = oracle.sample_weights(Z_TARGET, T, P)
    wq, _ = oracle.sample_weights(Z_DRAFT, T, P)
    p, q = _dist(wp), _dist(wq)
    n = 20000
    counts = np.zeros(len(p))
    for c in range(n):
        toks, _ = oracle.spec_sample([Z_DRAFT], [Z_TARGET, Z_TARGET], T, P, seed=2024, pos=3 * c)
        counts[toks[0]] += 1
    m = p > 0
    assert np.all(counts[~m] == 0)
    chi2_p = np.sum((counts[m] - n * p[m]) ** 2 / (n * p[m]))
    assert chi2_p < 25.0
    mq = q > 0
    assert np.sum((counts[mq] - n * q[mq]) ** 2 / (n * q[mq])) > 500.0   # the test can tell p from q


def test_equal_draft_and_target_accepts_everything():
    """q == p: every draft is accepted and the step emits the drafts plus the
    sampler's pick from the last target row, i.e. exactly what sampled
    decoding of the target would emit with the same (seed, position)."""
    rng = np.random.default_rng(9)
    rows = (rng.standard_normal((5, 50)) * 2).astype(np.float32)
    for pos in range(0, 400, 7):
        toks, drafts = oracle.spec_sample(rows[:4], rows, 0.9, 0.95, seed=11, pos=pos)
        assert toks[:4] == drafts
        assert toks == [oracle.sample(rows[i], 0.9, 0.95, oracle.sample_uniform(11, pos + i))[0] for i in range(5)]


def test_disjoint_supports_draw_from_target():
    """Disjoint nuclei: p(d) = 0, so every draft is rejected and the residual
    is p itself — the pick equals the plain sampler's for u = k_res / 2^24."""
    zq = np.array([5.0, 5.0, -30, -30, -30, -30], dtype=np.float32)
    zp = np.array([-30, -30, 1.0, 0.0, 0.5, -0.3], dtype=np.float32)
    T, P = 1.0, 0.999
    wq, _ = oracle.sample_weights(zq, T, P)
    wp, _ = oracle.sample_weights(zp, T, P)
    assert not np.any((wq > 0) & (wp > 0))
    for pos in range(300):
        toks, drafts = oracle.spec_sample([zq, zq], [zp, zp, zp], T, P, seed=5, pos=pos)
        assert len(toks) == 1 and drafts[0] in (0, 1)
        k_res = oracle.spec_uniforms(5, pos)[1]
        assert toks[0] == oracle.sample(zp, T, P, k_res / 2**24)[0]
