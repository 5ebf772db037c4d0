"""Pins for the oracle's non-greedy sampler (temperature + nucleus / top-p;
"ntransformer - moteur d'inférence NVMe-to-GPU…", "Architecture et structure
du code": inference/ sampler) and its counter-based uniform (CPU only).

Each check ties the sampler to something other than itself: the published
SplitMix64 output sequence, a distribution worked by hand, the reduction to
greedy decoding, a frequency test against softmax, tie order, and the
temperature identity softmax(z / T)."""
import numpy as np
import pytest

import oracle

GOLDEN = 0x9E3779B97F4A7C15


def test_splitmix64_published_sequence():
    # the first outputs of SplitMix64 started from state 0 (Steele, Lea & Flood 2014)
    outs = [oracle.splitmix64((k * GOLDEN) & (2**64 - 1)) for k in range(3)]
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_uniform_is_24_bit_grid_in_unit_interval():
    us = [oracle.sample_uniform(1234, c) for c in range(2000)]
    assert all(0.0 <= u < 1.0 for u in us)
    assert all(float(u * 2**24).is_integer() for u in us)
    assert abs(np.mean(us) - 0.5) < 4 * (1 / np.sqrt(12)) / np.sqrt(len(us))


def test_hand_worked_nucleus():
    """z = [2, 1, 0, -1], T = 1: p = [0.644, 0.237, 0.087, 0.032]; top-p 0.7
    keeps tokens 0 and 1 (0.644 < 0.7 <= 0.881), renormalised to
    [0.731, 0.269]."""
    z = [2.0, 1.0, 0.0, -1.0]
    assert oracle.sample(z, 1.0, 0.7, 0.5) == (0, 2)
    assert oracle.sample(z, 1.0, 0.7, 0.72) == (0, 2)
    assert oracle.sample(z, 1.0, 0.7, 0.74) == (1, 2)
    assert oracle.sample(z, 1.0, 0.7, 0.999) == (1, 2)
    # top-p 0.9 adds token 2 (0.881 < 0.9 <= 0.968)
    assert oracle.sample(z, 1.0, 0.9, 0.999)[1] == 3


@pytest.mark.parametrize("u", [0.0, 0.3, 0.999])
def test_greedy_limits(u):
    rng = np.random.default_rng(1)
    z = rng.standard_normal(1000).astype(np.float32)
    best = int(np.argmax(z))
    assert oracle.sample(z, 0.0, 0.9, u) == (best, 1)          # T <= 0: argmax
    assert oracle.sample(z, 1.0, 1e-9, u) == (best, 1)         # tiny top-p: the top token only


def test_frequencies_match_softmax():
    """top_p = 1: over many counters the token frequencies follow softmax(z / T)."""
    z = np.array([1.5, 0.2, -0.4, 0.9, -2.0, 0.0], dtype=np.float32)
    T, n = 0.8, 60000
    p = np.exp((z - z.max()) / T)
    p /= p.sum()
    counts = np.zeros(len(z))
    for c in range(n):
        t, k = oracle.sample(z, T, 1.0, oracle.sample_uniform(99, c))
        assert k == len(z)
        counts[t] += 1
    chi2 = np.sum((counts - n * p) ** 2 / (n * p))
    assert chi2 < 25.0   # 5 degrees of freedom: p ~ 1e-4


def test_ties_go_to_lower_index():
    z = [1.0, 1.0, 1.0, 1.0]
    assert oracle.sample(z, 1.0, 0.5, 0.2) == (0, 2)
    assert oracle.sample(z, 1.0, 0.5, 0.7) == (1, 2)
    assert oracle.sample(z, 1.0, 0.51, 0.9) == (2, 3)


def test_temperature_is_logit_scaling():
    rng = np.random.default_rng(2)
    z = (rng.standard_normal(500) * 3).astype(np.float32)
    for u in (0.1, 0.5, 0.9):
        assert oracle.sample(z, 2.0, 0.8, u) == oracle.sample((z / 2).astype(np.float32), 1.0, 0.8, u)
