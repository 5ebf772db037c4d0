"""The seeded generator: deterministic, counter-based, and drawing the
distributions the workloads state (CPU only)."""
import numpy as np

import synth


def test_deterministic_and_stream_separated():
    a = synth.quant_matrix(synth.Q8_0, 16, 256, seed=0, stream=0)
    b = synth.quant_matrix(synth.Q8_0, 16, 256, seed=0, stream=0)
    c = synth.quant_matrix(synth.Q8_0, 16, 256, seed=0, stream=1)
    d = synth.quant_matrix(synth.Q8_0, 16, 256, seed=1, stream=0)
    assert np.array_equal(a, b) and not np.array_equal(a, c) and not np.array_equal(a, d)
    # counter-based: the first rows of a taller matrix are the same bytes
    e = synth.quant_matrix(synth.Q8_0, 32, 256, seed=0, stream=0)
    assert np.array_equal(e[:16], a)


def test_q8_0_distributions():
    W = synth.quant_matrix(synth.Q8_0, 512, 4096, seed=0, stream=0).reshape(-1, 34)
    d = W[:, :2].copy().view(np.float16).astype(np.float64).ravel()
    q = W[:, 2:].view(np.int8).astype(np.int64)
    assert q.min() == -127 and q.max() == 127
    assert abs(q.mean()) < 0.1 and abs(q.std() - np.sqrt((255 ** 2 - 1) / 12)) < 0.2
    assert (d >= 0).all()
    # |N(0,1)| * 0.02 has mean 0.02 * sqrt(2/pi)
    assert abs(d.mean() - 0.02 * np.sqrt(2 / np.pi)) < 2e-4


def test_normals():
    x = synth.normal_f32(200000, seed=0, stream=1)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    g = synth.normal_f32(100000, seed=1, stream=2, mean=1.0, std=0.02)
    assert abs(g.mean() - 1) < 1e-3 and abs(g.std() - 0.02) < 1e-3
    h = synth.normal_f16(100000, seed=1, stream=3)
    assert h.dtype == np.float16 and abs(h.astype(np.float64).std() - 1) < 0.01


def test_model_specs():
    s = synth.model_spec("llama8b_q8_0")
    # 8B: per-layer Q8_0 weights 218,103,808 weights * 34/32 bytes
    assert s.layer_bytes() == (4096 * 4096 * 2 + 1024 * 4096 * 2 + 3 * 14336 * 4096) * 34 // 32
    s70 = synth.model_spec("llama70b_q6_k_streamed")
    assert s70.layer_bytes() == 701_890_560
    m = synth.model_spec("llama70b_q4_k_m")
    assert m.fmt["wv"] == synth.Q6_K and m.fmt["wd"] == synth.Q6_K and m.fmt["wq"] == synth.Q4_K
