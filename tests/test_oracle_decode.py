"""Pins for the oracle's whole decode step (CPU only).

The step is a composition of the pinned pieces.  Here it is checked against a
brute-force numpy restatement on a tiny model (dense dequantised matrices,
RoPE as complex multiplication, softmax with numpy), against the special case
"every layer skipped" (embedding -> final norm -> head), and for its KV-cache
writes.
"""
import numpy as np

import oracle
import synth


def _dense(spec, hm, li, t):
    r, c = spec.tensor_shape(t)
    return oracle.dequant(spec.fmt[t], hm.layers[li][t], r, c).astype(np.float64)


def _rms(x, g, eps):
    return x / np.sqrt(np.mean(x * x) + eps) * g.astype(np.float64)


def _rope_complex(v, n_heads, hd, pos, theta):
    z = v.reshape(n_heads, hd // 2, 2)
    c = z[..., 0] + 1j * z[..., 1]
    freq = theta ** (-np.arange(0, hd, 2) / hd)
    c = c * np.exp(1j * pos * freq)
    return np.stack([c.real, c.imag], axis=-1).reshape(-1)


def _f16_round(v):
    return v.astype(np.float32).astype(np.float16)


def _numpy_step(spec, hm, kc, vc, token, pos):
    d, hd, H, G = spec.d_model, spec.head_dim, spec.n_qh, spec.n_kvh
    r, c = spec.tensor_shape("embd")
    x = oracle.dequant(spec.fmt["embd"], hm.embd, r, c, row0=token, nrows=1)[0].astype(np.float64)
    for li in range(spec.n_layers):
        L = hm.layers[li]
        xn = _rms(x, L["attn_norm"], spec.eps)
        q = _dense(spec, hm, li, "wq") @ xn
        k = _dense(spec, hm, li, "wk") @ xn
        v = _dense(spec, hm, li, "wv") @ xn
        q = _rope_complex(q, H, hd, pos, spec.theta)
        k = _rope_complex(k, G, hd, pos, spec.theta)
        kc[li, :, pos, :] = _f16_round(k.reshape(G, hd))
        vc[li, :, pos, :] = _f16_round(v.reshape(G, hd))
        o = np.empty(H * hd)
        for h in range(H):
            g = h // (H // G)
            Kh = kc[li, g, :pos + 1].astype(np.float64)
            Vh = vc[li, g, :pos + 1].astype(np.float64)
            s = Kh @ q[h * hd:(h + 1) * hd] / np.sqrt(hd)
            p = np.exp(s - s.max())
            p /= p.sum()
            o[h * hd:(h + 1) * hd] = p @ Vh
        x = x + _dense(spec, hm, li, "wo") @ o
        xn = _rms(x, L["ffn_norm"], spec.eps)
        gt = _dense(spec, hm, li, "wg") @ xn
        up = _dense(spec, hm, li, "wu") @ xn
        x = x + _dense(spec, hm, li, "wd") @ (gt / (1 + np.exp(-gt)) * up)
    xn = _rms(x, hm.out_norm, spec.eps)
    r, c = spec.tensor_shape("out")
    return oracle.dequant(spec.fmt["out"], hm.out, r, c).astype(np.float64) @ xn


def _model(name):
    spec = synth.model_spec(name)
    hm = synth.make_host_model(spec)
    return spec, hm


def test_decode_step_matches_numpy_restatement():
    for name in ("tiny_q8_0", "tiny_q4_k_m"):
        spec, hm = _model(name)
        om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
        kc, vc = hm.kcache.copy(), hm.vcache.copy()
        tok, pos = spec.first_token, spec.n_prefill
        for step in range(2):
            got = om.step(tok, pos)
            ref = _numpy_step(spec, hm, kc, vc, tok, pos)
            assert np.allclose(got, ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())
            # the KV writes agree bit for bit (both round fp64 -> fp32 -> f16)
            diff = np.abs(om.kcache[:, :, pos].astype(np.float64) - kc[:, :, pos].astype(np.float64))
            assert (diff <= np.abs(kc[:, :, pos].astype(np.float64)) * 2 ** -10).all()
            tok, pos = int(np.argmax(got)), pos + 1


def test_decode_step_all_layers_skipped_is_head_of_embedding():
    spec, hm = _model("tiny_q4_0")
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    tok = 5
    got = om.step(tok, spec.n_prefill, skip=np.ones(spec.n_layers, np.uint8))
    r, c = spec.tensor_shape("embd")
    x = oracle.dequant(spec.fmt["embd"], hm.embd, r, c, row0=tok, nrows=1)[0].astype(np.float64)
    ref = oracle.gemv(spec.fmt["out"], hm.out, _rms(x, hm.out_norm, spec.eps), r, c)
    assert np.allclose(got, ref, rtol=1e-12)
    # skipped layers write no KV
    assert np.array_equal(om.kcache, hm.kcache)


def test_decode_cos_reported_for_executed_layers():
    spec, hm = _model("tiny_q8_0")
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    skip = np.zeros(spec.n_layers, np.uint8)
    skip[1] = 1
    _, cos = om.step(1, spec.n_prefill, skip=skip, want_cos=True)
    assert np.isnan(cos[1]) and np.all(np.abs(cos[[0, 2]]) <= 1.0)
