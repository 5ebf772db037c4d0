"""Speculative sampling with sampled drafts ("ntransformer - moteur
d'inférence NVMe-to-GPU…", "Fonctionnalités principales": self-speculative
decoding; "Architecture et structure du code": inference/ sampler) on the GPU
vs the oracle, and the multi-CTA sampler at its edges.

Teacher-forced: the oracle takes the GPU's draft and verify logits of each
step and re-derives every decision — the draft picks, the acceptance tests
u < p/q, the residual draw, the last token — from its own definition; the
tokens must agree.  Separately, the verify rows of the emitted tokens must
match the oracle model run on the emitted sequence (so the device state and
the KV cache advance correctly), and a draft with every layer must
reproduce plain sampled decoding."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import dev, host, need_gpu, torch

pytestmark = pytest.mark.gpu

T, P, SEED = 0.8, 0.9, 77


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    from block_quantized_gemv_nt_gb300 import nt
    c = nt.Context(0)
    yield c
    c.sync()
    c.close()


def _models(ctx, name):
    from block_quantized_gemv_nt_gb300 import engine
    spec = synth.model_spec(name)
    hm = synth.make_host_model(spec)
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    gm = engine.DeviceModel(ctx, spec, hm)
    return spec, hm, gm, om


@pytest.mark.parametrize("name,k,n_draft", [("tiny_q8_0", 4, 2), ("small_q4_k_m", 3, 1), ("tiny_q6_k", 6, 1),
                                            ("tiny_q4_k_m", 5, 3)])
def test_spec_sampled_matches_oracle(ctx, name, k, n_draft):
    spec, hm, gm, om = _models(ctx, name)
    gm.set_sampler(T, P, SEED)
    tok, pos = spec.first_token, spec.n_prefill
    agree, steps, worst, counts, rejections = 0, 0, 0.0, [], 0
    for step in range(6):
        if pos + k >= spec.kv_cap:
            break
        toks, cnt, vl = gm.spec_step(tok if step == 0 else -1, pos, k, n_draft)
        n = int(cnt.item())
        out = host(toks)[:n].tolist()
        V = host(vl).reshape(k + 1, spec.vocab)
        D = host(gm.draft_logits).reshape(k, spec.vocab)
        assert 1 <= n <= k + 1
        ref, drafts = oracle.spec_sample(D, V, T, P, SEED, pos)
        agree += out == ref
        steps += 1
        rejections += n <= k
        # the kept drafts are the oracle's draft picks from the GPU's draft logits
        assert out[:n - 1] == drafts[:n - 1]
        # verify rows of the emitted sequence against the oracle model
        seq = [tok] + out[:-1]
        for i in range(n):
            r = om.step(seq[i], pos + i)
            worst = max(worst, np.max(np.abs(V[i].astype(np.float64) - r)) / r.std())
        counts.append(n)
        tok, pos = out[-1], pos + n
    gm.close()
    print(f"{name}: tokens/step {counts}, agree {agree}/{steps}, worst {worst:.2e}")
    assert agree >= steps - 1
    assert worst <= 2e-2


def test_spec_sampled_full_draft_is_sampled_decoding(ctx):
    """A draft with every layer is the model itself (p = q up to the
    rounding of the M = 1 and M = k + 1 paths): every draft is kept and the
    output is the plain sampled decode with the same seed."""
    from block_quantized_gemv_nt_gb300 import engine
    name, k, n_tok = "tiny_q4_k", 4, 15
    spec = synth.model_spec(name)
    hm = synth.make_host_model(spec)
    ga = engine.DeviceModel(ctx, spec, hm)
    ga.set_sampler(T, P, SEED)
    plain = []
    for i in range(n_tok):
        ga.step(spec.first_token if i == 0 else -1, spec.n_prefill)
        plain.append(int(ga.next_token.item()))
    ga.close()
    gb = engine.DeviceModel(ctx, spec, hm)
    gb.set_sampler(T, P, SEED)
    got, counts = [], []
    while len(got) < n_tok:
        toks, cnt, _ = gb.spec_step(spec.first_token if not got else -1, spec.n_prefill, k, spec.n_layers)
        n = int(cnt.item())
        got += host(toks)[:n].tolist()
        counts.append(n)
    gb.close()
    assert got[:n_tok] == plain
    assert sum(c == k + 1 for c in counts) >= len(counts) - 1, counts


def test_spec_sampled_then_greedy_again(ctx):
    """Switching the sampler off returns the step to the greedy rule (a
    separate graph), and back."""
    spec, hm, gm, om = _models(ctx, "tiny_q8_0")
    gm.set_sampler(T, P, SEED)
    toks, cnt, _ = gm.spec_step(spec.first_token, spec.n_prefill, 3, 2)
    gm.set_sampler(0.0, 1.0, 0)
    toks, cnt, vl = gm.spec_step(spec.first_token, spec.n_prefill, 3, 2)
    n = int(cnt.item())
    out = host(toks)[:n].tolist()
    V = host(vl)
    assert out == [int(np.argmax(V[i])) for i in range(n)]
    gm.close()


# ---- the sampler's cross-CTA paths ------------------------------------------
def test_sample_ties_span_ctas(ctx):
    """50,000 equal logits (49 CTA ranges): the nucleus is the first
    ceil(top_p n) tokens in index order, the pick floor(u * that count)."""
    from block_quantized_gemv_nt_gb300 import nt
    n = 50000
    z = np.full(n, 0.25, dtype=np.float32)
    zd = dev(z)
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    for c in range(12):
        nt.nt_sample(ctx, zd, n, 1.0, 0.5, 3, c, out)
        u = oracle.sample_uniform(3, c)
        want = oracle.sample(z, 1.0, 0.5, u)[0]
        assert want == int(np.floor(u * 25000))
        assert int(out.item()) == want


def test_sample_largest_row(ctx):
    """n = 1,024,000, the largest row (256 CTA ranges of 4000 logits)."""
    from block_quantized_gemv_nt_gb300 import nt
    n = 1024000
    z = synth.normal_f32(n, seed=8, stream=2) * 2.0
    zd = dev(z)
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    for c, (t, p) in enumerate([(1.0, 0.9), (0.5, 0.3), (2.0, 1.0)]):
        nt.nt_sample(ctx, zd, n, t, p, 21, c, out)
        u = oracle.sample_uniform(21, c)
        tok = int(out.item())
        assert tok in {oracle.sample(z, t, p, min(max(u + d, 0.0), 1 - 2**-24))[0] for d in (-1e-6, 0.0, 1e-6)}
    with pytest.raises(nt.NtError) as ei:
        nt.nt_sample(ctx, torch.zeros(n + 1, device="cuda"), n + 1, 1.0, 0.9, 0, 0, out)
    assert ei.value.status == nt.NT_ERR_INVALID_ARG
