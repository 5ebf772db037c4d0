"""Whole decode step on the GPU (one CUDA-graph replay per token) vs the fp64
oracle, teacher-forced: the oracle is fed the GPU's token sequence and logits
are compared step by step.

Bar: max |logit error| <= 2e-2 * std(oracle logits) at every step, and greedy
argmax identical on >= 99% of steps (for the short runs here: every step)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import need_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    from block_quantized_gemv_nt_gb300 import nt
    c = nt.Context(0)
    yield c
    c.sync()
    c.close()


def _run(ctx, name, n_steps, skip=None, continue_on_device=False, layers=None):
    from block_quantized_gemv_nt_gb300 import engine
    spec = synth.model_spec(name)
    hm = synth.make_host_model(spec)
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    gm = engine.DeviceModel(ctx, spec, hm)
    tok, pos = spec.first_token, spec.n_prefill
    worst, agree = 0.0, 0
    for step in range(n_steps):
        if continue_on_device and step > 0:
            logits = gm.step(-1, 0, skip)
        else:
            logits = gm.step(tok, pos, skip)
        got = logits.cpu().numpy().astype(np.float64)
        ref = om.step(tok, pos, skip)
        err = np.max(np.abs(got - ref)) / ref.std()
        worst = max(worst, err)
        g_arg = int(np.argmax(got))
        agree += g_arg == int(np.argmax(ref))
        assert int(gm.next_token.item()) == g_arg
        tok, pos = g_arg, pos + 1
    ctx.sync()
    # the KV written by the GPU matches the oracle's: one f16 ulp of the value plus
    # the fp32 GEMV rounding relative to the scale of the head (cancellation)
    kg = gm.layers[0]["kcache"].cpu().numpy().astype(np.float64)
    ko = om.kcache[0].astype(np.float64)
    P0 = spec.n_prefill
    if skip is None or not skip[0]:
        new_o, new_g = ko[:, P0:P0 + n_steps], kg[:, P0:P0 + n_steps]
        scale = np.sqrt(np.mean(new_o ** 2, axis=-1, keepdims=True))
        assert np.all(np.abs(new_g - new_o) <= np.abs(new_o) * 2 ** -10 + 1e-4 * scale)
    gm.close()
    print(f"{name}: worst max|err|/std = {worst:.2e}, argmax agree {agree}/{n_steps}")
    return worst, agree


@pytest.mark.parametrize("name", ["tiny_q8_0", "tiny_q4_0", "tiny_q4_k", "tiny_q5_k", "tiny_q6_k", "tiny_q4_k_m",
                                  "tiny_f16", "tiny_f32"])
def test_decode_tiny(ctx, name):
    worst, agree = _run(ctx, name, 6)
    assert worst <= 2e-2 and agree == 6


@pytest.mark.parametrize("name", ["small_q8_0", "small_q4_k_m"])
def test_decode_small(ctx, name):
    worst, agree = _run(ctx, name, 5)
    assert worst <= 2e-2 and agree == 5


def test_decode_continues_on_device(ctx):
    worst, agree = _run(ctx, "small_q8_0", 6, continue_on_device=True)
    assert worst <= 2e-2 and agree == 6


def test_decode_with_skip_mask(ctx):
    spec = synth.model_spec("small_q4_k_m")
    skip = np.zeros(spec.n_layers, np.uint8)
    skip[1] = skip[2] = 1
    worst, agree = _run(ctx, "small_q4_k_m", 4, skip=skip)
    assert worst <= 2e-2 and agree == 4


def test_graph_replay_is_deterministic(ctx):
    from block_quantized_gemv_nt_gb300 import engine
    spec = synth.model_spec("tiny_q4_k_m")
    hm = synth.make_host_model(spec)
    gm = engine.DeviceModel(ctx, spec, hm)
    a = gm.step(3, spec.n_prefill).clone()
    b = gm.step(3, spec.n_prefill).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    gm.close()


def test_layer_skip_calibration(ctx):
    from block_quantized_gemv_nt_gb300 import engine
    spec = synth.model_spec("small_q4_k_m")
    hm = synth.make_host_model(spec)
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    gm = engine.DeviceModel(ctx, spec, hm)
    P = spec.n_prefill
    mask, cos = gm.calibrate(spec.first_token, P, n_skip=2)
    ref_logits, ref_cos = om.step(spec.first_token, P, want_cos=True)
    assert np.max(np.abs(cos - ref_cos)) <= 1e-4
    # the mask is the oracle's selection rule applied to the GPU's cosines
    assert np.array_equal(mask, oracle.layer_skip_select(cos.astype(np.float64), 2))
    got = gm.logits.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref_logits)) <= 2e-2 * ref_logits.std()
    # decode with the chosen mask: same function as the oracle running that mask
    tok = int(np.argmax(got))
    g2 = gm.step(tok, P + 1, mask).cpu().numpy().astype(np.float64)
    r2 = om.step(tok, P + 1, mask)
    assert np.max(np.abs(g2 - r2)) <= 2e-2 * r2.std()
    assert int(np.argmax(g2)) == int(np.argmax(r2))
    gm.close()


def test_decode_bad_args(ctx):
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec = synth.model_spec("tiny_q8_0")
    hm = synth.make_host_model(spec)
    gm = engine.DeviceModel(ctx, spec, hm)
    for tok, pos in [(spec.vocab, 5), (1, spec.kv_cap), (1, -1)]:
        with pytest.raises(nt.NtError) as ei:
            gm.step(tok, pos)
        assert ei.value.status == nt.NT_ERR_INVALID_ARG
    gm.close()


@pytest.mark.slow
def test_decode_llama8b_q8_0_full_size(ctx):
    """The 8B Q8_0 workload (seed 1, 1024 prefilled positions): the first two
    greedy steps at full size against the oracle."""
    worst, agree = _run(ctx, "llama8b_q8_0", 2)
    assert worst <= 2e-2 and agree == 2


@pytest.mark.slow
def test_decode_llama70b_q4_k_m_full_size(ctx):
    """The 70B Q4_K_M workload (seed 2, 4096 prefilled positions, attn_v and
    ffn_down in Q6_K): two greedy steps at full size against the oracle; then
    the 20-of-80 layer skip: calibration cosines against the oracle's, the
    mask from the selection rule, and one masked step against the oracle
    running that mask."""
    from block_quantized_gemv_nt_gb300 import engine
    spec = synth.model_spec("llama70b_q4_k_m")
    hm = synth.make_host_model(spec)
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    gm = engine.DeviceModel(ctx, spec, hm)
    P = spec.n_prefill
    tok = spec.first_token
    for i in range(2):
        got = gm.step(tok, P + i).cpu().numpy().astype(np.float64)
        ref = om.step(tok, P + i)
        assert np.max(np.abs(got - ref)) <= 2e-2 * ref.std()
        assert int(np.argmax(got)) == int(np.argmax(ref))
        tok = int(np.argmax(got))
    # calibration on the next position (all layers run), then one masked step
    mask, cos = gm.calibrate(tok, P + 2, n_skip=20)
    ref_logits, ref_cos = om.step(tok, P + 2, want_cos=True)
    assert np.max(np.abs(cos - ref_cos)) <= 1e-4
    assert int(mask.sum()) == 20
    assert np.array_equal(mask, oracle.layer_skip_select(cos.astype(np.float64), 20))
    tok = int(np.argmax(gm.logits.cpu().numpy()))
    got = gm.step(tok, P + 3, mask).cpu().numpy().astype(np.float64)
    ref = om.step(tok, P + 3, mask)
    assert np.max(np.abs(got - ref)) <= 2e-2 * ref.std()
    assert int(np.argmax(got)) == int(np.argmax(ref))
    gm.close()
