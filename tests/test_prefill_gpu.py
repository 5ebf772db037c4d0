"""Prompt prefill on the GPU (the step before decoding: "ntransformer - moteur
d'inférence NVMe-to-GPU…", "Fonctionnalités principales", KV cache): chunks of
up to 16 prompt tokens (8 when a GEMM of the model takes the integer form)
through the M-vector GEMMs and causal multi-query attention, against the fp64
oracle run token by token (teacher-forced).

Pins: the K/V the prefill writes for every prompt position match the
oracle's — layer 0 to one f16 ulp plus the fp32 GEMV rounding; deeper layers
to the decode tolerance (2e-2 of the head's RMS), because attention in these
random models has near-ties that amplify rounding-level differences with
depth — the logits after the last prompt token match the oracle's within the
decode tolerance, and decoding continues from the prefilled state like the
oracle."""
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


def _prompt(spec, n, stream):
    raw = synth.random_bytes(4 * n, seed=spec.seed, stream=stream).view(np.uint32)
    return (raw % spec.vocab).astype(np.int32)


@pytest.mark.parametrize("name,n,pos0", [("tiny_q4_k_m", 20, 37), ("tiny_q8_0", 8, 0), ("small_q6_k", 13, 300),
                                         ("tiny_f16", 3, 40), ("small_q4_k_m_r1", 11, 290),
                                         ("tiny_q8_0", 1, 0), ("tiny_q8_0", 37, 5), ("small_q4_k_m_r1", 20, 270)])
def test_prefill_matches_oracle(ctx, name, n, pos0):
    from block_quantized_gemv_nt_gb300 import engine
    spec = synth.model_spec(name)
    blobs = engine.HostBlobs(spec) if spec.n_resident >= 0 else None
    hm = synth.make_host_model(spec, out_view=blobs.view if blobs else None)
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    gm = engine.DeviceModel(ctx, spec, hm, blobs=blobs)
    prompt = _prompt(spec, n, 777)
    got = gm.prefill(prompt, pos0).cpu().numpy().astype(np.float64)
    for i, t in enumerate(prompt):
        ref = om.step(int(t), pos0 + i)
    assert np.max(np.abs(got - ref)) <= 2e-2 * ref.std()
    assert int(gm.next_token.item()) == int(np.argmax(got)) == int(np.argmax(ref))
    # the K/V of every prompt position, every layer
    torch.cuda.synchronize()
    worst = []   # per layer: the largest |delta| / (head RMS), K and V together
    for li in range(spec.n_layers):
        w = 0.0
        for which in ("kcache", "vcache"):
            g = gm.layers[li][which].cpu().numpy().astype(np.float64)[:, pos0:pos0 + n]
            o = getattr(om, which)[li].astype(np.float64)[:, pos0:pos0 + n]
            scale = np.sqrt(np.mean(o ** 2, axis=-1, keepdims=True))
            bar = np.abs(o) * 2 ** -10 + 1e-4 * scale if li == 0 else 2e-2 * scale
            ratio = np.abs(g - o) / bar
            where = np.unravel_index(np.argmax(ratio), ratio.shape)
            assert ratio.max() <= 1.0, (li, which, float(ratio.max()), where, float(g[where]), float(o[where]))
            w = max(w, float(np.max(np.abs(g - o) / scale)))
        worst.append(w)
    print(f"prefill K/V {name} n={n}: worst |delta|/rms per layer", " ".join(f"{v:.2e}" for v in worst))
    # decoding continues from the prefilled state
    tok = int(np.argmax(got))
    for step in range(3):
        g = gm.step(-1, 0).cpu().numpy().astype(np.float64)
        r = om.step(tok, pos0 + n + step)
        assert np.max(np.abs(g - r)) <= 2e-2 * r.std()
        assert int(np.argmax(g)) == int(np.argmax(r))
        tok = int(np.argmax(r))
    gm.close()


@pytest.mark.parametrize("name,chunk", [("tiny_q8_0", 16), ("tiny_q4_k_m", 8), ("small_q6_k", 16),
                                        ("tiny_f16", 8), ("tiny_q4_0", 8), ("small_q4_k_m_r1", 16)])
def test_prefill_chunk(ctx, name, chunk):
    """16 prompt tokens per pass when every GEMM of the model takes the
    tensor-core form (Q8_0 / Q4_K / Q6_K with rows of a multiple of 16 bytes,
    streamed layers in aligned slots included), 8 when one takes the integer
    form: the tiny Q4_K_M model's Q6_K rows of 512 and 768 columns are 420
    and 630 bytes."""
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec = synth.model_spec(name)
    blobs = engine.HostBlobs(spec) if spec.n_resident >= 0 else None
    hm = synth.make_host_model(spec, out_view=blobs.view if blobs else None)
    gm = engine.DeviceModel(ctx, spec, hm, blobs=blobs)
    assert nt.nt_model_prefill_chunk(ctx, gm.handle) == chunk
    gm.close()


def test_prefill_bad_args(ctx):
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec = synth.model_spec("tiny_q8_0")
    gm = engine.DeviceModel(ctx, spec, synth.make_host_model(spec))
    for toks, pos0 in [([], 0), ([1, 2], spec.kv_cap - 1), ([spec.vocab], 0), ([-1], 0), ([1], -1)]:
        with pytest.raises(nt.NtError) as ei:
            nt.nt_prefill(ctx, gm.handle, toks, pos0, gm.logits)
        assert ei.value.status == nt.NT_ERR_INVALID_ARG
    gm.close()


def test_prefill_tokens_free_on_return(ctx):
    """The prompt is read before nt_prefill returns, from page-locked memory
    too: overwriting the caller's array right after the call (the GPU still
    busy on the stream) changes nothing, and two prefills enqueued back to back
    on one stream each see their own tokens."""
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec = synth.model_spec("tiny_q8_0")
    hm = synth.make_host_model(spec)
    a, b = _prompt(spec, 12, 5), _prompt(spec, 12, 6)
    st = torch.cuda.Stream()
    ref = []
    for p in (a, b):
        g = engine.DeviceModel(ctx, spec, hm)
        torch.cuda.synchronize()
        g.prefill(p, 30, stream=st)
        st.synchronize()
        ref.append(g.logits.clone())
        g.close()
    gm = engine.DeviceModel(ctx, spec, hm)
    pinned = torch.from_numpy(a.copy()).pin_memory()
    torch.cuda.synchronize()
    out = []
    with torch.cuda.stream(st):
        nt.nt_debug_host_delay(ctx, st, 100_000)  # keep the stream busy so the upload cannot have run yet
        for p in (a, b):
            pinned.numpy()[:] = p
            ctx.check(nt._lib.nt_prefill(ctx.handle, gm.handle, pinned.data_ptr(), len(p), 30, gm.logits.data_ptr(),
                                         None, st.cuda_stream))
            pinned.numpy()[:] = 0
            out.append(gm.logits.clone())
    st.synchronize()
    for g, r in zip(out, ref):
        assert torch.equal(g, r)
    gm.close()


@pytest.mark.slow
def test_prefill_llama8b_q8_0_full_size(ctx):
    """The 8B Q8_0 prefill workload at full size: the first 17 tokens of its
    prompt (one chunk of 16 and a ragged one) at the position it starts from,
    against the oracle run token by token — the logits after the prompt, the
    K/V the prefill wrote in the first and the last layer, and one decode
    step continued from the prefilled state."""
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec = synth.model_spec("llama8b_q8_0")
    n, n_bench = 17, 256
    hm = synth.make_host_model(spec)
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    gm = engine.DeviceModel(ctx, spec, hm)
    assert nt.nt_model_prefill_chunk(ctx, gm.handle) == 16
    raw = synth.random_bytes(4 * n_bench, seed=spec.seed, stream=777).view(np.uint32)
    prompt = (raw % spec.vocab).astype(np.int32)[:n]
    pos0 = max(0, min(spec.n_prefill, spec.kv_cap - n_bench))
    got = gm.prefill(prompt, pos0).cpu().numpy().astype(np.float64)
    for i, t in enumerate(prompt):
        ref = om.step(int(t), pos0 + i)
    assert np.max(np.abs(got - ref)) <= 2e-2 * ref.std()
    assert int(np.argmax(got)) == int(np.argmax(ref))
    torch.cuda.synchronize()
    for li in (0, spec.n_layers - 1):
        for which in ("kcache", "vcache"):
            g = gm.layers[li][which].cpu().numpy().astype(np.float64)[:, pos0:pos0 + n]
            o = getattr(om, which)[li].astype(np.float64)[:, pos0:pos0 + n]
            scale = np.sqrt(np.mean(o ** 2, axis=-1, keepdims=True))
            bar = np.abs(o) * 2 ** -10 + 1e-4 * scale if li == 0 else 2e-2 * scale
            assert np.all(np.abs(g - o) <= bar), (li, which)
    tok = int(np.argmax(got))
    g = gm.step(-1, 0).cpu().numpy().astype(np.float64)
    r = om.step(tok, pos0 + n)
    assert np.max(np.abs(g - r)) <= 2e-2 * r.std()
    assert int(np.argmax(g)) == int(np.argmax(r))
    gm.close()
