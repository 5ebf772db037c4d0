"""Self-speculative decoding ("ntransformer - moteur d'inférence NVMe-to-GPU…",
"Fonctionnalités principales": the VRAM-resident layers draft, the whole
model verifies) on the GPU: the M-vector verify GEMM and the causal
multi-query attention against the fp64 oracle, then whole speculative steps.

Pins: every emitted token is the oracle's greedy argmax for the sequence
emitted so far (teacher-forced), each verify row's logits match the
oracle's step logits, and the spec output equals plain greedy decoding of
the same model token for token."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import dev, host, need_gpu, rel_l2, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    from block_quantized_gemv_nt_gb300 import nt
    c = nt.Context(0)
    yield c
    c.sync()
    c.close()


# ---- verify GEMM ----------------------------------------------------------
@pytest.mark.parametrize("fmt", [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q5_K, synth.Q6_K, synth.F16, synth.F32])
@pytest.mark.parametrize("rows,cols,M", [(300, 2304, 5), (257, 4608, 1), (64, 2048, 8), (1000, 512, 3)])
def test_gemm_q_matches_oracle(ctx, fmt, rows, cols, M):
    """Y[m] = W X[m] for M vectors; columns cut into 2048-wide parts (ragged
    last part) and odd row counts (ragged last row group)."""
    from block_quantized_gemv_nt_gb300 import nt
    W = synth.quant_matrix(fmt, rows, cols, seed=21, stream=fmt)
    X = synth.normal_f32(M * cols, seed=21, stream=50 + M).reshape(M, cols)
    res = synth.normal_f32(M * rows, seed=21, stream=60).reshape(M, rows)
    Y = torch.empty(M, rows, dtype=torch.float32, device="cuda")
    Yr = dev(res)
    nt.nt_gemm_q(ctx, fmt, dev(W), dev(X), Y, rows, cols, M)
    nt.nt_gemm_q(ctx, fmt, dev(W), dev(X), Yr, rows, cols, M, residual=Yr)
    torch.cuda.synchronize()
    for m in range(M):
        ref = oracle.gemv(fmt, W, X[m].astype(np.float64), rows, cols)
        assert rel_l2(host(Y[m]), ref) <= 1e-3
        assert rel_l2(host(Yr[m]), ref + res[m]) <= 1e-3


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.Q6_K, synth.Q8_0])
def test_gemm_q_rmsnorm_prologue(ctx, fmt):
    from block_quantized_gemv_nt_gb300 import nt
    rows, cols, M = 200, 4096, 5
    W = synth.quant_matrix(fmt, rows, cols, seed=22, stream=fmt)
    X = synth.normal_f32(M * cols, seed=22, stream=70).reshape(M, cols) * 30
    g = synth.normal_f32(cols, seed=22, stream=71, mean=1.0, std=0.02)
    Y = torch.empty(M, rows, dtype=torch.float32, device="cuda")
    nt.nt_gemm_q(ctx, fmt, dev(W), dev(X), Y, rows, cols, M, norm_g=dev(g), eps=1e-5)
    torch.cuda.synchronize()
    for m in range(M):
        xn = oracle.rmsnorm(X[m].astype(np.float64), g, 1e-5)
        assert rel_l2(host(Y[m]), oracle.gemv(fmt, W, xn, rows, cols)) <= 1e-3


def test_gemm_q_one_vector_equals_gemv(ctx):
    """M = 1 computes the same function as the decode GEMV (same precision)."""
    from block_quantized_gemv_nt_gb300 import nt
    fmt, rows, cols = synth.Q6_K, 512, 8192
    W = dev(synth.quant_matrix(fmt, rows, cols, seed=23, stream=1))
    x = dev(synth.normal_f32(cols, seed=23, stream=2))
    a = torch.empty(rows, device="cuda")
    b = torch.empty(1, rows, device="cuda")
    nt.nt_gemv_q(ctx, fmt, W, x, a, rows, cols)
    nt.nt_gemm_q(ctx, fmt, W, x, b, rows, cols, 1)
    torch.cuda.synchronize()
    assert rel_l2(host(b[0]), host(a).astype(np.float64)) <= 1e-6


@pytest.mark.parametrize("fmt", [synth.Q8_0, synth.Q4_K, synth.Q6_K])
@pytest.mark.parametrize("rows,cols,M", [(300, 2304, 16), (257, 4608, 9), (64, 2048, 12), (1000, 512, 16),
                                         (4096, 4096, 16)])
def test_gemm_q_sixteen_vectors(ctx, fmt, rows, cols, M):
    """M 9..16 (two MMA N-tiles of 8 vectors, the prompt-chunk width) against
    the oracle, with the fused RMSNorm on half the cases; ragged parts, row
    tiles and vector counts.  The tensor-core form needs rows of a multiple of
    16 bytes: Q6_K's 210-byte blocks take column counts of a multiple of 2048."""
    from block_quantized_gemv_nt_gb300 import nt
    if fmt == synth.Q6_K:
        cols = max(2048, cols // 2048 * 2048)
    W = synth.quant_matrix(fmt, rows, cols, seed=24, stream=fmt)
    X = synth.normal_f32(M * cols, seed=24, stream=80 + M).reshape(M, cols) * 3
    g = synth.normal_f32(cols, seed=24, stream=81, mean=1.0, std=0.02)
    norm = (rows + M) % 2 == 0
    res = synth.normal_f32(M * rows, seed=24, stream=82).reshape(M, rows)
    Y = torch.empty(M, rows, dtype=torch.float32, device="cuda")
    Yr = dev(res)
    nt.nt_gemm_q(ctx, fmt, dev(W), dev(X), Y, rows, cols, M, norm_g=dev(g) if norm else None, eps=1e-5)
    nt.nt_gemm_q(ctx, fmt, dev(W), dev(X), Yr, rows, cols, M, residual=Yr, norm_g=dev(g) if norm else None,
                 eps=1e-5)
    torch.cuda.synchronize()
    for m in range(M):
        x = X[m].astype(np.float64)
        if norm:
            x = oracle.rmsnorm(x, g, 1e-5)
        ref = oracle.gemv(fmt, W, x, rows, cols)
        assert rel_l2(host(Y[m]), ref) <= 1e-3, m
        assert rel_l2(host(Yr[m]), ref + res[m]) <= 1e-3, m


def test_gemm_q_bad_args(ctx):
    from block_quantized_gemv_nt_gb300 import nt
    W = torch.zeros(64 * 34 * 8, dtype=torch.uint8, device="cuda")
    X = torch.zeros(17 * 256, device="cuda")
    Y = torch.zeros(17 * 64, device="cuda")
    for M, cols in [(0, 256), (17, 256), (2, 100)]:
        with pytest.raises(nt.NtError) as ei:
            nt.nt_gemm_q(ctx, synth.Q8_0, W, X, Y, 64, cols, M)
        assert ei.value.status == nt.NT_ERR_INVALID_ARG
    # more than 8 vectors only in the tensor-core form: not for Q4_0
    W4 = torch.zeros(64 * 18 * 8, dtype=torch.uint8, device="cuda")
    with pytest.raises(nt.NtError) as ei:
        nt.nt_gemm_q(ctx, synth.Q4_0, W4, X, Y, 64, 256, 9)
    assert ei.value.status == nt.NT_ERR_INVALID_ARG


# ---- causal multi-query attention -------------------------------------------
@pytest.mark.parametrize("H,G,n_pos0,nq,stride", [(64, 8, 4097, 5, 4168), (32, 8, 1, 5, 16), (8, 2, 45, 3, 60),
                                                  (16, 4, 300, 8, 1000)])
def test_attn_verify_matches_oracle(ctx, H, G, n_pos0, nq, stride):
    from block_quantized_gemv_nt_gb300 import nt
    hd = 128
    q = synth.normal_f32(nq * H * hd, 31, 1).reshape(nq, H * hd) * 3
    K = synth.normal_f16(G * stride * hd, 31, 2).reshape(G, stride, hd)
    V = synth.normal_f16(G * stride * hd, 31, 3).reshape(G, stride, hd)
    out = torch.empty(nq, H * hd, dtype=torch.float32, device="cuda")
    nt.nt_attn_verify(ctx, dev(q), dev(K), dev(V), out, H, G, hd, n_pos0, nq, stride)
    torch.cuda.synchronize()
    for i in range(nq):
        ref = oracle.attn_decode(q[i].astype(np.float64), K, V, H, G, hd, n_pos0 + i, stride)
        assert rel_l2(host(out[i]), ref) <= 1e-4, i


def test_attn_verify_bad_args(ctx):
    from block_quantized_gemv_nt_gb300 import nt
    q = torch.zeros(9 * 32 * 128, device="cuda")
    K = torch.zeros(8 * 10 * 128, dtype=torch.float16, device="cuda")
    for n_pos0, nq in [(5, 0), (5, 9), (8, 4)]:  # 8 + 4 - 1 > kv_stride 10
        with pytest.raises(nt.NtError):
            nt.nt_attn_verify(ctx, q, K, K, q, 32, 8, 128, n_pos0, nq, 10)


# ---- whole speculative steps --------------------------------------------------
def _spec_model(ctx, name):
    from block_quantized_gemv_nt_gb300 import engine
    spec = synth.model_spec(name)
    blobs = engine.HostBlobs(spec) if spec.n_resident >= 0 else None
    hm = synth.make_host_model(spec, out_view=blobs.view if blobs else None)
    gm = engine.DeviceModel(ctx, spec, hm, blobs=blobs)
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    return spec, hm, gm, om


def _run_spec_vs_oracle(ctx, name, k, n_draft, n_steps):
    spec, hm, gm, om = _spec_model(ctx, name)
    tok, pos = spec.first_token, spec.n_prefill
    emitted, counts, worst, agree, total = [], [], 0.0, 0, 0
    for step in range(n_steps):
        toks, cnt, vl = gm.spec_step(tok if step == 0 else -1, pos, k, n_draft)
        n = int(cnt.item())
        out = host(toks)[:n].tolist()
        vl = host(vl).astype(np.float64)
        assert 1 <= n <= k + 1
        seq = [tok] + out[:-1]  # the verify rows whose outputs were emitted
        for i in range(n):
            ref = om.step(seq[i], pos + i)
            worst = max(worst, np.max(np.abs(vl[i] - ref)) / ref.std())
            agree += int(np.argmax(ref)) == out[i]
            total += 1
        emitted += out
        counts.append(n)
        tok, pos = out[-1], pos + n
    gm.close()
    return emitted, counts, worst, agree, total


@pytest.mark.parametrize("name,k,n_draft", [("tiny_q8_0", 4, 2), ("tiny_q4_k_m", 4, 3), ("small_q4_k_m", 3, 3),
                                            ("tiny_q6_k", 7, 1), ("tiny_q8_0", 1, 2)])
def test_spec_step_matches_oracle(ctx, name, k, n_draft):
    emitted, counts, worst, agree, total = _run_spec_vs_oracle(ctx, name, k, n_draft, 4)
    print(f"{name}: tokens/step {counts}, worst max|err|/std {worst:.2e}, agree {agree}/{total}")
    assert worst <= 2e-2 and agree == total


def test_spec_full_depth_draft_accepts_everything(ctx):
    """A draft with every layer is the model itself: each step keeps all k
    drafts plus the bonus token (up to fp32 near-ties between the M = 1 and
    M = k + 1 paths)."""
    spec = synth.model_spec("tiny_q4_k")
    emitted, counts, worst, agree, total = _run_spec_vs_oracle(ctx, "tiny_q4_k", 4, spec.n_layers, 4)
    assert worst <= 2e-2 and agree == total
    assert sum(c == 5 for c in counts) >= 3, counts


def test_spec_equals_plain_greedy(ctx):
    """The speculative output is the greedy decode of the same model."""
    from block_quantized_gemv_nt_gb300 import engine
    name, k, n_draft, n_tok = "small_q8_0", 4, 3, 14
    spec = synth.model_spec(name)
    hm = synth.make_host_model(spec)
    ga = engine.DeviceModel(ctx, spec, hm)
    greedy = []
    tok, pos = spec.first_token, spec.n_prefill
    for i in range(n_tok):
        ga.step(tok if i == 0 else -1, pos)
        greedy.append(int(ga.next_token.item()))
    ga.close()
    gb = engine.DeviceModel(ctx, spec, hm)
    got = []
    step = 0
    while len(got) < n_tok:
        toks, cnt, _ = gb.spec_step(spec.first_token if step == 0 else -1, spec.n_prefill, k, n_draft)
        got += host(toks)[:int(cnt.item())].tolist()
        step += 1
    gb.close()
    assert got[:n_tok] == greedy


def test_spec_step_streamed_model(ctx):
    """Draft = the resident layer; the verify pass streams the other layers."""
    emitted, counts, worst, agree, total = _run_spec_vs_oracle(ctx, "small_q6_k_r1", 4, 0, 3)
    assert worst <= 2e-2 and agree == total


def test_spec_step_bad_args(ctx):
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec = synth.model_spec("tiny_q8_0")
    hm = synth.make_host_model(spec)
    gm = engine.DeviceModel(ctx, spec, hm)
    t = torch.zeros(8, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    for tok, pos, k, nd in [(1, 5, 0, 1), (1, 5, 8, 1), (1, 5, 2, 4), (1, spec.kv_cap - 2, 2, 1), (spec.vocab, 5, 2, 1)]:
        with pytest.raises(nt.NtError) as ei:
            nt.nt_spec_step(ctx, gm.handle, tok, pos, k, nd, t, n)
        assert ei.value.status == nt.NT_ERR_INVALID_ARG
    gm.close()


@pytest.mark.parametrize("name,k,n_draft", [("tiny_q4_k_m", 4, 1), ("small_q8_0", 3, 2)])
def test_spec_accept_rule_with_the_draft_chain(ctx, name, k, n_draft):
    """The drafts are greedy decode steps of the first n_draft layers (the
    same kernels as a decode step with the deeper layers skipped), and the
    step keeps draft i+1 exactly while it equals verify output i: emitted
    tokens 0..n-1 are drafts 1..n, and draft n+1 (if any) differs from
    emitted token n."""
    from block_quantized_gemv_nt_gb300 import engine
    spec = synth.model_spec(name)
    hm = synth.make_host_model(spec)
    gd = engine.DeviceModel(ctx, spec, hm)   # runs the draft chain alone
    gs = engine.DeviceModel(ctx, spec, hm)   # runs the speculative steps
    skip = np.zeros(spec.n_layers, np.uint8)
    skip[n_draft:] = 1
    tok, pos = spec.first_token, spec.n_prefill
    for step in range(4):
        drafts, t = [tok], tok
        for i in range(k):
            gd.step(t, pos + i, skip)
            t = int(gd.next_token.item())
            drafts.append(t)
        toks, cnt, _ = gs.spec_step(tok, pos, k, n_draft)
        n_out = int(cnt.item())
        out = host(toks)[:n_out].tolist()
        n = n_out - 1
        assert out[:n] == drafts[1:n + 1]
        if n < k:
            assert drafts[n + 1] != out[n]
        # the draft model's KV at the accepted positions must hold the real
        # tokens before the next draft chain: replay them through it
        for i, t in enumerate([tok] + out[:-1]):
            gd.step(t, pos + i, skip)
        tok, pos = out[-1], pos + n_out
    gd.close()
    gs.close()
