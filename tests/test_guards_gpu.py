"""Guard canaries: every kernel writes its outputs and nothing next to them.

Each output buffer sits between two 64-element guard regions filled with a
fixed bit pattern; after the call (and a synchronize) the guards must be
unchanged bit for bit, and the output itself fully written (no canary left
inside it).  Shapes cover ragged row groups, single rows, split-K parts and
the largest cases the tests use elsewhere.  This is the stand-in for a memory
sanitizer, which is not available here."""
import numpy as np
import pytest

import synth
from gpu_util import dev, need_gpu, torch

pytestmark = pytest.mark.gpu

GUARD = 64
CANARY_BITS = 0x5A5AA5A5  # as float32: a finite value no kernel produces by chance here


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    from block_quantized_gemv_nt_gb300 import nt
    c = nt.Context(0)
    yield c
    c.sync()
    c.close()


def _guarded(n, dtype=torch.float32):
    buf = torch.full((n + 2 * GUARD,), CANARY_BITS, dtype=torch.int32, device="cuda")
    if dtype == torch.float32:
        buf = buf.view(torch.float32)
    return buf, buf[GUARD:GUARD + n]


def _check(buf, n):
    torch.cuda.synchronize()
    bits = buf.view(torch.int32)
    assert torch.all(bits[:GUARD] == CANARY_BITS), "write before the output"
    assert torch.all(bits[GUARD + n:] == CANARY_BITS), "write after the output"
    assert not torch.any(bits[GUARD:GUARD + n] == CANARY_BITS), "output element left unwritten"


FMTS = [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q5_K, synth.Q6_K, synth.F16, synth.F32]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,cols", [(1, 256), (5, 512), (257, 2048), (1000, 4096)])
def test_gemv_outputs(ctx, fmt, rows, cols):
    from block_quantized_gemv_nt_gb300 import nt
    W = dev(synth.quant_matrix(fmt, rows, cols, seed=31, stream=fmt))
    Wu = dev(synth.quant_matrix(fmt, rows, cols, seed=31, stream=10 + fmt))
    x = dev(synth.normal_f32(cols, seed=31, stream=20))
    buf, y = _guarded(rows)
    nt.nt_gemv_q(ctx, fmt, W, x, y, rows, cols)
    _check(buf, rows)
    buf, h = _guarded(rows)
    nt.nt_gemv_q_swiglu(ctx, fmt, W, Wu, x, h, rows, cols)
    _check(buf, rows)
    M = 3
    X = dev(synth.normal_f32(M * cols, seed=31, stream=21))
    buf, Y = _guarded(M * rows)
    nt.nt_gemm_q(ctx, fmt, W, X, Y, rows, cols, M)
    _check(buf, M * rows)
    buf, d = _guarded(rows * cols)
    nt.nt_dequant_rows(ctx, fmt, W, 0, rows, cols, d)
    _check(buf, rows * cols)


@pytest.mark.parametrize("H,G,n_pos,stride", [(32, 8, 1, 16), (32, 8, 1088, 1096), (64, 8, 4097, 4168), (8, 2, 45, 60)])
def test_attention_output(ctx, H, G, n_pos, stride):
    from block_quantized_gemv_nt_gb300 import nt
    hd = 128
    q = dev(synth.normal_f32(H * hd, seed=32, stream=1))
    K = torch.from_numpy(synth.normal_f32(G * stride * hd, seed=32, stream=2)).half().cuda()
    V = torch.from_numpy(synth.normal_f32(G * stride * hd, seed=32, stream=3)).half().cuda()
    buf, out = _guarded(H * hd)
    nt.nt_attn_decode(ctx, q, K, V, out, H, G, hd, n_pos, stride)
    _check(buf, H * hd)


@pytest.mark.parametrize("n", [7, 128256])
def test_sampler_and_argmax_output(ctx, n):
    from block_quantized_gemv_nt_gb300 import nt
    z = dev(synth.normal_f32(n, seed=33, stream=1))
    for T in (0.0, 0.8):
        buf, out = _guarded(1, torch.int32)
        nt.nt_sample(ctx, z, n, T, 0.9, 5, 1, out)
        _check(buf, 1)
    buf, out = _guarded(1, torch.int32)
    nt.nt_argmax(ctx, z, n, out)
    _check(buf, 1)


def test_decode_and_spec_outputs(ctx):
    """A whole decode step writes the logits row and the next token, a
    speculative step at most k + 1 tokens and their count."""
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec = synth.model_spec("tiny_q8_0")
    hm = synth.make_host_model(spec)
    gm = engine.DeviceModel(ctx, spec, hm)
    lbuf, logits = _guarded(spec.vocab)
    tbuf, tok = _guarded(1, torch.int32)
    nt.nt_decode_step(ctx, gm.handle, spec.first_token, spec.n_prefill, None, logits, tok)
    _check(lbuf, spec.vocab)
    _check(tbuf, 1)
    k = 3
    obuf, toks = _guarded(k + 1, torch.int32)
    cbuf, cnt = _guarded(1, torch.int32)
    nt.nt_spec_step(ctx, gm.handle, spec.first_token, spec.n_prefill, k, 2, toks, cnt)
    torch.cuda.synchronize()
    n = int(cnt.item())
    assert 1 <= n <= k + 1
    bits = obuf.view(torch.int32)
    assert torch.all(bits[:GUARD] == CANARY_BITS) and torch.all(bits[GUARD + k + 1:] == CANARY_BITS)
    assert not torch.any(bits[GUARD:GUARD + n] == CANARY_BITS)
    _check(cbuf, 1)
    gm.close()
