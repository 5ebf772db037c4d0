"""The allocation-free attention entry point, nt_attn_decode_static.

Some callers cannot allocate device memory: code that runs while a stream is
being captured into a CUDA graph in a mode that forbids allocation, and hosts
that hand out device memory only from their own pool.  Such callers cannot
create an nt_ctx (it allocates its scratch), so this entry point keeps its
scratch in a fixed array inside the library.  These tests check that it
computes the same attention as the context entry point and as the fp64
oracle, on two calls in a row, that its size limit holds exactly where the
header says, and that a device-side wait that runs out shows in the output
without spoiling the next call.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.  It must pass alone in a fresh process too,
so the first call here is also the entry point's first call on the device."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import dev, host, need_gpu, rel_l2, torch

pytestmark = pytest.mark.gpu


def _cache(G, stride, hd, seed):
    K = synth.normal_f16(G * stride * hd, seed, 1).reshape(G, stride, hd)
    V = synth.normal_f16(G * stride * hd, seed, 2).reshape(G, stride, hd)
    return K, V


def test_static_attention_matches_context_attention_and_oracle():
    need_gpu()
    from block_quantized_gemv_nt_gb300 import nt
    ctx = nt.Context(0)
    H, G, hd, stride = 64, 8, 128, 4168
    Kh, Vh = _cache(G, stride, hd, 21)
    K, V = dev(Kh), dev(Vh)
    for call, n_pos in enumerate([4097, 733]):          # two calls in a row share the scratch
        qh = synth.normal_f32(H * hd, 21, 10 + call) * 3
        q = dev(qh)
        ref = torch.empty(H * hd, dtype=torch.float32, device="cuda")
        got = torch.full((H * hd,), float("nan"), dtype=torch.float32, device="cuda")
        nt.nt_attn_decode(ctx, q, K, V, ref, H, G, hd, n_pos, stride)
        nt.nt_attn_decode_static(q, K, V, got, H, G, hd, n_pos, stride)
        torch.cuda.synchronize()
        want = oracle.attn_decode(qh.astype(np.float64), Kh, Vh, H, G, hd, n_pos, stride)
        assert rel_l2(host(got), want) <= 1e-4
        assert rel_l2(host(got), host(ref)) <= 1e-4
    ctx.sync()
    ctx.close()


def test_static_attention_size_limit():
    """64 q heads over 8 KV heads: 15,872 cached positions is the largest
    stride whose split partials fit the fixed 4 MiB (accepted, and correct);
    16,000 (within the attention's own 16,384 limit) does not fit and is
    refused before anything is enqueued."""
    need_gpu()
    from block_quantized_gemv_nt_gb300 import nt
    H, G, hd, stride = 64, 8, 128, 15872
    Kh, Vh = _cache(G, stride, hd, 22)
    K, V = dev(Kh), dev(Vh)
    qh = synth.normal_f32(H * hd, 22, 3) * 3
    q = dev(qh)
    got = torch.full((H * hd,), float("nan"), dtype=torch.float32, device="cuda")
    nt.nt_attn_decode_static(q, K, V, got, H, G, hd, stride, stride)
    torch.cuda.synchronize()
    want = oracle.attn_decode(qh.astype(np.float64), Kh, Vh, H, G, hd, stride, stride)
    assert rel_l2(host(got), want) <= 1e-4
    big = torch.zeros(G * 16000 * hd, dtype=torch.float16, device="cuda")
    before = got.clone()
    with pytest.raises(nt.NtError) as ei:
        nt.nt_attn_decode_static(q, big, big, got, H, G, hd, 1, 16000)
    assert ei.value.status == nt.NT_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.equal(got, before)      # nothing was enqueued
    with pytest.raises(nt.NtError) as ei:  # and far beyond: 128 q heads over 64 KV heads, a huge stride
        nt.nt_attn_decode_static(q, big, big, got, 128, 64, hd, 1, 1 << 22)
    assert ei.value.status == nt.NT_ERR_INVALID_ARG


def test_static_attention_timeout_shows_as_nan_then_clears():
    """A device-side wait that runs out (made to run out by the test hook: the
    armed launch issues no copies, so nothing ever completes its barrier; no
    GPU fault or hang) leaves this call's output NaN — there is no context to
    report it — and the next call, unarmed, is correct again."""
    need_gpu()
    from block_quantized_gemv_nt_gb300 import nt
    H, G, hd, stride, n_pos = 32, 8, 128, 1100, 1088
    Kh, Vh = _cache(G, stride, hd, 23)
    K, V = dev(Kh), dev(Vh)
    qh = synth.normal_f32(H * hd, 23, 4)
    q = dev(qh)
    out = torch.zeros(H * hd, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    nt.nt_debug_stall_waits(1)
    try:
        nt.nt_attn_decode_static(q, K, V, out, H, G, hd, n_pos, stride)
        torch.cuda.synchronize()
    finally:
        nt.nt_debug_stall_waits(0)
    assert torch.isnan(out).all()
    nt.nt_attn_decode_static(q, K, V, out, H, G, hd, n_pos, stride)
    torch.cuda.synchronize()
    want = oracle.attn_decode(qh.astype(np.float64), Kh, Vh, H, G, hd, n_pos, stride)
    assert rel_l2(host(out), want) <= 1e-4
