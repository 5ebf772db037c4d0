"""The allocation-free attention entry point (fixed scratch compiled into the
library, no context) gives the same result as nt_attn_decode.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.  It must pass alone in a fresh process too,
so the first call here is also the entry point's first call on the device."""
import numpy as np
import pytest

import synth
from gpu_util import dev, host, need_gpu, rel_l2, torch

pytestmark = pytest.mark.gpu


def test_static_attention_matches_context_attention():
    need_gpu()
    from block_quantized_gemv_nt_gb300 import nt
    ctx = nt.Context(0)
    H, G, hd, stride = 64, 8, 128, 4168
    K = dev(synth.normal_f16(G * stride * hd, 21, 1).reshape(G, stride, hd))
    V = dev(synth.normal_f16(G * stride * hd, 21, 2).reshape(G, stride, hd))
    for call, n_pos in enumerate([4097, 733]):          # two calls in a row share the scratch
        q = dev(synth.normal_f32(H * hd, 21, 10 + call) * 3)
        ref = torch.empty(H * hd, dtype=torch.float32, device="cuda")
        got = torch.full((H * hd,), float("nan"), dtype=torch.float32, device="cuda")
        nt.nt_attn_decode(ctx, q, K, V, ref, H, G, hd, n_pos, stride)
        nt.nt_attn_decode_static(q, K, V, got, H, G, hd, n_pos, stride)
        torch.cuda.synchronize()
        assert rel_l2(host(got), host(ref)) <= 1e-4
    ctx.sync()
    ctx.close()


def test_static_attention_rejects_oversized_shapes():
    need_gpu()
    from block_quantized_gemv_nt_gb300 import nt
    q = torch.zeros(128 * 128, device="cuda")
    K = torch.zeros(8 * 16 * 128, dtype=torch.float16, device="cuda")
    with pytest.raises(nt.NtError) as ei:   # 128 q heads over 64 KV heads with a huge stride: beyond the 4 MiB
        nt.nt_attn_decode_static(q, K, K, q, 128, 64, 128, 1, 1 << 22)
    assert ei.value.status == nt.NT_ERR_INVALID_ARG
