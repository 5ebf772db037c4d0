"""The decode step's CUDA graphs and the reproducibility of its results.

- Graphs are keyed on what changes their kernels (skip mask, sampler,
  outputs given or not), not on the caller's output buffers: a caller that
  passes freshly allocated logits and token tensors on every call (the usual
  torch pattern) keeps the graph count constant, and every step is
  bit-identical to the same steps written into one fixed buffer.
- Quant-GEMV plans fix their arithmetic by the shape alone (the tuner only
  times launch shapes that leave every addition unchanged), so two fresh
  processes decode the full-size 8B Q8_0 workload to bit-identical logits.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import synth
from gpu_util import need_gpu, torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    from block_quantized_gemv_nt_gb300 import nt
    c = nt.Context(0)
    yield c
    c.sync()
    c.close()


def test_fresh_output_buffers_do_not_grow_the_graph_cache(ctx):
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec = synth.model_spec("tiny_q4_k_m")
    hm = synth.make_host_model(spec)
    ref = engine.DeviceModel(ctx, spec, hm)
    WINDOW = spec.kv_cap - spec.n_prefill - 1   # steps that fit the KV cache after the prefill
    want = []
    for i in range(200):
        lg = ref.step(spec.first_token, spec.n_prefill) if i % WINDOW == 0 else ref.step(-1, 0)
        want.append(lg.clone())
    torch.cuda.synchronize()
    gm = engine.DeviceModel(ctx, spec, hm)
    counts = set()
    for i in range(200):
        logits = torch.empty(spec.vocab, dtype=torch.float32, device="cuda")   # a new buffer every call
        tok = torch.empty(1, dtype=torch.int32, device="cuda")
        if i % WINDOW == 0:   # restart inside the KV cache
            nt.nt_decode_step(ctx, gm.handle, spec.first_token, spec.n_prefill, None, logits, tok)
        else:
            nt.nt_decode_step(ctx, gm.handle, -1, 0, None, logits, tok)
        assert torch.equal(logits, want[i]), i
        assert int(tok.item()) == int(torch.argmax(want[i]).item())
        counts.add(nt.nt_model_graph_count(ctx, gm.handle))
    assert counts == {1}
    # a step without a token output and a masked step are graphs of their own, and only those
    logits = torch.empty(spec.vocab, dtype=torch.float32, device="cuda")
    nt.nt_decode_step(ctx, gm.handle, -1, 0, None, logits, None)
    mask = np.zeros(spec.n_layers, dtype=np.uint8)
    mask[1] = 1
    for _ in range(3):
        nt.nt_decode_step(ctx, gm.handle, -1, 0, mask, torch.empty_like(logits), None)
    torch.cuda.synchronize()
    assert nt.nt_model_graph_count(ctx, gm.handle) == 3
    gm.close()
    ref.close()


def test_fresh_spec_step_buffers_do_not_grow_the_graph_cache(ctx):
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec = synth.model_spec("tiny_q8_0")
    hm = synth.make_host_model(spec)
    k = 3
    runs = []
    for fresh in (False, True):
        gm = engine.DeviceModel(ctx, spec, hm)
        toks = torch.zeros(k + 1, dtype=torch.int32, device="cuda")
        cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
        lg = torch.zeros((2 * k + 1) * spec.vocab, dtype=torch.float32, device="cuda")
        seq = []
        for i in range(20):
            if fresh:
                toks = torch.empty(k + 1, dtype=torch.int32, device="cuda")
                cnt = torch.empty(1, dtype=torch.int32, device="cuda")
                lg = torch.empty((2 * k + 1) * spec.vocab, dtype=torch.float32, device="cuda")
            t0, p0 = (spec.first_token, spec.n_prefill) if i == 0 else (-1, 0)
            nt.nt_spec_step(ctx, gm.handle, t0, p0, k, 1, toks, cnt, lg)
            n = int(cnt.item())
            seq.append((toks[:n].clone(), lg[:(k + 1) * spec.vocab].clone()))
        assert nt.nt_model_graph_count(ctx, gm.handle) == 1
        runs.append(seq)
        gm.close()
    for (ta, la), (tb, lb) in zip(*runs):
        assert torch.equal(ta, tb)
        assert torch.equal(la, lb)


REPRO = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[2])
import synth
from block_quantized_gemv_nt_gb300 import engine, nt
spec = synth.model_spec("llama8b_q8_0")
hm = synth.make_host_model(spec)
ctx = nt.Context(0)
gm = engine.DeviceModel(ctx, spec, hm)
out = [gm.step(spec.first_token, spec.n_prefill).cpu().numpy().copy()]
for _ in range(19):
    out.append(gm.step(-1, 0).cpu().numpy().copy())
np.save(sys.argv[1], np.stack(out))
print("\n".join(nt.nt_ctx_gemv_plans(ctx)))
gm.close()
ctx.close()
"""


@pytest.mark.slow
def test_processes_decode_bit_identically(tmp_path):
    """Full-size 8B Q8_0, 20 greedy steps, in three fresh processes: two that
    tune their GEMV plans themselves, and one forced onto other launch
    shapes (8 warps, 24 KB stages, no tuning).  Every logit is
    bit-identical: the plans differ only in how the work is launched."""
    need_gpu()
    envs = [{"NT_GEMV_TUNE": "1"}, {"NT_GEMV_TUNE": "1"},
            {"NT_GEMV_TUNE": "0", "NT_GEMV_WARPS": "8", "NT_GEMV_STAGE_MAX": "24576"}]
    outs = []
    for i, extra in enumerate(envs):
        path = str(tmp_path / f"logits{i}.npy")
        r = subprocess.run([sys.executable, "-c", REPRO, path, ROOT], capture_output=True, text=True, timeout=900,
                           env={**os.environ, **extra})
        assert r.returncode == 0, r.stdout + r.stderr
        print(extra, "\n" + r.stdout)
        outs.append(np.load(path))
    assert outs[0].shape == (20, synth.model_spec("llama8b_q8_0").vocab)
    for o in outs[1:]:
        diff = outs[0].view(np.uint32) != o.view(np.uint32)
        assert not diff.any(), [int(d.sum()) for d in diff]
