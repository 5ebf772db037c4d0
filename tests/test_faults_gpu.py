"""Failure detection of the layer-streaming engine, made on the host: no GPU
fault, trap or hang is ever induced.

- A fault-injection hook makes the nth layer copy request fail before
  anything is enqueued: the error reaches the caller, the slot bookkeeping
  stays as it was, and a retry works (for a direct nt_stream_layer and for a
  decode step whose graph capture hits the failure).
- A deadline-bounded stream wait returns NT_ERR_TIMEOUT while a host
  callback keeps the stream busy, and NT_OK once it is done; the context
  stays usable.
- The device-side bounded waits themselves: a test hook makes the next
  launch of the quant GEMV or the decode attention issue no bulk copies, so
  its mbarrier is never completed (nothing is in flight, nothing faults); the
  wait gives up after a few tries, the kernel raises the context's flag and
  returns, nt_ctx_sync reports NT_ERR_TIMEOUT, and the next launch on the
  same context is correct."""
import time

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
    nt.nt_debug_fail_copy(c, -1)
    c.sync()
    c.close()


def _models(ctx, name, stream_slots=0):
    from block_quantized_gemv_nt_gb300 import engine
    spec = synth.model_spec(name)
    blobs = engine.HostBlobs(spec, stream_slots)
    hm = synth.make_host_model(spec, out_view=blobs.view)
    gm = engine.DeviceModel(ctx, spec, hm, blobs=blobs, stream_slots=stream_slots)
    return spec, hm, gm


def test_injected_copy_failure_then_retry(ctx):
    from block_quantized_gemv_nt_gb300 import nt
    spec, hm, gm = _models(ctx, "small_q4_k_m_r1")
    blobs = gm.blobs
    st = torch.cuda.Stream()
    _, _, before = nt.nt_model_slot(ctx, gm.handle, 1)
    nt.nt_debug_fail_copy(ctx, 0)
    with pytest.raises(nt.NtError) as ei:
        nt.nt_stream_layer(ctx, gm.handle, 3, blobs.blob[3], blobs.nbytes, 1, st)
    assert ei.value.status == nt.NT_ERR_CUDA and "injected" in str(ei.value)
    st.synchronize()
    assert nt.nt_model_slot(ctx, gm.handle, 1)[2] == before  # nothing was copied, nothing recorded
    nt.nt_stream_layer(ctx, gm.handle, 3, blobs.blob[3], blobs.nbytes, 1, st)  # the hook fired once
    st.synchronize()
    assert nt.nt_model_slot(ctx, gm.handle, 1)[2] == 3
    gm.close()


@pytest.mark.parametrize("nth", [0, 1])
def test_decode_step_capture_failure_then_retry(ctx, nth):
    """The nth copy of the first streamed step fails while its graph is being
    captured: the step reports it and keeps no graph; the retry captures
    again and decodes exactly like the same model held resident."""
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec, hm, gs = _models(ctx, "small_q6_k_r1")
    rspec = synth.model_spec("small_q6_k")
    gr = engine.DeviceModel(ctx, rspec, hm)
    tok, pos = spec.first_token, spec.n_prefill
    nt.nt_debug_fail_copy(ctx, nth)
    with pytest.raises(nt.NtError) as ei:
        gs.step(tok, pos)
    assert ei.value.status == nt.NT_ERR_CUDA and "injected" in str(ei.value)
    slots = [nt.nt_model_slot(ctx, gs.handle, i)[2] for i in range(gs.n_slots)]
    assert slots == [-1] * gs.n_slots  # no copy of the aborted pass is recorded
    out = []
    for model in (gs, gr):
        t, p = tok, pos
        seq = []
        for i in range(3):
            lg = model.step(t, p) if i == 0 else model.step(-1, 0)
            seq.append(lg.clone())
            t, p = int(model.next_token.item()), p + 1
        out.append(seq)
    torch.cuda.synchronize()
    for a, b in zip(*out):
        assert torch.equal(a, b)
    gs.close()
    gr.close()


def test_stream_sync_deadline(ctx):
    from block_quantized_gemv_nt_gb300 import nt
    st = torch.cuda.Stream()
    nt.nt_debug_host_delay(ctx, st, 300_000)
    t0 = time.perf_counter()
    with pytest.raises(nt.NtError) as ei:
        nt.nt_stream_sync(ctx, st, 20_000)
    assert ei.value.status == nt.NT_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 0.25
    nt.nt_stream_sync(ctx, st, 5_000_000)
    assert time.perf_counter() - t0 >= 0.29
    # the context is still usable
    x = torch.randn(1000, device="cuda")
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    nt.nt_argmax(ctx, x, 1000, out)
    torch.cuda.synchronize()
    assert int(out.item()) == int(torch.argmax(x).item())
    with pytest.raises(nt.NtError) as ei:
        nt.nt_stream_sync(ctx, st, -1)
    assert ei.value.status == nt.NT_ERR_INVALID_ARG


def _stalled_then_clean(ctx, launch):
    """launch() once armed (the wait runs out), then once clean."""
    from block_quantized_gemv_nt_gb300 import nt
    ctx.sync()
    nt.nt_debug_stall_waits(1)
    try:
        launch()
    finally:
        nt.nt_debug_stall_waits(0)
    with pytest.raises(nt.NtError) as ei:
        ctx.sync()
    assert ei.value.status == nt.NT_ERR_TIMEOUT
    launch()
    ctx.sync()   # the flag was taken: a clean launch reports nothing


def test_attention_wait_timeout_is_reported(ctx):
    from block_quantized_gemv_nt_gb300 import nt
    H, G, hd, stride, n_pos = 32, 8, 128, 1100, 1088
    Kh = synth.normal_f16(G * stride * hd, 31, 1).reshape(G, stride, hd)
    Vh = synth.normal_f16(G * stride * hd, 31, 2).reshape(G, stride, hd)
    qh = synth.normal_f32(H * hd, 31, 3)
    K, V, q = dev(Kh), dev(Vh), dev(qh)
    out = torch.zeros(H * hd, dtype=torch.float32, device="cuda")
    _stalled_then_clean(ctx, lambda: nt.nt_attn_decode(ctx, q, K, V, out, H, G, hd, n_pos, stride))
    want = oracle.attn_decode(qh.astype(np.float64), Kh, Vh, H, G, hd, n_pos, stride)
    assert rel_l2(host(out), want) <= 1e-4


@pytest.mark.parametrize("fmt", [0, 2, 4])
def test_gemv_wait_timeout_is_reported(ctx, fmt):
    from block_quantized_gemv_nt_gb300 import nt
    rows, cols = 3000, 4096
    W = synth.quant_matrix(fmt, rows, cols, seed=32, stream=fmt)
    x = synth.normal_f32(cols, seed=32, stream=99)
    Wd, xd = dev(W), dev(x)
    y = torch.zeros(rows, dtype=torch.float32, device="cuda")
    nt.nt_gemv_q(ctx, fmt, Wd, xd, y, rows, cols)   # plan tuning happens on this first call, unarmed
    _stalled_then_clean(ctx, lambda: nt.nt_gemv_q(ctx, fmt, Wd, xd, y, rows, cols))
    want = oracle.gemv(fmt, W, x.astype(np.float64), rows, cols)
    assert rel_l2(host(y), want) <= 1e-3
