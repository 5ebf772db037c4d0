"""Layer streaming from page-locked host memory (the SLEP double-buffered
pipeline and the pinned-RAM tier of "ntransformer - moteur d'inférence
NVMe-to-GPU…", "Fonctionnalités principales" and "Performances et structure
de cache"), on the GPU.

Pins: a streamed model runs the same kernels on the same bytes as the
resident one, so its logits are bit-identical to the resident model's, for
any slot count; and it matches the fp64 oracle within the decode tolerance.
"""
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


def _models(ctx, name, stream_slots=0):
    """(spec, host model, streamed device model): the streamed layers' host
    arrays are views of the page-locked blobs."""
    from block_quantized_gemv_nt_gb300 import engine
    spec = synth.model_spec(name)
    blobs = engine.HostBlobs(spec, stream_slots)
    hm = synth.make_host_model(spec, out_view=blobs.view)
    gm = engine.DeviceModel(ctx, spec, hm, blobs=blobs, stream_slots=stream_slots)
    return spec, hm, gm


def _greedy(gm, spec, n, skip=None):
    out = []
    tok, pos = spec.first_token, spec.n_prefill
    for i in range(n):
        lg = gm.step(tok, pos, skip) if i == 0 else gm.step(-1, 0, skip)
        out.append(lg.clone())
        tok, pos = int(gm.next_token.item()), pos + 1
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name,slots", [("tiny_q4_k_m_r0", 0), ("small_q6_k_r1", 0), ("small_q6_k_r1", 3),
                                        ("small_q4_k_m_r2", 1)])
def test_streamed_equals_resident_bit_exact(ctx, name, slots):
    from block_quantized_gemv_nt_gb300 import engine
    spec, hm, gs = _models(ctx, name, slots)
    rspec = synth.model_spec(name.rsplit("_r", 1)[0])
    gr = engine.DeviceModel(ctx, rspec, hm)
    a = _greedy(gs, spec, 4)
    b = _greedy(gr, rspec, 4)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    # the streamed layers' KV went to the same caches as the resident model's
    for li in range(spec.n_layers):
        assert torch.equal(gs.layers[li]["kcache"], gr.layers[li]["kcache"])
        assert torch.equal(gs.layers[li]["vcache"], gr.layers[li]["vcache"])
    gs.close()
    gr.close()


@pytest.mark.parametrize("name", ["tiny_q4_k_m_r0", "small_q6_k_r1"])
def test_streamed_decode_matches_oracle(ctx, name):
    spec, hm, gm = _models(ctx, name)
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    tok, pos = spec.first_token, spec.n_prefill
    for _ in range(5):
        got = gm.step(tok, pos).cpu().numpy().astype(np.float64)
        ref = om.step(tok, pos)
        assert np.max(np.abs(got - ref)) <= 2e-2 * ref.std()
        assert int(np.argmax(got)) == int(np.argmax(ref))
        tok, pos = int(np.argmax(got)), pos + 1
    gm.close()


def test_streamed_decode_with_skip_mask(ctx):
    """Skipped streamed layers are not copied; the rest still match the oracle
    running the same mask."""
    spec, hm, gm = _models(ctx, "small_q4_k_m_r1")
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    skip = np.zeros(spec.n_layers, np.uint8)
    skip[2] = 1
    tok, pos = spec.first_token, spec.n_prefill
    for _ in range(3):
        got = gm.step(tok, pos, skip).cpu().numpy().astype(np.float64)
        ref = om.step(tok, pos, skip)
        assert np.max(np.abs(got - ref)) <= 2e-2 * ref.std()
        assert int(np.argmax(got)) == int(np.argmax(ref))
        tok, pos = int(np.argmax(got)), pos + 1
    gm.close()


def test_streamed_calibration(ctx):
    """Calibration runs the streaming schedule eagerly (no graph)."""
    spec, hm, gm = _models(ctx, "small_q6_k_r1")
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    mask, cos = gm.calibrate(spec.first_token, spec.n_prefill, n_skip=1)
    _, ref_cos = om.step(spec.first_token, spec.n_prefill, want_cos=True)
    assert np.max(np.abs(cos - ref_cos)) <= 1e-4
    gm.close()


def test_stream_layer_copies_the_blob(ctx):
    """nt_stream_layer lands the blob bytes in the slot: every matrix read back
    from the slot dequantises exactly like the host copy."""
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec, hm, gm = _models(ctx, "small_q4_k_m_r1")
    blobs = gm.blobs
    st = torch.cuda.Stream()
    nt.nt_stream_layer(ctx, gm.handle, 3, blobs.blob[3], blobs.nbytes, 1, st)
    st.synchronize()
    base, nbytes, occupant = nt.nt_model_slot(ctx, gm.handle, 1)
    assert nbytes == blobs.nbytes and occupant == 3
    for i, name in enumerate(engine.LAYER):
        rows, cols = spec.tensor_shape(name)
        n = min(rows, 64)
        got = torch.empty(n * cols, device="cuda")
        ref = torch.empty(n * cols, device="cuda")
        host = torch.from_numpy(hm.layers[3][name][:n]).cuda()
        nt.nt_dequant_rows(ctx, spec.fmt[name], base + blobs.offsets[i], 0, n, cols, got)
        nt.nt_dequant_rows(ctx, spec.fmt[name], host, 0, n, cols, ref)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), name
    gm.close()


def test_stream_bad_args(ctx):
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec, hm, gm = _models(ctx, "tiny_q8_0_r1")
    blobs = gm.blobs
    st = torch.cuda.Stream()
    cases = [
        dict(layer=0, slot=0, nbytes=blobs.nbytes),        # resident layer
        dict(layer=1, slot=2, nbytes=blobs.nbytes),        # slot out of range
        dict(layer=1, slot=0, nbytes=blobs.nbytes - 256),  # wrong size
    ]
    for c in cases:
        with pytest.raises(nt.NtError) as ei:
            nt.nt_stream_layer(ctx, gm.handle, c["layer"], blobs.blob[1], c["nbytes"], c["slot"], st)
        assert ei.value.status == nt.NT_ERR_INVALID_ARG
    pageable = torch.empty(blobs.nbytes, dtype=torch.uint8)
    with pytest.raises(nt.NtError) as ei:
        nt.nt_stream_layer(ctx, gm.handle, 1, pageable, blobs.nbytes, 0, st)
    assert ei.value.status == nt.NT_ERR_INVALID_ARG
    # a layer with some weight pointers and a host blob is refused at model init
    layers = [dict(L) for L in gm.layers]
    layers[1]["wq"] = gm.layers[0]["wq"]
    with pytest.raises(nt.NtError) as ei:
        nt.nt_model_init(ctx, engine.model_desc(spec), layers, gm.embd, gm.out, gm.out_norm)
    assert ei.value.status == nt.NT_ERR_INVALID_ARG
    # a pageable host blob is refused too
    layers = [dict(L) for L in gm.layers]
    layers[1]["host_blob"] = pageable
    with pytest.raises(nt.NtError) as ei:
        nt.nt_model_init(ctx, engine.model_desc(spec), layers, gm.embd, gm.out, gm.out_norm)
    assert ei.value.status == nt.NT_ERR_INVALID_ARG
    gm.close()


@pytest.mark.slow
def test_llama70b_q6_k_streamed_full_size(ctx):
    """The streamed 70B all-Q6_K workload (seed 3, 4096 prefilled positions,
    layers 0..25 resident, 26..79 streamed from page-locked host memory):
    the weights kept in HBM fit the 24 GB cap; one greedy streamed step, then
    one self-speculative step (k = 4, the resident layers draft) against the
    oracle, teacher-forced on the emitted tokens."""
    spec, hm, gm = _models(ctx, "llama70b_q6_k_streamed")
    assert gm.hbm_weight_bytes() <= 24e9
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    P = spec.n_prefill
    got = gm.step(spec.first_token, P).cpu().numpy().astype(np.float64)
    ref = om.step(spec.first_token, P)
    assert np.max(np.abs(got - ref)) <= 2e-2 * ref.std()
    assert int(np.argmax(got)) == int(np.argmax(ref))
    tok = int(np.argmax(got))
    toks, cnt, vl = gm.spec_step(tok, P + 1, 4)
    n = int(cnt.item())
    out = toks.cpu().numpy()[:n].tolist()
    vl = vl.cpu().numpy().astype(np.float64)
    seq = [tok] + out[:-1]
    for i in range(n):
        ref = om.step(seq[i], P + 1 + i)
        assert np.max(np.abs(vl[i] - ref)) <= 2e-2 * ref.std()
        assert int(np.argmax(ref)) == out[i]
    gm.close()


def test_planned_residency_decodes_like_resident(ctx):
    """The planner's split for a budget of the head and two layers with one
    slot keeps layer 0 resident (layers 1 and 2 share the slot); the model
    built from that plan holds exactly the planned bytes in HBM and decodes
    bit-identically to the all-resident model."""
    from block_quantized_gemv_nt_gb300 import engine, nt
    base = synth.model_spec("tiny_q4_k_m")
    sizes = nt.nt_plan_residency(engine.model_desc(base), 10**12)
    plan = nt.nt_plan_residency(engine.model_desc(base, 1), sizes.fixed_bytes + 2 * sizes.layer_bytes)
    assert plan.n_resident == 1 and plan.stream_slots == 1
    spec, hm, gs = _models(ctx, f"tiny_q4_k_m_r{plan.n_resident}", stream_slots=1)
    # the model keeps exactly the planned weight bytes in HBM (its embedding table is in host memory)
    assert gs.hbm_weight_bytes() == plan.total_bytes
    gr = engine.DeviceModel(ctx, base, hm)
    for x, y in zip(_greedy(gs, spec, 3), _greedy(gr, base, 3)):
        assert torch.equal(x, y)
    gs.close()
    gr.close()


@pytest.mark.parametrize("where", ["tmp", "shm"])
def test_model_file_streams_like_resident(ctx, tmp_path, where):
    """The host-file tier: a model written to a file, mapped read-only, its
    streamed layers page-locked in the mapping (else in a private mapping of
    it, else copied once into page-locked memory), decodes bit-identically to
    the same model held resident, and matches the fp64 oracle reading the
    file's own mapped bytes (teacher-forced on the GPU's tokens)."""
    import os
    from block_quantized_gemv_nt_gb300 import engine, modelfile
    spec = synth.model_spec("small_q4_k_m_r1")
    hm = synth.make_host_model(spec)
    d = str(tmp_path) if where == "tmp" or not os.path.isdir("/dev/shm") else "/dev/shm"
    path = os.path.join(d, f"nt_test_{os.getpid()}.ntq")
    modelfile.write_model(path, spec, hm)
    try:
        mf = modelfile.ModelFile(path)
        fb = modelfile.FileBlobs(ctx, mf, spec.n_resident)
        print("tier:", fb.tier, "rungs:", fb.rung_of)
        assert fb.tier in ("mmap pinned", "mmap pinned private", "CPU memcpy")
        hf = synth.HostModel(mf.spec, mf.layers, mf.embd, mf.out, mf.out_norm, hm.kcache, hm.vcache)
        gf = engine.DeviceModel(ctx, mf.spec, hf, blobs=fb)
        base = synth.model_spec("small_q4_k_m")
        gr = engine.DeviceModel(ctx, base, hm)
        got = _greedy(gf, spec, 4)
        for x, y in zip(got, _greedy(gr, base, 4)):
            assert torch.equal(x, y)
        # the oracle on the bytes the file holds (its own mapping), fed the GPU's tokens
        om = oracle.Model(mf.spec, mf.layers, mf.embd, mf.out, mf.out_norm, hm.kcache, hm.vcache)
        tok, pos = spec.first_token, spec.n_prefill
        for lg in got:
            g = lg.cpu().numpy().astype(np.float64)
            ref = om.step(tok, pos)
            assert np.max(np.abs(g - ref)) <= 2e-2 * ref.std()
            assert int(np.argmax(g)) == int(np.argmax(ref))
            tok, pos = int(np.argmax(g)), pos + 1
        del om
        gf.close()
        gr.close()
        fb.close()
        mf.close()
    finally:
        os.unlink(path)


def test_model_file_cpu_copy_rung(ctx, tmp_path):
    """The third rung on the hardware: with both in-place rungs refused (the
    host-side hook), every streamed range takes one CPU copy into page-locked
    memory, or the lock fails with NT_ERR_CUDA when no copy is allowed; the
    model streamed from those copies decodes bit-identically to the same
    model held resident."""
    import os
    from block_quantized_gemv_nt_gb300 import engine, modelfile, nt
    spec = synth.model_spec("small_q4_k_m_r1")
    hm = synth.make_host_model(spec)
    path = os.path.join(str(tmp_path), "m.ntq")
    modelfile.write_model(path, spec, hm)
    mf = modelfile.ModelFile(path)
    nt.nt_debug_file_refuse_in_place(True)
    try:
        with pytest.raises(nt.NtError) as ei:
            modelfile.FileBlobs(ctx, mf, spec.n_resident, allow_copy=False)
        assert ei.value.status == nt.NT_ERR_CUDA
        fb = modelfile.FileBlobs(ctx, mf, spec.n_resident)
    finally:
        nt.nt_debug_file_refuse_in_place(False)
    assert fb.tier == "CPU memcpy" and set(fb.rung_of.values()) == {"CPU memcpy"}
    assert len(fb.rung_of) == spec.n_layers - spec.n_resident + 1   # the streamed layers and the embedding table
    hf = synth.HostModel(mf.spec, mf.layers, mf.embd, mf.out, mf.out_norm, hm.kcache, hm.vcache)
    gf = engine.DeviceModel(ctx, mf.spec, hf, blobs=fb)
    base = synth.model_spec("small_q4_k_m")
    gr = engine.DeviceModel(ctx, base, hm)
    for x, y in zip(_greedy(gf, spec, 3), _greedy(gr, base, 3)):
        assert torch.equal(x, y)
    gf.close()
    gr.close()
    fb.close()
    mf.close()


def test_model_file_lock(ctx, tmp_path):
    """nt_file_lock hands out page-locked ranges holding the entry's bytes
    (in place, or NT_ERR_CUDA when in-place locking is refused and no copy
    is allowed); locking again returns the same range; the file cannot be
    closed while a range is locked; unlocking twice or locking an unknown
    entry is refused."""
    import ctypes
    import os
    from block_quantized_gemv_nt_gb300 import modelfile, nt
    spec = synth.model_spec("tiny_q8_0")
    path = os.path.join(str(tmp_path), "m.ntq")
    modelfile.write_model(path, spec, synth.make_host_model(spec, with_kv=False))
    data = open(path, "rb").read()
    f = nt.nt_file_open(path)
    held = []
    try:
        try:
            a, rung = nt.nt_file_lock(ctx, f, "blob.0", allow_copy=False)
            held.append("blob.0")
            assert nt.FILE_RUNGS[rung] in ("mmap pinned", "mmap pinned private")
        except nt.NtError as e:
            assert e.status == nt.NT_ERR_CUDA
        a, rung = nt.nt_file_lock(ctx, f, "blob.1")
        held.append("blob.1")
        print("rung:", nt.FILE_RUNGS[rung])
        assert nt.nt_file_lock(ctx, f, "blob.1") == (a, rung)
        _, off, n = nt.nt_file_entry(f, "blob.1")
        assert a % 4096 == 0 and ctypes.string_at(a, n) == data[off:off + n]
        with pytest.raises(nt.NtError) as ei:
            nt.nt_file_lock(ctx, f, "blob.99")
        assert ei.value.status == nt.NT_ERR_INVALID_ARG
        with pytest.raises(nt.NtError):
            nt.nt_file_close(f)
        nt.nt_file_unlock(ctx, f, "blob.1")
        held.remove("blob.1")
        with pytest.raises(nt.NtError) as ei:
            nt.nt_file_unlock(ctx, f, "blob.1")
        assert ei.value.status == nt.NT_ERR_INVALID_ARG
    finally:
        for name in held:
            nt.nt_file_unlock(ctx, f, name)
        nt.nt_file_close(f)
