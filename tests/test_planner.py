"""The resident-layer planner (3-tier caching of "Ntransformer" (en.unwiki.net),
About: VRAM-resident layers first, then pinned RAM; "36 vs 26" layers for
Q4_K_M vs Q6_K on the pages' card).  Pure host arithmetic in libnt.so, so
these run without a GPU; the expected numbers are worked out below from the
block sizes."""
import pytest

import synth


def _plan(name, budget, embd_in_hbm=False, slots=0):
    from block_quantized_gemv_nt_gb300 import engine, nt
    spec = synth.model_spec(name)
    return spec, nt.nt_plan_residency(engine.model_desc(spec, slots), budget, embd_in_hbm)


def test_q6_k_70b_at_24_gb():
    # layer: 2*8192^2 + 2*1024*8192 + 3*28672*8192 weights at 210 B / 256 = 701,890,560 B
    # head: 128256 rows x 32 blocks x 210 B = 861,880,320 B; 2 slots
    spec, p = _plan("llama70b_q6_k_streamed", 24 * 10**9)
    assert p.layer_bytes == 701_890_560
    assert p.fixed_bytes == 861_880_320
    assert p.stream_slots == 2
    assert p.n_resident == (24 * 10**9 - 861_880_320 - 2 * 701_890_560) // 701_890_560 == 30
    assert p.total_bytes == 861_880_320 + 32 * 701_890_560 <= 24 * 10**9


def test_q4_k_m_fits_more_layers_than_q6_k():
    """At the budget where Q6_K keeps the pages' 26 layers, Q4_K_M keeps 8
    more: 34 (the pages, with their own overheads, report 36 vs 26)."""
    # Q4_K_M layer: Q,O 8192^2 and K 1024x8192 at 144/256 B, V 1024x8192 and
    # down 8192x28672 at 210/256 B, gate+up 2x28672x8192 at 144/256 B
    q4km_layer = 2 * 37_748_736 + 4_718_592 + 6_881_280 + 2 * 132_120_576 + 192_675_840
    budget = 861_880_320 + 28 * 701_890_560          # Q6_K: head + 26 layers + 2 slots
    _, p6 = _plan("llama70b_q6_k_streamed", budget)
    spec, p4 = _plan("llama70b_q4_k_m", budget)
    assert p6.n_resident == 26
    assert p4.layer_bytes == q4km_layer == 544_014_336
    assert p4.fixed_bytes == 128_256 * 32 * 144
    assert p4.n_resident == (budget - p4.fixed_bytes - 2 * q4km_layer) // q4km_layer == 34


def test_everything_fits_streams_nothing():
    spec, p = _plan("llama8b_q8_0", 10**12)
    assert p.n_resident == spec.n_layers and p.stream_slots == 0
    assert p.total_bytes == p.fixed_bytes + spec.n_layers * p.layer_bytes


def test_nothing_fits_streams_everything():
    spec, p = _plan("llama8b_q8_0", 10)
    assert p.n_resident == 0 and p.stream_slots == 2


def test_embedding_in_hbm_and_slot_count():
    _, a = _plan("llama8b_q8_0", 8 * 10**9)
    _, b = _plan("llama8b_q8_0", 8 * 10**9, embd_in_hbm=True)
    emb = 128_256 * (4096 // 32) * 34
    assert b.fixed_bytes == a.fixed_bytes + emb
    assert b.n_resident == (8 * 10**9 - b.fixed_bytes - 2 * b.layer_bytes) // b.layer_bytes
    _, c = _plan("llama8b_q8_0", 6 * 10**9, slots=4)
    assert c.stream_slots == 4
    assert c.n_resident == (6 * 10**9 - c.fixed_bytes - 4 * c.layer_bytes) // c.layer_bytes


def test_bad_descriptor():
    from block_quantized_gemv_nt_gb300 import engine, nt
    d = engine.model_desc(synth.model_spec("tiny_q8_0"))
    d.fmt_out = 9
    with pytest.raises(nt.NtError) as ei:
        nt.nt_plan_residency(d, 10**9)
    assert ei.value.status == nt.NT_ERR_UNSUPPORTED_FMT
