"""The benchmark's launch counts and byte counts (CPU only).

The launch list of one 8B Q8_0 decode step, captured with ncu on a GB300
(the embedding row to the argmax, one full step), holds 195 kernels: 32
layers of Q/K/V, attention split and combine, O, gate/up and down, then the
LM head and the argmax, with the embedding in front.  The count the
benchmark claims is pinned to that.  The per-token bytes are pinned to the
block sizes of the formats."""
import bench
import synth


def test_decode_launches_match_the_captured_step():
    spec = synth.model_spec("llama8b_q8_0")
    assert bench.decode_kernels_per_step(spec, spec.n_layers) == 195


def test_decode_launches_mixed_formats_skip_and_sampler():
    spec = synth.model_spec("llama70b_q4_k_m")
    # Q/K share Q4_K, V is Q6_K: two Q/K/V launches per layer
    assert bench.decode_kernels_per_step(spec, 80) == 2 + 80 * 7 + 1
    assert bench.decode_kernels_per_step(spec, 60) == 2 + 60 * 7 + 1
    assert bench.decode_kernels_per_step(spec, 80, sampled=True) == 2 + 80 * 7 + 6


def test_step_bytes_8b():
    """8B Q8_0: 32 layers of 6144x4096 + 4096x4096 + 2 x 14336x4096 +
    4096x14336 weights at 34 bytes per 32, plus the 128256x4096 head."""
    spec = synth.model_spec("llama8b_q8_0")
    per_row = lambda cols: cols // 32 * 34  # noqa: E731
    layer = 6144 * per_row(4096) + 4096 * per_row(4096) + 2 * 14336 * per_row(4096) + 4096 * per_row(14336)
    weights = 32 * layer + 128256 * per_row(4096)
    got = bench.step_bytes(spec)
    # the step also reads one embedding row and the KV cache; the weights are all but a few percent
    assert weights <= got <= weights * 1.03, (got, weights)


def test_verify_layer_launches():
    """A verify or prefill layer: every GEMM is its kernel and the epilogue that
    adds the column parts; a normed GEMM in the tensor-core form (Q8_0 / Q4_K /
    Q6_K) has the RMSNorm scalars' kernel in front; attention is split +
    combine."""
    assert bench.verify_layer_launches(synth.model_spec("llama8b_q8_0")) == 3 + 2 + 2 + 3 + 2
    # Q/K in Q4_K and V in Q6_K: two normed Q/K/V launches
    assert bench.verify_layer_launches(synth.model_spec("llama70b_q4_k_m")) == 2 * 3 + 2 + 2 + 3 + 2
    # F16 takes the integer form: no RMSNorm kernel
    assert bench.verify_layer_launches(synth.model_spec("tiny_f16")) == 2 + 2 + 2 + 2 + 2
