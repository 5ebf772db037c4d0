"""RMSNorm, RoPE + KV append, split-K decode attention, softmax, SwiGLU,
argmax and cosine similarity on the GPU vs the fp64 oracle, through the C ABI."""
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


def _nt():
    from block_quantized_gemv_nt_gb300 import nt
    return nt


@pytest.mark.parametrize("n", [1, 512, 4096, 8192, 5000])
def test_rmsnorm(ctx, n):
    nt = _nt()
    x = synth.normal_f32(n, 1, 1) * 1e5
    g = synth.normal_f32(n, 1, 2, mean=1.0, std=0.02)
    y = torch.empty(n, dtype=torch.float32, device="cuda")
    nt.nt_rmsnorm(ctx, dev(x), dev(g), y, n, 1e-5)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm(x.astype(np.float64), g, 1e-5)
    assert np.max(np.abs(host(y) - ref)) <= 1e-5 * np.max(np.abs(ref))


@pytest.mark.parametrize("pos", [0, 1, 1024, 4159])
def test_rope(ctx, pos):
    nt = _nt()
    q = synth.normal_f32(32 * 128, 2, 1) * 90
    k = synth.normal_f32(8 * 128, 2, 2) * 90
    qd, kd = dev(q), dev(k)
    nt.nt_rope(ctx, qd, kd, 32, 8, 128, pos, 500000.0)
    torch.cuda.synchronize()
    for got, src, nh in ((qd, q, 32), (kd, k, 8)):
        ref = oracle.rope(src, nh, 128, pos, 500000.0)
        assert np.max(np.abs(host(got) - ref)) <= 2e-6 * np.max(np.abs(ref))


def test_rope_kv_append(ctx):
    nt = _nt()
    H, G, hd, stride, pos = 8, 2, 128, 40, 37
    q = synth.normal_f32(H * hd, 3, 1) * 90
    k = synth.normal_f32(G * hd, 3, 2) * 90
    v = synth.normal_f32(G * hd, 3, 3) * 90
    kc = torch.zeros(G * stride * hd, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    qd = dev(q)
    nt.nt_rope_kv_append(ctx, qd, dev(k), dev(v), kc, vc, H, G, hd, pos, stride, 500000.0)
    torch.cuda.synchronize()
    kref = oracle.rope(k, G, hd, pos, 500000.0).reshape(G, hd)
    K = host(kc).reshape(G, stride, hd).astype(np.float64)
    V = host(vc).reshape(G, stride, hd).astype(np.float64)
    # f16 storage: within one binary16 ulp of the fp64 value
    assert np.all(np.abs(K[:, pos] - kref) <= np.abs(kref) * 2 ** -10 + 1e-7)
    assert np.array_equal(V[:, pos], v.reshape(G, hd).astype(np.float16).astype(np.float64))
    assert not np.any(K[:, :pos]) and not np.any(K[:, pos + 1:])
    qref = oracle.rope(q, H, hd, pos, 500000.0)
    assert np.max(np.abs(host(qd) - qref)) <= 2e-6 * np.max(np.abs(qref))


@pytest.mark.parametrize("H,G,n_pos,stride", [(32, 8, 1, 16), (32, 8, 1025, 1160), (64, 8, 4097, 4168),
                                              (8, 2, 45, 45), (16, 4, 300, 1000), (8, 8, 7, 9)])
def test_attention(ctx, H, G, n_pos, stride):
    nt = _nt()
    hd = 128
    q = synth.normal_f32(H * hd, 4, 1) * 3
    K = synth.normal_f16(G * stride * hd, 4, 2).reshape(G, stride, hd)
    V = synth.normal_f16(G * stride * hd, 4, 3).reshape(G, stride, hd)
    out = torch.empty(H * hd, dtype=torch.float32, device="cuda")
    nt.nt_attn_decode(ctx, dev(q), dev(K), dev(V), out, H, G, hd, n_pos, stride)
    torch.cuda.synchronize()
    ref = oracle.attn_decode(q.astype(np.float64), K, V, H, G, hd, n_pos, stride)
    e = rel_l2(host(out), ref)
    assert e <= 1e-4, e
    if n_pos == 1:
        assert np.allclose(host(out).reshape(H, hd), np.repeat(V[:, 0].astype(np.float32), H // G, axis=0))


def test_attention_repeated_launches_reset_counters(ctx):
    nt = _nt()
    H, G, hd, stride = 32, 8, 128, 700
    K = synth.normal_f16(G * stride * hd, 5, 2).reshape(G, stride, hd)
    V = synth.normal_f16(G * stride * hd, 5, 3).reshape(G, stride, hd)
    Kd, Vd = dev(K), dev(V)
    for it, n_pos in enumerate([1, 700, 333, 64]):
        q = synth.normal_f32(H * hd, 5, 10 + it)
        out = torch.empty(H * hd, dtype=torch.float32, device="cuda")
        nt.nt_attn_decode(ctx, dev(q), Kd, Vd, out, H, G, hd, n_pos, stride)
        torch.cuda.synchronize()
        ref = oracle.attn_decode(q.astype(np.float64), K, V, H, G, hd, n_pos, stride)
        assert rel_l2(host(out), ref) <= 1e-4


def test_attention_bad_args(ctx):
    nt = _nt()
    q = torch.zeros(32 * 128, device="cuda")
    K = torch.zeros(8 * 10 * 128, dtype=torch.float16, device="cuda")
    for args in [(32, 8, 64, 5, 10), (30, 8, 128, 5, 10), (32, 8, 128, 0, 10), (32, 8, 128, 11, 10)]:
        with pytest.raises(nt.NtError):
            nt.nt_attn_decode(ctx, q, K, K, q, *args)


@pytest.mark.parametrize("n", [1, 7, 1025, 70000])
def test_softmax(ctx, n):
    nt = _nt()
    x = synth.normal_f32(n, 6, 1) * 20
    y = torch.empty(n, dtype=torch.float32, device="cuda")
    nt.nt_softmax(ctx, dev(x), y, n)
    torch.cuda.synchronize()
    ref = oracle.softmax(x)
    assert np.max(np.abs(host(y) - ref)) <= 1e-5 * ref.max() + 1e-30
    assert abs(host(y).astype(np.float64).sum() - 1) < 1e-4


def test_swiglu(ctx):
    nt = _nt()
    n = 14336
    g = synth.normal_f32(n, 7, 1) * 50
    g[:4] = [0.0, -1000.0, 1000.0, -90.0]
    u = synth.normal_f32(n, 7, 2) * 50
    h = torch.empty(n, dtype=torch.float32, device="cuda")
    nt.nt_swiglu(ctx, dev(g), dev(u), h, n)
    torch.cuda.synchronize()
    hh = host(h)
    ref = oracle.swiglu(g.astype(np.float64), u.astype(np.float64))
    assert not np.any(np.isnan(hh))
    assert np.max(np.abs(hh - ref) / (np.abs(ref) + 1e-3)) <= 1e-5


@pytest.mark.parametrize("n", [1, 5, 128256, 1000003])
def test_argmax(ctx, n):
    nt = _nt()
    v = synth.normal_f32(n, 8, n % 1000) * 90
    if n > 10:
        m = v.max() + 1.0
        v[n // 3] = m
        v[n // 2] = m       # tie: the lower index wins
    out = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):      # twice: the scratch key must reset itself
        nt.nt_argmax(ctx, dev(v), n, out)
        torch.cuda.synchronize()
        assert int(host(out)[0]) == oracle.argmax(v)


def test_cos_sim(ctx):
    nt = _nt()
    a = synth.normal_f32(8192, 9, 1) * 1e6
    b = a + synth.normal_f32(8192, 9, 2) * 1e5
    out = torch.empty(1, dtype=torch.float32, device="cuda")
    nt.nt_cos_sim(ctx, dev(a), dev(b), 8192, out)
    torch.cuda.synchronize()
    assert abs(float(host(out)[0]) - oracle.cos_sim(a, b)) <= 1e-6


def test_small_ops_reject_misaligned_vectors(ctx):
    """A float pointer off its 4-byte boundary is refused on the host with
    NT_ERR_ALIGNMENT; nothing is launched and the output keeps its bytes."""
    nt = _nt()
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    good, bad = buf.data_ptr(), buf.data_ptr() + 2
    calls = [
        lambda p: nt.nt_softmax(ctx, p, good, 16),
        lambda p: nt.nt_softmax(ctx, good, p, 16),
        lambda p: nt.nt_swiglu(ctx, p, good, good + 1024, 16),
        lambda p: nt.nt_swiglu(ctx, good, good, p, 16),
        lambda p: nt.nt_cos_sim(ctx, p, good, 16, good + 1024),
        lambda p: nt.nt_cos_sim(ctx, good, good, 16, p),
        lambda p: nt.nt_rmsnorm(ctx, p, good, good + 1024, 16, 1e-5),
        lambda p: nt.nt_rope(ctx, p, None, 1, 1, 128, 3, 10000.0),
        lambda p: nt.nt_rope(ctx, good, p, 1, 1, 128, 3, 10000.0),
    ]
    for call in calls:
        with pytest.raises(nt.NtError) as ei:
            call(bad)
        assert ei.value.status == nt.NT_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert int(buf.count_nonzero().item()) == 0
