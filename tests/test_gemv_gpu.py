"""Quant GEMV and dequantisation on the GPU vs the fp64 oracle, through the C ABI.

Bar: dequantised weights bit-exact (all seven formats: the five block formats
and plain F16 / F32); GEMV relative L2 error <= 1e-3 of the fp64 oracle (the
stated tolerance)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import dev, host, need_gpu, rel_l2, torch

pytestmark = pytest.mark.gpu
TOL = 1e-3
FMTS = [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q5_K, synth.Q6_K, synth.F16, synth.F32]


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


def _case(fmt, rows, cols, seed=0, offset=0):
    W = synth.quant_matrix(fmt, rows, cols, seed=seed, stream=fmt)
    x = synth.normal_f32(cols, seed=seed, stream=50 + fmt)
    Wd = dev(np.concatenate([np.zeros(offset, np.uint8), W.ravel()]))[offset:] if offset else dev(W)
    return W, x, Wd, dev(x)


@pytest.mark.parametrize("fmt", FMTS)
def test_dequant_bit_exact(ctx, fmt):
    nt = _nt()
    be = synth.BLOCK_ELEMS[fmt]
    rows, cols = 37, 8 * be
    W = synth.quant_matrix(fmt, rows, cols, seed=1, stream=fmt)
    out = torch.empty(rows * cols, dtype=torch.float32, device="cuda")
    nt.nt_dequant_rows(ctx, fmt, dev(W), 0, rows, cols, out)
    torch.cuda.synchronize()
    ref = oracle.dequant(fmt, W, rows, cols)
    assert np.array_equal(host(out).view(np.uint32), ref.ravel().view(np.uint32))
    # a row range in the middle
    out2 = torch.empty(5 * cols, dtype=torch.float32, device="cuda")
    nt.nt_dequant_rows(ctx, fmt, dev(W), 11, 5, cols, out2)
    torch.cuda.synchronize()
    assert np.array_equal(host(out2).view(np.uint32), ref[11:16].ravel().view(np.uint32))


SHAPES = [(1, None), (7, 256), (333, 4096), (1027, 8192), (64, 28672), (130, 14336), (5, 2048)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_gemv_parity(ctx, fmt, rows, cols):
    nt = _nt()
    cols = cols or synth.BLOCK_ELEMS[fmt]
    W, x, Wd, xd = _case(fmt, rows, cols)
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    nt.nt_gemv_q(ctx, fmt, Wd, xd, y, rows, cols)
    torch.cuda.synchronize()
    ref = oracle.gemv(fmt, W, x.astype(np.float64), rows, cols)
    e = rel_l2(host(y), ref)
    print(f"{synth.FMT_NAMES[fmt]} {rows}x{cols} rel_l2={e:.2e}")
    assert e <= TOL


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_unaligned_path(ctx, fmt):
    """W starting 2 bytes past a 16-byte boundary takes the plain-load path."""
    nt = _nt()
    rows, cols = 45, 2048
    W, x, Wd, xd = _case(fmt, rows, cols, seed=2, offset=2)
    assert Wd.data_ptr() % 16 == 2
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    nt.nt_gemv_q(ctx, fmt, Wd, xd, y, rows, cols)
    torch.cuda.synchronize()
    assert rel_l2(host(y), oracle.gemv(fmt, W, x.astype(np.float64), rows, cols)) <= TOL


@pytest.mark.parametrize("fmt,cols", [(synth.Q8_0, 96), (synth.Q4_0, 160), (synth.Q6_K, 768)])
def test_gemv_rows_not_multiple_of_16_bytes(ctx, fmt, cols):
    nt = _nt()
    rows = 19
    W, x, Wd, xd = _case(fmt, rows, cols, seed=3)
    assert (cols // synth.BLOCK_ELEMS[fmt] * synth.BLOCK_BYTES[fmt]) % 16 != 0
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    nt.nt_gemv_q(ctx, fmt, Wd, xd, y, rows, cols)
    torch.cuda.synchronize()
    assert rel_l2(host(y), oracle.gemv(fmt, W, x.astype(np.float64), rows, cols)) <= TOL


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_residual_and_multi_with_norm(ctx, fmt):
    nt = _nt()
    cols = 4096
    rows = [300, 77, 129]
    Ws = [synth.quant_matrix(fmt, r, cols, seed=4, stream=10 + i) for i, r in enumerate(rows)]
    x = synth.normal_f32(cols, seed=4, stream=20) * 30
    g = synth.normal_f32(cols, seed=4, stream=21, mean=1.0, std=0.02)
    res = [synth.normal_f32(r, seed=4, stream=30 + i) for i, r in enumerate(rows)]
    ys = [dev(r.copy()) for r in res]
    nt.nt_gemv_q_multi(ctx, fmt, [(dev(W), y, y, r) for W, y, r in zip(Ws, ys, rows)], dev(x), cols,
                       norm_g=dev(g), eps=1e-5)
    torch.cuda.synchronize()
    xn = oracle.rmsnorm(x.astype(np.float64), g, 1e-5)
    for W, y, r, rr in zip(Ws, ys, rows, res):
        ref = oracle.gemv(fmt, W, xn, r, cols, residual=rr.astype(np.float64))
        assert rel_l2(host(y), ref) <= TOL


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,cols,norm", [(333, 4096, False), (1, 256, False), (96, 28672, False),
                                            (1001, 4096, True)])
def test_gemv_swiglu(ctx, fmt, rows, cols, norm):
    nt = _nt()
    Wg = synth.quant_matrix(fmt, rows, cols, seed=5, stream=1)
    Wu = synth.quant_matrix(fmt, rows, cols, seed=5, stream=2)
    x = synth.normal_f32(cols, seed=5, stream=3) * 0.05
    g = synth.normal_f32(cols, seed=5, stream=4, mean=1.0, std=0.02)
    h = torch.empty(rows, dtype=torch.float32, device="cuda")
    nt.nt_gemv_q_swiglu(ctx, fmt, dev(Wg), dev(Wu), dev(x), h, rows, cols, norm_g=dev(g) if norm else None, eps=1e-5)
    torch.cuda.synchronize()
    xin = oracle.rmsnorm(x.astype(np.float64), g, 1e-5) if norm else x.astype(np.float64)
    gg = oracle.gemv(fmt, Wg, xin, rows, cols)
    u = oracle.gemv(fmt, Wu, xin, rows, cols)
    assert rel_l2(host(h), oracle.swiglu(gg, u)) <= TOL


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,cols", [(8192, 8192), (28672, 8192), (8192, 28672), (1024, 8192)])
def test_gemv_sweep_shapes_full(ctx, fmt, rows, cols):
    """The format-sweep workload shapes, every row checked against the oracle."""
    nt = _nt()
    W, x, Wd, xd = _case(fmt, rows, cols, seed=100 + fmt)
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    nt.nt_gemv_q(ctx, fmt, Wd, xd, y, rows, cols)
    torch.cuda.synchronize()
    e = rel_l2(host(y), oracle.gemv(fmt, W, x.astype(np.float64), rows, cols))
    print(f"{synth.FMT_NAMES[fmt]} {rows}x{cols} rel_l2={e:.2e}")
    assert e <= TOL


def test_gemv_q8_0_4096_config(ctx):
    """Q8_0 4096 x 4096, seed 0: every output against the oracle."""
    nt = _nt()
    W = synth.quant_matrix(synth.Q8_0, 4096, 4096, seed=0, stream=0)
    x = synth.normal_f32(4096, seed=0, stream=1)
    y = torch.empty(4096, dtype=torch.float32, device="cuda")
    nt.nt_gemv_q(ctx, synth.Q8_0, dev(W), dev(x), y, 4096, 4096)
    torch.cuda.synchronize()
    assert rel_l2(host(y), oracle.gemv(synth.Q8_0, W, x.astype(np.float64), 4096, 4096)) <= TOL


def test_gemv_empty_and_bad_args(ctx):
    nt = _nt()
    x = torch.zeros(256, dtype=torch.float32, device="cuda")
    y = torch.zeros(4, dtype=torch.float32, device="cuda")
    W = torch.zeros(4 * 34 * 8, dtype=torch.uint8, device="cuda")
    nt.nt_gemv_q(ctx, synth.Q8_0, W, x, y, 0, 256)              # rows = 0: nothing to do
    for fmt, cols, code in [(7, 256, nt.NT_ERR_UNSUPPORTED_FMT), (synth.Q8_0, 40, nt.NT_ERR_INVALID_ARG),
                            (synth.Q4_K, 128, nt.NT_ERR_INVALID_ARG)]:
        with pytest.raises(nt.NtError) as ei:
            nt.nt_gemv_q(ctx, fmt, W, x, y, 4, cols)
        assert ei.value.status == code
    with pytest.raises(nt.NtError) as ei:
        nt.nt_gemv_q(ctx, synth.Q8_0, W, x[1:], y, 4, 32)        # x not 16-byte aligned
    assert ei.value.status == nt.NT_ERR_ALIGNMENT
    with pytest.raises(nt.NtError) as ei:
        nt.nt_gemv_q(ctx, synth.Q8_0, W[1:], x, y, 4, 32)        # odd weight pointer
    assert ei.value.status == nt.NT_ERR_ALIGNMENT
    ctx.sync()
