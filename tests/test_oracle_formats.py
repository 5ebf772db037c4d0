"""Pins for the oracle's block formats and GEMV (CPU only).

Each check ties the oracle to something other than itself: hand-packed golden
blocks (tests/golden/blocks.json, fields chosen by hand, values from the
closed forms), K-quant blocks packed from random fields by the same golden
encoder, IEEE binary16 as implemented by numpy, the sizes the pages print, and
brute force / special cases of the dot product.
"""
import os

import numpy as np
import pytest

import oracle
import synth

FMTS = {"Q8_0": 0, "Q4_0": 1, "Q4_K": 2, "Q5_K": 3, "Q6_K": 4}


# --- binary16 -------------------------------------------------------------
def test_half_decode_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_float_to_half_rne_matches_numpy():
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(100.0),
        (rng.standard_normal(5000) * 1e-5).astype(np.float32),          # subnormal halves
        np.array([65504, 65519.99, 65520, -65520, 1e-8, 2 ** -25, 2 ** -24, 3 * 2 ** -25,
                  1 + 2 ** -11, 1 + 3 * 2 ** -11, 0.0, -0.0], dtype=np.float32),  # ties and edges
    ])
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)


# --- block layouts --------------------------------------------------------
@pytest.mark.parametrize("name,elems,nbytes", [("Q8_0", 32, 34), ("Q4_0", 32, 18), ("Q4_K", 256, 144),
                                               ("Q5_K", 256, 176), ("Q6_K", 256, 210), ("F16", 32, 64),
                                               ("F32", 32, 128)])
def test_block_geometry(name, elems, nbytes):
    fmt = FMTS.get(name, {"F16": 5, "F32": 6}.get(name))
    assert oracle.block_elems(fmt) == elems
    assert oracle.block_bytes(fmt) == nbytes


# --- the float formats ("Ntransformer" (en.unwiki.net), About: F16, F32) -----
def test_f16_rows_decode_like_numpy():
    """F16 weights are IEEE binary16 values, row-major: numpy's float16 view of
    the same bytes (every bit pattern but NaN) is the reference."""
    bits = np.arange(65536, dtype=np.uint16)
    bits = bits[~np.isnan(bits.view(np.float16))]
    n = len(bits) // 32 * 32
    W = bits[:n].view(np.uint8).reshape(n // 32, 64)
    got = oracle.dequant(5, W, n // 32, 32)
    ref = bits[:n].view(np.float16).astype(np.float32).reshape(n // 32, 32)
    assert np.array_equal(got, ref)


def test_f32_rows_are_the_bytes():
    x = synth.normal_f32(4 * 96, seed=9, stream=9)
    got = oracle.dequant(6, x.view(np.uint8).reshape(4, 96 * 4), 4, 96)
    assert np.array_equal(got, x.reshape(4, 96))


@pytest.mark.parametrize("fmt", [5, 6])
def test_float_format_gemv_is_plain_matvec(fmt):
    """y = W x with W the float matrix itself (numpy fp64 matvec, same column order)."""
    rows, cols = 9, 160
    W = synth.quant_matrix(fmt, rows, cols, seed=5, stream=fmt)
    x = synth.normal_f32(cols, seed=5, stream=50).astype(np.float64)
    dense = (W.view(np.float16) if fmt == 5 else W.view(np.float32)).astype(np.float64).reshape(rows, cols)
    y = oracle.gemv(fmt, W, x, rows, cols)
    assert np.allclose(y, dense @ x, rtol=1e-13, atol=1e-15)


def test_float_format_generator_statistics():
    """The generator's plain weights are N(0, scale^2): mean and std within a
    few standard errors at 64k samples."""
    for fmt, view in ((5, np.float16), (6, np.float32)):
        W = synth.quant_matrix(fmt, 256, 256, seed=11, stream=1, scale_std=0.5)
        v = W.view(view).astype(np.float64).ravel()
        assert abs(v.mean()) < 4 * 0.5 / np.sqrt(v.size)
        assert abs(v.std() - 0.5) < 0.01


def test_q6_k_layer_size_matches_page():
    """ "Ntransformer" (en.unwiki.net), NVMe direct section: a 70B Q6_K layer is about 670 MB."""
    d, f, kv = 8192, 28672, 1024
    weights = 2 * d * d + 2 * kv * d + 3 * f * d
    nbytes = weights // oracle.block_elems(4) * oracle.block_bytes(4)
    assert nbytes == 701_890_560
    assert abs(nbytes / 2 ** 20 - 670) < 1.0          # 669.4 MiB


@pytest.mark.parametrize("name", list(FMTS))
def test_golden_block_quants_and_values(golden_blocks, name):
    g = golden_blocks[name]
    fmt = FMTS[name]
    raw = bytes.fromhex(g["hex"])
    assert len(raw) == oracle.block_bytes(fmt)
    q = oracle.quants(fmt, raw)
    assert list(q) == g["q"]
    vals = oracle.dequant(fmt, np.frombuffer(raw, np.uint8), 1, oracle.block_elems(fmt))[0]
    assert np.array_equal(vals.astype(np.float64), np.array(g["values"], dtype=np.float64))


@pytest.mark.parametrize("name", ["Q4_K", "Q5_K"])
def test_golden_kquant_scale_min(golden_blocks, name):
    g = golden_blocks[name]
    raw = bytes.fromhex(g["hex"])
    for j in range(8):
        assert oracle.kquant_scale_min(raw[4:16], j) == (g["sc"][j], g["m"][j])


def test_closed_forms_on_random_blocks():
    """Q8_0 = d*q and Q4_0 = d*(q-8) exactly, for random blocks: recompute from the bytes with numpy."""
    for fmt, off in ((0, 0), (1, 8)):
        W = synth.quant_matrix(fmt, 64, 256, seed=5, stream=3)
        deq = oracle.dequant(fmt, W, 64, 256)
        blocks = W.reshape(-1, oracle.block_bytes(fmt))
        d = blocks[:, :2].copy().view(np.float16).astype(np.float32).ravel()
        if fmt == 0:
            q = blocks[:, 2:].view(np.int8).astype(np.float32)
        else:
            qs = blocks[:, 2:]
            q = np.concatenate([qs & 15, qs >> 4], axis=1).astype(np.float32) - off
        ref = (d[:, None] * q).reshape(64, 256)
        assert np.array_equal(deq, ref)


def test_kquant_value_ranges_random():
    """sc, m in 0..63 and 4/5/6-bit quants stay in range for arbitrary bytes."""
    raw = synth.random_bytes(176 * 50, seed=9, stream=1)
    for b in range(50):
        blk = raw[176 * b:176 * (b + 1)].tobytes()
        for j in range(8):
            sc, m = oracle.kquant_scale_min(blk[4:16], j)
            assert 0 <= sc < 64 and 0 <= m < 64
        assert oracle.quants(3, blk).max() < 32
        assert oracle.quants(2, blk[:144]).max() < 16
        assert oracle.quants(4, blk[:210]).max() < 64


def test_kquant_scale_bits_are_a_bijection():
    """The 96 bits of scales[12] carry the 8 (sc, m) pairs exactly once: flipping any
    single bit changes exactly one of the 16 six-bit fields."""
    base = bytes(12)
    f0 = [oracle.kquant_scale_min(base, j) for j in range(8)]
    seen = set()
    for byte in range(12):
        for bit in range(8):
            s = bytearray(base)
            s[byte] ^= 1 << bit
            f = [oracle.kquant_scale_min(bytes(s), j) for j in range(8)]
            diff = [(j, k) for j in range(8) for k in range(2) if f[j][k] != f0[j][k]]
            assert len(diff) == 1
            j, k = diff[0]
            delta = f[j][k] - f0[j][k]
            assert delta > 0 and (delta & (delta - 1)) == 0
            seen.add((j, k, delta))
    assert len(seen) == 96


# --- GEMV -----------------------------------------------------------------
@pytest.mark.parametrize("fmt", range(7))
def test_gemv_brute_force_small(fmt):
    be = oracle.block_elems(fmt)
    rows, cols = 5, 2 * be
    W = synth.quant_matrix(fmt, rows, cols, seed=3, stream=fmt)
    x = synth.normal_f32(cols, seed=3, stream=100 + fmt)
    y = oracle.gemv(fmt, W, x, rows, cols)
    dense = oracle.dequant(fmt, W, rows, cols).astype(np.float64)
    ref = np.array([sum(float(dense[r, c]) * float(x[c]) for c in range(cols)) for r in range(rows)])
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("fmt", range(7))
def test_gemv_one_hot_returns_column(fmt):
    be = oracle.block_elems(fmt)
    rows, cols = 7, 3 * be
    W = synth.quant_matrix(fmt, rows, cols, seed=4, stream=fmt)
    dense = oracle.dequant(fmt, W, rows, cols)
    for k in (0, 1, be - 1, be, cols - 1):
        e = np.zeros(cols)
        e[k] = 1.0
        assert np.array_equal(oracle.gemv(fmt, W, e, rows, cols), dense[:, k].astype(np.float64))


def test_gemv_all_ones_is_sum():
    """Q8_0 blocks with d = 1 and q = 1 everywhere: y[r] = sum(x)."""
    rows, cols = 3, 96
    blk = bytes([0x00, 0x3C]) + bytes([1] * 32)
    W = np.frombuffer(blk * (rows * cols // 32), np.uint8).copy()
    x = synth.normal_f32(cols, seed=1, stream=1).astype(np.float64)
    y = oracle.gemv(0, W, x, rows, cols)
    assert np.allclose(y, np.sum(x), rtol=1e-14)


def test_gemv_residual_added():
    W = synth.quant_matrix(0, 4, 64, seed=2, stream=2)
    x = synth.normal_f32(64, seed=2, stream=3)
    r = np.arange(4, dtype=np.float64)
    assert np.allclose(oracle.gemv(0, W, x, 4, 64, residual=r) - oracle.gemv(0, W, x, 4, 64), r, atol=1e-9)


def test_gemv_rejects_ragged_cols():
    W = np.zeros(34 * 4, np.uint8)
    with pytest.raises(ValueError):
        oracle.gemv(0, W, np.zeros(40), 4, 40)


def _golden_packers():
    import importlib.util
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "make_golden.py")
    spec = importlib.util.spec_from_file_location("make_golden", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _f16(bits):
    return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_kquant_random_fields_roundtrip(fmt):
    """K-quant blocks packed from random fields by the golden encoder (its own
    code, written from the GGUF layout) decode in the oracle to those fields
    and to the closed forms: d*sc*q - dmin*m (Q4_K, Q5_K), d*sc*(q-32)
    (Q6_K), each the fp32 rounding of the exact value.  d and dmin are
    normal f16 values of either sign in [2^-10, 2^5), so the exact value fits
    an fp64."""
    mg = _golden_packers()
    rng = np.random.default_rng(20 + fmt)
    for _ in range(60):
        def rand_half():
            return int(rng.integers(0, 2)) << 15 | int(rng.integers(5, 20)) << 10 | int(rng.integers(0, 1024))
        d_bits, dmin_bits = rand_half(), rand_half()
        d, dmin = _f16(d_bits), _f16(dmin_bits)
        if fmt == 4:
            sc = [int(v) for v in rng.integers(-128, 128, 16)]
            q = [int(v) for v in rng.integers(0, 64, 256)]
            raw = bytes(mg.pack_q6_k(d_bits, sc, q))
            exact = [d * sc[(i // 128) * 8 + (i % 128) // 16] * (q[i] - 32) for i in range(256)]
        else:
            sc = [int(v) for v in rng.integers(0, 64, 8)]
            mn = [int(v) for v in rng.integers(0, 64, 8)]
            q = [int(v) for v in rng.integers(0, 16 if fmt == 2 else 32, 256)]
            raw = bytes((mg.pack_q4_k if fmt == 2 else mg.pack_q5_k)(d_bits, dmin_bits, sc, mn, q))
            for j in range(8):
                assert oracle.kquant_scale_min(raw[4:16], j) == (sc[j], mn[j])
            exact = [d * sc[i // 32] * q[i] - dmin * mn[i // 32] for i in range(256)]
        assert len(raw) == oracle.block_bytes(fmt)
        assert list(oracle.quants(fmt, raw)) == q
        got = oracle.dequant(fmt, np.frombuffer(raw, np.uint8), 1, 256)[0]
        assert np.array_equal(got, np.array(exact, dtype=np.float64).astype(np.float32))
