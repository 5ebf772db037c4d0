"""CPU oracle for the block-quantized decode path — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (``block_quantized_gemv_nt_gb300``)
never imports it and shares no code with it.

``oracle.c`` holds the arithmetic (fp64, plain loops, one function per step,
each citing the page passage it follows); this file is ctypes marshalling.
Every function here is pinned by ``tests/test_oracle_*.py`` against closed
forms, hand-worked golden blocks, brute force and invariants.  Parity of the
whole decode step composes the pinned pieces and is otherwise pinned only by
itself (see the design notes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

Q8_0, Q4_0, Q4_K, Q5_K, Q6_K, F16, F32 = 0, 1, 2, 3, 4, 5, 6


def build(force: bool = False) -> str:
    """Compile oracle.c (plain C, OpenMP over rows only, no FMA contraction)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


class _QT(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("w", ctypes.c_void_p)]


class _Layer(ctypes.Structure):
    _fields_ = [(n, _QT) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd")] + [
        ("attn_norm", ctypes.c_void_p), ("ffn_norm", ctypes.c_void_p)]


class _Model(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_qh", ctypes.c_int),
                ("n_kvh", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("eps", ctypes.c_double), ("theta", ctypes.c_double),
                ("kv_cap", ctypes.c_int64), ("embd", _QT), ("out", _QT), ("out_norm", ctypes.c_void_p),
                ("layers", ctypes.POINTER(_Layer)), ("kcache", ctypes.c_void_p), ("vcache", ctypes.c_void_p)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        vp, i64, ci, cd = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.or_block_elems.argtypes = [ci]
        L.or_block_bytes.argtypes = [ci]
        L.or_half_to_double.argtypes = [ctypes.c_uint16]
        L.or_half_to_double.restype = cd
        L.or_float_to_half.argtypes = [ctypes.c_float]
        L.or_float_to_half.restype = ctypes.c_uint16
        L.or_kquant_scale_min.argtypes = [vp, ci, ctypes.POINTER(ci), ctypes.POINTER(ci)]
        L.or_quant_of.argtypes = [ci, vp, ci]
        L.or_dequant_block.argtypes = [ci, vp, vp]
        L.or_dequant_rows.argtypes = [ci, vp, i64, i64, i64, vp]
        L.or_gemv.argtypes = [ci, vp, vp, vp, i64, i64, vp]
        L.or_rmsnorm.argtypes = [vp, vp, i64, cd, vp]
        L.or_rope.argtypes = [vp, ci, ci, i64, cd]
        L.or_softmax.argtypes = [vp, i64]
        L.or_attn_decode.argtypes = [vp, vp, vp, vp, ci, ci, ci, i64, i64]
        L.or_silu.argtypes = [cd]
        L.or_silu.restype = cd
        L.or_swiglu.argtypes = [vp, vp, vp, i64]
        L.or_argmax.argtypes = [vp, i64]
        L.or_argmax.restype = i64
        L.or_cos_sim.argtypes = [vp, vp, i64]
        L.or_cos_sim.restype = cd
        L.or_layer_skip_select.argtypes = [vp, ci, ci, vp]
        L.or_decode_step.argtypes = [ctypes.POINTER(_Model), ctypes.c_int32, i64, vp, vp, vp]
        L.or_set_num_threads.argtypes = [ci]
        L.or_splitmix64.argtypes = [ctypes.c_uint64]
        L.or_splitmix64.restype = ctypes.c_uint64
        L.or_sample_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.or_sample_uniform.restype = ctypes.c_double
        L.or_sample.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                ctypes.POINTER(ctypes.c_int64)]
        L.or_sample.restype = ctypes.c_int64
        u64, u32 = ctypes.c_uint64, ctypes.c_uint32
        L.or_sample_weights.argtypes = [vp, i64, cd, cd, vp]
        L.or_sample_weights.restype = u64
        L.or_spec_uniforms.argtypes = [u64, u64, ctypes.POINTER(u32), ctypes.POINTER(u32)]
        L.or_spec_accept.argtypes = [u64, u64, u64, u64, u32]
        L.or_spec_accept.restype = ci
        L.or_spec_residual.argtypes = [vp, u64, vp, u64, i64, u32]
        L.or_spec_residual.restype = i64
        _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def block_elems(fmt: int) -> int:
    return lib().or_block_elems(fmt)


def block_bytes(fmt: int) -> int:
    return lib().or_block_bytes(fmt)


def half_to_double(bits: int) -> float:
    return lib().or_half_to_double(bits)


def float_to_half(x: float) -> int:
    return lib().or_float_to_half(x)


def kquant_scale_min(scales12: bytes, j: int) -> tuple[int, int]:
    buf = (ctypes.c_uint8 * 12).from_buffer_copy(bytes(scales12))
    sc, m = ctypes.c_int(), ctypes.c_int()
    lib().or_kquant_scale_min(ctypes.addressof(buf), j, ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def quants(fmt: int, block: bytes) -> np.ndarray:
    """Integer quant of every element of one block."""
    buf = (ctypes.c_uint8 * len(block)).from_buffer_copy(bytes(block))
    n = block_elems(fmt)
    return np.array([lib().or_quant_of(fmt, ctypes.addressof(buf), i) for i in range(n)], dtype=np.int64)


def dequant(fmt: int, W: np.ndarray, rows: int, cols: int, row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """fp32 dequantised rows [row0, row0+nrows) of a rows x cols block matrix."""
    nrows = rows - row0 if nrows is None else nrows
    W, wp = _c(W, np.uint8)
    out = np.empty((nrows, cols), dtype=np.float32)
    if lib().or_dequant_rows(fmt, wp, row0, nrows, cols, out.ctypes.data):
        raise ValueError("bad format or cols")
    return out


def gemv(fmt: int, W: np.ndarray, x: np.ndarray, rows: int, cols: int, residual=None) -> np.ndarray:
    """fp64 y = W x (+ residual)."""
    W, wp = _c(W, np.uint8)
    x, xp = _c(x, np.float64)
    y = np.empty(rows, dtype=np.float64)
    rp = None
    if residual is not None:
        residual, rp = _c(residual, np.float64)
    if lib().or_gemv(fmt, wp, xp, y.ctypes.data, rows, cols, rp):
        raise ValueError("bad format or cols")
    return y


def rmsnorm(x, g, eps: float) -> np.ndarray:
    x, xp = _c(x, np.float64)
    g, gp = _c(g, np.float32)
    y = np.empty_like(x)
    lib().or_rmsnorm(xp, gp, x.size, eps, y.ctypes.data)
    return y


def rope(v, n_heads: int, head_dim: int, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, dtype=np.float64, copy=True).ravel()
    lib().or_rope(v.ctypes.data, n_heads, head_dim, pos, theta)
    return v


def softmax(s) -> np.ndarray:
    s = np.array(s, dtype=np.float64, copy=True).ravel()
    lib().or_softmax(s.ctypes.data, s.size)
    return s


def attn_decode(q, Kc, Vc, n_qh: int, n_kvh: int, head_dim: int, n_pos: int, kv_stride: int) -> np.ndarray:
    """Kc/Vc: float16 arrays [n_kvh, kv_stride, head_dim]."""
    q, qp = _c(q, np.float64)
    Kc, kp = _c(np.asarray(Kc, dtype=np.float16).view(np.uint16), np.uint16)
    Vc, vp_ = _c(np.asarray(Vc, dtype=np.float16).view(np.uint16), np.uint16)
    out = np.empty(n_qh * head_dim, dtype=np.float64)
    if lib().or_attn_decode(qp, kp, vp_, out.ctypes.data, n_qh, n_kvh, head_dim, n_pos, kv_stride):
        raise ValueError("bad attention arguments")
    return out


def silu(z: float) -> float:
    return lib().or_silu(z)


def swiglu(gate, up) -> np.ndarray:
    gate, gp = _c(gate, np.float64)
    up, upp = _c(up, np.float64)
    h = np.empty_like(gate)
    lib().or_swiglu(gp, upp, h.ctypes.data, gate.size)
    return h


def argmax(v) -> int:
    v, vp_ = _c(v, np.float64)
    return int(lib().or_argmax(vp_, v.size))


def splitmix64(z: int) -> int:
    return int(lib().or_splitmix64(ctypes.c_uint64(z & 0xFFFFFFFFFFFFFFFF)))


def sample_uniform(seed: int, counter: int) -> float:
    return float(lib().or_sample_uniform(ctypes.c_uint64(seed), ctypes.c_uint64(counter)))


def sample(logits, temperature: float, top_p: float, u: float):
    """Nucleus sample of fp32 logits with uniform u; returns (token, nucleus size)."""
    z = np.ascontiguousarray(np.asarray(logits, dtype=np.float32))
    k = ctypes.c_int64(0)
    t = int(lib().or_sample(z.ctypes.data, z.size, float(temperature), float(top_p), float(u), ctypes.byref(k)))
    if t < 0:
        raise RuntimeError("or_sample failed")
    return t, int(k.value)


def sample_weights(logits, temperature: float, top_p: float):
    """The sampler's distribution as integer weights: (w uint64 [n], W) with
    w[i] = token i's weight inside the nucleus, else 0, and W = sum w."""
    z = np.ascontiguousarray(np.asarray(logits, dtype=np.float32))
    w = np.zeros(z.size, dtype=np.uint64)
    W = int(lib().or_sample_weights(z.ctypes.data, z.size, float(temperature), float(top_p), w.ctypes.data))
    if W == 0:
        raise RuntimeError("or_sample_weights failed")
    return w, W


def spec_uniforms(seed: int, counter: int) -> tuple[int, int]:
    """The two 24-bit uniforms (k_acc, k_res) of speculative sampling at
    (seed, counter)."""
    a, r = ctypes.c_uint32(), ctypes.c_uint32()
    lib().or_spec_uniforms(ctypes.c_uint64(seed), ctypes.c_uint64(counter), ctypes.byref(a), ctypes.byref(r))
    return int(a.value), int(r.value)


def spec_accept(wq_d: int, Wq: int, wp_d: int, Wp: int, k_acc: int) -> bool:
    """Speculative sampling's acceptance test u < p(d) / q(d), u = k_acc / 2^24."""
    return bool(lib().or_spec_accept(wq_d, Wq, wp_d, Wp, k_acc))


def spec_residual(wp, Wp: int, wq, Wq: int, k_res: int) -> int:
    """Token drawn from max(0, p - q) with uniform k_res / 2^24 (-1: empty)."""
    wp = np.ascontiguousarray(wp, dtype=np.uint64)
    wq = np.ascontiguousarray(wq, dtype=np.uint64)
    return int(lib().or_spec_residual(wp.ctypes.data, Wp, wq.ctypes.data, Wq, wp.size, k_res))


def spec_sample(draft_logits, verify_logits, temperature: float, top_p: float, seed: int, pos: int):
    """Speculative sampling over one step, teacher-forced on given logits.

    draft_logits [k][vocab]: the draft model's logits at positions pos .. pos+k-1
    (row i is the distribution of draft token i + 1); verify_logits [k+1][vocab]:
    the target's at pos .. pos+k.  Draft i + 1 is the sampler's pick from row i
    with the sampler's uniform at counter pos + i.  Returns (tokens, drafts):
    the accepted drafts, then the residual draw at the first rejection or,
    with every draft accepted, the sampler's pick from the last target row
    (counter pos + k)."""
    k = len(draft_logits)
    drafts = [sample(draft_logits[i], temperature, top_p, sample_uniform(seed, pos + i))[0] for i in range(k)]
    out = []
    for i, d in enumerate(drafts):
        wq, Wq = sample_weights(draft_logits[i], temperature, top_p)
        wp, Wp = sample_weights(verify_logits[i], temperature, top_p)
        k_acc, k_res = spec_uniforms(seed, pos + i)
        if spec_accept(int(wq[d]), Wq, int(wp[d]), Wp, k_acc):
            out.append(d)
            continue
        out.append(spec_residual(wp, Wp, wq, Wq, k_res))
        return out, drafts
    out.append(sample(verify_logits[k], temperature, top_p, sample_uniform(seed, pos + k))[0])
    return out, drafts


def cos_sim(a, b) -> float:
    a, ap = _c(a, np.float64)
    b, bp = _c(b, np.float64)
    return float(lib().or_cos_sim(ap, bp, a.size))


def layer_skip_select(cos_l, n_skip: int) -> np.ndarray:
    cos_l, cp = _c(cos_l, np.float64)
    mask = np.zeros(cos_l.size, dtype=np.uint8)
    lib().or_layer_skip_select(cp, cos_l.size, n_skip, mask.ctypes.data)
    return mask


def set_num_threads(n: int) -> None:
    lib().or_set_num_threads(n)


def num_threads() -> int:
    return lib().or_num_threads()


class Model:
    """Oracle view of a model held in host numpy arrays (weights are only read;
    the oracle keeps its own copy of the KV cache and writes into it).

    ``spec`` needs n_layers, d_model, n_qh, n_kvh, head_dim, ffn, vocab, eps,
    theta, kv_cap and fmt; ``layers`` is a list of dicts with wq..wd byte
    arrays and attn_norm/ffn_norm fp32 arrays.
    """

    def __init__(self, spec, layers, embd, out, out_norm, kcache, vcache):
        self.spec = spec
        self._keep = [layers, embd, out, out_norm]
        self.kcache = np.array(kcache, dtype=np.float16, copy=True)
        self.vcache = np.array(vcache, dtype=np.float16, copy=True)
        L = len(layers)
        arr = (_Layer * L)()
        for i, ld in enumerate(layers):
            for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
                a = ld[n]
                assert a.flags.c_contiguous and a.dtype == np.uint8
                setattr(arr[i], n, _QT(spec.fmt[n], a.ctypes.data))
            for n in ("attn_norm", "ffn_norm"):
                a = ld[n]
                assert a.flags.c_contiguous and a.dtype == np.float32
                setattr(arr[i], n, a.ctypes.data)
        self._layers = arr
        m = _Model()
        m.n_layers, m.d_model, m.n_qh, m.n_kvh = L, spec.d_model, spec.n_qh, spec.n_kvh
        m.head_dim, m.ffn, m.vocab = spec.head_dim, spec.ffn, spec.vocab
        m.eps, m.theta, m.kv_cap = spec.eps, spec.theta, spec.kv_cap
        m.embd = _QT(spec.fmt["embd"], embd.ctypes.data)
        m.out = _QT(spec.fmt["out"], out.ctypes.data)
        m.out_norm = out_norm.ctypes.data
        m.layers = arr
        m.kcache = self.kcache.ctypes.data
        m.vcache = self.vcache.ctypes.data
        self._m = m

    def step(self, token: int, pos: int, skip=None, want_cos: bool = False):
        """One decode step; returns fp64 logits (and per-layer cos if asked)."""
        logits = np.empty(self.spec.vocab, dtype=np.float64)
        cos = np.full(self._m.n_layers, np.nan) if want_cos else None
        sp = None
        if skip is not None:
            skip = np.ascontiguousarray(skip, dtype=np.uint8)
            sp = skip.ctypes.data
        rc = lib().or_decode_step(ctypes.byref(self._m), token, pos, sp, logits.ctypes.data,
                                  cos.ctypes.data if cos is not None else None)
        if rc:
            raise RuntimeError(f"or_decode_step failed ({rc})")
        return (logits, cos) if want_cos else logits
