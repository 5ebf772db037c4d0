"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws numbers (see ``synth.c``): block bytes with random
fields, fp32/f16 normal arrays, and the descriptions of the synthetic Llama
workloads (shapes, per-tensor formats, seeds).  It holds none of the method's
arithmetic, so importing it couples neither side to the other.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libsynth.so")

# format ids (same numbering as the public C ABI's nt_fmt)
Q8_0, Q4_0, Q4_K, Q5_K, Q6_K, F16, F32 = 0, 1, 2, 3, 4, 5, 6
FMT_NAMES = {Q8_0: "Q8_0", Q4_0: "Q4_0", Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K", F16: "F16", F32: "F32"}
FMT_BY_NAME = {v: k for k, v in FMT_NAMES.items()}
# F16 / F32 rows are plain arrays, handled in units of 32 values
BLOCK_ELEMS = {Q8_0: 32, Q4_0: 32, Q4_K: 256, Q5_K: 256, Q6_K: 256, F16: 32, F32: 32}
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18, Q4_K: 144, Q5_K: 176, Q6_K: 210, F16: 64, F32: 128}


def build(force: bool = False) -> str:
    """Compile synth.c into a shared library beside this file."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        _lib.sy_fill_quant.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_uint64, ctypes.c_uint32, ctypes.c_double]
        _lib.sy_fill_quant.restype = ctypes.c_int
        _lib.sy_fill_normal_f32.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_double,
                                            ctypes.c_uint64, ctypes.c_uint32]
        _lib.sy_fill_normal_f16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_double,
                                            ctypes.c_uint64, ctypes.c_uint32]
        _lib.sy_fill_bytes.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32]
        _lib.sy_num_threads.restype = ctypes.c_int
        del u8p
    return _lib


def row_bytes(fmt: int, cols: int) -> int:
    return (cols // BLOCK_ELEMS[fmt]) * BLOCK_BYTES[fmt]


def quant_matrix(fmt: int, rows: int, cols: int, seed: int, stream: int, scale_std: float = 0.02,
                 out: np.ndarray | None = None) -> np.ndarray:
    """rows x cols block-quantized matrix as raw bytes, shape [rows, row_bytes].
    Block scales are f16(|N(0,1)| * scale_std); F16 / F32 weights are plain
    N(0, scale_std^2) values."""
    if cols % BLOCK_ELEMS[fmt]:
        raise ValueError("cols must be a multiple of the block size")
    rb = row_bytes(fmt, cols)
    if out is None:
        out = np.empty((rows, rb), dtype=np.uint8)
    assert out.nbytes == rows * rb and out.flags.c_contiguous
    rc = lib().sy_fill_quant(fmt, out.ctypes.data, rows, cols, seed, stream, scale_std)
    if rc != 0:
        raise ValueError("sy_fill_quant failed")
    return out


def normal_f32(n: int, seed: int, stream: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().sy_fill_normal_f32(out.ctypes.data, n, mean, std, seed, stream)
    return out


def normal_f16(n: int, seed: int, stream: int, std: float = 1.0) -> np.ndarray:
    """binary16 values as np.float16 (bit patterns written by synth.c)."""
    out = np.empty(n, dtype=np.uint16)
    lib().sy_fill_normal_f16(out.ctypes.data, n, std, seed, stream)
    return out.view(np.float16)


def random_bytes(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    lib().sy_fill_bytes(out.ctypes.data, n, seed, stream)
    return out


# ---------------------------------------------------------------------------
# Synthetic Llama workloads.  Shapes follow the Llama-3.1 8B / 70B geometry;
# weights are random (no trained checkpoint exists here).
# ---------------------------------------------------------------------------
LAYER_TENSORS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


@dataclass
class ModelSpec:
    name: str
    n_layers: int
    d_model: int
    n_qh: int
    n_kvh: int
    head_dim: int
    ffn: int
    vocab: int
    eps: float
    theta: float
    seed: int
    n_prefill: int            # positions of N(0,1) KV already in the cache
    n_gen: int                # tokens the workload decodes
    fmt: dict = field(default_factory=dict)   # per-tensor format (LAYER_TENSORS + "embd", "out")
    n_resident: int = -1      # layers kept in HBM (-1: all)
    first_token: int = 1

    def tensor_fmt(self, name: str) -> int:
        return self.fmt[name]

    def tensor_shape(self, name: str) -> tuple[int, int]:
        d, hd = self.d_model, self.head_dim
        return {
            "wq": (self.n_qh * hd, d), "wk": (self.n_kvh * hd, d), "wv": (self.n_kvh * hd, d),
            "wo": (d, self.n_qh * hd), "wg": (self.ffn, d), "wu": (self.ffn, d), "wd": (d, self.ffn),
            "embd": (self.vocab, d), "out": (self.vocab, d),
        }[name]

    # stream ids: every tensor gets its own counter space
    @staticmethod
    def stream_of(name: str, layer: int = -1) -> int:
        glob = {"embd": 1, "out": 2, "out_norm": 3}
        if layer < 0:
            return glob[name]
        per = {n: i for i, n in enumerate(LAYER_TENSORS + ("attn_norm", "ffn_norm"))}
        if name in ("kprefill", "vprefill"):
            return 8192 + 2 * layer + (name == "vprefill")
        return 16 + 16 * layer + per[name]

    @property
    def kv_cap(self) -> int:
        # room for the prefill, the generated tokens and a speculative window
        return self.n_prefill + self.n_gen + 8

    def layer_bytes(self) -> int:
        return sum(self.tensor_shape(t)[0] * row_bytes(self.fmt[t], self.tensor_shape(t)[1])
                   for t in LAYER_TENSORS)

    def weight_bytes(self) -> int:
        tot = self.n_layers * self.layer_bytes()
        r, c = self.tensor_shape("out")
        tot += r * row_bytes(self.fmt["out"], c)
        return tot


def _uniform_fmt(f: int) -> dict:
    return {t: f for t in LAYER_TENSORS + ("embd", "out")}


def _q4_k_m() -> dict:
    m = _uniform_fmt(Q4_K)
    m["wv"] = Q6_K
    m["wd"] = Q6_K
    return m


def model_spec(name: str) -> ModelSpec:
    # "<tiny_* or small_*>_r<N>": the same model with only layers 0..N-1 resident
    base, sep, tail = name.rpartition("_r")
    if sep and tail.isdigit() and (base.startswith("tiny_") or base.startswith("small_")):
        spec = model_spec(base)
        spec.name, spec.n_resident = name, int(tail)
        return spec
    if name == "llama8b_q8_0":
        return ModelSpec(name, 32, 4096, 32, 8, 128, 14336, 128256, 1e-5, 500000.0, seed=1,
                         n_prefill=1024, n_gen=128, fmt=_uniform_fmt(Q8_0))
    if name == "llama8b_q8_0_streamed":
        # the 8B workload's weights (same seed) with layers 16..31 streamed from host memory
        return ModelSpec(name, 32, 4096, 32, 8, 128, 14336, 128256, 1e-5, 500000.0, seed=1,
                         n_prefill=1024, n_gen=128, fmt=_uniform_fmt(Q8_0), n_resident=16)
    if name == "llama70b_q4_k_m":
        return ModelSpec(name, 80, 8192, 64, 8, 128, 28672, 128256, 1e-5, 500000.0, seed=2,
                         n_prefill=4096, n_gen=64, fmt=_q4_k_m())
    if name == "llama70b_q6_k_streamed":
        return ModelSpec(name, 80, 8192, 64, 8, 128, 28672, 128256, 1e-5, 500000.0, seed=3,
                         n_prefill=4096, n_gen=32, fmt=_uniform_fmt(Q6_K), n_resident=26)
    # small models with the same structure, for parity tests the oracle finishes in seconds
    if name.startswith("tiny_"):
        f = FMT_BY_NAME[name[5:].upper()] if name[5:].upper() in FMT_BY_NAME else None
        fm = _q4_k_m() if name == "tiny_q4_k_m" else _uniform_fmt(f)
        return ModelSpec(name, 3, 512, 8, 2, 128, 768, 1000, 1e-5, 500000.0, seed=7,
                         n_prefill=37, n_gen=32, fmt=fm)
    if name.startswith("small_"):
        f = FMT_BY_NAME[name[6:].upper()] if name[6:].upper() in FMT_BY_NAME else None
        fm = _q4_k_m() if name == "small_q4_k_m" else _uniform_fmt(f)
        return ModelSpec(name, 4, 2048, 16, 4, 128, 6144, 32000, 1e-5, 500000.0, seed=11,
                         n_prefill=300, n_gen=32, fmt=fm)
    raise KeyError(name)


@dataclass
class HostModel:
    """All bytes of a synthetic model in host memory (numpy)."""
    spec: ModelSpec
    layers: list            # list of dict name -> ndarray
    embd: np.ndarray
    out: np.ndarray
    out_norm: np.ndarray
    kcache: np.ndarray      # float16 [L, kvh, cap, hd]
    vcache: np.ndarray


def make_host_model(spec: ModelSpec, layers: range | None = None, with_kv: bool = True,
                    out_view=None) -> HostModel:
    """out_view(layer, name) may return a preallocated uint8 array [rows,
    row_bytes] to generate a weight matrix into (layer -1 for "embd"/"out"),
    or None for a fresh array."""
    s = spec.seed
    Ls = range(spec.n_layers) if layers is None else layers
    dst = (lambda li, t: None) if out_view is None else out_view
    lay = []
    for li in Ls:
        d = {}
        for t in LAYER_TENSORS:
            r, c = spec.tensor_shape(t)
            d[t] = quant_matrix(spec.fmt[t], r, c, s, spec.stream_of(t, li), out=dst(li, t))
        d["attn_norm"] = normal_f32(spec.d_model, s, spec.stream_of("attn_norm", li), 1.0, 0.02)
        d["ffn_norm"] = normal_f32(spec.d_model, s, spec.stream_of("ffn_norm", li), 1.0, 0.02)
        lay.append(d)
    r, c = spec.tensor_shape("embd")
    embd = quant_matrix(spec.fmt["embd"], r, c, s, spec.stream_of("embd"), out=dst(-1, "embd"))
    out = quant_matrix(spec.fmt["out"], r, c, s, spec.stream_of("out"), out=dst(-1, "out"))
    out_norm = normal_f32(spec.d_model, s, spec.stream_of("out_norm"), 1.0, 0.02)
    if with_kv:
        kc, vc = make_kv_cache(spec)
    else:
        kc = vc = None
    return HostModel(spec, lay, embd, out, out_norm, kc, vc)


def make_kv_cache(spec: ModelSpec, n_layers: int | None = None):
    L = spec.n_layers if n_layers is None else n_layers
    shape = (L, spec.n_kvh, spec.kv_cap, spec.head_dim)
    kc = np.zeros(shape, dtype=np.float16)
    vc = np.zeros(shape, dtype=np.float16)
    P = spec.n_prefill
    n = spec.n_kvh * P * spec.head_dim
    for li in range(L):
        kc[li, :, :P, :] = normal_f16(n, spec.seed, spec.stream_of("kprefill", li)).reshape(spec.n_kvh, P, -1)
        vc[li, :, :P, :] = normal_f16(n, spec.seed, spec.stream_of("vprefill", li)).reshape(spec.n_kvh, P, -1)
    return kc, vc
