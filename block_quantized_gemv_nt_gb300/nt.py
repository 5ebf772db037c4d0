"""ctypes binding of libnt.so — argument marshalling only.

Every function keeps the C name from include/nt.h and takes torch tensors
(device pointers via ``data_ptr()``) or plain ints; the stream defaults to
torch's current stream on the tensor's device.  All computation runs in the
CUDA kernels of libnt.so; if the library cannot be loaded, importing this
module raises — there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

Q8_0, Q4_0, Q4_K, Q5_K, Q6_K, F16, F32 = 0, 1, 2, 3, 4, 5, 6
FMT_NAMES = {Q8_0: "Q8_0", Q4_0: "Q4_0", Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K", F16: "F16", F32: "F32"}

NT_OK, NT_ERR_INVALID_ARG, NT_ERR_UNSUPPORTED_FMT, NT_ERR_ALIGNMENT, NT_ERR_CUDA, NT_ERR_OOM, NT_ERR_TIMEOUT = range(7)
STATUS_NAMES = ["NT_OK", "NT_ERR_INVALID_ARG", "NT_ERR_UNSUPPORTED_FMT", "NT_ERR_ALIGNMENT", "NT_ERR_CUDA",
                "NT_ERR_OOM", "NT_ERR_TIMEOUT"]


class NtError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else status}: {msg}")
        self.status = status


def library_path() -> str:
    return _build.SO


def _load():
    path = _build.SO
    if not os.path.exists(path) or _build._stale():
        _build.build()
    return ctypes.CDLL(path)


_lib = _load()

_vp, _i64, _ci, _cf, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class nt_gemv_job(ctypes.Structure):
    _fields_ = [("W_dev", _vp), ("y_dev", _vp), ("residual_dev", _vp), ("rows", _i64)]


def _sig(name, args, res=_ci):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = res
    return f


_sig("nt_ctx_create", [ctypes.POINTER(_vp), _ci, _sz])
_sig("nt_ctx_destroy", [_vp])
_sig("nt_ctx_sync", [_vp])
_sig("nt_last_error", [_vp], ctypes.c_char_p)
_sig("nt_block_bytes", [_ci])
_sig("nt_block_elems", [_ci])
_sig("nt_dequant_rows", [_vp, _ci, _vp, _i64, _i64, _i64, _vp, _vp])
_sig("nt_gemv_q", [_vp, _ci, _vp, _vp, _vp, _i64, _i64, _vp, _vp])
_sig("nt_gemv_q_swiglu", [_vp, _ci, _vp, _vp, _vp, _vp, _cf, _vp, _i64, _i64, _vp])
_sig("nt_gemv_q_multi", [_vp, _ci, ctypes.POINTER(nt_gemv_job), _ci, _vp, _vp, _cf, _i64, _vp])
_sig("nt_rmsnorm", [_vp, _vp, _vp, _vp, _i64, _cf, _vp])
_sig("nt_rope", [_vp, _vp, _vp, _ci, _ci, _ci, _i64, _cf, _vp])
_sig("nt_rope_kv_append", [_vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _i64, _i64, _cf, _vp])
_sig("nt_attn_decode", [_vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _i64, _i64, _vp])
_sig("nt_softmax", [_vp, _vp, _vp, _i64, _vp])
_sig("nt_swiglu", [_vp, _vp, _vp, _vp, _i64, _vp])
_sig("nt_argmax", [_vp, _vp, _i64, _vp, _vp])
_sig("nt_cos_sim", [_vp, _vp, _vp, _i64, _vp, _vp])


class nt_model_desc(ctypes.Structure):
    _fields_ = [(n, _ci) for n in ("n_layers", "d_model", "n_qh", "n_kvh", "head_dim", "ffn", "vocab")] + [
        ("eps", _cf), ("theta", _cf), ("kv_cap", _i64)] + [
        (n, _ci) for n in ("fmt_q", "fmt_k", "fmt_v", "fmt_o", "fmt_gate", "fmt_up", "fmt_down", "fmt_embd",
                           "fmt_out", "stream_slots")]


class nt_layer_ptrs(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "attn_norm", "ffn_norm", "kcache",
                                   "vcache", "host_blob")]


_sig("nt_model_init", [_vp, ctypes.POINTER(nt_model_desc), ctypes.POINTER(nt_layer_ptrs), _vp, _vp, _vp,
                       ctypes.POINTER(_vp)])
_sig("nt_model_destroy", [_vp, _vp])
_sig("nt_decode_step", [_vp, _vp, ctypes.c_int32, _i64, _vp, _vp, _vp, _vp])
_sig("nt_layer_skip_calibrate", [_vp, _vp, ctypes.c_int32, _i64, _ci, _vp, _vp, _vp, _vp, _vp])
_sig("nt_attn_decode_static", [_vp, _vp, _vp, _vp, _ci, _ci, _ci, _i64, _i64, _vp])
_sig("nt_layer_blob_layout", [ctypes.POINTER(nt_model_desc), ctypes.POINTER(_sz), ctypes.POINTER(_sz)])


class nt_residency_plan(ctypes.Structure):
    _fields_ = [("n_resident", _ci), ("stream_slots", _ci), ("layer_bytes", _sz), ("fixed_bytes", _sz),
                ("total_bytes", _sz)]


_sig("nt_plan_residency", [ctypes.POINTER(nt_model_desc), _sz, _ci, ctypes.POINTER(nt_residency_plan)])
_sig("nt_host_register", [_vp, _vp, _sz, _ci])
_sig("nt_host_unregister", [_vp, _vp])
_sig("nt_sample", [_vp, _vp, _i64, _cf, _cf, ctypes.c_uint64, ctypes.c_uint64, _vp, _vp])
_sig("nt_model_set_sampler", [_vp, _vp, _cf, _cf, ctypes.c_uint64])
_sig("nt_prefill", [_vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp])
_sig("nt_spec_step", [_vp, _vp, ctypes.c_int32, _i64, _ci, _ci, _vp, _vp, _vp, _vp])
_sig("nt_gemm_q", [_vp, _ci, _vp, _vp, _vp, _i64, _i64, _ci, _vp, _vp, _cf, _vp])
_sig("nt_attn_verify", [_vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _i64, _ci, _i64, _vp])
_sig("nt_stream_layer", [_vp, _vp, _ci, _vp, _sz, _ci, _vp])
_sig("nt_model_slot", [_vp, _vp, _ci, ctypes.POINTER(_vp), ctypes.POINTER(_sz), ctypes.POINTER(_ci)])
_sig("nt_stream_sync", [_vp, _vp, _i64])
_sig("nt_debug_fail_copy", [_vp, _ci])
_sig("nt_debug_host_delay", [_vp, _vp, _i64])
_sig("nt_debug_stall_waits", [_ci])
_sig("nt_ctx_gemv_plans", [_vp, _vp, _sz, ctypes.POINTER(_sz)])
_sig("nt_model_graph_count", [_vp, _vp, ctypes.POINTER(_ci)])
_sig("nt_model_prefill_chunk", [_vp, _vp, ctypes.POINTER(_ci)])
_sig("nt_file_open", [ctypes.c_char_p, ctypes.POINTER(_vp)])
_sig("nt_file_close", [_vp])
_sig("nt_file_desc", [_vp, ctypes.POINTER(nt_model_desc)])
_sig("nt_file_header", [_vp, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_sz)])
_sig("nt_file_entry", [_vp, ctypes.c_char_p, ctypes.POINTER(_vp), ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(_sz)])
_sig("nt_file_lock", [_vp, _vp, ctypes.c_char_p, _ci, ctypes.POINTER(_vp), ctypes.POINTER(_ci)])
_sig("nt_file_unlock", [_vp, _vp, ctypes.c_char_p])
_sig("nt_debug_file_refuse_in_place", [_ci])

EXPORTED = ["nt_ctx_create", "nt_ctx_destroy", "nt_ctx_sync", "nt_last_error", "nt_block_bytes", "nt_block_elems",
            "nt_dequant_rows", "nt_gemv_q", "nt_gemv_q_swiglu", "nt_gemv_q_multi", "nt_rmsnorm", "nt_rope",
            "nt_rope_kv_append", "nt_attn_decode", "nt_softmax", "nt_swiglu", "nt_argmax", "nt_cos_sim",
            "nt_model_init", "nt_model_destroy", "nt_decode_step", "nt_layer_skip_calibrate",
            "nt_attn_decode_static", "nt_layer_blob_layout", "nt_stream_layer", "nt_model_slot", "nt_spec_step",
            "nt_gemm_q", "nt_attn_verify", "nt_plan_residency", "nt_prefill", "nt_sample", "nt_model_set_sampler",
            "nt_host_register", "nt_host_unregister", "nt_stream_sync", "nt_debug_fail_copy", "nt_debug_host_delay",
            "nt_debug_stall_waits", "nt_ctx_gemv_plans", "nt_model_graph_count", "nt_model_prefill_chunk",
            "nt_file_open", "nt_file_close", "nt_file_desc", "nt_file_header", "nt_file_entry", "nt_file_lock",
            "nt_file_unlock", "nt_debug_file_refuse_in_place"]


def lib():
    return _lib


# ---------------------------------------------------------------------------
def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, like=None):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    dev = like.device if like is not None and hasattr(like, "device") else None
    return torch.cuda.current_stream(dev).cuda_stream


class Context:
    """Owns one nt_ctx (device scratch, events, graphs)."""

    def __init__(self, device: int = 0, scratch_bytes: int = 0):
        h = _vp()
        st = _lib.nt_ctx_create(ctypes.byref(h), device, scratch_bytes)
        if st != NT_OK:
            raise NtError(st, "nt_ctx_create failed: " + (_lib.nt_last_error(None) or b"").decode())
        self.handle = h.value
        self.device = device

    def check(self, status: int):
        if status != NT_OK:
            raise NtError(status, _lib.nt_last_error(self.handle).decode())
        return status

    def sync(self):
        return self.check(_lib.nt_ctx_sync(self.handle))

    def close(self):
        if self.handle:
            _lib.nt_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def nt_ctx_create(device: int = 0, scratch_bytes: int = 0) -> Context:
    return Context(device, scratch_bytes)


def nt_block_bytes(fmt: int) -> int:
    return _lib.nt_block_bytes(fmt)


def nt_block_elems(fmt: int) -> int:
    return _lib.nt_block_elems(fmt)


def nt_dequant_rows(ctx, fmt, W, row0, nrows, cols, out, stream=None):
    return ctx.check(_lib.nt_dequant_rows(ctx.handle, fmt, _ptr(W), row0, nrows, cols, _ptr(out), _stream(stream, out)))


def nt_gemv_q(ctx, fmt, W, x, y, rows, cols, residual=None, stream=None):
    return ctx.check(_lib.nt_gemv_q(ctx.handle, fmt, _ptr(W), _ptr(x), _ptr(y), rows, cols, _ptr(residual),
                                    _stream(stream, y)))


def nt_gemv_q_swiglu(ctx, fmt, Wg, Wu, x, h, rows, cols, norm_g=None, eps=0.0, stream=None):
    return ctx.check(_lib.nt_gemv_q_swiglu(ctx.handle, fmt, _ptr(Wg), _ptr(Wu), _ptr(x), _ptr(norm_g), eps, _ptr(h),
                                           rows, cols, _stream(stream, h)))


def nt_gemv_q_multi(ctx, fmt, jobs, x, cols, norm_g=None, eps=0.0, stream=None):
    """jobs: list of (W, y, residual_or_None, rows)."""
    arr = (nt_gemv_job * max(1, len(jobs)))()
    for i, (W, y, r, rows) in enumerate(jobs):
        arr[i] = nt_gemv_job(_ptr(W), _ptr(y), _ptr(r), rows)
    return ctx.check(_lib.nt_gemv_q_multi(ctx.handle, fmt, arr, len(jobs), _ptr(x), _ptr(norm_g), eps, cols,
                                          _stream(stream, x)))


def nt_rmsnorm(ctx, x, g, y, n, eps, stream=None):
    return ctx.check(_lib.nt_rmsnorm(ctx.handle, _ptr(x), _ptr(g), _ptr(y), n, eps, _stream(stream, y)))


def nt_rope(ctx, q, k, n_qh, n_kvh, head_dim, pos, theta, stream=None):
    return ctx.check(_lib.nt_rope(ctx.handle, _ptr(q), _ptr(k), n_qh, n_kvh, head_dim, pos, theta,
                                  _stream(stream, q)))


def nt_rope_kv_append(ctx, q, k, v, kcache, vcache, n_qh, n_kvh, head_dim, pos, kv_stride, theta, stream=None):
    return ctx.check(_lib.nt_rope_kv_append(ctx.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(kcache), _ptr(vcache), n_qh,
                                            n_kvh, head_dim, pos, kv_stride, theta, _stream(stream, q)))


def nt_attn_decode(ctx, q, kcache, vcache, out, n_qh, n_kvh, head_dim, n_pos, kv_stride, stream=None):
    return ctx.check(_lib.nt_attn_decode(ctx.handle, _ptr(q), _ptr(kcache), _ptr(vcache), _ptr(out), n_qh, n_kvh,
                                         head_dim, n_pos, kv_stride, _stream(stream, out)))


def nt_softmax(ctx, x, y, n, stream=None):
    return ctx.check(_lib.nt_softmax(ctx.handle, _ptr(x), _ptr(y), n, _stream(stream, y)))


def nt_swiglu(ctx, gate, up, h, n, stream=None):
    return ctx.check(_lib.nt_swiglu(ctx.handle, _ptr(gate), _ptr(up), _ptr(h), n, _stream(stream, h)))


def nt_argmax(ctx, v, n, out, stream=None):
    return ctx.check(_lib.nt_argmax(ctx.handle, _ptr(v), n, _ptr(out), _stream(stream, out)))


def nt_cos_sim(ctx, a, b, n, out, stream=None):
    return ctx.check(_lib.nt_cos_sim(ctx.handle, _ptr(a), _ptr(b), n, _ptr(out), _stream(stream, out)))


def nt_model_init(ctx, desc: nt_model_desc, layers, embd, out, out_norm) -> int:
    """layers: list of dicts with wq..wd, attn_norm, ffn_norm, kcache, vcache (tensors or int pointers)."""
    arr = (nt_layer_ptrs * len(layers))()
    for i, L in enumerate(layers):
        arr[i] = nt_layer_ptrs(*[_ptr(L.get(n)) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "attn_norm",
                                                          "ffn_norm", "kcache", "vcache", "host_blob")])
    h = _vp()
    ctx.check(_lib.nt_model_init(ctx.handle, ctypes.byref(desc), arr, _ptr(embd), _ptr(out), _ptr(out_norm),
                                 ctypes.byref(h)))
    return h.value


def nt_gemm_q(ctx, fmt, W, X, Y, rows, cols, M, residual=None, norm_g=None, eps=0.0, stream=None):
    return ctx.check(_lib.nt_gemm_q(ctx.handle, fmt, _ptr(W), _ptr(X), _ptr(Y), rows, cols, M, _ptr(residual),
                                    _ptr(norm_g), eps, _stream(stream, Y)))


def nt_attn_verify(ctx, q, kcache, vcache, out, n_qh, n_kvh, head_dim, n_pos0, n_query, kv_stride, stream=None):
    return ctx.check(_lib.nt_attn_verify(ctx.handle, _ptr(q), _ptr(kcache), _ptr(vcache), _ptr(out), n_qh, n_kvh,
                                         head_dim, n_pos0, n_query, kv_stride, _stream(stream, out)))


def nt_host_register(ctx, host_ptr: int, nbytes: int, read_only: bool = True):
    return ctx.check(_lib.nt_host_register(ctx.handle, host_ptr, nbytes, int(bool(read_only))))


def nt_host_unregister(ctx, host_ptr: int):
    return ctx.check(_lib.nt_host_unregister(ctx.handle, host_ptr))


# rungs of nt_file_lock, in the order of preference
FILE_RUNGS = ("mmap pinned", "mmap pinned private", "CPU memcpy")


def _no_ctx_check(status: int, what: str):
    """Raise for a failed call made without a context (its reason is the thread's nt_last_error(NULL))."""
    if status != NT_OK:
        raise NtError(status, what + ": " + (_lib.nt_last_error(None) or b"").decode())
    return status


def nt_file_open(path: str) -> int:
    """Open and check a model file; returns the nt_file handle."""
    h = _vp()
    _no_ctx_check(_lib.nt_file_open(os.fsencode(path), ctypes.byref(h)), "nt_file_open")
    return h.value


def nt_file_close(f: int):
    return _no_ctx_check(_lib.nt_file_close(f), "nt_file_close")


def nt_file_desc(f: int) -> nt_model_desc:
    d = nt_model_desc()
    _no_ctx_check(_lib.nt_file_desc(f, ctypes.byref(d)), "nt_file_desc")
    return d


def nt_file_header(f: int) -> str:
    t, n = ctypes.c_char_p(), _sz()
    _no_ctx_check(_lib.nt_file_header(f, ctypes.byref(t), ctypes.byref(n)), "nt_file_header")
    return ctypes.string_at(t, n.value).decode()


def nt_file_entry(f: int, name: str):
    """Returns (address in the read-only mapping, offset in the file, bytes) of entry `name`."""
    p, off, n = _vp(), ctypes.c_uint64(), _sz()
    st = _lib.nt_file_entry(f, name.encode(), ctypes.byref(p), ctypes.byref(off), ctypes.byref(n))
    if st != NT_OK:
        raise NtError(st, f"nt_file_entry: no entry {name}")
    return p.value, off.value, n.value


def nt_file_lock(ctx, f: int, name: str, allow_copy: bool = True):
    """Page-lock entry `name`; returns (page-locked address, rung index into FILE_RUNGS)."""
    p, rung = _vp(), _ci()
    ctx.check(_lib.nt_file_lock(ctx.handle, f, name.encode(), int(bool(allow_copy)), ctypes.byref(p),
                                ctypes.byref(rung)))
    return p.value, rung.value


def nt_file_unlock(ctx, f: int, name: str):
    return ctx.check(_lib.nt_file_unlock(ctx.handle, f, name.encode()))


def nt_debug_file_refuse_in_place(on: bool):
    """Test hook: nt_file_lock treats both in-place rungs as refused (host side only)."""
    st = _lib.nt_debug_file_refuse_in_place(int(bool(on)))
    if st != NT_OK:
        raise NtError(st, "nt_debug_file_refuse_in_place failed")
    return st


def nt_stream_sync(ctx, stream, timeout_us: int):
    """Wait at most timeout_us for `stream`; NtError(NT_ERR_TIMEOUT) when it stays busy."""
    return ctx.check(_lib.nt_stream_sync(ctx.handle, _stream(stream), timeout_us))


def nt_debug_fail_copy(ctx, nth: int):
    """Fault injection (host side): the nth following layer copy fails; -1 disarms."""
    return ctx.check(_lib.nt_debug_fail_copy(ctx.handle, nth))


def nt_debug_host_delay(ctx, stream, us: int):
    """A host callback that keeps `stream` busy for `us` microseconds."""
    return ctx.check(_lib.nt_debug_host_delay(ctx.handle, _stream(stream), us))


def nt_ctx_gemv_plans(ctx) -> list:
    """The quant-GEMV plans the context has chosen, one string per launch shape."""
    n = _sz()
    ctx.check(_lib.nt_ctx_gemv_plans(ctx.handle, None, 0, ctypes.byref(n)))
    buf = ctypes.create_string_buffer(n.value)
    ctx.check(_lib.nt_ctx_gemv_plans(ctx.handle, buf, n.value, ctypes.byref(n)))
    return [ln for ln in buf.value.decode().splitlines() if ln]


def nt_model_graph_count(ctx, model: int) -> int:
    n = _ci()
    ctx.check(_lib.nt_model_graph_count(ctx.handle, model, ctypes.byref(n)))
    return n.value


def nt_model_prefill_chunk(ctx, model: int) -> int:
    n = ctypes.c_int(0)
    ctx.check(_lib.nt_model_prefill_chunk(ctx.handle, model, ctypes.byref(n)))
    return n.value


def nt_debug_stall_waits(n: int):
    """Test hook: the next n eager launches of the copy-waiting kernels take
    their bounded-wait timeout path (no GPU fault or hang); 0 disarms."""
    st = _lib.nt_debug_stall_waits(n)
    if st != NT_OK:
        raise NtError(st, "nt_debug_stall_waits failed")
    return st


def nt_sample(ctx, logits, n: int, temperature: float, top_p: float, seed: int, counter: int, out, stream=None):
    return ctx.check(_lib.nt_sample(ctx.handle, _ptr(logits), n, temperature, top_p, seed, counter, _ptr(out),
                                    _stream(stream, out)))


def nt_model_set_sampler(ctx, model: int, temperature: float, top_p: float, seed: int):
    return ctx.check(_lib.nt_model_set_sampler(ctx.handle, model, temperature, top_p, seed))


def nt_prefill(ctx, model: int, tokens, pos0: int, logits, next_token=None, stream=None):
    """tokens: a sequence of ints (copied to an int32 host array)."""
    import numpy as np
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    return ctx.check(_lib.nt_prefill(ctx.handle, model, t.ctypes.data, t.size, pos0, _ptr(logits), _ptr(next_token),
                                     _stream(stream, logits)))


def nt_spec_step(ctx, model: int, token: int, pos: int, k: int, n_draft_layers: int, tokens_out, n_out,
                 logits=None, stream=None):
    return ctx.check(_lib.nt_spec_step(ctx.handle, model, token, pos, k, n_draft_layers, _ptr(tokens_out),
                                       _ptr(n_out), _ptr(logits), _stream(stream, tokens_out)))


def nt_plan_residency(desc: nt_model_desc, hbm_weight_budget: int, embd_in_hbm: bool = False) -> nt_residency_plan:
    p = nt_residency_plan()
    st = _lib.nt_plan_residency(ctypes.byref(desc), int(hbm_weight_budget), int(bool(embd_in_hbm)), ctypes.byref(p))
    if st != NT_OK:
        raise NtError(st, "nt_plan_residency failed")
    return p


def nt_layer_blob_layout(desc: nt_model_desc):
    """Returns (offsets of wq..wd [7 ints], blob bytes)."""
    off = (_sz * 7)()
    n = _sz()
    st = _lib.nt_layer_blob_layout(ctypes.byref(desc), off, ctypes.byref(n))
    if st != NT_OK:
        raise NtError(st, "nt_layer_blob_layout failed")
    return list(off), n.value


def nt_stream_layer(ctx, model: int, layer: int, host_src, nbytes: int, slot: int, copy_stream=None):
    return ctx.check(_lib.nt_stream_layer(ctx.handle, model, layer, _ptr(host_src), nbytes, slot,
                                          _stream(copy_stream)))


def nt_model_slot(ctx, model: int, slot: int):
    """Returns (slot device address, slot bytes, layer last copied into it)."""
    p, n, layer = _vp(), _sz(), _ci()
    ctx.check(_lib.nt_model_slot(ctx.handle, model, slot, ctypes.byref(p), ctypes.byref(n), ctypes.byref(layer)))
    return p.value, n.value, layer.value


def nt_model_destroy(ctx, model: int):
    return ctx.check(_lib.nt_model_destroy(ctx.handle, model))


def _mask_ptr(mask):
    if mask is None:
        return None, None
    import numpy as np
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    return m, m.ctypes.data


def nt_decode_step(ctx, model: int, token: int, pos: int, skip_mask, logits, next_token=None, stream=None):
    keep, mp = _mask_ptr(skip_mask)
    return ctx.check(_lib.nt_decode_step(ctx.handle, model, token, pos, mp, _ptr(logits), _ptr(next_token),
                                         _stream(stream, logits)))


def nt_layer_skip_calibrate(ctx, model: int, token: int, pos: int, n_skip: int, n_layers: int, logits,
                            next_token=None, stream=None):
    """Returns (skip_mask uint8[n_layers], cos float32[n_layers])."""
    import numpy as np
    mask = np.zeros(n_layers, dtype=np.uint8)
    cos = np.zeros(n_layers, dtype=np.float32)
    ctx.check(_lib.nt_layer_skip_calibrate(ctx.handle, model, token, pos, n_skip, mask.ctypes.data,
                                           cos.ctypes.data, _ptr(logits), _ptr(next_token),
                                           _stream(stream, logits)))
    return mask, cos


def nt_attn_decode_static(q, kcache, vcache, out, n_qh, n_kvh, head_dim, n_pos, kv_stride, stream=None):
    """Decode attention without a context or any allocation (fixed scratch inside
    the library); raises NtError on a non-OK status."""
    st = _lib.nt_attn_decode_static(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(out), n_qh, n_kvh, head_dim, n_pos,
                                    kv_stride, _stream(stream, out))
    if st != NT_OK:
        raise NtError(st, "nt_attn_decode_static failed")
    return st
