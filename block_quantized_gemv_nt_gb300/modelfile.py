"""Model files: the host-file tier of the 3-tier cache ("Ntransformer"
(en.unwiki.net), About: VRAM-resident layers, pinned RAM, NVMe/mmap
fallback; the "mmap pinned" data path).

A GGUF-style single-file container of a model's weights, laid out so that a
streamed layer is one contiguous, page-aligned range of the file:

    offset 0   b"NTQF", u32 version (1), u64 header length H
    offset 16  H bytes of UTF-8 JSON: the model description, the blob layout
               and every entry's (offset, bytes)
    data       entries at 4096-byte-aligned offsets: "embd", "out",
               "out_norm", and per layer l: "blob.l" (its seven weight
               matrices in the library's blob layout, nt_layer_blob_layout),
               "attn_norm.l", "ffn_norm.l"

``write_model`` writes it; reading is native (libnt.so: nt_file_open,
nt_file_entry, nt_file_lock), so a C caller has the whole tier too.
``ModelFile`` opens the file through that reader.  Resident layers are
uploaded from the mapping; the streamed layers' blobs (and the embedding
table) are page-locked where they lie, so the streaming engine copies them
to HBM exactly as it copies pinned RAM.  ``FileBlobs`` (nt_file_lock) takes
the first rung that the operating system and driver accept, in the pages'
order of preference:

  "mmap pinned"          the read-only shared mapping, registered read-only;
  "mmap pinned private"  a private, writable, pre-faulted mapping of the
                         range (copy-on-write: the file is never written),
                         registered without the read-only flag;
  "CPU memcpy"           one CPU copy of the range into page-locked memory.

The KV cache is runtime state, not part of the file.
"""
from __future__ import annotations

import json
import mmap
import struct
from dataclasses import asdict

import numpy as np

from . import nt

MAGIC = b"NTQF"
VERSION = 1
ALIGN = 4096
LAYER = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def _up(n: int, a: int = ALIGN) -> int:
    return (n + a - 1) // a * a


def _row_bytes(fmt: int, cols: int) -> int:
    return cols // nt.nt_block_elems(fmt) * nt.nt_block_bytes(fmt)


class FileSpec:
    """The model description stored in a file: the fields of the spec it was
    written from, with the shape helpers the engine uses."""

    def __init__(self, fields: dict):
        self.__dict__.update(fields)
        self.fmt = {k: int(v) for k, v in self.fmt.items()}

    def tensor_shape(self, name: str):
        d, hd = self.d_model, self.head_dim
        return {"wq": (self.n_qh * hd, d), "wk": (self.n_kvh * hd, d), "wv": (self.n_kvh * hd, d),
                "wo": (d, self.n_qh * hd), "wg": (self.ffn, d), "wu": (self.ffn, d), "wd": (d, self.ffn),
                "embd": (self.vocab, d), "out": (self.vocab, d)}[name]

    @property
    def kv_cap(self) -> int:
        return self.n_prefill + self.n_gen + 8

    def layer_bytes(self) -> int:
        return sum(self.tensor_shape(t)[0] * _row_bytes(self.fmt[t], self.tensor_shape(t)[1]) for t in LAYER)


def write_model(path: str, spec, hm) -> None:
    """Write host model `hm` (synth.HostModel layout) of `spec` to `path`."""
    from .engine import model_desc
    offsets, blob_bytes = nt.nt_layer_blob_layout(model_desc(spec))
    entries = {}
    pieces = []  # (name, offset, writer)
    pos = 0

    def add(name, nbytes, fill):
        nonlocal pos
        entries[name] = [pos, int(nbytes)]
        pieces.append((pos, fill))
        pos = _up(pos + int(nbytes))

    add("embd", hm.embd.nbytes, lambda f: f.write(hm.embd.tobytes()))
    add("out", hm.out.nbytes, lambda f: f.write(hm.out.tobytes()))
    add("out_norm", hm.out_norm.nbytes, lambda f: f.write(hm.out_norm.tobytes()))
    for li, L in enumerate(hm.layers):
        def blob_writer(f, L=L):
            start = f.tell()
            for i, name in enumerate(LAYER):
                f.seek(start + offsets[i])
                f.write(np.ascontiguousarray(L[name]).tobytes())
        add(f"blob.{li}", blob_bytes, blob_writer)
        add(f"attn_norm.{li}", L["attn_norm"].nbytes, lambda f, L=L: f.write(L["attn_norm"].tobytes()))
        add(f"ffn_norm.{li}", L["ffn_norm"].nbytes, lambda f, L=L: f.write(L["ffn_norm"].tobytes()))
    fields = asdict(spec) if hasattr(spec, "__dataclass_fields__") else dict(vars(spec))
    header = json.dumps({"spec": fields, "blob_offsets": list(offsets), "blob_bytes": blob_bytes,
                         "entries": entries}).encode()
    data0 = _up(16 + len(header))
    with open(path, "wb") as f:
        f.write(MAGIC + struct.pack("<IQ", VERSION, len(header)) + header)
        for off, fill in pieces:
            f.seek(data0 + off)
            fill(f)
        f.truncate(data0 + pos)


class ModelFile:
    """A model file opened through the native reader (nt_file_open: the
    container, the header, the blob layout and every entry are checked
    there): ``spec``, ``handle`` (the nt_file), and numpy views of every
    entry (``layers`` as synth.HostModel lays them out, ``embd``, ``out``,
    ``out_norm``).  The views read a second read-only mapping of the same
    file (the same page-cache pages), so their lifetime follows Python's
    references rather than nt_file_close.  A file the reader refuses raises
    ValueError with its reason."""

    def __init__(self, path: str):
        self.path = path
        self.handle = None
        self._mm = None
        try:
            self.handle = nt.nt_file_open(path)
        except nt.NtError as e:
            raise ValueError(str(e)) from None
        try:
            self._open(path)
        except Exception:
            self.close()
            raise

    def _open(self, path: str) -> None:
        meta = json.loads(nt.nt_file_header(self.handle))
        self.spec = FileSpec(meta["spec"])
        self.blob_offsets, self.blob_bytes = meta["blob_offsets"], meta["blob_bytes"]
        self.entries = {k: nt.nt_file_entry(self.handle, k)[1:] for k in meta["entries"]}  # name -> (offset, bytes)
        with open(path, "rb") as f:
            self._mm = mmap.mmap(f.fileno(), 0, prot=mmap.PROT_READ)
        self._buf = buf = np.frombuffer(self._mm, dtype=np.uint8)
        s = self.spec

        def view(name, dtype=np.uint8, shape=None):
            off, n = self.entries[name]
            a = buf[off:off + n].view(dtype)
            return a.reshape(shape) if shape is not None else a

        def mat_shape(name):
            r, c = s.tensor_shape(name)
            return r, _row_bytes(s.fmt[name], c)

        self.embd = view("embd", shape=mat_shape("embd"))
        self.out = view("out", shape=mat_shape("out"))
        self.out_norm = view("out_norm", np.float32)
        self.layers = []
        for li in range(s.n_layers):
            off, _ = self.entries[f"blob.{li}"]
            d = {}
            for i, name in enumerate(LAYER):
                r, rb = mat_shape(name)
                o = off + self.blob_offsets[i]
                d[name] = buf[o:o + r * rb].reshape(r, rb)
            d["attn_norm"] = view(f"attn_norm.{li}", np.float32)
            d["ffn_norm"] = view(f"ffn_norm.{li}", np.float32)
            self.layers.append(d)

    def close(self):
        self.embd = self.out = self.out_norm = None
        self.layers = []
        self._buf = None
        if self._mm is not None:
            try:
                self._mm.close()
            except BufferError:
                pass  # views still alive elsewhere: the mapping closes with them
            self._mm = None
        if self.handle:
            nt.nt_file_close(self.handle)  # refused while a FileBlobs still holds page-locked entries
            self.handle = None


class FileBlobs:
    """The streamed layers of a model file, page-locked through the native
    reader (nt_file_lock): the same interface as engine.HostBlobs (``blob``
    maps a layer to its page-locked host address, ``embd`` is the embedding
    table's), so DeviceModel streams from the file.  ``rung_of`` records the
    rung each range took, ``tier`` the lowest taken."""

    def __init__(self, ctx: nt.Context, mf: ModelFile, n_resident: int, allow_copy: bool = True):
        self.ctx, self.mf = ctx, mf
        s = mf.spec
        self.layers = list(range(n_resident, s.n_layers))
        self.offsets, self.nbytes = mf.blob_offsets, mf.blob_bytes
        self.rung_of = {}  # entry name -> rung
        self.blob = {}
        try:
            for li in self.layers:
                self.blob[li] = self._lock(f"blob.{li}", allow_copy)
            self.embd = self._lock("embd", allow_copy) if self.layers else None
        except Exception:
            self.close()
            raise
        order = ("CPU memcpy", "mmap pinned private", "mmap pinned")
        self.tier = next((t for t in order if t in self.rung_of.values()), "mmap pinned")  # the lowest rung taken

    def _lock(self, name: str, allow_copy: bool) -> int:
        addr, rung = nt.nt_file_lock(self.ctx, self.mf.handle, name, allow_copy)
        self.rung_of[name] = nt.FILE_RUNGS[rung]
        return addr

    def close(self):
        for name in list(self.rung_of):
            nt.nt_file_unlock(self.ctx, self.mf.handle, name)
            del self.rung_of[name]
