"""Device-side model: places a synthetic host model's tensors in HBM (torch
allocations) and drives the C ABI's decode step.  Marshalling only: every
step of the computation runs in libnt.so's kernels."""
from __future__ import annotations

import numpy as np
import torch

from . import nt

LAYER = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def _h(a) -> torch.Tensor:
    """A host array as a tensor (read-only views, e.g. of a mapped file, are copied)."""
    return torch.from_numpy(a if a.flags.writeable else np.array(a))


def model_desc(spec, stream_slots: int = 0) -> nt.nt_model_desc:
    f = spec.fmt
    return nt.nt_model_desc(spec.n_layers, spec.d_model, spec.n_qh, spec.n_kvh, spec.head_dim, spec.ffn, spec.vocab,
                            spec.eps, spec.theta, spec.kv_cap, f["wq"], f["wk"], f["wv"], f["wo"], f["wg"], f["wu"],
                            f["wd"], f["embd"], f["out"], stream_slots)


def _row_bytes(spec, name):
    r, c = spec.tensor_shape(name)
    f = spec.fmt[name]
    return r, (c // nt.nt_block_elems(f)) * nt.nt_block_bytes(f)


class HostBlobs:
    """Page-locked host memory for the streamed layers of a model (layers
    n_resident..n_layers-1, each one blob in the library's blob layout) and,
    for streamed models, the embedding table.  ``view`` hands the generator
    numpy views to write the weights into, so they are never copied."""

    def __init__(self, spec, stream_slots: int = 0):
        self.spec = spec
        n_res = spec.n_layers if spec.n_resident < 0 else spec.n_resident
        self.layers = list(range(n_res, spec.n_layers))
        self.offsets, self.nbytes = nt.nt_layer_blob_layout(model_desc(spec, stream_slots))
        self.blob = {l: torch.empty(self.nbytes, dtype=torch.uint8, pin_memory=True) for l in self.layers}
        self.embd = None
        if self.layers:
            r, rb = _row_bytes(spec, "embd")
            self.embd = torch.empty((r, rb), dtype=torch.uint8, pin_memory=True)

    def view(self, layer: int, name: str):
        if layer < 0:
            return self.embd.numpy() if (name == "embd" and self.embd is not None) else None
        if layer not in self.blob:
            return None
        i = LAYER.index(name)
        r, rb = _row_bytes(self.spec, name)
        o = self.offsets[i]
        return self.blob[layer].numpy()[o:o + r * rb].reshape(r, rb)


class DeviceModel:
    """spec: shapes/formats; hm: host arrays (layers list of dicts, embd, out,
    out_norm, kcache/vcache float16 [L, kvh, cap, hd]).  With ``blobs`` the
    layers it holds are streamed from its page-locked host memory and the
    embedding table is read from host memory; their host arrays in ``hm``
    must be the blobs' views (make_host_model(..., out_view=blobs.view))."""

    def __init__(self, ctx: nt.Context, spec, hm, device: str = "cuda", blobs: HostBlobs | None = None,
                 stream_slots: int = 0):
        self.ctx, self.spec, self.blobs = ctx, spec, blobs
        self.n_slots = (stream_slots or 2) if (blobs is not None and blobs.layers) else 0
        dev = torch.device(device)
        self.layers = []
        for i, L in enumerate(hm.layers):
            if blobs is not None and i in blobs.blob:
                d = {n: _h(L[n]).to(dev) for n in ("attn_norm", "ffn_norm")}
                d["host_blob"] = blobs.blob[i]
            else:
                d = {n: _h(L[n]).to(dev) for n in LAYER + ("attn_norm", "ffn_norm")}
            d["kcache"] = torch.from_numpy(np.ascontiguousarray(hm.kcache[i])).to(dev)
            d["vcache"] = torch.from_numpy(np.ascontiguousarray(hm.vcache[i])).to(dev)
            self.layers.append(d)
        if blobs is not None and blobs.embd is not None:
            self.embd = blobs.embd
        else:
            self.embd = _h(hm.embd).to(dev)
        self.out = _h(hm.out).to(dev)
        self.out_norm = _h(hm.out_norm).to(dev)
        self.logits = torch.empty(spec.vocab, dtype=torch.float32, device=dev)
        self.next_token = torch.zeros(1, dtype=torch.int32, device=dev)
        self.handle = nt.nt_model_init(ctx, model_desc(spec, stream_slots), self.layers, self.embd, self.out,
                                       self.out_norm)

    def hbm_weight_bytes(self) -> int:
        """Weight bytes this model keeps in HBM: resident layers, LM head,
        embedding table when resident, streaming slots."""
        n = sum(t.numel() for L in self.layers for k, t in L.items() if k in LAYER)
        n += self.out.numel() + (self.embd.numel() if isinstance(self.embd, torch.Tensor) and self.embd.is_cuda else 0)
        return n + self.n_slots * (self.blobs.nbytes if self.blobs is not None else 0)

    def step(self, token: int, pos: int, skip=None, stream=None):
        """One decode step; token < 0 continues from the device state."""
        nt.nt_decode_step(self.ctx, self.handle, token, pos, skip, self.logits, self.next_token, stream)
        return self.logits

    def set_sampler(self, temperature: float, top_p: float = 1.0, seed: int = 0):
        """Later decode steps sample (temperature, top-p); temperature <= 0 is greedy."""
        nt.nt_model_set_sampler(self.ctx, self.handle, temperature, top_p, seed)

    def prefill(self, tokens, pos0: int, stream=None):
        """Run a prompt through the model (KV written for pos0 ..); returns the
        logits after its last token.  Decoding continues with step(-1, 0)."""
        nt.nt_prefill(self.ctx, self.handle, tokens, pos0, self.logits, self.next_token, stream)
        return self.logits

    def spec_step(self, token: int, pos: int, k: int, n_draft_layers: int = 0, stream=None):
        """One self-speculative step (token < 0 continues from the device
        state); returns (tokens [k + 1] int32 device tensor, count [1] int32
        device tensor, verify logits [k + 1, vocab]).  The first count tokens
        are the step's output."""
        if not hasattr(self, "spec_tokens"):
            dev = self.logits.device
            self.spec_tokens = torch.zeros(8, dtype=torch.int32, device=dev)
            self.spec_count = torch.zeros(1, dtype=torch.int32, device=dev)
            self.spec_logits = torch.empty(16, self.spec.vocab, dtype=torch.float32, device=dev)
        nt.nt_spec_step(self.ctx, self.handle, token, pos, k, n_draft_layers, self.spec_tokens, self.spec_count,
                        self.spec_logits, stream)
        # with the sampler set, the draft logits follow the verify rows
        self.draft_logits = self.spec_logits[k + 1:2 * k + 1]
        return self.spec_tokens, self.spec_count, self.spec_logits[:k + 1]

    def calibrate(self, token: int, pos: int, n_skip: int, stream=None):
        return nt.nt_layer_skip_calibrate(self.ctx, self.handle, token, pos, n_skip, self.spec.n_layers,
                                          self.logits, self.next_token, stream)

    def kv(self, layer: int):
        return self.layers[layer]["kcache"], self.layers[layer]["vcache"]

    def close(self):
        if self.handle:
            nt.nt_model_destroy(self.ctx, self.handle)
            self.handle = None
