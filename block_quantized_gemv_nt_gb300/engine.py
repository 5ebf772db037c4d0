"""Device-side model: places a synthetic host model's tensors in HBM (torch
allocations) and drives the C ABI's decode step.  Marshalling only: every
step of the computation runs in libnt.so's kernels."""
from __future__ import annotations

import numpy as np
import torch

from . import nt

LAYER = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def model_desc(spec) -> nt.nt_model_desc:
    f = spec.fmt
    return nt.nt_model_desc(spec.n_layers, spec.d_model, spec.n_qh, spec.n_kvh, spec.head_dim, spec.ffn, spec.vocab,
                            spec.eps, spec.theta, spec.kv_cap, f["wq"], f["wk"], f["wv"], f["wo"], f["wg"], f["wu"],
                            f["wd"], f["embd"], f["out"])


class DeviceModel:
    """spec: shapes/formats; hm: host arrays (layers list of dicts, embd, out,
    out_norm, kcache/vcache float16 [L, kvh, cap, hd])."""

    def __init__(self, ctx: nt.Context, spec, hm, device: str = "cuda"):
        self.ctx, self.spec = ctx, spec
        dev = torch.device(device)
        self.layers = []
        for i, L in enumerate(hm.layers):
            d = {n: torch.from_numpy(L[n]).to(dev) for n in LAYER + ("attn_norm", "ffn_norm")}
            d["kcache"] = torch.from_numpy(np.ascontiguousarray(hm.kcache[i])).to(dev)
            d["vcache"] = torch.from_numpy(np.ascontiguousarray(hm.vcache[i])).to(dev)
            self.layers.append(d)
        self.embd = torch.from_numpy(hm.embd).to(dev)
        self.out = torch.from_numpy(hm.out).to(dev)
        self.out_norm = torch.from_numpy(hm.out_norm).to(dev)
        self.logits = torch.empty(spec.vocab, dtype=torch.float32, device=dev)
        self.next_token = torch.zeros(1, dtype=torch.int32, device=dev)
        self.handle = nt.nt_model_init(ctx, model_desc(spec), self.layers, self.embd, self.out, self.out_norm)

    def step(self, token: int, pos: int, skip=None, stream=None):
        """One decode step; token < 0 continues from the device state."""
        nt.nt_decode_step(self.ctx, self.handle, token, pos, skip, self.logits, self.next_token, stream)
        return self.logits

    def calibrate(self, token: int, pos: int, n_skip: int, stream=None):
        return nt.nt_layer_skip_calibrate(self.ctx, self.handle, token, pos, n_skip, self.spec.n_layers,
                                          self.logits, self.next_token, stream)

    def kv(self, layer: int):
        return self.layers[layer]["kcache"], self.layers[layer]["vcache"]

    def close(self):
        if self.handle:
            nt.nt_model_destroy(self.ctx, self.handle)
            self.handle = None
