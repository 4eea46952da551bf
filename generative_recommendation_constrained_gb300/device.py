"""Device-memory plumbing around the C ABI: torch tensors hold the model,
workspace and outputs; the library's kernels do all the work."""
from __future__ import annotations

import numpy as np
import torch

from . import _lib as Z


def _to_device_weights(w: np.ndarray, w_dtype: str, device) -> torch.Tensor:
    if w_dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(device)
    if w_dtype == "bf16":      # uint16 bfloat16 bit patterns
        bits = np.ascontiguousarray(w, np.uint16).view(np.int16)
        return torch.from_numpy(bits).to(device).view(torch.bfloat16)
    if w_dtype == "f16":
        return torch.from_numpy(np.ascontiguousarray(w, np.float16)).to(device)
    raise ValueError(w_dtype)


def _f32(x, device):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)


class DeviceModel:
    """Uploads a synthetic model (C_s float32, W_s in its storage dtype) and,
    optionally, a light decoder's weights (deco: the hidden vectors then come
    from the decoder and the decode's input is the concept vectors), and
    builds the zg_model struct pointing at the device copies."""

    def __init__(self, model, device="cuda", deco=None):
        self.L, self.V, self.d, self.w_dtype = model.L, model.V, model.d, model.w_dtype
        self.C = [_f32(c, device) for c in model.C]
        self.W = [_to_device_weights(w, model.w_dtype, device) for w in model.W]
        dstruct = None
        if deco is not None:
            self.deco = {"E": [_f32(e, device) for e in deco.E], "P": _f32(deco.P, device)}
            for n in ("Wq", "Wk", "Wv", "Wo", "W1", "W2"):
                self.deco[n] = [_f32(w, device) for w in getattr(deco, n)]
            t = self.deco
            dstruct = Z.make_deco(deco.M, deco.heads, deco.ffn, [e.data_ptr() for e in t["E"]],
                                  t["P"].data_ptr(), *[[w.data_ptr() for w in t[n]]
                                                       for n in ("Wq", "Wk", "Wv", "Wo", "W1", "W2")])
        self.struct = Z.make_model(self.L, self.V, self.d, Z.DTYPES[self.w_dtype],
                                   [c.data_ptr() for c in self.C], [w.data_ptr() for w in self.W], dstruct)


class Decoder:
    """Workspace and outputs for repeated zg_decode calls with fixed shapes."""

    def __init__(self, idx, plan, dmodel: DeviceModel, B: int, beam: int, K: int, device="cuda"):
        self.idx, self.plan, self.dm = idx, plan, dmodel
        self.B, self.beam, self.K = B, beam, K
        self.ws_bytes = Z.zg_decode_workspace_size(idx, plan, dmodel.struct, B, beam, K)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.out_sids = torch.empty((B, K, dmodel.L), dtype=torch.int32, device=device)
        self.out_scores = torch.empty((B, K), dtype=torch.float32, device=device)

    def __call__(self, u: torch.Tensor, stream: int | None = None):
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        Z.zg_decode(self.idx, self.plan, self.dm.struct, u, self.B, self.beam, self.K, self.out_sids,
                    self.out_scores, self.ws, self.ws_bytes, stream)
        return self.out_sids, self.out_scores

    def trace(self, u: torch.Tensor, stream: int | None = None) -> list[dict]:
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        return Z.zg_decode_trace(self.idx, self.plan, self.dm.struct, u, self.B, self.beam, self.K,
                                 self.out_sids, self.out_scores, self.ws, self.ws_bytes, stream)
