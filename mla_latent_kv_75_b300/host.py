"""Host-side plumbing around libmla: device buffers, cache layout and one decode / prefill
step through the C ABI. Memory and streams come from PyTorch; every arithmetic step runs
in libmla's CUDA kernels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import (MLA_BF16, MLA_F32, make_cache, make_dims, make_weights, mla_append_cache,
               mla_decode_absorbed, mla_decode_step, mla_decode_step_workspace_size,
               mla_decode_workspace_size, mla_fast_path, mla_prefill, mla_prefill_workspace_size,
               mla_project_q, mla_project_q_workspace_size)

WEIGHT_NAMES = ("W_DQ", "W_UQ", "W_QR", "W_DKV", "W_KR", "W_UK", "W_UV")


def torch_dtype(dtype: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]


def abi_dtype(dtype: str) -> int:
    return {"bf16": MLA_BF16, "f32": MLA_F32}[dtype]


def to_device(a: np.ndarray, dtype: str, device="cuda", pin: bool = False) -> torch.Tensor:
    """Upload float32 values (bf16-exact for dtype "bf16") as a tensor of ``dtype``."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch_dtype(dtype))
    if device == "cpu":
        return t.pin_memory() if pin else t
    return t.to(device)


def dims_struct(dims, dtype: str, scale: float = 0.0):
    return make_dims(dims.d, dims.n_h, dims.d_hc, dims.d_hr, dims.d_c, dims.d_cq,
                     abi_dtype(dtype), dims.rope_base, scale)


@dataclass
class DeviceModel:
    """Weights of one MLA layer resident on the device."""
    dims: object
    dtype: str
    W: Dict[str, torch.Tensor]

    @classmethod
    def upload(cls, dims, dtype: str, W_np: Dict[str, np.ndarray], device="cuda"):
        return cls(dims, dtype, {k: to_device(W_np[k], dtype, device) for k in WEIGHT_NAMES})

    @property
    def abi_dims(self):
        return dims_struct(self.dims, self.dtype)

    @property
    def abi_weights(self):
        return make_weights(self.W)


class LatentCache:
    """Latent cache rows [capacity, d_c + d_h^R] with per-sequence row bases."""

    def __init__(self, dims, dtype: str, seq_base: Sequence[int], capacity: int, device="cuda",
                 fill: Optional[float] = None):
        self.dims, self.dtype = dims, dtype
        width = dims.d_c + dims.d_hr
        if fill is None:
            self.rows = torch.empty((capacity, width), dtype=torch_dtype(dtype), device=device)
        else:
            self.rows = torch.full((capacity, width), fill, dtype=torch_dtype(dtype), device=device)
        self.seq_base = torch.tensor(list(seq_base), dtype=torch.int64, device=device)
        self.capacity = capacity

    @property
    def abi(self):
        return make_cache(self.rows, self.seq_base, self.capacity)


def append_tokens(model: DeviceModel, cache: LatentCache, h: torch.Tensor, seq_idx: torch.Tensor,
                  pos: torch.Tensor, stream=None) -> None:
    c = cache.abi
    mla_append_cache(model.abi_dims, model.abi_weights, h, seq_idx, pos, h.shape[0], c, stream)


def fill_context(model: DeviceModel, cache: LatentCache, hidden_fn, seq_lens: Sequence[int],
                 upto_last: bool = True, chunk: int = 16384) -> None:
    """Append every sequence's context rows (positions 0..L-2 if upto_last, else 0..L-1),
    generating hidden states with ``hidden_fn(b, n) -> np.ndarray [n, d]`` chunk by chunk."""
    dev = cache.rows.device
    for b, L in enumerate(seq_lens):
        n_ctx = L - 1 if upto_last else L
        if n_ctx <= 0:
            continue
        h_all = hidden_fn(b, n_ctx)
        for s in range(0, n_ctx, chunk):
            e = min(n_ctx, s + chunk)
            h = to_device(h_all[s:e], model.dtype, dev)
            seq = torch.full((e - s,), b, dtype=torch.int32, device=dev)
            pos = torch.arange(s, e, dtype=torch.int32, device=dev)
            append_tokens(model, cache, h, seq, pos)


class DecodeStep:
    """Buffers and calls of one decode step: append the new tokens' rows, project their
    queries, run absorbed decode over ``seq_len`` rows per sequence. ``fused`` (tensor-core
    dims only) runs the step as the single mla_decode_step call (down-projections in one
    launch, query up-projection fused with the absorption); otherwise as the three calls
    mla_append_cache, mla_project_q and mla_decode_absorbed."""

    def __init__(self, model: DeviceModel, cache: LatentCache, seq_lens: Sequence[int],
                 max_len: Optional[int] = None, fused: bool = False):
        dev = cache.rows.device
        d = model.dims
        self.model, self.cache = model, cache
        self.B = len(seq_lens)
        self.max_len = int(max_len if max_len is not None else max(seq_lens))
        self.seq_len = torch.tensor(list(seq_lens), dtype=torch.int32, device=dev)
        self.pos = (self.seq_len - 1).to(torch.int32)
        self.seq_idx = torch.arange(self.B, dtype=torch.int32, device=dev)
        td = torch_dtype(model.dtype)
        self.q_c = torch.empty((self.B, d.n_h, d.d_hc), dtype=td, device=dev)
        self.q_r = torch.empty((self.B, d.n_h, d.d_hr), dtype=td, device=dev)
        self.o = torch.empty((self.B, d.n_h, d.d_hc), dtype=torch.float32, device=dev)
        self.qws_bytes = mla_project_q_workspace_size(model.abi_dims, self.B)
        self.qws = torch.empty(max(self.qws_bytes, 256), dtype=torch.uint8, device=dev)
        self.ws_bytes = mla_decode_workspace_size(model.abi_dims, self.B, self.max_len)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self._dims, self._w = model.abi_dims, model.abi_weights
        self._cache = cache.abi
        self.fused = bool(fused) and mla_fast_path(self._dims) == 1
        if self.fused:
            self.step_ws_bytes = mla_decode_step_workspace_size(self._dims, self.B, self.max_len)
            self.step_ws = torch.empty(max(self.step_ws_bytes, 256), dtype=torch.uint8, device=dev)

    def append(self, h_new: torch.Tensor, stream=None) -> None:
        mla_append_cache(self._dims, self._w, h_new, self.seq_idx, self.pos, self.B, self._cache,
                         stream)

    def project(self, h_new: torch.Tensor, stream=None) -> None:
        mla_project_q(self._dims, self._w, h_new, self.pos, self.B, self.qws, self.qws_bytes,
                      self.q_c, self.q_r, stream)

    def decode(self, stream=None, q_c=None, q_r=None) -> torch.Tensor:
        mla_decode_absorbed(self._dims, self._w, self.q_c if q_c is None else q_c,
                            self.q_r if q_r is None else q_r, self._cache, self.seq_len, self.B,
                            self.max_len, self.ws, self.ws_bytes, self.o, stream)
        return self.o

    def step(self, h_new: torch.Tensor, stream=None) -> torch.Tensor:
        if self.fused:
            mla_decode_step(self._dims, self._w, h_new, self.pos, self._cache, self.seq_len,
                            self.B, self.max_len, self.step_ws, self.step_ws_bytes, self.o, stream)
            return self.o
        self.append(h_new, stream)
        self.project(h_new, stream)
        return self.decode(stream)


class PrefillStep:
    """Buffers and the call of one causal prefill over sequences packed back to back."""

    def __init__(self, model: DeviceModel, cache: LatentCache, seq_lens: Sequence[int]):
        dev = cache.rows.device
        d = model.dims
        self.model, self.cache = model, cache
        self.B = len(seq_lens)
        self.n_tok = int(sum(seq_lens))
        self.max_T = int(max(seq_lens)) if seq_lens else 0
        cu = np.concatenate([[0], np.cumsum(seq_lens)]).astype(np.int32)
        self.cu = torch.tensor(cu, dtype=torch.int32, device=dev)
        self.o = torch.empty((self.n_tok, d.n_h, d.d_hc), dtype=torch.float32, device=dev)
        self.ws_bytes = mla_prefill_workspace_size(model.abi_dims, self.n_tok, self.B, self.max_T)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self._dims, self._w, self._cache = model.abi_dims, model.abi_weights, cache.abi

    def run(self, h: torch.Tensor, stream=None) -> torch.Tensor:
        mla_prefill(self._dims, self._w, h, self.cu, self.B, self.n_tok, self.max_T, self._cache,
                    self.ws, self.ws_bytes, self.o, stream)
        return self.o
