"""Seeded synthetic inputs for MLA (Multi-head Latent Attention) workloads.

This module only draws random numbers and lays them out; it contains none of the
method's arithmetic. Both the float64 oracle (test infrastructure) and the CUDA
library consume exactly the arrays produced here, so the two sides always see
identical inputs.

Workload shapes follow the symbol table of "MLA前向计算流程" (deepseek-tech-notes,
§符号): d=5120, n_h=128, d_h^C=128, d_h^R=64, d_c'=1536, d_c=512 for the
DeepSeek-V2-shaped cases, plus a tiny fp32 case.

Value distributions: every hidden state h_t ~ N(0, 1); every weight W ~ N(0, 1/fan_in)
where fan_in is the input width of W (stored [out, in], so y = W x).

Random streams: each tensor is drawn from its own stream,
``numpy.random.default_rng([seed, stream_id, index])``, so any tensor (for instance
one sequence's hidden states) can be regenerated alone. Values of bf16 workloads are
rounded to bfloat16 (round-to-nearest-even) once, here, and returned as float32
arrays holding exactly representable bf16 values; ``to_bf16_bits`` gives the raw
16-bit patterns that are uploaded to the device.
"""
from __future__ import annotations

from dataclasses import dataclass, field, asdict
from typing import Dict, List, Optional

import numpy as np

# Stream ids: one per tensor kind (fixed forever so that stored expectations stay valid).
_STREAM = {
    "W_DQ": 1, "W_UQ": 2, "W_QR": 3, "W_DKV": 4, "W_KR": 5, "W_UK": 6, "W_UV": 7,
    "lengths": 8, "h": 9, "aux": 10, "W_O": 11,
}

WEIGHT_NAMES = ("W_DQ", "W_UQ", "W_QR", "W_DKV", "W_KR", "W_UK", "W_UV")


@dataclass(frozen=True)
class Dims:
    """MLA dimensions in the notation of the symbol table (§符号)."""
    d: int          # hidden width d
    n_h: int        # attention heads n_h
    d_hc: int       # per-head content width d_h^C
    d_hr: int       # decoupled RoPE width d_h^R (shared key, per-head query)
    d_c: int        # KV joint latent rank d_c
    d_cq: int       # query latent rank d_c'
    rope_base: float = 10000.0

    @property
    def d_h(self) -> int:
        return self.d_hc + self.d_hr

    @property
    def row(self) -> int:
        """Width of one latent cache row: [c^KV ; k^R]."""
        return self.d_c + self.d_hr

    def weight_shapes(self) -> Dict[str, tuple]:
        return {
            "W_DQ": (self.d_cq, self.d),
            "W_UQ": (self.n_h * self.d_hc, self.d_cq),
            "W_QR": (self.n_h * self.d_hr, self.d_cq),
            "W_DKV": (self.d_c, self.d),
            "W_KR": (self.d_hr, self.d),
            "W_UK": (self.n_h * self.d_hc, self.d_c),
            "W_UV": (self.n_h * self.d_hc, self.d_c),
        }


V2 = Dims(d=5120, n_h=128, d_hc=128, d_hr=64, d_c=512, d_cq=1536)
TINY = Dims(d=64, n_h=4, d_hc=16, d_hr=8, d_c=32, d_cq=48)


@dataclass
class Workload:
    """One named workload: dims, dtype, and the per-sequence lengths.

    For decode workloads ``seq_lens[b]`` is the number of cache rows sequence b attends
    to after this step's append; the last of them (position seq_lens[b]-1) is the new
    token, whose hidden state is also the query's input. For prefill workloads it is
    the number of prompt tokens of sequence b (positions 0..T_b-1).
    """
    name: str
    dims: Dims
    dtype: str                     # "f32" or "bf16"
    kind: str                      # "decode" or "prefill"
    seq_lens: List[int]
    seed: int = 0
    note: str = ""

    @property
    def B(self) -> int:
        return len(self.seq_lens)

    @property
    def n_rows(self) -> int:
        return int(sum(self.seq_lens))

    def describe(self) -> dict:
        out = asdict(self)
        out["dims"] = asdict(self.dims)
        if len(self.seq_lens) > 8:
            out["seq_lens"] = {"B": self.B, "sum": self.n_rows,
                               "min": int(min(self.seq_lens)), "max": int(max(self.seq_lens))}
        return out


def ragged_lengths(seed: int, B: int, lo: int, hi: int) -> List[int]:
    """Per-sequence context lengths drawn uniformly from the integers [lo, hi]."""
    rng = np.random.default_rng([seed, _STREAM["lengths"]])
    return [int(x) for x in rng.integers(lo, hi + 1, B)]


def workload(name: str, seed: int = 0) -> Workload:
    """The named workloads (tiny fp32 check, V2-shaped decode and prefill cases)."""
    if name == "tiny_f32":
        # 64 context tokens at positions 0..63 plus one new token at position 64.
        return Workload(name, TINY, "f32", "decode", [65], seed,
                        "batch 1, 64 cached tokens + 1 decoded token")
    if name == "v2_decode_b16_l4096":
        return Workload(name, V2, "bf16", "decode", [4096] * 16, seed,
                        "batch 16, every sequence at context 4096")
    if name == "v2_decode_b1_l131072":
        return Workload(name, V2, "bf16", "decode", [131072], seed,
                        "batch 1 at context 131072")
    if name == "v2_decode_b4_l32768":
        return Workload(name, V2, "bf16", "decode", [32768] * 4, seed,
                        "batch 4 at context 32768")
    if name == "v2_decode_b128_ragged":
        lens = [L + 1 for L in ragged_lengths(seed, 128, 1024, 8192)]
        return Workload(name, V2, "bf16", "decode", lens, seed,
                        "batch 128, lengths U[1024,8192] + the appended token")
    if name == "v2_prefill_b2_t4096":
        return Workload(name, V2, "bf16", "prefill", [4096, 4096], seed,
                        "causal prefill, batch 2 x 4096 tokens")
    raise KeyError(name)


WORKLOADS = ("tiny_f32", "v2_decode_b16_l4096", "v2_decode_b1_l131072",
             "v2_decode_b4_l32768", "v2_decode_b128_ragged", "v2_prefill_b2_t4096")


# ---------------------------------------------------------------------------------
# bfloat16 storage (input preparation only)
# ---------------------------------------------------------------------------------

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); float32 result."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(x.shape)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Raw bf16 bit patterns (uint16) of float32 values that are already bf16-exact."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _finish(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(dtype)


def weights(dims: Dims, dtype: str, seed: int = 0) -> Dict[str, np.ndarray]:
    """All seven projection matrices, each [out, in], W ~ N(0, 1/in)."""
    out = {}
    for name, (o, i) in dims.weight_shapes().items():
        rng = np.random.default_rng([seed, _STREAM[name]])
        w = rng.standard_normal((o, i), dtype=np.float32) * np.float32(1.0 / np.sqrt(i))
        out[name] = _finish(w, dtype)
    return out


def output_weight(dims: Dims, dtype: str, seed: int = 0) -> np.ndarray:
    """The output projection W^O [d, n_h * d_h^C], W ~ N(0, 1/(n_h d_h^C)); drawn apart from
    the seven MLA matrices (it is 168 MB at the V2 widths)."""
    fan_in = dims.n_h * dims.d_hc
    rng = np.random.default_rng([seed, _STREAM["W_O"]])
    w = rng.standard_normal((dims.d, fan_in), dtype=np.float32) * np.float32(1.0 / np.sqrt(fan_in))
    return _finish(w, dtype)


def hidden(dims: Dims, dtype: str, seq: int, n: int, seed: int = 0, start: int = 0) -> np.ndarray:
    """Hidden states h of sequence ``seq`` at positions start..start+n-1, [n, d], ~N(0,1).

    Rows are drawn in position order from the sequence's own stream, so a prefix of a
    longer draw equals a shorter draw.
    """
    rng = np.random.default_rng([seed, _STREAM["h"], seq])
    if start:
        rng.standard_normal((start, dims.d), dtype=np.float32)  # advance the stream
    h = rng.standard_normal((n, dims.d), dtype=np.float32)
    return _finish(h, dtype)


def hidden_rows(dims: Dims, dtype: str, seq: int, positions, seed: int = 0) -> np.ndarray:
    """Hidden states of sequence ``seq`` at arbitrary positions (draws the prefix)."""
    positions = np.asarray(positions, dtype=np.int64)
    n = int(positions.max()) + 1 if positions.size else 0
    return hidden(dims, dtype, seq, n, seed)[positions]


def packed_layout(seq_lens, guard: int = 0) -> np.ndarray:
    """Row base of each sequence when sequences are packed back to back in one cache,
    optionally with ``guard`` spare rows after each sequence (used to poison gaps)."""
    base = np.zeros(len(seq_lens), dtype=np.int64)
    acc = 0
    for b, L in enumerate(seq_lens):
        base[b] = acc
        acc += int(L) + guard
    return base


def aux_normal(shape, seed: int = 0, index: int = 0, dtype: str = "f32", scale: float = 1.0) -> np.ndarray:
    """Extra N(0, scale^2) tensors for kernel-level tests (e.g. synthetic queries)."""
    rng = np.random.default_rng([seed, _STREAM["aux"], index])
    return _finish(rng.standard_normal(shape, dtype=np.float32) * np.float32(scale), dtype)
