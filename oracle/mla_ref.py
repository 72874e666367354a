"""Float64 CPU oracle for Multi-head Latent Attention (MLA). TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this module. The CUDA library never calls it and shares no code with it.

What it computes is the plain, explicit per-head definition of MLA, in the order and
notation of the pages:

* "MLA前向计算流程" (deepseek-tech-notes 02-MLA低秩注意力), §三分支计算 ① Query,
  ② Key, ③ Value, ④ 注意力与输出, and §符号 for the dimension names;
* the absorbed form used for decoding, from "从LLaMA到DeepSeek[01] - MLA（上）"
  §六 (associativity: transform the query once, multiply it with the cached latent).

Conventions (readings of the pages where they are silent or garbled):

* every matrix is stored [out, in] and applied as y = W x (§流程图 gives
  W^UQ as [16384 x 1536], W^QR as [8192 x 1536], W^KR as [64 x 5120]);
* the head-i block of W^UQ / W^UK / W^UV is rows i*d_h^C .. (i+1)*d_h^C-1, the head-i
  block of W^QR is rows i*d_h^R .. (i+1)*d_h^R-1;
* q^R is per head ([n_h, d_h^R], §流程图), k^R is one [d_h^R] vector shared by all
  heads (§三分支计算 ② Key);
* RoPE rotates consecutive pairs (2k, 2k+1) by the angle p * base^(-2k/d_h^R), with
  0-based positions p and base 10000 ("多头潜在注意力" article, §RoPE, pairs
  consecutive dimensions; the frequency schedule is the standard one);
* the softmax scale is 1/sqrt(d_h^C + d_h^R) and the sum runs over j = 1..t, the
  query token included (§三分支计算 ④);
* no W^O: the output is the per-head o_{t,i};
* no normalisation of the latents.

Everything is float64. The caller passes the exact values the GPU receives (already
rounded to the workload's storage type by the input generator).
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------------
# Storage rounding (the bf16 workloads store the latent cache and the query
# projections in bfloat16; the oracle rounds its own float64 values the same way)
# ---------------------------------------------------------------------------------

def round_bf16(x) -> np.ndarray:
    """Round float64 values directly to the nearest bfloat16 value (ties to even).

    bfloat16 keeps 8 significant bits: x = m * 2^e with 0.5 <= |m| < 1, so the kept
    value is rint(m * 2^8) * 2^(e-8). Values outside the bf16 normal range do not
    occur in these workloads.
    """
    x = _f64(x)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def store(x, dtype: str) -> np.ndarray:
    """Value after storage in ``dtype`` ("f32" keeps float64 precision for the oracle's
    purposes: the fp32 workload's tolerance is far above fp32 rounding)."""
    if dtype == "bf16":
        return round_bf16(x)
    return _f64(x)


# ---------------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------------

def rope_freqs(d_r: int, base: float) -> np.ndarray:
    """theta_k = base^(-2k/d_r), k = 0 .. d_r/2-1 (one angle step per consecutive pair)."""
    k = np.arange(d_r // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * k / d_r)


def rope(x, pos, base: float) -> np.ndarray:
    """Rotate consecutive pairs (x_{2k}, x_{2k+1}) of the last axis by pos * theta_k.

    ``pos`` broadcasts against x.shape[:-1]. [x', y'] = [x cos a - y sin a, x sin a + y cos a].
    """
    x = _f64(x)
    d_r = x.shape[-1]
    if d_r % 2:
        raise ValueError("RoPE width must be even")
    ang = _f64(pos)[..., None] * rope_freqs(d_r, base)
    c, s = np.cos(ang), np.sin(ang)
    xe, xo = x[..., 0::2], x[..., 1::2]
    out = np.empty(np.broadcast_shapes(x.shape, ang.shape[:-1] + (d_r,)), dtype=np.float64)
    out[..., 0::2] = xe * c - xo * s
    out[..., 1::2] = xe * s + xo * c
    return out


# ---------------------------------------------------------------------------------
# The three branches (§三分支计算)
# ---------------------------------------------------------------------------------

def kv_latent(h, W_DKV, W_KR, pos, base: float):
    """② Key / ③ Value compression: c^KV_t = W^DKV h_t, k^R_t = RoPE(W^KR h_t) at pos_t.

    h [n, d] -> c_kv [n, d_c], k_r [n, d_h^R]. These two are all that is cached
    (§KV Cache 里到底存什么: c^KV + the shared k^R, 512 + 64 = 576 values per token).
    """
    h = _f64(h)
    c_kv = h @ _f64(W_DKV).T
    k_r = rope(h @ _f64(W_KR).T, pos, base)
    return c_kv, k_r


def cache_rows(c_kv, k_r) -> np.ndarray:
    """One latent-cache row per token: [c^KV_t ; k^R_t]."""
    return np.concatenate([_f64(c_kv), _f64(k_r)], axis=-1)


def query(h, W_DQ, W_UQ, W_QR, pos, n_h: int, d_hc: int, d_hr: int, base: float):
    """① Query: c^Q = W^DQ h; q^C = W^UQ c^Q split per head; q^R = RoPE(W^QR c^Q) per head.

    h [n, d] -> q_c [n, n_h, d_h^C], q_r [n, n_h, d_h^R].
    """
    h = _f64(h)
    n = h.shape[0]
    c_q = h @ _f64(W_DQ).T
    q_c = (c_q @ _f64(W_UQ).T).reshape(n, n_h, d_hc)
    q_r = rope((c_q @ _f64(W_QR).T).reshape(n, n_h, d_hr), _f64(pos)[:, None], base)
    return q_c, q_r


def expand_kv(c_kv, W_UK, W_UV, n_h: int, d_hc: int, heads: Optional[Sequence[int]] = None):
    """② Key / ③ Value up-projection: k^C_{j,i} = W^UK_i c_j, v_{j,i} = W^UV_i c_j.

    c_kv [L, d_c] -> k_c, v [L, len(heads), d_h^C].
    """
    c = _f64(c_kv)
    W_UK = _f64(W_UK).reshape(n_h, d_hc, -1)
    W_UV = _f64(W_UV).reshape(n_h, d_hc, -1)
    if heads is not None:
        W_UK, W_UV = W_UK[list(heads)], W_UV[list(heads)]
    k_c = np.einsum("hdc,lc->lhd", W_UK, c)
    v = np.einsum("hdc,lc->lhd", W_UV, c)
    return k_c, v


def softmax(s, axis: int = -1) -> np.ndarray:
    """Naive softmax: subtract the maximum, exponentiate, divide by the sum."""
    s = _f64(s)
    e = np.exp(s - np.max(s, axis=axis, keepdims=True))
    return e / np.sum(e, axis=axis, keepdims=True)


def default_scale(d_hc: int, d_hr: int) -> float:
    """1/sqrt(d_h^C + d_h^R) (§三分支计算 ④)."""
    return 1.0 / math.sqrt(d_hc + d_hr)


def attend(q_c, q_r, k_c, k_r, v, scale: float) -> np.ndarray:
    """④ for one query token: o_i = sum_j softmax_j(q_i . k_{j,i} * scale) v_{j,i},
    with q_i = [q^C_i ; q^R_i] and k_{j,i} = [k^C_{j,i} ; k^R_j].

    q_c [H, d_hc], q_r [H, d_hr], k_c [L, H, d_hc], k_r [L, d_hr], v [L, H, d_hc] -> [H, d_hc].
    """
    s = (np.einsum("hd,lhd->hl", _f64(q_c), _f64(k_c))
         + np.einsum("hd,ld->hl", _f64(q_r), _f64(k_r))) * scale
    p = softmax(s, axis=-1)
    return np.einsum("hl,lhd->hd", p, _f64(v))


# ---------------------------------------------------------------------------------
# Decode (one query token per sequence) over the latent cache
# ---------------------------------------------------------------------------------

def decode_explicit(q_c, q_r, rows: List[np.ndarray], W_UK, W_UV, d_c: int,
                    scale: Optional[float] = None,
                    heads: Optional[Sequence[int]] = None) -> np.ndarray:
    """Non-absorbed decode: read c_j from the cache, up-project K/V per head, attend.

    q_c [B, n_h, d_hc], q_r [B, n_h, d_hr]; rows[b] = the L_b cache rows [L_b, d_c+d_hr]
    that sequence b attends to (positions 0..L_b-1, the query token's own row last).
    Returns o [B, len(heads), d_hc].
    """
    q_c, q_r = _f64(q_c), _f64(q_r)
    B, n_h, d_hc = q_c.shape
    d_hr = q_r.shape[-1]
    if scale is None:
        scale = default_scale(d_hc, d_hr)
    hs = list(range(n_h)) if heads is None else list(heads)
    out = np.zeros((B, len(hs), d_hc))
    for b in range(B):
        r = _f64(rows[b])
        if r.shape[0] == 0:
            continue
        k_c, v = expand_kv(r[:, :d_c], W_UK, W_UV, n_h, d_hc, hs)
        out[b] = attend(q_c[b, hs], q_r[b, hs], k_c, r[:, d_c:], v, scale)
    return out


def merge_query_absorption(W_UQ, W_UK, n_h: int, d_hc: int) -> np.ndarray:
    """The absorbed query map formed once ("从LLaMA到DeepSeek" §六: both factors are fixed):
    W^UQK_i = (W^UK_i)^T W^UQ_i for every head, stacked head by head.

    W_UQ [n_h*d_hc, d_cq], W_UK [n_h*d_hc, d_c] -> [n_h*d_c, d_cq].
    """
    uq = _f64(W_UQ).reshape(n_h, d_hc, -1)
    uk = _f64(W_UK).reshape(n_h, d_hc, -1)
    return np.einsum("hdl,hdc->hlc", uk, uq).reshape(-1, uq.shape[-1])


def output_projection(o, W_O) -> np.ndarray:
    """④ output: u_t = W^O [o_{t,1}; ...; o_{t,n_h}], the per-head outputs of token t
    concatenated head by head and mapped back to the hidden width.

    o [..., n_h, d_hc], W_O [d, n_h * d_hc] -> u [..., d].
    """
    o = _f64(o)
    return o.reshape(o.shape[:-2] + (o.shape[-2] * o.shape[-1],)) @ _f64(W_O).T


def absorb_query(q_c, W_UK, n_h: int, d_hc: int) -> np.ndarray:
    """q~_i = (W^UK_i)^T q^C_i, the latent-space query ("从LLaMA到DeepSeek" §六).

    q_c [..., n_h, d_hc] -> [..., n_h, d_c].
    """
    W = _f64(W_UK).reshape(n_h, d_hc, -1)
    return np.einsum("hdc,...hd->...hc", W, _f64(q_c))


def decode_absorbed(q_c, q_r, rows: List[np.ndarray], W_UK, W_UV, d_c: int,
                    scale: Optional[float] = None) -> np.ndarray:
    """Absorbed decode in float64 (used only to pin the explicit form by associativity):

    score_{i,j} = (q~_i . c_j + q^R_i . k^R_j) * scale, p = softmax_j,
    o~_i = sum_j p_{i,j} c_j, o_i = W^UV_i o~_i.
    """
    q_c, q_r = _f64(q_c), _f64(q_r)
    B, n_h, d_hc = q_c.shape
    d_hr = q_r.shape[-1]
    if scale is None:
        scale = default_scale(d_hc, d_hr)
    qt = absorb_query(q_c, W_UK, n_h, d_hc)
    W_UV = _f64(W_UV).reshape(n_h, d_hc, -1)
    out = np.zeros((B, n_h, d_hc))
    for b in range(B):
        r = _f64(rows[b])
        if r.shape[0] == 0:
            continue
        c, kr = r[:, :d_c], r[:, d_c:]
        s = (qt[b] @ c.T + q_r[b] @ kr.T) * scale
        p = softmax(s, axis=-1)
        o_lat = p @ c
        out[b] = np.einsum("hdc,hc->hd", W_UV, o_lat)
    return out


# ---------------------------------------------------------------------------------
# Prefill (non-absorbed, causal) for one sequence
# ---------------------------------------------------------------------------------

def prefill_sequence(h, W: Dict[str, np.ndarray], n_h: int, d_hc: int, d_hr: int, d_c: int,
                     base: float, cache_dtype: str = "f32", scale: Optional[float] = None,
                     heads: Optional[Sequence[int]] = None,
                     queries: Optional[Sequence[int]] = None):
    """Causal prefill of one sequence with positions 0..T-1 (MHA-style expansion).

    The latent cache rows [c^KV ; k^R] are produced first and held in ``cache_dtype``;
    K^C and V are expanded from those stored rows, so prefill and later decode steps
    read the same latent values. Queries come from h directly. Output o[t, i] for t in
    ``queries`` (default all) and i in ``heads`` (default all); also returns the rows.
    """
    h = _f64(h)
    T = h.shape[0]
    pos = np.arange(T, dtype=np.float64)
    c_kv, k_r = kv_latent(h, W["W_DKV"], W["W_KR"], pos, base)
    rows = store(cache_rows(c_kv, k_r), cache_dtype)
    hs = list(range(n_h)) if heads is None else list(heads)
    ts = list(range(T)) if queries is None else list(queries)
    if scale is None:
        scale = default_scale(d_hc, d_hr)
    h_q = h[ts]
    q_c, q_r = query(h_q, W["W_DQ"], W["W_UQ"], W["W_QR"], pos[ts], n_h, d_hc, d_hr, base)
    k_c, v = expand_kv(rows[:, :d_c], W["W_UK"], W["W_UV"], n_h, d_hc, hs)
    kr = rows[:, d_c:]
    out = np.zeros((len(ts), len(hs), d_hc))
    for n, t in enumerate(ts):
        out[n] = attend(q_c[n, hs], q_r[n, hs], k_c[: t + 1], kr[: t + 1], v[: t + 1], scale)
    return out, rows


# ---------------------------------------------------------------------------------
# Cache size arithmetic (§流程图 缓存总量, §KV Cache 里到底存什么; "从LLaMA到DeepSeek" §五)
# ---------------------------------------------------------------------------------

def cache_counts(n_h: int, d_hc: int, d_hr: int, d_c: int, d_cq: int) -> Dict[str, float]:
    """Values cached per token per layer, and the compression ratios, as the pages count them."""
    mha = 2 * n_h * d_hc                  # n_h keys + n_h values of width d_h^C
    mla = d_c + d_hr                      # c^KV + the shared k^R
    uncompressed = n_h * d_hc + d_hr      # MLA without the latent: per-head K^C plus shared k^R
    return {
        "mha": mha,
        "mla": mla,
        "mla_uncompressed": uncompressed,
        "mha_over_mla": mha / mla,
        "gqa_groups_equivalent": mla / (2 * d_hc),   # groups g with 2*g*d_h = MLA count
        "ratio_c_q": n_h * d_hc / d_cq,
        "ratio_c_kv": n_h * d_hc / d_c,
        "ratio_k_r": n_h * d_hr / d_hr,
    }


# ---------------------------------------------------------------------------------
# Top-k sparse selection before the decode ("MLA前向计算流程", version table, V3.2 + DSA
# row: MLA itself is unchanged; an indexer picks top-k over the latent sequence and the core
# attention still runs MLA over what was picked)
# ---------------------------------------------------------------------------------

def select_topk(scores, L: int, k: int) -> np.ndarray:
    """Positions of the k largest index scores among positions 0..L-1, in increasing position
    order. Equal scores rank the lower position first (-0.0 equals +0.0); L <= k selects every
    position. The indexer that produces the scores is not defined by the pages: they are an
    input here."""
    s = np.asarray(scores, dtype=np.float64)[:L]
    if L <= k:
        return np.arange(L)
    order = np.lexsort((np.arange(L), -s))  # primary key: score, descending; then position
    return np.sort(order[:k])


def decode_sparse(q_c, q_r, rows: List[np.ndarray], scores: List[np.ndarray], k: int, W_UK,
                  W_UV, d_c: int, scale: Optional[float] = None,
                  heads: Optional[Sequence[int]] = None) -> np.ndarray:
    """Decode of sequence b over its selected rows only: the same per-head attention as
    ``decode_explicit`` with rows[b] replaced by rows[b][select_topk(scores[b], L_b, k)].
    Every head attends to the same selected positions (the selection is over the shared
    latent sequence)."""
    picked = [_f64(r)[select_topk(sc, len(r), k)] for r, sc in zip(rows, scores)]
    return decode_explicit(q_c, q_r, picked, W_UK, W_UV, d_c, scale=scale, heads=heads)
