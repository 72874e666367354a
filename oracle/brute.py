"""Pure-Python scalar MLA for tiny shapes. TEST INFRASTRUCTURE ONLY.

An independent restatement of the explicit per-head formulas of "MLA前向计算流程"
§三分支计算 ①–④ with nothing but Python floats, loops and ``math``: no numpy, no
matrix routines, no shared helpers with ``oracle.mla_ref``. It exists to pin the
vectorised oracle (a transposed operand, a wrong head slice, a dropped RoPE term or a
wrong softmax axis in one of them shows up as a mismatch between the two).
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence


def _matvec(W: List[List[float]], x: Sequence[float]) -> List[float]:
    """y_o = sum_k W[o][k] x[k] for W stored [out][in]."""
    out = []
    for row in W:
        acc = 0.0
        for k in range(len(x)):
            acc += row[k] * x[k]
        out.append(acc)
    return out


def _rope(x: Sequence[float], p: int, base: float) -> List[float]:
    """Rotate (x[2k], x[2k+1]) by p * base^(-2k/len(x))."""
    n = len(x)
    y = [0.0] * n
    for k in range(n // 2):
        a = p * base ** (-2.0 * k / n)
        c, s = math.cos(a), math.sin(a)
        y[2 * k] = x[2 * k] * c - x[2 * k + 1] * s
        y[2 * k + 1] = x[2 * k] * s + x[2 * k + 1] * c
    return y


def _rows(W, lo: int, hi: int):
    return [W[r] for r in range(lo, hi)]


def token_branches(h: Sequence[float], W: Dict[str, list], p: int, dims: dict):
    """All per-token vectors of §三分支计算 for one token at position p."""
    n_h, d_hc, d_hr, base = dims["n_h"], dims["d_hc"], dims["d_hr"], dims["rope_base"]
    c_q = _matvec(W["W_DQ"], h)
    c_kv = _matvec(W["W_DKV"], h)
    k_r = _rope(_matvec(W["W_KR"], h), p, base)
    q_c, q_r, k_c, v = [], [], [], []
    for i in range(n_h):
        q_c.append(_matvec(_rows(W["W_UQ"], i * d_hc, (i + 1) * d_hc), c_q))
        q_r.append(_rope(_matvec(_rows(W["W_QR"], i * d_hr, (i + 1) * d_hr), c_q), p, base))
        k_c.append(_matvec(_rows(W["W_UK"], i * d_hc, (i + 1) * d_hc), c_kv))
        v.append(_matvec(_rows(W["W_UV"], i * d_hc, (i + 1) * d_hc), c_kv))
    return {"c_kv": c_kv, "k_r": k_r, "q_c": q_c, "q_r": q_r, "k_c": k_c, "v": v}


def attention_output(tok: List[dict], t: int, i: int, scale: float) -> List[float]:
    """o_{t,i} = sum_{j<=t} softmax_j((q_{t,i} . k_{j,i}) * scale) v_{j,i}."""
    q = tok[t]["q_c"][i] + tok[t]["q_r"][i]
    s = []
    for j in range(t + 1):
        k = tok[j]["k_c"][i] + tok[j]["k_r"]
        acc = 0.0
        for a, b in zip(q, k):
            acc += a * b
        s.append(acc * scale)
    m = max(s)
    e = [math.exp(x - m) for x in s]
    z = sum(e)
    d_hc = len(tok[0]["v"][i])
    o = [0.0] * d_hc
    for j in range(t + 1):
        w = e[j] / z
        for dd in range(d_hc):
            o[dd] += w * tok[j]["v"][i][dd]
    return o


def prefill(h_rows: List[Sequence[float]], W: Dict[str, list], dims: dict):
    """Causal MLA over one sequence at positions 0..T-1: outputs o[t][i][:] and the
    cache rows [c^KV ; k^R] of every token."""
    scale = 1.0 / math.sqrt(dims["d_hc"] + dims["d_hr"])
    tok = [token_branches(h, W, p, dims) for p, h in enumerate(h_rows)]
    o = [[attention_output(tok, t, i, scale) for i in range(dims["n_h"])]
         for t in range(len(h_rows))]
    rows = [t["c_kv"] + t["k_r"] for t in tok]
    return o, rows


def to_lists(W: dict) -> Dict[str, list]:
    """Convert array-like weights to nested Python lists of floats."""
    return {k: [[float(x) for x in row] for row in v] for k, v in W.items()}


def output_projection(o_heads: List[List[float]], W_O: List[List[float]]) -> List[float]:
    """u = W^O [o_1; ...; o_{n_h}] for one token, with scalar loops: element k of head i is
    input column i * d_hc + k of W^O."""
    d_hc = len(o_heads[0])
    u = []
    for row in W_O:
        acc = 0.0
        for i, oi in enumerate(o_heads):
            for k in range(d_hc):
                acc += row[i * d_hc + k] * oi[k]
        u.append(acc)
    return u


def merge_query_absorption(W_UQ: List[List[float]], W_UK: List[List[float]], n_h: int,
                           d_hc: int) -> List[List[float]]:
    """(W^UK_i)^T W^UQ_i for every head with scalar loops: row i*d_c + l, column c is
    sum over d of W^UK[i*d_hc + d][l] * W^UQ[i*d_hc + d][c]."""
    d_c, d_cq = len(W_UK[0]), len(W_UQ[0])
    out = []
    for i in range(n_h):
        for l in range(d_c):
            row = []
            for c in range(d_cq):
                acc = 0.0
                for d in range(d_hc):
                    acc += W_UK[i * d_hc + d][l] * W_UQ[i * d_hc + d][c]
                row.append(acc)
            out.append(row)
    return out


def select_topk(scores: Sequence[float], k: int) -> List[int]:
    """k rounds of 'take the largest remaining score, the lowest position among equals',
    then the picked positions in increasing order."""
    left = list(range(len(scores)))
    picked = []
    for _ in range(min(k, len(scores))):
        best = left[0]
        for j in left[1:]:
            if scores[j] > scores[best]:
                best = j
        picked.append(best)
        left.remove(best)
    return sorted(picked)


def sparse_attention_output(tok: List[dict], t: int, selected: Sequence[int], i: int,
                            scale: float) -> List[float]:
    """o_{t,i} over the selected key positions only: softmax over j in ``selected`` of
    (q_{t,i} . k_{j,i}) * scale, weights applied to v_{j,i}."""
    q = tok[t]["q_c"][i] + tok[t]["q_r"][i]
    s = []
    for j in selected:
        k = tok[j]["k_c"][i] + tok[j]["k_r"]
        acc = 0.0
        for a, b in zip(q, k):
            acc += a * b
        s.append(acc * scale)
    m = max(s)
    e = [math.exp(x - m) for x in s]
    z = sum(e)
    o = [0.0] * len(tok[0]["v"][i])
    for w_j, j in zip(e, selected):
        for dd in range(len(o)):
            o[dd] += (w_j / z) * tok[j]["v"][i][dd]
    return o
