"""Shared test helpers: tolerances, error metrics, and oracle expectations for workloads.

Expected values come only from ``oracle`` (float64) on inputs from ``mla_inputs``.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

import mla_inputs as mi
from oracle import mla_ref as ref

# Tolerances (max|err| / max|ref|, RMS relative error) per storage type.
TOL = {"bf16": (1e-2, 3e-3), "f32": (1e-5, 1e-5)}


def rel_errors(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    err = got - want
    denom = np.max(np.abs(want))
    max_rel = float(np.max(np.abs(err)) / denom) if denom > 0 else float(np.max(np.abs(err)))
    ss = float(np.sum(want * want))
    rms_rel = float(np.sqrt(np.sum(err * err) / ss)) if ss > 0 else float(np.sqrt(np.mean(err * err)))
    return max_rel, rms_rel


def assert_close(got, want, dtype: str, what: str = ""):
    max_rel, rms_rel = rel_errors(got, want)
    tmax, trms = TOL[dtype]
    assert max_rel <= tmax and rms_rel <= trms, (
        "%s: max_rel %.3e (tol %.0e), rms_rel %.3e (tol %.0e)" % (what, max_rel, tmax, rms_rel, trms))
    return max_rel, rms_rel


def oracle_weights(dims, dtype):
    W = mi.weights(dims, dtype)
    return W, {k: v.astype(np.float64) for k, v in W.items()}


def oracle_sequence_rows(dims, dtype, W64, seq: int, L: int, seed: int = 0):
    """Cache rows of sequence ``seq`` at positions 0..L-1 (stored in ``dtype``) and the
    float64 values before storage."""
    h = mi.hidden(dims, dtype, seq, L, seed)
    c, kr = ref.kv_latent(h, W64["W_DKV"], W64["W_KR"], np.arange(L), dims.rope_base)
    exact = ref.cache_rows(c, kr)
    return ref.store(exact, dtype), exact, h


def oracle_query(dims, dtype, W64, h_row, pos: int):
    q_c, q_r = ref.query(h_row[None, :], W64["W_DQ"], W64["W_UQ"], W64["W_QR"], [pos], dims.n_h,
                         dims.d_hc, dims.d_hr, dims.rope_base)
    return ref.store(q_c[0], dtype), ref.store(q_r[0], dtype), q_c[0], q_r[0]


def oracle_decode_step(wl: mi.Workload, W64, seqs: Optional[Sequence[int]] = None,
                       heads: Optional[Sequence[int]] = None):
    """Expected decode outputs of a workload for sequences ``seqs`` and ``heads``: each
    sequence's rows 0..L-1 come from its hidden states (the last one is the new token),
    the query from the new token; cache rows and q are held in the workload's dtype."""
    dims, dtype = wl.dims, wl.dtype
    seqs = list(range(wl.B)) if seqs is None else list(seqs)
    out = {"o": [], "rows": [], "rows_exact": [], "q_c": [], "q_r": [], "q_c_exact": [],
           "q_r_exact": []}
    for b in seqs:
        L = wl.seq_lens[b]
        rows, exact, h = oracle_sequence_rows(dims, dtype, W64, b, L, wl.seed)
        q_c, q_r, q_c_x, q_r_x = oracle_query(dims, dtype, W64, h[L - 1], L - 1)
        o = ref.decode_explicit(q_c[None], q_r[None], [rows], W64["W_UK"], W64["W_UV"], dims.d_c,
                                heads=heads)
        out["o"].append(o[0])
        out["rows"].append(rows)
        out["rows_exact"].append(exact)
        out["q_c"].append(q_c)
        out["q_r"].append(q_r)
        out["q_c_exact"].append(q_c_x)
        out["q_r_exact"].append(q_r_x)
    return out
