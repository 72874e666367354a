"""Pins for the float64 oracle, against what the MLA pages and the mathematics fix.

None of these re-types the oracle's formula: each checks it against an independent
fact (a printed figure, a closed form, an invariant, brute force, or the absorbed form).
"""
import json
import math
import os

import numpy as np
import pytest

import mla_inputs as mi
from oracle import brute
from oracle import mla_ref as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")

# A shape small enough for pure-Python loops, with every width distinct so that a
# transposed or mis-sliced operand cannot go unnoticed.
MICRO = mi.Dims(d=7, n_h=3, d_hc=5, d_hr=4, d_c=6, d_cq=9)


def _dims_dict(d):
    return {"n_h": d.n_h, "d_hc": d.d_hc, "d_hr": d.d_hr, "rope_base": d.rope_base}


def _seq(dims, T, dtype="f32", seq=0):
    W = mi.weights(dims, dtype)
    h = mi.hidden(dims, dtype, seq, T)
    return W, h


# ------------------------------------------------------------------ page figures

def test_cache_counts_match_printed_figures():
    g = json.load(open(GOLDEN))
    v2 = g["v2_dims"]["value"]
    c = ref.cache_counts(v2["n_h"], v2["d_hc"], v2["d_hr"], v2["d_c"], v2["d_cq"])
    pc = g["cache_values_per_token"]["value"]
    assert c["mha"] == pc["mha"]
    assert c["mla"] == pc["mla"]
    assert c["mla_uncompressed"] == pc["mla_uncompressed"]
    assert round(c["mha_over_mla"]) == pc["mha_over_mla_approx"]
    assert c["gqa_groups_equivalent"] == g["gqa_groups_equivalent"]["value"]
    r = g["compression_ratios"]["value"]
    assert round(c["ratio_c_q"]) == r["c_q"]
    assert c["ratio_c_kv"] == r["c_kv"]
    assert c["ratio_k_r"] == r["k_r"]
    assert v2["d_h"] == v2["d_hc"] + v2["d_hr"]
    # absorbed per-head product width: d_c vs d_h^C
    assert v2["d_c"] // v2["d_hc"] == g["absorbed_width_factor"]["value"]


def test_weight_and_head_shapes_match_printed_shapes():
    g = json.load(open(GOLDEN))
    shapes = mi.V2.weight_shapes()
    for name, shp in g["weight_shapes"]["value"].items():
        assert list(shapes[name]) == shp
    # query shapes per head and the shared k^R, from a real (tiny-token) run at V2 widths
    W = {k: np.zeros(v, dtype=np.float32) for k, v in shapes.items()}
    h = np.zeros((1, mi.V2.d))
    q_c, q_r = ref.query(h, W["W_DQ"], W["W_UQ"], W["W_QR"], [0], 128, 128, 64, 1e4)
    _, k_r = ref.kv_latent(h, W["W_DKV"], W["W_KR"], [0], 1e4)
    ps = g["per_head_query_shapes"]["value"]
    assert list(q_c.shape[1:]) == ps["q_c"] and list(q_r.shape[1:]) == ps["q_r"]
    assert list(k_r.shape[1:]) == ps["k_r"]


# ------------------------------------------------------------------ RoPE

def test_rope_is_identity_at_position_zero():
    x = mi.aux_normal((5, 16), index=1)
    np.testing.assert_array_equal(ref.rope(x, np.zeros(5), 1e4), x.astype(np.float64))


def test_rope_rotates_unit_vectors_by_the_frequency_schedule():
    # e_{2k} at position p must land on (cos(p*theta_k), sin(p*theta_k)) in slots (2k, 2k+1)
    # with theta_k = 10000^(-2k/d); nothing else may move (consecutive-pair interleaving).
    d = 8
    for k in range(d // 2):
        e = np.zeros(d)
        e[2 * k] = 1.0
        p = 7
        y = ref.rope(e, p, 10000.0)
        th = p * 10000.0 ** (-2.0 * k / d)
        want = np.zeros(d)
        want[2 * k], want[2 * k + 1] = math.cos(th), math.sin(th)
        np.testing.assert_allclose(y, want, atol=1e-15)
        # the odd slot of the pair rotates into (-sin, cos)
        e = np.zeros(d)
        e[2 * k + 1] = 1.0
        y = ref.rope(e, p, 10000.0)
        want = np.zeros(d)
        want[2 * k], want[2 * k + 1] = -math.sin(th), math.cos(th)
        np.testing.assert_allclose(y, want, atol=1e-15)


def test_rope_preserves_norm_and_depends_only_on_relative_position():
    x = mi.aux_normal((64,), index=2).astype(np.float64)
    y = mi.aux_normal((64,), index=3).astype(np.float64)
    for p in (0, 1, 17, 4095, 131071):
        assert abs(np.linalg.norm(ref.rope(x, p, 1e4)) - np.linalg.norm(x)) < 1e-12
    for p, q in ((5, 2), (100, 97), (131071, 131068)):
        a = ref.rope(x, p, 1e4) @ ref.rope(y, q, 1e4)
        b = ref.rope(x, p - q, 1e4) @ y
        assert abs(a - b) < 1e-9


# ------------------------------------------------------------------ softmax / attention

def test_softmax_rows_sum_to_one():
    s = mi.aux_normal((17, 333), index=4, scale=8.0)
    p = ref.softmax(s)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
    assert (p > 0).all()


def test_two_key_attention_is_logistic_in_the_scaled_score_gap():
    # With two keys the weights are sigma(Delta) and 1-sigma(Delta), Delta being the score
    # gap times 1/sqrt(d_h^C + d_h^R); this fixes the scale and the [content; rope] concat.
    rng = np.random.default_rng(5)
    H, dc, dr = 2, 3, 2
    q_c, q_r = rng.standard_normal((H, dc)), rng.standard_normal((H, dr))
    k_c, k_r = rng.standard_normal((2, H, dc)), rng.standard_normal((2, dr))
    v = rng.standard_normal((2, H, dc))
    scale = 1.0 / math.sqrt(dc + dr)
    o = ref.attend(q_c, q_r, k_c, k_r, v, scale)
    for i in range(H):
        s0 = (sum(q_c[i] * k_c[0, i]) + sum(q_r[i] * k_r[0])) * scale
        s1 = (sum(q_c[i] * k_c[1, i]) + sum(q_r[i] * k_r[1])) * scale
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        np.testing.assert_allclose(o[i], w0 * v[0, i] + (1 - w0) * v[1, i], rtol=1e-13)


def test_length_one_context_returns_v_exactly():
    dims = mi.V2
    W = mi.weights(mi.Dims(d=64, n_h=128, d_hc=128, d_hr=64, d_c=512, d_cq=96), "bf16")
    rows = [mi.aux_normal((1, dims.row), index=5, dtype="bf16").astype(np.float64)]
    q_c = mi.aux_normal((1, 128, 128), index=6, dtype="bf16")
    q_r = mi.aux_normal((1, 128, 64), index=7, dtype="bf16")
    o = ref.decode_explicit(q_c, q_r, rows, W["W_UK"], W["W_UV"], 512)
    v = (W["W_UV"].astype(np.float64).reshape(128, 128, 512) @ rows[0][0, :512])
    np.testing.assert_array_equal(o[0], v)


# ------------------------------------------------------------------ absorption

@pytest.mark.parametrize("dims,L", [(MICRO, 5), (mi.TINY, 65),
                                    (mi.Dims(d=32, n_h=128, d_hc=128, d_hr=64, d_c=512, d_cq=64), 37)])
def test_absorbed_equals_explicit(dims, L):
    """Associativity ("从LLaMA到DeepSeek" §六): (W^UK_i^T q) . c == q . (W^UK_i c), and the same
    for W^UV on the output side; the two decode forms must agree to float64 rounding."""
    W = mi.weights(dims, "f32")
    B = 3
    rows = [mi.aux_normal((L - b, dims.row), index=10 + b).astype(np.float64) for b in range(B)]
    q_c = mi.aux_normal((B, dims.n_h, dims.d_hc), index=20)
    q_r = mi.aux_normal((B, dims.n_h, dims.d_hr), index=21)
    a = ref.decode_explicit(q_c, q_r, rows, W["W_UK"], W["W_UV"], dims.d_c)
    b = ref.decode_absorbed(q_c, q_r, rows, W["W_UK"], W["W_UV"], dims.d_c)
    assert np.max(np.abs(a - b)) / np.max(np.abs(a)) <= 1e-12


def test_heads_attend_differently_with_the_same_query():
    """"从LLaMA到DeepSeek" §四: two heads given the same query still weight the tokens
    differently because each makes its own K from the shared latent."""
    dims = MICRO
    W = mi.weights(dims, "f32")
    rows = mi.aux_normal((6, dims.row), index=30).astype(np.float64)
    q = mi.aux_normal((dims.d_hc,), index=31)
    k_c, _ = ref.expand_kv(rows[:, :dims.d_c], W["W_UK"], W["W_UV"], dims.n_h, dims.d_hc)
    p0 = ref.softmax(k_c[:, 0] @ q)
    p1 = ref.softmax(k_c[:, 1] @ q)
    assert np.max(np.abs(p0 - p1)) > 1e-3


# ------------------------------------------------------------------ brute force

@pytest.mark.parametrize("dims,T", [(MICRO, 4), (mi.TINY, 9)])
def test_vectorised_prefill_matches_scalar_brute_force(dims, T):
    W, h = _seq(dims, T)
    o, rows = ref.prefill_sequence(h, W, dims.n_h, dims.d_hc, dims.d_hr, dims.d_c, dims.rope_base)
    ob, rb = brute.prefill([list(map(float, r)) for r in h], brute.to_lists(W), _dims_dict(dims))
    np.testing.assert_allclose(rows, np.array(rb), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o, np.array(ob), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("dims", [MICRO, mi.TINY])
def test_output_projection_matches_scalar_brute_force(dims):
    """u = W^O [o_1; ...; o_{n_h}]: the head-major concatenation against scalar loops, on
    shapes where every width differs (a head/feature transposition cannot go unnoticed)."""
    W_O = mi.output_weight(dims, "f32")
    assert W_O.shape == (dims.d, dims.n_h * dims.d_hc)
    o = mi.aux_normal((3, dims.n_h, dims.d_hc), index=40)
    u = ref.output_projection(o, W_O)
    Wl = [[float(x) for x in row] for row in W_O]
    for t in range(3):
        ub = brute.output_projection([[float(x) for x in oi] for oi in o[t]], Wl)
        np.testing.assert_allclose(u[t], ub, rtol=1e-12, atol=1e-12)
    # one head's output reaches u only through its own block of W^O
    one = np.zeros((dims.n_h, dims.d_hc))
    one[1, 2] = 1.0
    np.testing.assert_allclose(ref.output_projection(one, W_O), W_O[:, dims.d_hc + 2], atol=0)


def test_merged_absorption_matches_brute_force_and_associativity():
    """W^UQK_i = (W^UK_i)^T W^UQ_i: scalar loops on a shape with distinct widths, and applying
    the merged map to c^Q gives the absorbed query of the explicit two-step form."""
    dims = MICRO
    W = mi.weights(dims, "f32")
    M = ref.merge_query_absorption(W["W_UQ"], W["W_UK"], dims.n_h, dims.d_hc)
    assert M.shape == (dims.n_h * dims.d_c, dims.d_cq)
    Mb = brute.merge_query_absorption(brute.to_lists({"a": W["W_UQ"]})["a"],
                                      brute.to_lists({"a": W["W_UK"]})["a"], dims.n_h, dims.d_hc)
    np.testing.assert_allclose(M, np.array(Mb), rtol=1e-12, atol=1e-12)
    h = mi.hidden(dims, "f32", 0, 3).astype(np.float64)
    c_q = h @ W["W_DQ"].T.astype(np.float64)
    q_c, _ = ref.query(h, W["W_DQ"], W["W_UQ"], W["W_QR"], [0, 1, 2], dims.n_h, dims.d_hc,
                       dims.d_hr, dims.rope_base)
    q_t = ref.absorb_query(q_c, W["W_UK"], dims.n_h, dims.d_hc)
    q_t_merged = (c_q @ M.T).reshape(3, dims.n_h, dims.d_c)
    np.testing.assert_allclose(q_t_merged, q_t, rtol=1e-12, atol=1e-12)


def test_tiny_decode_matches_scalar_brute_force():
    """The fp32 tiny workload end to end (64 cached tokens + one new token at position 64)."""
    wl = mi.workload("tiny_f32")
    dims = wl.dims
    T = wl.seq_lens[0]
    W, h = _seq(dims, T)
    pos = np.arange(T)
    c, kr = ref.kv_latent(h, W["W_DKV"], W["W_KR"], pos, dims.rope_base)
    rows = ref.cache_rows(c, kr)
    q_c, q_r = ref.query(h[-1:], W["W_DQ"], W["W_UQ"], W["W_QR"], pos[-1:], dims.n_h,
                         dims.d_hc, dims.d_hr, dims.rope_base)
    o = ref.decode_explicit(q_c, q_r, [rows], W["W_UK"], W["W_UV"], dims.d_c)
    Wl = brute.to_lists(W)
    dd = _dims_dict(dims)
    tok = [brute.token_branches(list(map(float, h[p])), Wl, p, dd) for p in range(T)]
    scale = 1.0 / math.sqrt(dims.d_hc + dims.d_hr)
    for i in range(dims.n_h):
        np.testing.assert_allclose(o[0, i], brute.attention_output(tok, T - 1, i, scale),
                                   rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------------ structure

def test_prefill_is_causal_and_agrees_with_decode():
    dims = MICRO
    T = 6
    W, h = _seq(dims, T)
    o, rows = ref.prefill_sequence(h, W, dims.n_h, dims.d_hc, dims.d_hr, dims.d_c, dims.rope_base)
    # perturbing a later token leaves every earlier output unchanged
    h2 = h.copy()
    h2[4] += 1.0
    o2, _ = ref.prefill_sequence(h2, W, dims.n_h, dims.d_hc, dims.d_hr, dims.d_c, dims.rope_base)
    np.testing.assert_array_equal(o[:4], o2[:4])
    assert np.max(np.abs(o[4:] - o2[4:])) > 1e-6
    # the last prefill output equals a decode step over the same cache rows
    q_c, q_r = ref.query(h[-1:], W["W_DQ"], W["W_UQ"], W["W_QR"], [T - 1], dims.n_h,
                         dims.d_hc, dims.d_hr, dims.rope_base)
    od = ref.decode_explicit(q_c, q_r, [rows], W["W_UK"], W["W_UV"], dims.d_c)
    np.testing.assert_allclose(o[-1], od[0], rtol=1e-12, atol=1e-13)


def test_decoupled_rope_makes_scores_depend_on_relative_position_only():
    """Shifting every position (queries and keys) by the same offset leaves decode unchanged:
    the rotations of q^R and k^R cancel up to the position difference."""
    dims = MICRO
    T = 5
    W, h = _seq(dims, T)
    outs = []
    for off in (0, 1000):
        pos = np.arange(T) + off
        c, kr = ref.kv_latent(h, W["W_DKV"], W["W_KR"], pos, dims.rope_base)
        q_c, q_r = ref.query(h[-1:], W["W_DQ"], W["W_UQ"], W["W_QR"], pos[-1:], dims.n_h,
                             dims.d_hc, dims.d_hr, dims.rope_base)
        outs.append(ref.decode_explicit(q_c, q_r, [ref.cache_rows(c, kr)], W["W_UK"], W["W_UV"],
                                        dims.d_c))
    np.testing.assert_allclose(outs[0], outs[1], rtol=1e-9, atol=1e-12)


def test_k_rope_comes_from_h_not_from_the_latent():
    """§三分支计算 ② Key: k^R = RoPE(W^KR h_t), from h, not from c^KV. Zeroing W^DKV must
    leave k^R untouched."""
    dims = MICRO
    W, h = _seq(dims, 3)
    c1, kr1 = ref.kv_latent(h, W["W_DKV"], W["W_KR"], np.arange(3), dims.rope_base)
    c2, kr2 = ref.kv_latent(h, np.zeros_like(W["W_DKV"]), W["W_KR"], np.arange(3), dims.rope_base)
    np.testing.assert_array_equal(kr1, kr2)
    assert not np.any(c2)


# ------------------------------------------------------------------ storage rounding

def test_round_bf16_closed_cases():
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -7, -(1 + 2 ** -8 + 2 ** -20),
                  3.0, 2 ** -130 * 0 + 1e-3])
    y = ref.round_bf16(x)
    assert y[0] == 1.0
    assert y[1] == 1.0                      # tie -> even
    assert y[2] == 1 + 2 ** -6              # tie -> even (upward)
    assert y[3] == 1 + 2 ** -7              # representable
    assert y[4] == -(1 + 2 ** -7)           # above the tie -> away
    assert y[5] == 3.0
    # 1e-3 lies between two bf16 neighbours; the result is one of them and within half a spacing
    assert abs(y[6] - 1e-3) <= 2 ** -10 * 2 ** -8


def test_round_bf16_agrees_with_the_generators_float32_rounding():
    # two independent implementations (float64 frexp here, float32 bit twiddling in the
    # input generator) agree on values that are exactly representable in float32
    x = mi.aux_normal((10000,), index=40, scale=3.0)
    np.testing.assert_array_equal(ref.round_bf16(x.astype(np.float64)),
                                  mi.round_to_bf16(x).astype(np.float64))


# ------------------------------------------------------------------ top-k sparse selection

def test_topk_selection_matches_scalar_brute_force():
    """Scores from a small set (many ties, -0.0 beside +0.0) against k rounds of 'largest
    remaining, lowest position first'."""
    rng = np.random.default_rng(7)
    values = np.array([-2.5, -1.0, -0.0, 0.0, 0.5, 3.0], dtype=np.float32)
    for L in (1, 2, 5, 17, 40):
        for k in (1, 2, 3, 8, 16, 64):
            s = rng.choice(values, L)
            want = brute.select_topk([float(x) for x in s], k)
            got = ref.select_topk(s, L, k)
            assert list(got) == want, (L, k)


def test_topk_selection_special_cases():
    L, k = 10, 4
    assert list(ref.select_topk(np.zeros(L), L, k)) == [0, 1, 2, 3]  # all tied: lowest first
    assert list(ref.select_topk(np.arange(L, dtype=float), L, k)) == [6, 7, 8, 9]
    assert list(ref.select_topk(-np.arange(L, dtype=float), L, k)) == [0, 1, 2, 3]
    assert list(ref.select_topk(np.arange(L, dtype=float), L, L + 3)) == list(range(L))
    assert list(ref.select_topk(np.arange(L, dtype=float), 0, k)) == []
    # only the first L scores count: larger scores past L are ignored
    s = np.array([1.0, 2.0, 3.0, 100.0, 200.0])
    assert list(ref.select_topk(s, 3, 2)) == [1, 2]
    # -inf and huge values order like any other scores
    s = np.array([-np.inf, 3e38, -3e38, np.inf, 0.0])
    assert list(ref.select_topk(s, 5, 2)) == [1, 3]


def _micro_tokens(T, seed=0):
    dims = MICRO
    W, h = _seq(dims, T, seq=seed)
    pos = np.arange(T)
    c, kr = ref.kv_latent(h, W["W_DKV"], W["W_KR"], pos, dims.rope_base)
    rows = ref.cache_rows(c, kr)
    q_c, q_r = ref.query(h[-1:], W["W_DQ"], W["W_UQ"], W["W_QR"], pos[-1:], dims.n_h,
                         dims.d_hc, dims.d_hr, dims.rope_base)
    return dims, W, h, rows, q_c, q_r


def test_sparse_decode_matches_scalar_brute_force():
    T, k = 9, 4
    dims, W, h, rows, q_c, q_r = _micro_tokens(T)
    scores = np.random.default_rng(3).standard_normal(T)
    o = ref.decode_sparse(q_c, q_r, [rows], [scores], k, W["W_UK"], W["W_UV"], dims.d_c)
    Wl = brute.to_lists(W)
    dd = _dims_dict(dims)
    tok = [brute.token_branches(list(map(float, h[p])), Wl, p, dd) for p in range(T)]
    sel = brute.select_topk([float(x) for x in scores], k)
    scale = 1.0 / math.sqrt(dims.d_hc + dims.d_hr)
    for i in range(dims.n_h):
        np.testing.assert_allclose(o[0, i], brute.sparse_attention_output(tok, T - 1, sel, i,
                                                                          scale),
                                   rtol=1e-11, atol=1e-12)


def test_sparse_decode_with_k_at_least_the_length_is_the_dense_decode():
    T = 7
    dims, W, h, rows, q_c, q_r = _micro_tokens(T, seed=1)
    scores = np.random.default_rng(4).standard_normal(T)
    dense = ref.decode_explicit(q_c, q_r, [rows], W["W_UK"], W["W_UV"], dims.d_c)
    for k in (T, T + 5):
        sparse = ref.decode_sparse(q_c, q_r, [rows], [scores], k, W["W_UK"], W["W_UV"],
                                   dims.d_c)
        np.testing.assert_array_equal(sparse, dense)


def test_sparse_decode_with_one_selected_row_returns_its_value():
    """k = 1: the softmax over one key is 1, so o_i = W^UV_i c_{j*} for the top-scored j*."""
    T = 8
    dims, W, h, rows, q_c, q_r = _micro_tokens(T, seed=2)
    scores = np.zeros(T)
    scores[5] = 2.0
    o = ref.decode_sparse(q_c, q_r, [rows], [scores], 1, W["W_UK"], W["W_UV"], dims.d_c)
    c5 = rows[5, :dims.d_c]
    for i in range(dims.n_h):
        Wv = W["W_UV"][i * dims.d_hc:(i + 1) * dims.d_hc].astype(np.float64)
        want = [sum(float(Wv[r, c]) * float(c5[c]) for c in range(dims.d_c))
                for r in range(dims.d_hc)]
        np.testing.assert_allclose(o[0, i], want, rtol=1e-12, atol=1e-13)
