"""GPU parity of the top-k sparse decode ("MLA前向计算流程", version table, V3.2 + DSA row: an
indexer picks top-k positions of the latent sequence, MLA runs unchanged over them) against
the float64 oracle: the selection bit for bit, the decode over the picked rows within the bf16
tolerance, and the k >= length case bit for bit against the dense decode."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import mla_latent_kv_75_b300 as mla
from mla_latent_kv_75_b300 import host
from oracle import mla_ref as ref
from helpers import TOL, assert_close, oracle_weights, rel_errors

pytestmark = pytest.mark.gpu


def _scores(lens, stride, kind, seed):
    """Index scores [B, stride] float32 with the given value mix; entries past a sequence's
    length hold +inf so that reading past the length would show up as a wrong pick."""
    rng = np.random.default_rng(seed)
    s = np.full((len(lens), stride), np.inf, dtype=np.float32)
    for b, L in enumerate(lens):
        if kind == "normal":
            v = rng.standard_normal(L).astype(np.float32)
        elif kind == "ties":  # few distinct values, both zeros among them
            v = rng.choice(np.array([-1.5, -0.0, 0.0, 0.25, 2.0], dtype=np.float32), L)
        else:  # "extremes": infinities, huge and tiny magnitudes, denormals
            v = rng.choice(np.array([-np.inf, -3e38, -1e-40, 1e-40, 1e-30, 3e38, np.inf],
                                    dtype=np.float32), L)
        s[b, :L] = v
    return s


def _select(scores, lens, k):
    B, stride = scores.shape
    max_len = max(lens) if lens else 0
    sel = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    mla.mla_select_topk(torch.tensor(scores, device="cuda"), stride,
                        torch.tensor(lens, dtype=torch.int32, device="cuda"), B, max_len, k, sel,
                        cnt)
    assert mla.mla_get_device_status() == 0
    return sel.cpu().numpy(), cnt.cpu().numpy()


@pytest.mark.parametrize("kind", ["normal", "ties", "extremes"])
@pytest.mark.parametrize("k", [1, 64, 2048])
def test_select_topk_is_bit_exact(kind, k):
    """Lengths around k, lengths that leave some CTAs of the cluster with short or empty
    slices (40000 positions over three CTAs), and an empty sequence."""
    lens = [0, 1, 5, k - 1 if k > 1 else 1, k, k + 1, 3000, 4097, 16385, 40000]
    stride = max(lens) + 3
    scores = _scores(lens, stride, kind, seed=k)
    sel, cnt = _select(scores, lens, k)
    for b, L in enumerate(lens):
        want = ref.select_topk(scores[b], L, k)
        assert cnt[b] == len(want) == min(L, k)
        np.testing.assert_array_equal(sel[b, :cnt[b]], want, err_msg="seq %d (L=%d)" % (b, L))
        assert np.all(sel[b, cnt[b]:] == -7)  # entries past the count are not written


def _sparse_setup(lens, guard=2, seed=300):
    dims = mi.V2
    W, W64 = oracle_weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    base = mi.packed_layout(lens, guard=guard)
    cap = int(base[-1] + lens[-1] + guard)
    rows_np = mi.aux_normal((cap, dims.row), index=seed, dtype="bf16")
    cache = host.LatentCache(dims, "bf16", base, cap)
    cache.rows.copy_(host.to_device(rows_np, "bf16"))
    q_c = mi.aux_normal((len(lens), dims.n_h, dims.d_hc), index=seed + 1, dtype="bf16")
    q_r = mi.aux_normal((len(lens), dims.n_h, dims.d_hr), index=seed + 2, dtype="bf16")
    return dims, W64, model, base, rows_np, cache, q_c, q_r


def _sparse_decode(dims, model, cache, q_c, q_r, lens, scores, k):
    B = len(lens)
    max_len = max(lens)
    d = model.abi_dims
    ws_bytes = mla.mla_decode_sparse_workspace_size(d, B, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    o = torch.full((B, dims.n_h, dims.d_hc), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_absorbed_sparse(d, model.abi_weights, host.to_device(q_c, "bf16"),
                                   host.to_device(q_r, "bf16"), cache.abi,
                                   torch.tensor(lens, dtype=torch.int32, device="cuda"), B,
                                   max_len, torch.tensor(scores, device="cuda"), scores.shape[1],
                                   k, ws, ws_bytes, o)
    assert mla.mla_get_device_status() == 0
    return o.cpu().numpy().astype(np.float64)


def test_sparse_decode_matches_oracle():
    """Ragged lengths below, at and above k; scores with ties, so the tie rule decides which
    rows are attended."""
    lens = [1, 100, 256, 257, 1000, 5000]
    k = 256
    dims, W64, model, base, rows_np, cache, q_c, q_r = _sparse_setup(lens)
    scores = _scores(lens, max(lens), "ties", seed=11)
    o = _sparse_decode(dims, model, cache, q_c, q_r, lens, scores, k)
    rows = [rows_np[base[b]: base[b] + L].astype(np.float64) for b, L in enumerate(lens)]
    want = ref.decode_sparse(q_c, q_r, rows, list(scores), k, W64["W_UK"], W64["W_UV"],
                             dims.d_c)
    assert_close(o, want, "bf16", "sparse decode o")


def test_sparse_decode_with_large_k_equals_the_dense_decode_bitwise():
    lens = [3, 500, 4100]
    dims, W64, model, base, rows_np, cache, q_c, q_r = _sparse_setup(lens, seed=320)
    scores = _scores(lens, max(lens), "normal", seed=12)
    o_sparse = _sparse_decode(dims, model, cache, q_c, q_r, lens, scores, max(lens) + 5)
    step = host.DecodeStep(model, cache, lens)
    o_dense = step.decode(q_c=host.to_device(q_c, "bf16"), q_r=host.to_device(q_r, "bf16"))
    assert mla.mla_get_device_status() == 0
    np.testing.assert_array_equal(o_sparse, o_dense.cpu().numpy().astype(np.float64))


def test_sparse_decode_one_long_sequence_many_picks():
    """1 x 20000 rows with k = 2048: the packed rows span several 48-row tiles per pair."""
    lens = [20000]
    k = 2048
    dims, W64, model, base, rows_np, cache, q_c, q_r = _sparse_setup(lens, seed=340)
    scores = _scores(lens, lens[0], "normal", seed=13)
    o = _sparse_decode(dims, model, cache, q_c, q_r, lens, scores, k)
    rows = [rows_np[base[0]: base[0] + lens[0]].astype(np.float64)]
    heads = [0, 37, 127]
    want = ref.decode_sparse(q_c, q_r, rows, list(scores), k, W64["W_UK"], W64["W_UV"],
                             dims.d_c, heads=heads)
    assert_close(o[:, heads], want, "bf16", "sparse decode o (1 x 20000, k 2048)")


def test_sparse_decode_tiny_f32_matches_oracle():
    dims = mi.TINY
    lens = [1, 9, 40, 65]
    k = 12
    W, W64 = oracle_weights(dims, "f32")
    model = host.DeviceModel.upload(dims, "f32", W)
    base = mi.packed_layout(lens, guard=1)
    cap = int(base[-1] + lens[-1] + 1)
    rows_np = mi.aux_normal((cap, dims.row), index=360)
    cache = host.LatentCache(dims, "f32", base, cap)
    cache.rows.copy_(torch.tensor(rows_np, dtype=torch.float32))
    q_c = mi.aux_normal((len(lens), dims.n_h, dims.d_hc), index=361)
    q_r = mi.aux_normal((len(lens), dims.n_h, dims.d_hr), index=362)
    scores = _scores(lens, max(lens), "ties", seed=14)
    B = len(lens)
    d = model.abi_dims
    ws_bytes = mla.mla_decode_sparse_workspace_size(d, B, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    o = torch.full((B, dims.n_h, dims.d_hc), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_absorbed_sparse(d, model.abi_weights, torch.tensor(q_c, dtype=torch.float32,
                                                                      device="cuda"),
                                   torch.tensor(q_r, dtype=torch.float32, device="cuda"),
                                   cache.abi, torch.tensor(lens, dtype=torch.int32,
                                                           device="cuda"),
                                   B, max(lens), torch.tensor(scores, device="cuda"),
                                   scores.shape[1], k, ws, ws_bytes, o)
    assert mla.mla_get_device_status() == 0
    rows = [rows_np[base[b]: base[b] + L] for b, L in enumerate(lens)]
    want = ref.decode_sparse(q_c, q_r, rows, list(scores), k, W64["W_UK"], W64["W_UV"],
                             dims.d_c)
    mr, _ = rel_errors(o.cpu().numpy().astype(np.float64), want)
    assert mr <= TOL["f32"][0], mr


def test_select_topk_long_sequence_walks_several_rounds():
    """150000 positions: eight CTAs of 18750 positions each, walked in two rounds of 16384
    re-read from L2, against the oracle bit for bit; ties and a short second sequence too."""
    lens = [150000, 7]
    k = 2048
    scores = _scores(lens, max(lens), "ties", seed=21)
    sel, cnt = _select(scores, lens, k)
    for b, L in enumerate(lens):
        want = ref.select_topk(scores[b], L, k)
        assert cnt[b] == len(want)
        np.testing.assert_array_equal(sel[b, :cnt[b]], want)
