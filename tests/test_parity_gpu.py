"""GPU parity: libmla (through the C ABI) against the float64 oracle on the same seeded inputs,
at sizes the oracle finishes in seconds that still span several tiles and ragged tails."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import mla_latent_kv_75_b300 as mla
from mla_latent_kv_75_b300 import host
from oracle import mla_ref as ref
from helpers import TOL, assert_close, oracle_decode_step, oracle_weights, rel_errors

pytestmark = pytest.mark.gpu

SMALL_V2_LENS = [1, 77, 300, 129, 128, 640]


def run_decode_workload(wl, guard=0, poison=None):
    """Build the cache on the GPU (context rows by append), then one full decode step."""
    dims, dtype = wl.dims, wl.dtype
    W = mi.weights(dims, dtype)
    model = host.DeviceModel.upload(dims, dtype, W)
    base = mi.packed_layout(wl.seq_lens, guard)
    cap = int(base[-1] + wl.seq_lens[-1] + guard)
    cache = host.LatentCache(dims, dtype, base, cap, fill=poison)
    host.fill_context(model, cache, lambda b, n: mi.hidden(dims, dtype, b, n, wl.seed), wl.seq_lens)
    step = host.DecodeStep(model, cache, wl.seq_lens)
    h_new = np.stack([mi.hidden(dims, dtype, b, L, wl.seed)[L - 1] for b, L in enumerate(wl.seq_lens)])
    o = step.step(host.to_device(h_new, dtype))
    assert mla.mla_get_device_status() == 0
    return step, cache, base, o.float().cpu().numpy()


def gpu_rows(cache, base, lens, b):
    r = cache.rows[int(base[b]): int(base[b]) + lens[b]].float().cpu().numpy()
    return r.astype(np.float64)


def test_tiny_f32_decode_end_to_end():
    wl = mi.workload("tiny_f32")
    step, cache, base, o = run_decode_workload(wl)
    _, W64 = oracle_weights(wl.dims, wl.dtype)
    exp = oracle_decode_step(wl, W64)
    tol = TOL["f32"][0]
    mr, _ = rel_errors(gpu_rows(cache, base, wl.seq_lens, 0), exp["rows"][0])
    assert mr <= tol
    mr, _ = rel_errors(step.q_c.cpu().numpy()[0], exp["q_c"][0])
    assert mr <= tol
    mr, _ = rel_errors(step.q_r.cpu().numpy()[0], exp["q_r"][0])
    assert mr <= tol
    mr, _ = rel_errors(o[0], exp["o"][0])
    assert mr <= tol, mr


def test_v2_small_ragged_decode_end_to_end_with_poisoned_gaps():
    """Ragged lengths (1 row, partial tiles, exact tile multiples); the rows between sequences
    hold NaN, so any row read across a sequence boundary would poison the result."""
    wl = mi.Workload("v2_small", mi.V2, "bf16", "decode", SMALL_V2_LENS)
    step, cache, base, o = run_decode_workload(wl, guard=8, poison=float("nan"))
    _, W64 = oracle_weights(wl.dims, wl.dtype)
    exp = oracle_decode_step(wl, W64)
    for b in range(wl.B):
        got = gpu_rows(cache, base, wl.seq_lens, b)
        assert_close(got, exp["rows_exact"][b], "bf16", "cache rows seq %d" % b)
        # the stored values are the bf16 rounding of the exact rows, up to fp32 accumulation
        # flipping a rounding decision (one ulp) on a tiny fraction of elements
        assert np.mean(got == exp["rows"][b]) > 0.99
    qc = step.q_c.float().cpu().numpy().astype(np.float64)
    qr = step.q_r.float().cpu().numpy().astype(np.float64)
    assert_close(qc, np.stack(exp["q_c_exact"]), "bf16", "q_c")
    assert_close(qr, np.stack(exp["q_r_exact"]), "bf16", "q_r")
    assert_close(o, np.stack(exp["o"]), "bf16", "decode o")


def test_v2_decode_on_synthetic_cache_and_queries():
    """Decode alone: cache rows and queries straight from the generator (bf16), including a
    sequence of length 0 (o = 0) and lengths straddling tile boundaries."""
    dims = mi.V2
    lens = [0, 1, 2, 255, 256, 257, 1000]
    W, W64 = oracle_weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    base = mi.packed_layout(lens, guard=3)
    cap = int(base[-1] + lens[-1] + 3)
    rows_np = mi.aux_normal((cap, dims.row), index=100, dtype="bf16")
    cache = host.LatentCache(dims, "bf16", base, cap)
    cache.rows.copy_(host.to_device(rows_np, "bf16"))
    q_c = mi.aux_normal((len(lens), dims.n_h, dims.d_hc), index=101, dtype="bf16")
    q_r = mi.aux_normal((len(lens), dims.n_h, dims.d_hr), index=102, dtype="bf16")
    step = host.DecodeStep(model, cache, lens)
    o = step.decode(q_c=host.to_device(q_c, "bf16"), q_r=host.to_device(q_r, "bf16"))
    assert mla.mla_get_device_status() == 0
    o = o.cpu().numpy()
    rows = [rows_np[base[b]: base[b] + L].astype(np.float64) for b, L in enumerate(lens)]
    want = ref.decode_explicit(q_c, q_r, rows, W64["W_UK"], W64["W_UV"], dims.d_c)
    assert np.all(o[0] == 0.0)
    assert_close(o[1:], want[1:], "bf16", "decode o")
    # length 1 returns v = W^UV_i c_0 (up to the tolerance of the bf16 path)
    assert_close(o[1], want[1], "bf16", "length-1 decode")


def test_v2_decode_many_short_sequences_spanning_split():
    """More non-empty sequences than SM pairs: the tensor-core decode then gives each pair a
    contiguous range of the concatenated tile list, so pairs cross sequence boundaries (query
    re-load mid-range, one partial slot per segment). Lengths are short and ragged, some below
    one tile, some exactly at tile multiples; checked on a subset of heads."""
    dims = mi.V2
    rng = np.random.default_rng(7)
    lens = [int(x) for x in rng.integers(1, 200, 150)]
    lens[3], lens[10], lens[20] = 48, 96, 1
    W, W64 = oracle_weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    base = mi.packed_layout(lens, guard=1)
    cap = int(base[-1] + lens[-1] + 1)
    rows_np = mi.aux_normal((cap, dims.row), index=110, dtype="bf16")
    cache = host.LatentCache(dims, "bf16", base, cap)
    cache.rows.copy_(host.to_device(rows_np, "bf16"))
    q_c = mi.aux_normal((len(lens), dims.n_h, dims.d_hc), index=111, dtype="bf16")
    q_r = mi.aux_normal((len(lens), dims.n_h, dims.d_hr), index=112, dtype="bf16")
    step = host.DecodeStep(model, cache, lens)
    o = step.decode(q_c=host.to_device(q_c, "bf16"), q_r=host.to_device(q_r, "bf16"))
    assert mla.mla_get_device_status() == 0
    o = o.cpu().numpy()
    heads = [0, 63, 127]
    rows = [rows_np[base[b]: base[b] + L].astype(np.float64) for b, L in enumerate(lens)]
    want = ref.decode_explicit(q_c, q_r, rows, W64["W_UK"], W64["W_UV"], dims.d_c, heads=heads)
    assert_close(o[:, heads], want, "bf16", "decode o (spanning split)")


def test_v2_decode_one_long_sequence_split_over_every_pair():
    """One sequence longer than 74 tiles of 48 rows: every SM pair takes a contiguous share of
    it, so the merge combines 74 partial results (more than one warp's worth of slots, with a
    ragged last tile). Checked on a subset of heads."""
    dims = mi.V2
    lens = [74 * 48 + 1000 + 17]
    W, W64 = oracle_weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    base = mi.packed_layout(lens, guard=2)
    cap = int(base[-1] + lens[-1] + 2)
    rows_np = mi.aux_normal((cap, dims.row), index=120, dtype="bf16")
    cache = host.LatentCache(dims, "bf16", base, cap)
    cache.rows.copy_(host.to_device(rows_np, "bf16"))
    q_c = mi.aux_normal((1, dims.n_h, dims.d_hc), index=121, dtype="bf16")
    q_r = mi.aux_normal((1, dims.n_h, dims.d_hr), index=122, dtype="bf16")
    step = host.DecodeStep(model, cache, lens)
    o = step.decode(q_c=host.to_device(q_c, "bf16"), q_r=host.to_device(q_r, "bf16"))
    assert mla.mla_get_device_status() == 0
    o = o.cpu().numpy()
    heads = [0, 1, 64, 127]
    rows = [rows_np[base[0]: base[0] + lens[0]].astype(np.float64)]
    want = ref.decode_explicit(q_c, q_r, rows, W64["W_UK"], W64["W_UV"], dims.d_c, heads=heads)
    assert_close(o[:, heads], want, "bf16", "decode o (one long sequence)")


def test_tiny_f32_prefill():
    dims = mi.TINY
    lens = [33, 1, 70]
    W, W64 = oracle_weights(dims, "f32")
    model = host.DeviceModel.upload(dims, "f32", W)
    base = mi.packed_layout(lens)
    cache = host.LatentCache(dims, "f32", base, int(sum(lens)))
    pre = host.PrefillStep(model, cache, lens)
    h = np.concatenate([mi.hidden(dims, "f32", b, L) for b, L in enumerate(lens)])
    o = pre.run(host.to_device(h, "f32")).cpu().numpy()
    assert mla.mla_get_device_status() == 0
    s = 0
    for b, L in enumerate(lens):
        want, rows = ref.prefill_sequence(h[s:s + L], W64, dims.n_h, dims.d_hc, dims.d_hr,
                                          dims.d_c, dims.rope_base, "f32")
        mr, _ = rel_errors(o[s:s + L], want)
        assert mr <= TOL["f32"][0], (b, mr)
        got_rows = cache.rows[base[b]: base[b] + L].cpu().numpy()
        mr, _ = rel_errors(got_rows, rows)
        assert mr <= TOL["f32"][0]
        s += L


def test_v2_small_prefill():
    dims = mi.V2
    lens = [130, 61, 1]
    W, W64 = oracle_weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    base = mi.packed_layout(lens, guard=2)
    cache = host.LatentCache(dims, "bf16", base, int(base[-1] + lens[-1] + 2), fill=float("nan"))
    pre = host.PrefillStep(model, cache, lens)
    h = np.concatenate([mi.hidden(dims, "bf16", b, L) for b, L in enumerate(lens)])
    o = pre.run(host.to_device(h, "bf16")).cpu().numpy()
    assert mla.mla_get_device_status() == 0
    s = 0
    got, want = [], []
    for b, L in enumerate(lens):
        w_o, rows = ref.prefill_sequence(h[s:s + L], W64, dims.n_h, dims.d_hc, dims.d_hr,
                                         dims.d_c, dims.rope_base, "bf16")
        got.append(o[s:s + L])
        want.append(w_o)
        got_rows = cache.rows[base[b]: base[b] + L].float().cpu().numpy()
        assert np.mean(got_rows == rows) > 0.99
        s += L
    assert_close(np.concatenate(got), np.concatenate(want), "bf16", "prefill o")


def test_device_status_reports_capacity_and_length_violations():
    dims = mi.V2
    W = mi.weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    cache = host.LatentCache(dims, "bf16", [0, 10], 16, fill=0.0)
    h = host.to_device(mi.hidden(dims, "bf16", 0, 2), "bf16")
    seq = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    pos = torch.tensor([3, 6], dtype=torch.int32, device="cuda")  # row 16 is past capacity
    host.append_tokens(model, cache, h, seq, pos)
    assert mla.mla_get_device_status() == 3
    assert torch.count_nonzero(cache.rows[0:3]) == 0 and torch.count_nonzero(cache.rows[3]) > 0
    assert mla.mla_get_device_status() == 0  # cleared by the previous read
    step = host.DecodeStep(model, cache, [4, 6], max_len=5)  # 6 > max_len
    q = host.to_device(mi.aux_normal((2, 128, 128), index=3, dtype="bf16"), "bf16")
    qr = host.to_device(mi.aux_normal((2, 128, 64), index=4, dtype="bf16"), "bf16")
    step.decode(q_c=q, q_r=qr)
    assert mla.mla_get_device_status() == 8


def test_repeated_calls_are_bitwise_deterministic():
    wl = mi.Workload("v2_det", mi.V2, "bf16", "decode", [300, 1030])
    step, cache, base, o1 = run_decode_workload(wl)
    o2 = step.decode().cpu().numpy()
    assert np.array_equal(o1, o2)
