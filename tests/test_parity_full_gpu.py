"""GPU parity at the full workload sizes, in the launch configuration bench.py times, on
sampled outputs the oracle computes one by one (sampled sequences x sampled heads)."""
import numpy as np
import pytest

import mla_inputs as mi
import mla_latent_kv_75_b300 as mla
from mla_latent_kv_75_b300 import host
from oracle import mla_ref as ref
from helpers import assert_close, oracle_decode_step, oracle_weights

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

HEADS = [0, 1, 37, 64, 101, 127]


def build_and_step(wl):
    dims, dtype = wl.dims, wl.dtype
    W = mi.weights(dims, dtype)
    model = host.DeviceModel.upload(dims, dtype, W)
    base = mi.packed_layout(wl.seq_lens)
    cache = host.LatentCache(dims, dtype, base, wl.n_rows)
    host.fill_context(model, cache, lambda b, n: mi.hidden(dims, dtype, b, n, wl.seed), wl.seq_lens)
    step = host.DecodeStep(model, cache, wl.seq_lens)
    h_new = np.stack([mi.hidden_rows(dims, dtype, b, [L - 1], wl.seed)[0]
                      for b, L in enumerate(wl.seq_lens)])
    o = step.step(host.to_device(h_new, dtype)).cpu().numpy()
    assert mla.mla_get_device_status() == 0
    return o, cache, base


@pytest.mark.parametrize("name,seqs", [
    ("v2_decode_b16_l4096", [0, 7, 15]),
    ("v2_decode_b1_l131072", [0]),
    ("v2_decode_b4_l32768", [0, 3]),
    ("v2_decode_b128_ragged", [0, 5, 63, 127]),
])
def test_full_size_decode_sampled(name, seqs):
    wl = mi.workload(name)
    o, cache, base = build_and_step(wl)
    _, W64 = oracle_weights(wl.dims, wl.dtype)
    exp = oracle_decode_step(wl, W64, seqs=seqs, heads=HEADS)
    got = np.stack([o[b][HEADS] for b in seqs])
    assert_close(got, np.stack(exp["o"]), "bf16", name)
    # last row of every sampled sequence (the appended token) matches the oracle's row
    for k, b in enumerate(seqs):
        L = wl.seq_lens[b]
        row = cache.rows[int(base[b]) + L - 1].float().cpu().numpy().astype(np.float64)
        assert_close(row, exp["rows_exact"][k][L - 1], "bf16", "appended row")
    assert np.all(np.isfinite(o))


def test_full_size_prefill_sampled():
    wl = mi.workload("v2_prefill_b2_t4096")
    dims, dtype = wl.dims, wl.dtype
    W, W64 = oracle_weights(dims, dtype)
    model = host.DeviceModel.upload(dims, dtype, W)
    base = mi.packed_layout(wl.seq_lens)
    cache = host.LatentCache(dims, dtype, base, wl.n_rows)
    pre = host.PrefillStep(model, cache, wl.seq_lens)
    hs = [mi.hidden(dims, dtype, b, L, wl.seed) for b, L in enumerate(wl.seq_lens)]
    o = pre.run(host.to_device(np.concatenate(hs), dtype)).cpu().numpy()
    assert mla.mla_get_device_status() == 0
    queries = [0, 1, 127, 128, 1000, 2047, 4095]
    s = 0
    for b, L in enumerate(wl.seq_lens):
        want, rows = ref.prefill_sequence(hs[b], W64, dims.n_h, dims.d_hc, dims.d_hr, dims.d_c,
                                          dims.rope_base, dtype, heads=HEADS, queries=queries)
        got = o[s + np.array(queries)][:, HEADS]
        assert_close(got, want, dtype, "prefill seq %d" % b)
        got_rows = cache.rows[int(base[b]): int(base[b]) + L].float().cpu().numpy()
        assert np.mean(got_rows == rows) > 0.99
        s += L
