"""GPU parity of the fused decode path against the float64 oracle: the query projection with
the absorption applied (mla_project_q_absorbed: q~ = (W^UK_i)^T W^UQ_i c^Q without q^C in
global memory, "从LLaMA到DeepSeek[01] - MLA（上）" §六) and the one-call decode step
(mla_decode_step: down-projections in one launch, fused query, latent decode)."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import mla_latent_kv_75_b300 as mla
from mla_latent_kv_75_b300 import host
from oracle import mla_ref as ref
from helpers import assert_close, oracle_decode_step, oracle_weights

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [16, 150])
def test_project_q_absorbed_matches_oracle(n):
    """n = 16 runs the 32-token tile, n = 150 two 128-token tiles (the second ragged);
    positions spread to 10^5 exercise the RoPE angles."""
    dims = mi.V2
    W, W64 = oracle_weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    h = mi.aux_normal((n, dims.d), index=200 + n, dtype="bf16")
    pos = np.random.default_rng(n).integers(0, 100000, n).astype(np.int32)
    pos[0] = 0
    d = model.abi_dims
    ws_bytes = mla.mla_project_q_workspace_size(d, n)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    q_t = torch.full((n, dims.n_h, dims.d_c), float("nan"), dtype=torch.bfloat16, device="cuda")
    q_r = torch.full((n, dims.n_h, dims.d_hr), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.mla_project_q_absorbed(d, model.abi_weights, host.to_device(h, "bf16"),
                               torch.tensor(pos, device="cuda"), n, ws, ws_bytes, q_t, q_r)
    assert mla.mla_get_device_status() == 0
    q_c, q_r_want = ref.query(h, W64["W_DQ"], W64["W_UQ"], W64["W_QR"], pos, dims.n_h, dims.d_hc,
                              dims.d_hr, dims.rope_base)
    q_t_want = ref.absorb_query(q_c, W64["W_UK"], dims.n_h, dims.d_hc)
    got_t = q_t.float().cpu().numpy().astype(np.float64)
    got_r = q_r.float().cpu().numpy().astype(np.float64)
    assert_close(got_t, q_t_want, "bf16", "q~")
    assert_close(got_r, q_r_want, "bf16", "q^R")


def test_fused_decode_step_end_to_end_with_poisoned_gaps():
    """mla_decode_step on ragged lengths (1 row, partial tiles, tile multiples); rows between
    sequences hold NaN. The appended row, and o, match the oracle."""
    lens = [1, 77, 300, 129, 128, 640]
    wl = mi.Workload("v2_small", mi.V2, "bf16", "decode", lens)
    dims = wl.dims
    W, W64 = oracle_weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    base = mi.packed_layout(lens, guard=8)
    cap = int(base[-1] + lens[-1] + 8)
    cache = host.LatentCache(dims, "bf16", base, cap, fill=float("nan"))
    host.fill_context(model, cache, lambda b, n: mi.hidden(dims, "bf16", b, n), lens)
    step = host.DecodeStep(model, cache, lens, fused=True)
    assert step.fused
    h_new = np.stack([mi.hidden(dims, "bf16", b, L)[L - 1] for b, L in enumerate(lens)])
    o = step.step(host.to_device(h_new, "bf16")).cpu().numpy()
    assert mla.mla_get_device_status() == 0
    exp = oracle_decode_step(wl, W64)
    for b, L in enumerate(lens):
        row = cache.rows[int(base[b]) + L - 1].float().cpu().numpy().astype(np.float64)
        assert_close(row, exp["rows_exact"][b][L - 1], "bf16", "appended row seq %d" % b)
    assert_close(o, np.stack(exp["o"]), "bf16", "fused decode step o")
    # the guard rows after every sequence are untouched
    for b, L in enumerate(lens):
        g = cache.rows[int(base[b]) + L: int(base[b]) + L + 8].float()
        assert torch.isnan(g).all()


def test_fused_step_equals_three_call_step():
    """The one-call step and the three-call step (append, project, decode) agree to the
    precision of their shared rounding points; the latent decode of the absorbed query equals
    mla_decode_absorbed of the same query."""
    lens = [33, 500, 4100]
    dims = mi.V2
    W, _ = oracle_weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    outs = []
    for fused in (False, True):
        base = mi.packed_layout(lens)
        cache = host.LatentCache(dims, "bf16", base, int(sum(lens)))
        host.fill_context(model, cache, lambda b, n: mi.hidden(dims, "bf16", b, n), lens)
        step = host.DecodeStep(model, cache, lens, fused=fused)
        h_new = np.stack([mi.hidden(dims, "bf16", b, L)[L - 1] for b, L in enumerate(lens)])
        outs.append(step.step(host.to_device(h_new, "bf16")).cpu().numpy().astype(np.float64))
        assert mla.mla_get_device_status() == 0
    assert_close(outs[1], outs[0], "bf16", "fused vs three-call step")


def test_decode_absorbed_latent_rejects_fp32_dims():
    dims = mi.TINY
    d = host.dims_struct(dims, "f32")
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_decode_step_workspace_size(d, 1, 65)
    assert ei.value.status == 2
