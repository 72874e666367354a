"""GPU parity of the pre-merged absorbed query ("从LLaMA到DeepSeek[01] - MLA（上）" §六: W^UQ and
W^UK are fixed, so W^UQK_i = (W^UK_i)^T W^UQ_i can be formed once): the merged weights and the
query projection that uses them, against the float64 oracle."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import mla_latent_kv_75_b300 as mla
from mla_latent_kv_75_b300 import host
from oracle import mla_ref as ref
from helpers import TOL, assert_close, oracle_weights, rel_errors

pytestmark = pytest.mark.gpu


def _merge(dims, dtype, model):
    W_UQK = torch.empty((dims.n_h * dims.d_c, dims.d_cq), dtype=host.torch_dtype(dtype),
                        device="cuda")
    mla.mla_merge_query_absorption(model.abi_dims, model.W["W_UQ"], model.W["W_UK"], W_UQK)
    assert mla.mla_get_device_status() == 0
    return W_UQK


def _project(dims, dtype, model, W_UQK, h, pos):
    n = h.shape[0]
    d = model.abi_dims
    ws_bytes = mla.mla_project_q_workspace_size(d, n)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    td = host.torch_dtype(dtype)
    q_t = torch.full((n, dims.n_h, dims.d_c), float("nan"), dtype=td, device="cuda")
    q_r = torch.full((n, dims.n_h, dims.d_hr), float("nan"), dtype=td, device="cuda")
    mla.mla_project_q_premerged(d, model.abi_weights, W_UQK, host.to_device(h, dtype),
                                torch.tensor(pos, device="cuda"), n, ws, ws_bytes, q_t, q_r)
    assert mla.mla_get_device_status() == 0
    return (q_t.float().cpu().numpy().astype(np.float64),
            q_r.float().cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("n", [16, 150])
def test_premerged_query_matches_oracle(n):
    dims = mi.V2
    W, W64 = oracle_weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    W_UQK = _merge(dims, "bf16", model)
    # the merged map itself: one bf16 rounding of the exact product
    want_m = ref.merge_query_absorption(W64["W_UQ"], W64["W_UK"], dims.n_h, dims.d_hc)
    rows = [0, 511, 512 * 77 + 3, 512 * 128 - 1]
    assert_close(W_UQK[rows].float().cpu().numpy().astype(np.float64), want_m[rows], "bf16",
                 "merged W^UQK rows")
    h = mi.aux_normal((n, dims.d), index=500 + n, dtype="bf16")
    pos = np.random.default_rng(n + 1).integers(0, 50000, n).astype(np.int32)
    got_t, got_r = _project(dims, "bf16", model, W_UQK, h, pos)
    q_c, q_r = ref.query(h, W64["W_DQ"], W64["W_UQ"], W64["W_QR"], pos, dims.n_h, dims.d_hc,
                         dims.d_hr, dims.rope_base)
    assert_close(got_t, ref.absorb_query(q_c, W64["W_UK"], dims.n_h, dims.d_hc), "bf16", "q~")
    assert_close(got_r, q_r, "bf16", "q^R")


def test_premerged_query_tiny_f32_matches_oracle():
    dims = mi.TINY
    W, W64 = oracle_weights(dims, "f32")
    model = host.DeviceModel.upload(dims, "f32", W)
    W_UQK = _merge(dims, "f32", model)
    h = mi.aux_normal((5, dims.d), index=520)
    pos = np.array([0, 1, 7, 64, 300], dtype=np.int32)
    got_t, got_r = _project(dims, "f32", model, W_UQK, h, pos)
    q_c, q_r = ref.query(h, W64["W_DQ"], W64["W_UQ"], W64["W_QR"], pos, dims.n_h, dims.d_hc,
                         dims.d_hr, dims.rope_base)
    for got, want in ((got_t, ref.absorb_query(q_c, W64["W_UK"], dims.n_h, dims.d_hc)),
                      (got_r, q_r)):
        mr, _ = rel_errors(got, want)
        assert mr <= TOL["f32"][0], mr
