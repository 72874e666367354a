"""GPU parity of the output projection u_t = W^O [o_{t,1}; ...; o_{t,n_h}] ("MLA前向计算流程"
§三分支计算 ④) against the float64 oracle, on the tensor-core path (V2 widths, bf16 W^O, o as a
hi/lo bf16 pair) and the SIMT path (tiny fp32 config), and end to end after a decode."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import mla_latent_kv_75_b300 as mla
from mla_latent_kv_75_b300 import host
from oracle import mla_ref as ref
from helpers import TOL, assert_close, oracle_decode_step, oracle_weights, rel_errors

pytestmark = pytest.mark.gpu


def _run(dims, dtype, o_np, W_O):
    d = host.dims_struct(dims, dtype)
    n = o_np.shape[0]
    o = torch.tensor(o_np, dtype=torch.float32, device="cuda")
    w = host.to_device(W_O, dtype)
    ws_bytes = mla.mla_output_projection_workspace_size(d, n)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    u = torch.full((n, dims.d), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_output_projection(d, w, o, n, ws, ws_bytes, u)
    assert mla.mla_get_device_status() == 0
    return u.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("n", [16, 300])
def test_output_projection_v2_matches_oracle(n):
    """o enters the MMA as hi + lo (to ~2^-16) against the exact bf16 W^O with fp32
    accumulation over K = 16384, so the result is held to 1e-4 (the bf16-storage bar is 1e-2)."""
    dims = mi.V2
    W_O = mi.output_weight(dims, "bf16")
    o = mi.aux_normal((n, dims.n_h, dims.d_hc), index=400 + n)
    got = _run(dims, "bf16", o, W_O)
    want = ref.output_projection(o, W_O)
    max_rel, rms_rel = rel_errors(got, want)
    assert max_rel <= 1e-4 and rms_rel <= 1e-4, (max_rel, rms_rel)


def test_output_projection_tiny_f32_matches_oracle():
    dims = mi.TINY
    W_O = mi.output_weight(dims, "f32")
    o = mi.aux_normal((7, dims.n_h, dims.d_hc), index=410)
    got = _run(dims, "f32", o, W_O)
    want = ref.output_projection(o, W_O)
    mr, _ = rel_errors(got, want)
    assert mr <= TOL["f32"][0], mr


def test_decode_then_output_projection_end_to_end():
    """u of every sequence's new token after a decode step, against the oracle's decode and
    output projection."""
    lens = [1, 300, 129, 640]
    wl = mi.Workload("v2_small", mi.V2, "bf16", "decode", lens)
    dims = wl.dims
    W, W64 = oracle_weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    cache = host.LatentCache(dims, "bf16", mi.packed_layout(lens), int(sum(lens)))
    host.fill_context(model, cache, lambda b, n: mi.hidden(dims, "bf16", b, n), lens)
    step = host.DecodeStep(model, cache, lens, fused=True)
    h_new = np.stack([mi.hidden(dims, "bf16", b, L)[L - 1] for b, L in enumerate(lens)])
    o = step.step(host.to_device(h_new, "bf16")).cpu().numpy()
    assert mla.mla_get_device_status() == 0
    W_O = mi.output_weight(dims, "bf16")
    u = _run(dims, "bf16", o, W_O)
    want = ref.output_projection(np.stack(oracle_decode_step(wl, W64)["o"]), W_O)
    assert_close(u, want, "bf16", "u after decode")
