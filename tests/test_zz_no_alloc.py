"""mla_decode_absorbed_static: decode for callers that cannot allocate device memory.

Such callers (a plugin inside a framework that owns all device allocations, or a loop that
must not call cudaMalloc after start-up) get their scratch from a fixed array compiled into
the library instead of a workspace they allocate. These tests call that entry point through
the C ABI and check that it returns what mla_decode_absorbed returns with a caller-allocated
workspace, on two calls in a row, and that an oversized problem is refused before launching.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import mla_latent_kv_75_b300 as mla
from mla_latent_kv_75_b300 import host
from helpers import assert_close

pytestmark = pytest.mark.gpu


def _setup(lens, index0, model=None):
    dims = mi.V2
    if model is None:
        model = host.DeviceModel.upload(dims, "bf16", mi.weights(dims, "bf16"))
    base = mi.packed_layout(lens, guard=2)
    cap = int(base[-1] + lens[-1] + 2)
    cache = host.LatentCache(dims, "bf16", base, cap)
    cache.rows.copy_(host.to_device(mi.aux_normal((cap, dims.row), index=index0, dtype="bf16"),
                                    "bf16"))
    q_c = host.to_device(mi.aux_normal((len(lens), dims.n_h, dims.d_hc), index=index0 + 1,
                                       dtype="bf16"), "bf16")
    q_r = host.to_device(mi.aux_normal((len(lens), dims.n_h, dims.d_hr), index=index0 + 2,
                                       dtype="bf16"), "bf16")
    return model, cache, q_c, q_r


def _static_vs_workspace(model, cache, q_c, q_r, lens, tol="bf16"):
    step = host.DecodeStep(model, cache, lens)
    want = step.decode(q_c=q_c, q_r=q_r).clone()
    assert mla.mla_get_device_status() == 0
    o = torch.full_like(want, float("nan"))
    mla.mla_decode_absorbed_static(model.abi_dims, model.abi_weights, q_c, q_r, cache.abi,
                                   step.seq_len, step.B, step.max_len, o)
    assert mla.mla_get_device_status() == 0
    assert_close(o.cpu().numpy().astype(np.float64), want.cpu().numpy().astype(np.float64), tol,
                 "static-scratch decode")


def test_static_scratch_decode_matches_workspace_decode_on_two_calls():
    lens = [1, 300, 1500, 64]
    model, cache, q_c, q_r = _setup(lens, 500)
    step = host.DecodeStep(model, cache, lens)
    want = step.decode(q_c=q_c, q_r=q_r).clone()
    assert mla.mla_get_device_status() == 0
    want_np = want.cpu().numpy().astype(np.float64)
    for _ in range(2):
        o = torch.full_like(want, float("nan"))
        mla.mla_decode_absorbed_static(model.abi_dims, model.abi_weights, q_c, q_r, cache.abi,
                                       step.seq_len, step.B, step.max_len, o)
        assert mla.mla_get_device_status() == 0
        assert_close(o.cpu().numpy().astype(np.float64), want_np, "bf16", "static-scratch decode")


def test_static_scratch_refuses_problems_above_its_capacity():
    dims = mi.V2
    d = host.dims_struct(dims, "bf16")
    B, max_len = 128, 8193
    assert mla.mla_decode_workspace_size(d, B, max_len) > mla.MLA_STATIC_WS_BYTES
    model, cache, q_c, q_r = _setup([4], 510)
    seq_len = torch.full((B,), 4, dtype=torch.int32, device="cuda")
    o = torch.zeros((B, dims.n_h, dims.d_hc), dtype=torch.float32, device="cuda")
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_decode_absorbed_static(model.abi_dims, model.abi_weights, q_c, q_r, cache.abi,
                                       seq_len, B, max_len, o)
    assert ei.value.status == 7
    assert torch.count_nonzero(o) == 0


def test_static_scratch_large_spanning_call_then_small_call():
    """The array keeps the previous call's contents. A 31-sequence call whose work split crosses
    sequence boundaries (one long sequence and thirty short ones: many partial slots), then a
    3-sequence call that uses few: the second must not read anything the first left behind."""
    lens_big = [74 * 48 * 3] + [5] * 30
    model, cache, q_c, q_r = _setup(lens_big, 530)
    _static_vs_workspace(model, cache, q_c, q_r, lens_big)
    lens_small = [700, 1, 96]
    _, cache2, q_c2, q_r2 = _setup(lens_small, 540, model)
    _static_vs_workspace(model, cache2, q_c2, q_r2, lens_small)


def test_static_scratch_tiny_fp32_call():
    """The SIMT path (fp32, other widths) through the same array."""
    dims = mi.TINY
    W = mi.weights(dims, "f32")
    model = host.DeviceModel.upload(dims, "f32", W)
    lens = [65, 9]
    base = mi.packed_layout(lens)
    cap = int(sum(lens))
    cache = host.LatentCache(dims, "f32", base, cap)
    cache.rows.copy_(host.to_device(mi.aux_normal((cap, dims.row), index=550), "f32"))
    q_c = host.to_device(mi.aux_normal((2, dims.n_h, dims.d_hc), index=551), "f32")
    q_r = host.to_device(mi.aux_normal((2, dims.n_h, dims.d_hr), index=552), "f32")
    _static_vs_workspace(model, cache, q_c, q_r, lens, tol="f32")
