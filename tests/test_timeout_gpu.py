"""Failure detection on the GPU without a fault: a bounded wait inside the decode attention
kernel is made to run out (it waits for a barrier phase that nothing completes, with a 1 ms
limit). The kernel must report MLA_ERR_TIMEOUT through the device status word, leave no copy
or MMA in flight, and the next call on the same device must run normally and match the
oracle."""
import numpy as np
import pytest

import mla_inputs as mi
import mla_latent_kv_75_b300 as mla
from mla_latent_kv_75_b300 import host
from oracle import mla_ref as ref
from helpers import assert_close, oracle_weights

pytestmark = pytest.mark.gpu

MLA_ERR_TIMEOUT = 6


def _decode_setup(lens):
    dims = mi.V2
    W, W64 = oracle_weights(dims, "bf16")
    model = host.DeviceModel.upload(dims, "bf16", W)
    base = mi.packed_layout(lens)
    cap = int(base[-1] + lens[-1])
    rows_np = mi.aux_normal((cap, dims.row), index=300, dtype="bf16")
    cache = host.LatentCache(dims, "bf16", base, cap)
    cache.rows.copy_(host.to_device(rows_np, "bf16"))
    q_c = mi.aux_normal((len(lens), dims.n_h, dims.d_hc), index=301, dtype="bf16")
    q_r = mi.aux_normal((len(lens), dims.n_h, dims.d_hr), index=302, dtype="bf16")
    step = host.DecodeStep(model, cache, lens)
    rows = [rows_np[base[b]: base[b] + L].astype(np.float64) for b, L in enumerate(lens)]
    return step, q_c, q_r, rows, W64


@pytest.mark.parametrize("lens", [[5000], [300, 2000, 4096, 17]])
def test_bounded_wait_runs_out_and_the_next_call_is_clean(lens):
    step, q_c, q_r, rows, W64 = _decode_setup(lens)
    qc_d, qr_d = host.to_device(q_c, "bf16"), host.to_device(q_r, "bf16")
    assert mla.mla_get_device_status() == 0
    mla.mla_debug_arm_wait_timeout(1_000_000)  # 1 ms
    step.decode(q_c=qc_d, q_r=qr_d)
    assert mla.mla_get_device_status() == MLA_ERR_TIMEOUT
    # the hook is one-shot: the next call is a normal decode
    o = step.decode(q_c=qc_d, q_r=qr_d).cpu().numpy()
    assert mla.mla_get_device_status() == 0
    heads = [0, 45, 127]
    want = ref.decode_explicit(q_c, q_r, rows, W64["W_UK"], W64["W_UV"], mi.V2.d_c, heads=heads)
    assert_close(o[:, heads], want, "bf16", "decode after a timed-out call")
