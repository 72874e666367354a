"""MLA_DEBUG: with it set, every launch of the library is followed by a check of the stream
and of the device status word, reported on stderr with the kernel's name. Run in child
processes because the variable is read once per process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CLEAN_RUN = r"""
import numpy as np, torch
import mla_inputs as mi
import mla_latent_kv_75_b300 as mla
from mla_latent_kv_75_b300 import host
dims = mi.V2
model = host.DeviceModel.upload(dims, "bf16", mi.weights(dims, "bf16"))
lens = [5, 130]
cache = host.LatentCache(dims, "bf16", mi.packed_layout(lens), sum(lens))
host.fill_context(model, cache, lambda b, n: mi.hidden(dims, "bf16", b, n), lens)
step = host.DecodeStep(model, cache, lens, fused=True)
h = np.stack([mi.hidden(dims, "bf16", b, L)[L - 1] for b, L in enumerate(lens)])
step.step(host.to_device(h, "bf16"))
assert mla.mla_get_device_status() == 0
print("done")
"""

LENGTH_VIOLATION = r"""
import torch
import mla_inputs as mi
import mla_latent_kv_75_b300 as mla
from mla_latent_kv_75_b300 import host
dims = mi.V2
model = host.DeviceModel.upload(dims, "bf16", mi.weights(dims, "bf16"))
cache = host.LatentCache(dims, "bf16", [0, 10], 16, fill=0.0)
step = host.DecodeStep(model, cache, [4, 6], max_len=5)  # 6 > max_len: clamped and flagged
q = host.to_device(mi.aux_normal((2, 128, 128), index=3, dtype="bf16"), "bf16")
qr = host.to_device(mi.aux_normal((2, 128, 64), index=4, dtype="bf16"), "bf16")
step.decode(q_c=q, q_r=qr)
print("status", int(mla.mla_get_device_status()))
"""


def _run(code):
    env = dict(os.environ, MLA_DEBUG="1", PYTHONPATH=ROOT)
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=600)


def test_debug_checks_report_nothing_on_a_clean_step():
    r = _run(CLEAN_RUN)
    assert r.returncode == 0, r.stderr
    assert "done" in r.stdout
    assert "mla:" not in r.stderr, r.stderr


def test_debug_checks_name_the_kernel_that_latched_a_status():
    r = _run(LENGTH_VIOLATION)
    assert r.returncode == 0, r.stderr
    assert "status 8" in r.stdout
    assert "mla: after" in r.stderr and "device status 8" in r.stderr, r.stderr
