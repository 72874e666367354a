"""The bench's roofline arithmetic on CPU: algorithmic bytes and FLOPs per kernel from first
principles, the bound a kernel is judged against, and the fractions the JSON line reports."""
import pytest

import bench
import mla_inputs as mi

PEAKS = {"hbm_gbs": 6500.0, "bf16_tflops": 1756.5, "bf16_tflops_sustained": 1352.2,
         "source": "test"}


def test_attention_bytes_and_flops_per_cached_row():
    """Per cached row: 576 bf16 values read once (1152 B) and 2 n_h (576 + 512) FLOPs (scores
    over the 576-wide row, then P times the 512-wide latent); plus the query read once."""
    wl = mi.workload("v2_decode_b16_l4096")
    c = bench.decode_kernel_costs(wl)["decode_attn"]
    rows = 16 * 4096
    assert c["bytes"] == rows * 1152 + 16 * 128 * 576 * 2
    assert c["flops"] == rows * 278528
    # under the ridge (about 270 FLOP/B at these peaks): judged against HBM
    assert c["flops"] / c["bytes"] < PEAKS["bf16_tflops"] * 1e12 / (PEAKS["hbm_gbs"] * 1e9)


def test_weight_bytes_of_the_projection_kernels():
    wl = mi.workload("v2_decode_b16_l4096")
    c = bench.decode_kernel_costs(wl)
    w = {  # bf16 weight bytes at the V2 widths
        "W_DKV+W_KR": (512 + 64) * 5120 * 2, "W_DQ": 1536 * 5120 * 2,
        "W_UQ+W_QR": (16384 + 8192) * 1536 * 2, "W_UK": 16384 * 512 * 2, "W_UV": 16384 * 512 * 2}
    assert c["down"]["bytes"] > w["W_DKV+W_KR"] + w["W_DQ"]
    assert c["down"]["bytes"] - (w["W_DKV+W_KR"] + w["W_DQ"]) < 1 << 20  # activations only
    assert c["q_absorb"]["bytes"] - (w["W_UQ+W_QR"] + w["W_UK"]) < 4 << 20
    assert c["unabsorb"]["bytes"] == w["W_UV"] + 16 * 128 * 128 * 4


def test_roofline_object_and_kernel_table_agree():
    wl = mi.workload("v2_decode_b16_l4096")
    costs = bench.decode_kernel_costs(wl)
    launches = [("decode_attn", 0.044), ("decode_attn", 0.046), ("unabsorb", 0.014)]
    per, table = bench.kernel_table(launches, costs, PEAKS)
    r = bench.roofline_of("decode_attn", per, costs, PEAKS, wl.name)
    achieved = costs["decode_attn"]["bytes"] / 45e-6 / 1e9
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(achieved, abs=0.1)
    assert r["frac"] == pytest.approx(achieved / 6500.0, abs=1e-4)
    assert table["decode_attn"]["roofline_frac"] == pytest.approx(r["frac"], abs=1e-4)
    assert table["decode_attn"]["launches"] == 2
    assert table["decode_attn"]["share"] + table["unabsorb"]["share"] == pytest.approx(1.0)


def test_call_block_floor_is_the_slower_of_bytes_and_flops():
    wl = mi.workload("v2_decode_b16_l4096")
    costs = bench.decode_kernel_costs(wl)
    per = {"absorb": [0.010], "decode_attn": [0.044], "unabsorb": [0.014]}
    blk = bench.call_block(bench.DECODE_CALL_KERNELS, per, costs, PEAKS, 16 * 4096 * 1152)
    b = sum(costs[k]["bytes"] for k in ("absorb", "decode_attn", "unabsorb"))
    f = sum(costs[k]["flops"] for k in ("absorb", "decode_attn", "unabsorb"))
    floor = max(b / 6500e9, f / 1756.5e12)
    assert blk["floor_us"] == pytest.approx(floor * 1e6, abs=0.01)
    assert blk["us"] == pytest.approx(68.0, abs=1e-6)
    assert blk["roofline_frac"] == pytest.approx(floor / 68e-6, abs=1e-4)
    assert blk["kernels"] == ["absorb", "decode_attn", "unabsorb"]  # the SIMT merge did not run
