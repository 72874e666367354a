#!/usr/bin/env python3
"""Benchmark of the MLA hot path on B300: one decode step of the V2-shaped batch-16,
context-4096 workload (append the 16 new tokens' latent rows, project their queries,
weight-absorbed decode over the latent cache), the same step on the long-context and ragged
decode workloads (one block each under "configs"), plus the causal-prefill workload.

Prints ONE JSON line. ``--impl reference`` times the float64 CPU oracle instead (the
baseline arm). Under torchrun every rank runs its own replica of the workload (decode
sequences are independent; no data-path collective) and rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mla_inputs as mi  # noqa: E402

ROW_BYTES_BF16 = (512 + 64) * 2
DEFAULT_WORKLOAD = "v2_decode_b16_l4096"
EXTRA_DECODE_WORKLOADS = ("v2_decode_b1_l131072", "v2_decode_b4_l32768", "v2_decode_b128_ragged")
PREFILL_WORKLOAD = "v2_prefill_b2_t4096"
L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------- accounting
def decode_kernel_costs(wl: mi.Workload):
    """Algorithmic bytes and flops of each kernel of one decode step (inputs read once,
    outputs written once; split partials and other scratch traffic are not counted)."""
    d = wl.dims
    e = 2 if wl.dtype == "bf16" else 4
    B = wl.B
    rows = wl.n_rows
    nc, nr = d.n_h * d.d_hc, d.n_h * d.d_hr
    out = {
        "append": dict(bytes=(d.row * d.d + B * d.d + B * d.row) * e,
                       flops=2 * B * d.d * d.row),
        "q_down": dict(bytes=(d.d_cq * d.d + B * d.d) * e + B * d.d_cq * 4,
                       flops=2 * B * d.d * d.d_cq),
        "q_up": dict(bytes=(nc + nr) * d.d_cq * e + B * d.d_cq * 4 + B * (nc + nr) * e,
                     flops=2 * B * d.d_cq * (nc + nr)),
        "absorb": dict(bytes=nc * d.d_c * e + B * nc * e + B * d.n_h * d.d_c * e,
                       flops=2 * B * d.n_h * d.d_hc * d.d_c),
        # fused step: append + c^Q in one launch (W^DKV, W^KR, W^DQ read once) ...
        "down": dict(bytes=((d.row + d.d_cq) * d.d + B * d.d + B * d.row) * e + B * d.d_cq * 4,
                     flops=2 * B * d.d * (d.row + d.d_cq)),
        # ... and the query up-projection with the absorption applied (q^C stays on chip)
        "q_absorb": dict(bytes=((nc + nr) * d.d_cq + nc * d.d_c) * e
                         + B * d.d_cq * 4 + B * (d.n_h * d.d_c + nr) * e,
                         flops=2 * B * d.d_cq * (nc + nr) + 2 * B * d.n_h * d.d_hc * d.d_c),
        "decode_attn": dict(bytes=rows * d.row * e + B * d.n_h * (d.d_c + d.d_hr) * e,
                            flops=rows * (2 * d.n_h * d.row + 2 * d.n_h * d.d_c)),
        # merge of the split partials + W^UV: one SIMT kernel (decode_combine) or one
        # tensor-core kernel (unabsorb); only the one that ran is counted
        "decode_combine": dict(bytes=nc * d.d_c * e + B * d.n_h * d.d_hc * 4,
                               flops=2 * B * d.n_h * d.d_hc * d.d_c),
        "unabsorb": dict(bytes=nc * d.d_c * e + B * d.n_h * d.d_hc * 4,
                         flops=2 * B * d.n_h * d.d_hc * d.d_c),
    }
    return out


DECODE_CALL_KERNELS = ("absorb", "decode_attn", "decode_combine", "unabsorb")


def build_info():
    """Source identity of this run: the commit recorded by the library build (a copy of the
    tree may run without .git), else the current commit, plus a hash of the CUDA sources."""
    import hashlib
    info = {}
    try:
        info = json.load(open(os.path.join(ROOT, "_build", "build_info.json")))
    except Exception:
        try:
            info["git"] = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"], capture_output=True,
                                         text=True, timeout=10).stdout.strip() or None
        except Exception:
            info["git"] = None
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "mla_latent_kv_75_b300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    info["sources_sha1"] = h.hexdigest()
    return info


def prefill_flops(wl: mi.Workload):
    d = wl.dims
    n = wl.n_rows
    attn = sum(d.n_h * T * (T + 1) // 2 * 2 * (d.d_h + d.d_hc) for T in wl.seq_lens)
    proj = 2 * n * d.d * (d.d_cq + d.row) + 2 * n * d.d_cq * d.n_h * (d.d_hc + d.d_hr)
    expand = 2 * n * d.d_c * d.n_h * d.d_hc * 2
    return attn, proj + expand


def measured_traffic(kernel, workload):
    """DRAM bytes per launch of ``kernel`` from the committed ncu capture, or None when there
    is none for this workload or the kernel source changed since it was taken."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[kernel]
        src = open(os.path.join(ROOT, rec["source"]), "rb").read()
        if rec["workload"] != workload or hashlib.sha1(src).hexdigest() != rec["sha1"]:
            return None
        return int(rec["bytes"])
    except Exception:
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        p = json.load(open(path))
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "source": "fallback"}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["unsampled"]}
        loaded = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle arm
def oracle_decode_sample(wl: mi.Workload, budget_s: float, n_heads: int = 16,
                         max_seqs: int = 0):
    """Time the float64 oracle on whole sequences of the decode workload, restricted to
    ``n_heads`` evenly spaced heads: the new token's latent row and query, then the explicit
    per-head decode (K/V up-projection of every cached row) over all L rows. Sequences are
    added until about ``budget_s`` seconds of CPU work (at least one; at most ``max_seqs`` if
    set). The oracle's cost is linear in the number of heads, so the returned cache GB/s is
    scaled to the full head count; the sample description says what ran."""
    from oracle import mla_ref as ref
    d = wl.dims
    W = {k: v.astype(np.float64) for k, v in mi.weights(d, wl.dtype).items()}
    heads = list(range(0, d.n_h, max(1, d.n_h // n_heads)))[:n_heads]
    done_rows, spent, seqs = 0, 0.0, 0
    for b, L in enumerate(wl.seq_lens):
        h = mi.hidden(d, wl.dtype, b, L, wl.seed)
        c, kr = ref.kv_latent(h[:-1], W["W_DKV"], W["W_KR"], np.arange(L - 1), d.rope_base)
        ctx = ref.store(ref.cache_rows(c, kr), wl.dtype)            # cache fill: not timed
        t0 = time.perf_counter()
        c1, kr1 = ref.kv_latent(h[-1:], W["W_DKV"], W["W_KR"], [L - 1], d.rope_base)
        rows = np.concatenate([ctx, ref.store(ref.cache_rows(c1, kr1), wl.dtype)])
        q_c, q_r = ref.query(h[-1:], W["W_DQ"], W["W_UQ"], W["W_QR"], [L - 1], d.n_h, d.d_hc,
                             d.d_hr, d.rope_base)
        ref.decode_explicit(ref.store(q_c, wl.dtype), ref.store(q_r, wl.dtype), [rows],
                            W["W_UK"], W["W_UV"], d.d_c, heads=heads)
        spent += time.perf_counter() - t0
        done_rows += L
        seqs += 1
        if spent >= budget_s or (max_seqs and seqs >= max_seqs):
            break
    frac = len(heads) / d.n_h
    gbs = done_rows * d.row * (2 if wl.dtype == "bf16" else 4) * frac / spent / 1e9
    return gbs, spent, ("%d of %d sequences (%d cache rows), %d of %d heads; GB/s scaled to all "
                        "heads (the oracle's cost is linear in the head count)"
                        % (seqs, wl.B, done_rows, len(heads), d.n_h))


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        return int(max(n)) if n else os.cpu_count()
    except Exception:
        return os.cpu_count()


def run_reference(args, rank):
    """The baseline arm: the float64 CPU oracle (there is no other implementation of this path
    to compare with), timed on the host cores, one sequence x 8 heads per step."""
    if rank != 0:
        return
    wl = mi.workload(args.workload)
    for _ in range(args.warmup):
        oracle_decode_sample(wl, 0.0, n_heads=2, max_seqs=1)
    vals, times, sample = [], [], ""
    for _ in range(args.steps):
        v, t, sample = oracle_decode_sample(wl, 0.0, n_heads=8, max_seqs=1)
        vals.append(v)
        times.append(t)
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": metric_name(), "value": sig(value), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.mean(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl), "timing": ORACLE_TIMING,
        "cpu_baseline": {"value": sig(value), "unit": "GB/s", "cores": blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": sig(value), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (the job's time is that of its slowest rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, unit_bytes: int, steps: int, total_ms: float) -> float:
    """Whole-job GB/s: the bytes that all ranks processed over the slowest rank's time."""
    return world * unit_bytes * steps / (total_ms * 1e-3) / 1e9


# ----------------------------------------------------------------------------- GPU arm
def metric_name():
    return "MLA decode cache GB/s + TFLOP/s (% roofline) on 1 B300; prefill TFLOP/s"


def workload_config(wl):
    """The workload; identical in both arms (how each arm runs it is under "timing")."""
    return {"workload": wl.name, "B": wl.B, "context": int(max(wl.seq_lens)),
            "cache_rows": wl.n_rows, "dims": "d=5120 n_h=128 d_hc=128 d_hr=64 d_c=512 d_cq=1536",
            "step": "append B new rows + project B queries (absorbed) + decode over the latent "
                    "cache (mla_decode_step)"}


GPU_TIMING = {"launch": "CUDA graph of the library calls (e2e: eager calls + H2D/D2H copies)",
              "l2": "flushed between timed steps (256 MB write, then 256 MB read)"}
ORACLE_TIMING = {"launch": "float64 CPU oracle (explicit per-head form) on the host cores"}


def sig(x, n=4):
    """x rounded to n significant digits (the CPU baselines are far below 1 GB/s)."""
    return float("%.*g" % (n, x))


def setup_decode(wl, dev):
    """Device weights, the latent cache filled by mla_append_cache over every context token,
    and two steps over it: the one-call fused step and the three-call step."""
    import torch
    from mla_latent_kv_75_b300 import host
    d = wl.dims
    W = mi.weights(d, wl.dtype)
    model = host.DeviceModel.upload(d, wl.dtype, W, dev)
    base = mi.packed_layout(wl.seq_lens)
    cache = host.LatentCache(d, wl.dtype, base, wl.n_rows, device=dev)
    host.fill_context(model, cache, lambda b, n: mi.hidden(d, wl.dtype, b, n, wl.seed),
                      wl.seq_lens)
    step = host.DecodeStep(model, cache, wl.seq_lens, fused=True)
    step3 = host.DecodeStep(model, cache, wl.seq_lens)
    h_new = np.stack([mi.hidden_rows(d, wl.dtype, b, [L - 1], wl.seed)[0]
                      for b, L in enumerate(wl.seq_lens)])
    h_dev = host.to_device(h_new, wl.dtype, dev)
    h_host = host.to_device(h_new, wl.dtype, "cpu", pin=True)
    o_host = torch.empty(step.o.shape, dtype=step.o.dtype).pin_memory()
    torch.cuda.synchronize()
    return step, step3, h_dev, h_host, o_host


def time_steps(fn, steps, flush, trace_capacity=0, hold_ms=0.0):
    """Run ``steps`` steps, each bracketed by CUDA events on the current stream, with an L2
    flush before each (outside the events). Returns per-step ms and the kernel trace.
    ``hold_ms`` > 0 enqueues a sleep kernel of about that length before each step (outside the
    events) so that the whole step is queued before the GPU reaches it."""
    import torch
    import mla_latent_kv_75_b300 as mla
    st = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    trace = mla.KernelTrace(trace_capacity) if trace_capacity else None
    if trace:
        trace.__enter__()
    cycles = int(hold_ms * 1e-3 * 2.0e9)
    for k in range(steps):
        flush()
        if cycles:
            torch.cuda._sleep(cycles)
        evs[k][0].record(st)
        fn()
        evs[k][1].record(st)
    if trace:
        trace.__exit__(None, None, None)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    return ms, (trace.launches() if trace else [])


def kernel_table(launches, costs, peaks):
    """Per-kernel launches, mean device time, share of traced time and, for kernels with an
    algorithmic cost, GB/s, TFLOP/s and the fraction of their own roofline."""
    per = {}
    for name, t in launches:
        per.setdefault(name, []).append(t)
    total = sum(sum(v) for v in per.values()) or 1.0
    kernels = {}
    for name, ts in per.items():
        avg_ms = statistics.mean(ts)
        entry = {"launches": len(ts), "avg_us": round(avg_ms * 1e3, 3),
                 "share": round(sum(ts) / total, 4)}
        c = costs.get(name)
        if c and c["bytes"] > 0:
            floor_s = max(c["bytes"] / (peaks["hbm_gbs"] * 1e9),
                          c["flops"] / (peaks["bf16_tflops"] * 1e12))
            entry.update({"alg_bytes": c["bytes"], "alg_flops": c["flops"],
                          "GB_s": round(c["bytes"] / (avg_ms * 1e-3) / 1e9, 1),
                          "TFLOP_s": round(c["flops"] / (avg_ms * 1e-3) / 1e12, 2),
                          "roofline_frac": round(floor_s / (avg_ms * 1e-3), 4)})
        kernels[name] = entry
    return per, kernels


def roofline_of(name, per, costs, peaks, workload):
    """Roofline object of kernel ``name``: algorithmic bytes (or flops) per launch over its mean
    CUDA-event duration, against the measured peak of the bound it sits under."""
    c = costs[name]
    avg_s = statistics.mean(per[name]) * 1e-3
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if c["flops"] / c["bytes"] < ridge:
        achieved = c["bytes"] / avg_s / 1e9
        r = {"kernel": name, "bound": "hbm", "achieved": round(achieved, 1),
             "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        achieved = c["flops"] / avg_s / 1e12
        r = {"kernel": name, "bound": "tensor", "achieved": round(achieved, 2),
             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
             "frac": round(achieved / peaks["bf16_tflops"], 4)}
    r["peak_source"] = peaks["source"]
    r["traffic"] = measured_traffic(name, workload)
    return r


def call_block(names, per, costs, peaks, cache_bytes):
    """Time, floor and roofline fraction of a group of kernels (one library call)."""
    dec = [n for n in names if n in per]
    dec_s = sum(statistics.mean(per[n]) for n in dec) * 1e-3
    if dec_s <= 0:
        return None
    dec_bytes = sum(costs[n]["bytes"] for n in dec)
    dec_flops = sum(costs[n]["flops"] for n in dec)
    floor_s = max(dec_bytes / (peaks["hbm_gbs"] * 1e9), dec_flops / (peaks["bf16_tflops"] * 1e12))
    return {"kernels": dec, "us": round(dec_s * 1e6, 2), "floor_us": round(floor_s * 1e6, 2),
            "alg_bytes": dec_bytes, "alg_flops": dec_flops,
            "cache_GB_s": round(cache_bytes / dec_s / 1e9, 1),
            "TFLOP_s": round(dec_flops / dec_s / 1e12, 2), "roofline_frac": round(floor_s / dec_s, 4)}


def measure_decode(wl, args, dev, peaks, flush, world, steps, want_cpu, cpu_seconds,
                   cpu_heads=16, cpu_max_seqs=0):
    """One decode workload: the graph-timed step (the one-call fused step, mla_decode_step; the
    three-call step beside it), per-kernel device times of both, the e2e step and (rank 0, one
    GPU) the oracle on a bounded sample. Frees its device buffers on return."""
    import torch
    import mla_latent_kv_75_b300 as mla

    step, step3, h_dev, h_host, o_host = setup_decode(wl, dev)

    def e2e_step():
        h_dev.copy_(h_host, non_blocking=True)
        step.step(h_dev)
        o_host.copy_(step.o, non_blocking=True)

    def graph_of(st):
        for _ in range(max(3, args.warmup)):
            flush()
            st.step(h_dev)
        assert mla.mla_get_device_status() == 0
        if args.no_graph:
            return lambda: st.step(h_dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st.step(h_dev)
        for _ in range(max(3, args.warmup)):
            flush()
            g.replay()
        torch.cuda.synchronize()
        return g.replay

    # The timed decode step is a CUDA graph of the library's launches (how a decode loop runs in
    # production: no host work between kernels).
    run_f, run_3 = graph_of(step), graph_of(step3)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    ms, _ = time_steps(run_f, steps, flush)
    ms3, _ = time_steps(run_3, steps, flush)
    # Per-kernel device times: the same steps as eager library calls, each enqueued behind a
    # sleep kernel so that the host never starves the GPU between launches; CUDA event pairs
    # around every launch (on its stream) then time the kernels alone.
    _, launches = time_steps(lambda: step.step(h_dev), steps, flush, trace_capacity=64 * steps,
                             hold_ms=0.5)
    _, launches3 = time_steps(lambda: step3.step(h_dev), steps, flush,
                              trace_capacity=64 * steps, hold_ms=0.5)
    torch.cuda.synchronize()
    assert mla.mla_get_device_status() == 0
    total_ms = max_over_ranks(sum(ms), world, dev)
    total3_ms = max_over_ranks(sum(ms3), world, dev)

    for _ in range(3):
        flush()
        e2e_step()
    e2e_ms, _ = time_steps(e2e_step, steps, flush)
    e2e_total = max_over_ranks(sum(e2e_ms), world, dev)

    costs = decode_kernel_costs(wl)
    e = 2 if wl.dtype == "bf16" else 4
    cache_bytes = wl.n_rows * wl.dims.row * e
    per, kernels = kernel_table(launches, costs, peaks)
    per3, kernels3 = kernel_table(launches3, costs, peaks)
    step_flops = sum(costs[n]["flops"] for n in per if n in costs)
    step_bytes = sum(costs[n]["bytes"] for n in per if n in costs)
    dominant = max(per, key=lambda n: sum(per[n])) if per else None
    roofline = roofline_of(dominant, per, costs, peaks, wl.name) if dominant in costs else None
    out = {
        "value": round(job_rate(world, cache_bytes, steps, total_ms), 2), "unit": "GB/s",
        "ms_per_step": round(total_ms / steps, 4), "steps": steps,
        "tflops": round(world * step_flops * steps / (total_ms * 1e-3) / 1e12, 3),
        "step_alg_bytes": step_bytes,
        "step_roofline_frac": round(step_bytes / (peaks["hbm_gbs"] * 1e9) / (total_ms / steps * 1e-3), 4),
        "config": workload_config(wl), "roofline": roofline,
        # the mla_decode_absorbed call (absorb + attention + merge/un-absorb), from the
        # three-call step; and the latent decode of the fused step (attention + merge/un-absorb)
        "decode_call": call_block(DECODE_CALL_KERNELS, per3, costs, peaks, cache_bytes),
        "decode_latent_call": call_block(("decode_attn", "decode_combine", "unabsorb"), per, costs,
                                         peaks, cache_bytes),
        "kernels": kernels, "gpu_launches": len(launches),
        "three_call_step": {"ms_per_step": round(total3_ms / steps, 4),
                            "value": round(job_rate(world, cache_bytes, steps, total3_ms), 2),
                            "kernels": kernels3},
        "e2e": {"value": round(job_rate(world, cache_bytes, steps, e2e_total), 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h_host.numel() * h_host.element_size()),
                "d2h_bytes_per_step": int(o_host.numel() * o_host.element_size()),
                "ms_per_step": round(e2e_total / steps, 4), "call": "mla_decode_step"},
        "fast_path": mla.mla_fast_path(step.model.abi_dims),
    }
    del run_f, run_3, step, step3, h_dev, h_host, o_host
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if want_cpu:
        v, spent, sample = oracle_decode_sample(wl, cpu_seconds, n_heads=cpu_heads,
                                               max_seqs=cpu_max_seqs)
        out["cpu_baseline"] = {"value": sig(v), "unit": "GB/s", "cores": blas_threads(),
                               "kind": "oracle", "sample": sample, "seconds": round(spent, 2)}
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import mla_latent_kv_75_b300 as mla  # noqa: F401  (fails loudly without the library)

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clean_buf = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        # Write a buffer larger than L2, then read another: no step data stays in L2, and no
        # dirty flush lines are left for the timed step to write back.
        flush_buf.zero_()
        clean_buf.sum()

    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    with ClockSampler(torch.cuda.current_device()) as clk:
        main = measure_decode(mi.workload(args.workload), args, dev, peaks, flush, world,
                              args.steps, want_cpu, args.cpu_seconds)
        configs = {}
        if not args.no_extra_configs and args.workload == DEFAULT_WORKLOAD:
            for name in EXTRA_DECODE_WORKLOADS:
                configs[name] = measure_decode(mi.workload(name), args, dev, peaks, flush, world,
                                               max(1, min(args.steps, args.extra_steps)), want_cpu,
                                               args.extra_cpu_seconds, cpu_heads=4, cpu_max_seqs=1)
    clocks = clk.summary()

    prefill = None
    if not args.no_prefill:
        prefill = run_prefill(args, dev, peaks, flush)
    out_proj = query_variants = sparse = None
    if not args.no_extra_configs:
        out_proj = run_output_projection(args, dev, peaks, flush)
        query_variants = run_query_variants(args, dev, peaks, flush)
        sparse = run_sparse_decode(args, dev, peaks, flush)

    if rank == 0:
        line = {
            "metric": metric_name(), "value": main["value"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": main["config"], "timing": GPU_TIMING,
            "tflops": main["tflops"], "roofline": main["roofline"],
            "decode_call": main["decode_call"], "decode_latent_call": main["decode_latent_call"],
            "step_roofline_frac": main["step_roofline_frac"], "kernels": main["kernels"],
            "three_call_step": main["three_call_step"], "configs": configs, "prefill": prefill,
            "output_projection": out_proj, "query_variants": query_variants,
            "sparse_decode": sparse,
            "cpu_baseline": main.get("cpu_baseline"), "e2e": main["e2e"],
            "gpu_launches": main["gpu_launches"], "clocks": clocks, "fast_path": main["fast_path"],
            "build": build_info(),
        }
        print(json.dumps(line), flush=True)


def run_output_projection(args, dev, peaks, flush):
    """u = W^O [o_1; ...; o_{n_h}] at the decode batch (16 tokens: W^O streaming, HBM-bound)
    and at the prefill size (8192 tokens: tensor-bound), through mla_output_projection."""
    import torch
    import mla_latent_kv_75_b300 as mla
    from mla_latent_kv_75_b300 import host
    d = mi.V2
    dims = host.dims_struct(d, "bf16")
    W_O = host.to_device(mi.output_weight(d, "bf16"), "bf16", dev)
    K = d.n_h * d.d_hc
    out = {}
    for n in (16, 8192):
        o = torch.randn((n, K), device=dev, dtype=torch.float32)
        u = torch.empty((n, d.d), device=dev, dtype=torch.float32)
        ws_bytes = mla.mla_output_projection_workspace_size(dims, n)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        call = lambda: mla.mla_output_projection(dims, W_O, o, n, ws, ws_bytes, u)
        for _ in range(3):
            flush()
            call()
        assert mla.mla_get_device_status() == 0
        steps = max(1, min(args.steps, 10))
        ms, launches = time_steps(call, steps, flush, trace_capacity=4 * steps, hold_ms=0.5)
        per = {}
        for name, t in launches:
            per.setdefault(name, []).append(t)
        t_s = statistics.mean(ms) * 1e-3
        alg_bytes = d.d * K * 2 + n * K * 4 + n * d.d * 4
        flops = 2 * n * K * d.d
        floor_s = max(alg_bytes / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
        out["n%d" % n] = {"us": round(t_s * 1e6, 2), "alg_bytes": alg_bytes, "alg_flops": flops,
                          "GB_s": round(alg_bytes / t_s / 1e9, 1),
                          "TFLOP_s": round(flops / t_s / 1e12, 2),
                          "roofline_frac": round(floor_s / t_s, 4),
                          "kernels_us": {k: round(statistics.mean(v) * 1e3, 2)
                                         for k, v in per.items()}}
        del o, u, ws
    del W_O
    torch.cuda.empty_cache()
    return out


def run_query_variants(args, dev, peaks, flush):
    """The absorbed decode query two ways, at 16 and 128 tokens: the fused two-product kernel
    (mla_project_q_absorbed: W^UQ, W^QR and W^UK streamed, 92 MB) against the pre-merged map
    (mla_project_q_premerged: W^UQK = (W^UK_i)^T W^UQ_i formed once, 201 MB, with W^QR); both
    include the c^Q down-projection. Per-call device time and the call's HBM roofline."""
    import torch
    import mla_latent_kv_75_b300 as mla
    from mla_latent_kv_75_b300 import host
    d = mi.V2
    model = host.DeviceModel.upload(d, "bf16", mi.weights(d, "bf16"), dev)
    dims, w = model.abi_dims, model.abi_weights
    W_UQK = torch.empty((d.n_h * d.d_c, d.d_cq), dtype=torch.bfloat16, device=dev)
    mla.mla_merge_query_absorption(dims, model.W["W_UQ"], model.W["W_UK"], W_UQK)
    assert mla.mla_get_device_status() == 0
    wbytes = {"fused": (d.d_cq * d.d + d.n_h * (d.d_hc + d.d_hr) * d.d_cq + d.n_h * d.d_hc * d.d_c) * 2,
              "premerged": (d.d_cq * d.d + d.n_h * (d.d_c + d.d_hr) * d.d_cq) * 2}
    out = {"weight_bytes": wbytes}
    for n in (16, 128):
        h = torch.randn((n, d.d), device=dev).to(torch.bfloat16)
        pos = torch.arange(n, dtype=torch.int32, device=dev) * 37
        ws_bytes = mla.mla_project_q_workspace_size(dims, n)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        q_t = torch.empty((n, d.n_h, d.d_c), dtype=torch.bfloat16, device=dev)
        q_r = torch.empty((n, d.n_h, d.d_hr), dtype=torch.bfloat16, device=dev)
        calls = {"fused": lambda: mla.mla_project_q_absorbed(dims, w, h, pos, n, ws, ws_bytes, q_t, q_r),
                 "premerged": lambda: mla.mla_project_q_premerged(dims, w, W_UQK, h, pos, n, ws,
                                                                  ws_bytes, q_t, q_r)}
        res = {}
        for name, call in calls.items():
            for _ in range(3):
                flush()
                call()
            assert mla.mla_get_device_status() == 0
            steps = max(1, min(args.steps, 10))
            _, launches = time_steps(call, steps, flush, trace_capacity=4 * steps, hold_ms=0.5)
            per = {}
            for k, t in launches:
                per.setdefault(k, []).append(t)
            us = sum(statistics.mean(v) for v in per.values()) * 1e3
            alg = wbytes[name] + n * d.d * 2 + n * d.n_h * (d.d_c + d.d_hr) * 2
            res[name] = {"us": round(us, 2), "alg_bytes": alg,
                         "roofline_frac": round(alg / (peaks["hbm_gbs"] * 1e9) / (us * 1e-6), 4),
                         "kernels_us": {k: round(statistics.mean(v) * 1e3, 2) for k, v in per.items()}}
        out["n%d" % n] = res
    del model, W_UQK
    torch.cuda.empty_cache()
    return out


SPARSE_CASES = (("v2_decode_b16_l4096", 2048), ("v2_decode_b1_l131072", 2048))


def run_sparse_decode(args, dev, peaks, flush):
    """Top-k sparse decode (mla_decode_absorbed_sparse: selection on the index scores, gather of
    the picked rows, absorbed decode over them) on two decode workloads with k = 2048. The
    algorithmic bytes are the scores (4 B per cached position), the picked rows (1152 B each),
    W^UK and W^UV, q and o; the gather's copy is not counted. Synthetic N(0,1) rows, queries
    and scores."""
    import torch
    import mla_latent_kv_75_b300 as mla
    from mla_latent_kv_75_b300 import host
    d = mi.V2
    model = host.DeviceModel.upload(d, "bf16", mi.weights(d, "bf16"), dev)
    dims, w = model.abi_dims, model.abi_weights
    out = {}
    for name, k in SPARSE_CASES:
        wl = mi.workload(name)
        lens = wl.seq_lens
        B, max_len = wl.B, max(lens)
        g = torch.Generator(device=dev)
        g.manual_seed(5)
        cache = host.LatentCache(d, "bf16", mi.packed_layout(lens), wl.n_rows, device=dev)
        cache.rows.copy_(torch.randn(cache.rows.shape, device=dev, generator=g).to(torch.bfloat16))
        q_c = torch.randn((B, d.n_h, d.d_hc), device=dev, generator=g).to(torch.bfloat16)
        q_r = torch.randn((B, d.n_h, d.d_hr), device=dev, generator=g).to(torch.bfloat16)
        scores = torch.randn((B, max_len), device=dev, generator=g)
        seq_len = torch.tensor(lens, dtype=torch.int32, device=dev)
        ws_bytes = mla.mla_decode_sparse_workspace_size(dims, B, k)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        o = torch.empty((B, d.n_h, d.d_hc), dtype=torch.float32, device=dev)
        c = cache.abi
        call = lambda: mla.mla_decode_absorbed_sparse(dims, w, q_c, q_r, c, seq_len, B, max_len,
                                                      scores, max_len, k, ws, ws_bytes, o)
        for _ in range(3):
            flush()
            call()
        assert mla.mla_get_device_status() == 0
        steps = max(1, min(args.steps, 10))
        ms, launches = time_steps(call, steps, flush, trace_capacity=8 * steps, hold_ms=0.5)
        per = {}
        for kn, t in launches:
            per.setdefault(kn, []).append(t)
        us = sum(statistics.mean(v) for v in per.values()) * 1e3
        picked = sum(min(L, k) for L in lens)
        row_b = (d.d_c + d.d_hr) * 2
        alg = (sum(lens) * 4 + picked * row_b + 2 * d.n_h * d.d_hc * d.d_c * 2
               + B * d.n_h * (d.d_hc + d.d_hr) * 2 + B * d.n_h * d.d_hc * 4)
        flops = picked * 2 * d.n_h * (d.d_c + d.d_hr + d.d_c)
        floor_s = max(alg / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
        sel_us = statistics.mean(per["topk_select"]) * 1e3 if "topk_select" in per else None
        out["%s_k%d" % (name, k)] = {
            "us": round(us, 2), "call_us": round(statistics.mean(ms) * 1e3, 2),
            "picked_rows": picked, "alg_bytes": alg, "alg_flops": flops,
            "roofline_frac": round(floor_s / (us * 1e-6), 4),
            "select_GB_s": round(sum(lens) * 4 / (sel_us * 1e-6) / 1e9, 1) if sel_us else None,
            "kernels_us": {kn: round(statistics.mean(v) * 1e3, 2) for kn, v in per.items()}}
        del cache, ws, scores
        torch.cuda.empty_cache()
    del model
    torch.cuda.empty_cache()
    return out


def run_prefill(args, dev, peaks, flush):
    import torch
    from mla_latent_kv_75_b300 import host
    import mla_latent_kv_75_b300 as mla
    wl = mi.workload(PREFILL_WORKLOAD)
    d = wl.dims
    W = mi.weights(d, wl.dtype)
    model = host.DeviceModel.upload(d, wl.dtype, W, dev)
    cache = host.LatentCache(d, wl.dtype, mi.packed_layout(wl.seq_lens), wl.n_rows, device=dev)
    pre = host.PrefillStep(model, cache, wl.seq_lens)
    h = host.to_device(np.concatenate([mi.hidden(d, wl.dtype, b, L, wl.seed)
                                       for b, L in enumerate(wl.seq_lens)]), wl.dtype, dev)
    steps = max(1, min(args.steps, args.prefill_steps))
    for _ in range(3):
        pre.run(h)
    assert mla.mla_get_device_status() == 0
    ms, launches = time_steps(lambda: pre.run(h), steps, flush, trace_capacity=16 * steps)
    attn_f, other_f = prefill_flops(wl)
    per = {}
    for name, t in launches:
        per.setdefault(name, []).append(t)
    attn_ms = statistics.mean(per["prefill_attn"]) if "prefill_attn" in per else None
    step_ms = statistics.mean(ms)
    out = {"workload": wl.name, "ms_per_step": round(step_ms, 3),
           "TFLOP_s": round((attn_f + other_f) / (step_ms * 1e-3) / 1e12, 2),
           "attn_TFLOP_s": round(attn_f / (attn_ms * 1e-3) / 1e12, 2) if attn_ms else None,
           "attn_frac_of_peak": round(attn_f / (attn_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)
           if attn_ms else None,
           "kernels_us": {n: round(statistics.mean(v) * 1e3, 1) for n, v in per.items()}}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--prefill-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the decode step as eager library calls instead of a CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="skip the long-context and ragged decode workloads")
    ap.add_argument("--extra-steps", type=int, default=10,
                    help="timed steps of each extra decode workload")
    ap.add_argument("--extra-cpu-seconds", type=float, default=4.0)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
