#!/usr/bin/env python
"""Decode throughput of the 4-bit decode step on GB300.

One "step" is one batch-1 decode step of the whole hot path (embedding, every
layer's RMSNorm / q|k|v GEMV / RoPE + KV append / attention / o GEMV /
RMSNorm / gate|up GEMV / SwiGLU / down GEMV, final RMSNorm, LM head, argmax)
on seeded synthetic weights of the named shape. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl ours|reference]

--impl reference times the CPU oracle on the host cores (the pages publish no
runnable implementation). Multi-GPU runs are independent replicas (the
batch-1 step has no shardable data-parallel dimension): value = tokens of all
ranks / max elapsed over ranks.
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

import synth  # noqa: E402

METRIC = "decode tok/s (batch 1) and achieved HBM GB/s as % of GB300 roofline"


def args_():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", type=int, default=1)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--kv", default="bf16", choices=["bf16", "q8"],
                    help="K/V cache format: bf16, or the grouped int8 cache (LLM_KV_Q8)")
    ap.add_argument("--w4a8", action="store_true", help="int8 activation blocks in the batch-1 GEMVs (LLM_W4A8)")
    ap.add_argument("--phases", action="store_true",
                    help="per-phase breakdown of one grid-barrier step (builds a stamps variant of the library); "
                         "prints a table, not a bench line")
    ap.add_argument("--regions", type=int, default=5,
                    help="timed regions of K steps each (same positions); value = the median region")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers of the workload (small profiling cases; not a bench line)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# the sources a kernel's code comes from (the step kernel is defined in these headers)
KERNEL_SOURCES = {"step_kernel": ("common.cuh", "kernels.cuh", "attn_mma.cuh", "step.cuh", "step_kernels.cu")}


def src_sha(kernel="step_kernel"):
    """Hash of a kernel's sources: an ncu traffic figure is only used for the code it was taken on."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "bit_quantized_token_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(key):
    """DRAM bytes per launch from profiles/traffic.json, or None if absent or stale."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    t = json.load(open(p)).get(key)
    return t["traffic_bytes"] if t and t.get("src_sha") == src_sha(key.split()[0]) else None


def workload_desc(cfg, kv="bf16", w4a8=False):
    full = synth.workload(cfg["index"])["n_layers"] if "index" in cfg else cfg["n_layers"]
    layers = f"{cfg['n_layers']} layers" if cfg["n_layers"] == full else f"first {cfg['n_layers']} of {full} layers"
    acts = "int8 activation blocks (W4A8)" if w4a8 else "fp32 activations"
    cache = "grouped int8 KV (32-value groups, fp16 scales)" if kv == "q8" else "bf16 KV"
    return (f"{cfg['name']}: dim {cfg['dim']}, {layers}, {cfg['n_heads']}/{cfg['n_kv_heads']} heads, "
            f"head_dim {cfg['head_dim']}, ffn {cfg['ffn_dim']}, vocab {cfg['vocab']}, group-64 4-bit weights "
            f"(fp16 scale/min), {acts}, {cache}" + (", tied bf16 LM head" if cfg["tied"] else ""))


def kv_read_bytes(per_pos, positions):
    """Mean K/V bytes read per step when the steps run at the given positions."""
    return float(np.mean([(p + 1) * per_pos for p in positions]))


def model_flags(a):
    import bit_quantized_token_gb300 as bq
    return (bq.LLM_KV_Q8 if a.kv == "q8" else 0) | (bq.LLM_W4A8 if a.w4a8 else 0)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.seek(0)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().strip().splitlines():
            c = [x.strip() for x in line.split(",")]
            if len(c) < 9:
                continue
            try:
                sm.append(float(c[1]))
                mx = max(mx, float(c[2]))
            except ValueError:
                continue
            for n, v in zip(names, c[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.f.name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(cfg, w, prompt, seconds):
    """The oracle as it stands, on this host's cores, for a bounded sample."""
    import oracle

    m = oracle.OracleModel(cfg, w)
    n_pre = max(0, cfg.get("prefill_kv", 0))
    cache = m.new_cache(n_pre + len(prompt) + 1024)
    t0 = time.perf_counter()
    if n_pre:
        for l in range(cfg["n_layers"]):
            cache.fill(l, *synth.make_prefilled_kv(cfg, l, 0, n_pre))
        cache.set_len(n_pre)
        prompt = synth.make_first_tokens(cfg, 1)
    for t in prompt[:-1]:
        m.step(cache, int(t))
    tok, n = int(prompt[-1]), 0
    t1 = time.perf_counter()
    while n < 1024 and (n < 2 or time.perf_counter() - t1 < seconds):
        tok = oracle.argmax_f32(m.step(cache, tok))
        n += 1
    dt = time.perf_counter() - t1
    return {"value": n / dt, "unit": "tok/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": (f"{cfg['name']}: {len(prompt) + n_pre}-position context (untimed {time.perf_counter() - t0 - dt:.1f} s), "
                       f"then {n} greedy decode steps in {dt:.1f} s at positions {n_pre + len(prompt)}.."
                       f"{n_pre + len(prompt) + n - 1}")}


def max_over_ranks(ms, dist):
    """The slowest rank's timed-region length (ms); the replicas' own value without torch.distributed."""
    if not dist:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, ms):
    """Whole-job throughput: every rank's units over the slowest rank's time (weak scaling)."""
    return world * units_per_rank / (ms / 1000.0)


def run_reference(a, cfg, w, prompt, rank, world):
    if rank != 0:
        return
    cb = cpu_baseline(cfg, w, prompt, max(5.0, a.cpu_seconds))
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "tok/s", "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1000.0 / cb["value"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(cfg), "batch": 1, "prompt_len": len(prompt)},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_batched(a, cfg, w, rank, world, local, dist):
    """One decode step of every sequence of the batch per step (ragged pre-filled caches)."""
    import torch

    import bit_quantized_token_gb300 as bq

    B = cfg["batch"]
    lens = synth.make_kv_lengths(cfg, B)
    n_e2e = 8
    max_seq = int(lens.max()) + a.warmup + a.regions * a.steps + n_e2e + 8
    stream = torch.cuda.Stream()
    m = bq.Model(cfg, w, max_seq=max_seq, max_batch=B, stream=stream.cuda_stream, flags=model_flags(a))
    st = m.stats()
    for b in range(B):
        for l in range(cfg["n_layers"]):
            m.kv_write(b, l, 0, *synth.make_prefilled_kv(cfg, l, b, int(lens[b])))
    m.decode_step_batch(synth.make_first_tokens(cfg, B))
    for _ in range(a.warmup - 1):
        m.decode_step_batch(None)
    m.sync()
    per_pos = st["kv_bytes_per_pos"]  # the model's own cache format (bf16 or grouped int8)
    peak, peak_kind = peaks()
    clocks = ClockSampler(local)
    time.sleep(0.5)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    regions = []  # back to back: each region's caches are K positions longer than the last one's
    for r in range(a.regions):
        pos0 = lens + a.warmup + r * a.steps
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(a.steps):
            m.decode_step_batch(None)  # greedy tokens fed back on the device
        e1.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        ms_r = max_over_ranks(e0.elapsed_time(e1), dist)
        kv_r = float(np.mean([sum((int(pos0[b]) + i + 1) * per_pos for b in range(B)) for i in range(a.steps)]))
        regions.append((ms_r, kv_r))
    clk = clocks.stop()
    m.sync()
    order = sorted(range(len(regions)), key=lambda i: regions[i][0] / (st["weight_stream_bytes"] + regions[i][1]))
    ms, kv_step = regions[order[len(order) // 2]]  # the median region by time per byte
    tok_s = job_rate(world, B * a.steps, ms)
    bytes_step = st["weight_stream_bytes"] + kv_step
    gbs = bytes_step / (ms / a.steps / 1000.0) / 1e9
    # end to end: host tokens in, host greedy tokens out, every step
    am = np.zeros(B, np.int32)
    toks = synth.make_first_tokens(cfg, B)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        m.decode_step_batch(toks, None, am)
        toks = am.copy()
    e2e_s = time.perf_counter() - t0
    line = {
        "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": ms / a.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "i8" if a.w4a8 else "f32", "data": "synthetic",
        "config": {"workload": workload_desc(cfg, a.kv, a.w4a8), "batch": B, "kv_lengths": [int(lens.min()), int(lens.max())],
                   "kv_lengths_mean": float(lens.mean()), "l2": "inputs larger than L2: ~5.4 GB streamed per step",
                   "timed": "llm_decode_step_batch(NULL tokens): CUDA-graph replays, greedy tokens fed back on the device"},
        "hbm": {"bytes_per_step": bytes_step, "weight_bytes": st["weight_stream_bytes"], "kv_bytes_per_step": kv_step,
                "achieved_gbs": gbs, "frac_of_peak": gbs / peak, "peak_gbs": peak, "peak_kind": peak_kind},
        "roofline": {"kernel": "batched step (bgemv_kernel + battn_mma_kernel graph; attention reads ~90% of the bytes)",
                     "bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": None, "peak_kind": peak_kind},
        "e2e": {"value": world * B * n_e2e / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": 4 * B,
                "d2h_bytes_per_step": 4 * B, "steps": n_e2e,
                "call": "llm_decode_step_batch(host tokens -> host greedy tokens)"},
        "regions": {"n": len(regions), "ms_per_step": [r[0] / a.steps for r in regions],
                    "kv_bytes_per_step": [r[1] for r in regions],
                    "note": "consecutive regions (caches grow by K positions each); value, hbm and roofline "
                            "come from the median region by time per byte"},
        "gpu_launches": (5 * cfg["n_layers"] + 2) * a.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, w, synth.make_prompt(cfg, n=1), a.cpu_seconds)
    m.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def run_phases(a, cfg, w, prompt):
    """Where one batch-1 step's time goes, phase by phase (clock stamps of the grid-barrier step)."""
    import torch

    import bit_quantized_token_gb300 as bq

    lib = os.path.join(os.path.dirname(bq.LIB_PATH), "libllmq_phase_stamps.so")
    bq.build(out=lib, defines=["LLMQ_PHASE_STAMPS=1", "LLMQ_UNIT_STAMPS=1"])
    bq.LIB_PATH = lib
    torch.cuda.set_device(0)
    with bq.Model(cfg, w, max_seq=len(prompt) + 32, flags=model_flags(a)) as m:
        am = np.zeros(1, np.int32)
        m.prefill(0, prompt, None, am)
        g = m.decode_greedy(0, int(am[0]), 8)
        t = m.phase_times(0, int(g[-1]), 1).astype(np.float64)[0]  # [phase][cta][16]
    gt0, c0, gt1, c1 = t[0, :, 12], t[0, :, 13], t[0, :, 14], t[0, :, 15]
    rate = (gt1 - gt0) / (c1 - c0)  # ns per cycle, per SM
    T = lambda k: gt0[None, :] + (t[:, :, k] - c0[None, :]) * rate[None, :]
    bar, blt, und, arr = T(1), T(2), T(3), T(4)
    ghz = 1.0 / rate.mean()
    rows, prev = [], None
    for ph in range(t.shape[0]):
        if not (t[ph, :, 4] > 0).all():
            continue  # a phase the fused variant skips
        units = (t[ph, :, 3] > 0).all()
        r = {"phase": ph, "units": bool(units)}
        if prev is not None:
            last = arr[prev].max()
            r["barrier_after_last_arrival_us"] = float(np.median(bar[ph]) - last) / 1000
            r["span_us"] = float(arr[ph].max() - last) / 1000
        if units:
            r["build_us"] = float(np.median(blt[ph] - bar[ph])) / 1000
            r["units_us"] = float(np.median(und[ph] - blt[ph])) / 1000
            r["busiest_warp_wait_us"] = float(np.median(t[ph, :, 5])) / ghz / 1000
            r["busiest_warp_dot_us"] = float(np.median(t[ph, :, 6])) / ghz / 1000
        r["arrive_us"] = float(np.median(arr[ph] - (und[ph] if units else bar[ph]))) / 1000
        r["arrival_spread_us"] = float(arr[ph].max() - arr[ph].min()) / 1000
        rows.append(r)
        prev = ph
    print(f"{cfg['name']}: {len(rows)} phases, step {(gt1.max() - gt0.min()) / 1000:.1f} us (stamps build)")
    keys = ["barrier_after_last_arrival_us", "build_us", "units_us", "busiest_warp_wait_us", "busiest_warp_dot_us",
            "arrive_us", "arrival_spread_us", "span_us"]
    L = cfg["n_layers"]
    per = (len(rows) - 2) // L  # phases per layer; the last two are the LM head and the logit reduction
    names = (["q|k|v", "o (+attention)", "gate|up", "down"] if per == 4
             else ["q|k|v", "attention", "o", "gate|up", "down"])[:per]
    print("phase | " + " | ".join(k[:-3] for k in keys) + "  (us, median CTA, mean over layers 1..L-1)")
    fmt = lambda sel: " | ".join(
        f"{np.mean([r[k] for r in sel if k in r]):.2f}" if any(k in r for r in sel) else "-" for k in keys)
    for j in range(per):
        sel = [rows[l * per + j] for l in range(1, L)]
        print(f"{names[j]} | " + fmt(sel))
    print("LM head | " + fmt([rows[L * per]]))
    print("logits | " + fmt([rows[L * per + 1]]))


def main():
    a = args_()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")  # barrier only: the replicas exchange no data
    cfg = synth.workload(a.workload, **({"n_layers": a.layers} if a.layers else {}))
    w = synth.make_weights(cfg)
    prompt = synth.make_prompt(cfg)
    if a.phases:
        run_phases(a, cfg, w, prompt)
        return
    if a.impl == "reference":
        run_reference(a, cfg, w, prompt, rank, world)
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return

    import torch

    import bit_quantized_token_gb300 as bq

    torch.cuda.set_device(local)
    bq.build()
    assert a.warmup >= 3, "at least 3 warm-up steps"
    if cfg.get("batch", 1) > 1:
        run_batched(a, cfg, w, rank, world, local, dist)
        return
    n_e2e, n_kt, n_pf = 128, 3, 512
    n_pre = max(0, cfg.get("prefill_kv", 0))
    max_seq = max(n_pre + len(prompt) + 2 * (a.warmup + a.steps) + n_e2e + 8, n_pf + 8)
    stream = torch.cuda.Stream()  # the library launches on it; events are recorded on it
    m = bq.Model(cfg, w, max_seq=max_seq, stream=stream.cuda_stream, flags=model_flags(a))
    st = m.stats()
    kv_pre = [synth.make_prefilled_kv(cfg, l, 0, n_pre) for l in range(cfg["n_layers"])] if n_pre else None

    def fresh_sequence():
        # the same state before every timed region: the prompt (or the
        # pre-filled cache and its seeded first token), then W warm-up steps
        m.kv_reset(0)
        am = np.zeros(1, np.int32)
        if n_pre:
            for l in range(cfg["n_layers"]):
                m.kv_write(0, l, 0, *kv_pre[l])
            am[0] = synth.make_first_tokens(cfg, 1)[0]
        else:
            m.prefill(0, prompt, None, am)
        warm = m.decode_greedy(0, int(am[0]), a.warmup)
        return int(warm[-1])

    toks_dev = torch.empty(a.steps, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    time.sleep(0.5)
    region_ms = []
    for r in range(a.regions):
        tok = fresh_sequence()
        pos0 = m.kv_len(0)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        m.decode_greedy(0, tok, a.steps, toks_dev)
        e1.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        region_ms.append(max_over_ranks(e0.elapsed_time(e1), dist))
    clk = clocks.stop()
    m.sync()
    ms = statistics.median(region_ms)
    positions = list(range(pos0, pos0 + a.steps))
    tok = int(toks_dev[-1].item())
    tok_s = job_rate(world, a.steps, ms)
    bytes_tok = st["weight_stream_bytes"] + kv_read_bytes(st["kv_bytes_per_pos"], positions)
    peak, peak_kind = peaks()

    # dominant kernel: every 4-bit / bf16 GEMV of a step, back to back (582 MB > L2)
    g_ms, g_bytes = m.time_kernel(0, "all_gemv", -1, n_kt)
    g_gbs = g_bytes / (g_ms / 1000.0) / 1e9
    # kernel shares of one eagerly launched step (serialised, like an ncu launch list)
    share = None
    if a.kv == "bf16":  # the eager per-kernel profile runs the bf16-cache kernels
        prof = m.profile_step(0, tok)
        tot = sum(r["ms"] for r in prof)
        share = {}
        for r in prof:
            share[r["kind"]] = share.get(r["kind"], 0.0) + r["ms"] / tot
    # end to end through the public call: host token in, host argmax out,
    # every step; the inter-token latency of that loop, on the host clock and
    # between CUDA events recorded on the model's stream after each call
    am_h = np.zeros(1, np.int32)
    m.decode_step(0, tok, None, am_h)
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e + 1)]
    wall = []
    evs[0].record(stream)
    t0 = t_prev = time.perf_counter()
    for i in range(n_e2e):
        m.decode_step(0, int(am_h[0]), None, am_h)
        evs[i + 1].record(stream)
        t = time.perf_counter()
        wall.append(t - t_prev)
        t_prev = t
    e2e_s = time.perf_counter() - t0
    torch.cuda.synchronize()
    dev = [evs[i].elapsed_time(evs[i + 1]) / 1000.0 for i in range(n_e2e)]

    def pct(xs):
        us = np.asarray(xs) * 1e6
        return {"p50": float(np.percentile(us, 50)), "p95": float(np.percentile(us, 95)),
                "p99": float(np.percentile(us, 99)), "mean": float(us.mean())}

    e2e = {"value": world * n_e2e / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": 4, "d2h_bytes_per_step": 4,
           "steps": n_e2e, "call": "llm_decode_step(host token -> host argmax)"}
    itl = {"steps": n_e2e, "wall_us": pct(wall), "device_us": pct(dev),
           "positions": [pos0 + a.steps, pos0 + a.steps + n_e2e - 1],
           "call": "llm_decode_step(host token -> host argmax), one call per token"}

    # sampled choice (temperature 0.8, top-k 40, top-p 0.95, Philox draw): the
    # same device-fed loop with the sampling kernel in each step's graph
    # (from the same reset cache as the greedy regions: the same positions)
    m.set_sampling(0.8, 40, 0.95, 42)
    toks_s = torch.empty(a.steps, dtype=torch.int32, device="cuda")
    tok_s0 = fresh_sequence()
    warm_s = np.array([tok_s0], np.int32)
    torch.cuda.synchronize()
    e0.record(stream)
    m.decode_greedy(0, int(warm_s[-1]), a.steps, toks_s)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_s = e0.elapsed_time(e1)
    m.set_sampling(0.0)
    sampled = {"temperature": 0.8, "top_k": 40, "top_p": 0.95, "ms_per_step": ms_s / a.steps,
               "overhead_us_per_step": (ms_s - ms) / a.steps * 1000.0,
               "call": "llm_decode_greedy after llm_set_sampling (CUDA events)"}

    # prompt processing: a 512-token prompt, token by token (n graph steps) and
    # batched (chunks of 32 through the tensor-core pipeline); wall clock of the call
    prefill = None
    if n_pre == 0:
        pf_prompt = synth.make_prompt(cfg, n=n_pf)
        rates = {}
        for name, call in (("batched", m.prefill_batched), ("token_by_token", m.prefill)):
            m.kv_reset(0)
            call(0, pf_prompt[:64])  # warm
            m.kv_reset(0)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            call(0, pf_prompt, None, am_h)
            rates[name] = n_pf / (time.perf_counter() - t0)
        prefill = {"prompt_tokens": n_pf, "batched_tok_s": rates["batched"],
                   "token_by_token_tok_s": rates["token_by_token"],
                   "speedup": rates["batched"] / rates["token_by_token"],
                   "call": "llm_prefill_batched vs llm_prefill (wall clock of the call, host tokens in)"}

    if st["kernels_per_step"] == 1:
        # one persistent kernel per step: its launch duration is the step time
        roofline = {"kernel": "step_kernel (persistent decode step, one launch per token)", "bound": "hbm",
                    "achieved": bytes_tok / (ms / a.steps / 1000.0) / 1e9, "peak": peak, "unit": "GB/s",
                    "frac": bytes_tok / (ms / a.steps / 1000.0) / 1e9 / peak,
                    "traffic": ncu_traffic(f"step_kernel {cfg['name']}"),
                    "peak_kind": peak_kind, "bytes_per_launch": bytes_tok, "ms_per_launch": ms / a.steps}
    else:
        roofline = {"kernel": "gemv_kernel (4-bit dequant-GEMV stream of one step, back to back)", "bound": "hbm",
                    "achieved": g_gbs, "peak": peak, "unit": "GB/s", "frac": g_gbs / peak, "traffic": None,
                    "peak_kind": peak_kind, "bytes_per_launch": g_bytes, "ms_per_launch": g_ms}
    line = {
        "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": ms / a.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "i8" if a.w4a8 else "f32", "data": "synthetic",
        "config": {"workload": workload_desc(cfg, a.kv, a.w4a8), "batch": 1, "prompt_len": len(prompt),
                   "prefilled_positions": n_pre,
                   "positions": [positions[0], positions[-1]],
                   "l2": "inputs larger than L2: 582 MB of weights streamed per step vs 129 MB L2"
                   if a.workload in (1, 3) else "weights streamed per step exceed L2"
                   if st["weight_stream_bytes"] > 129e6 else "fits in L2",
                   "timed": "llm_decode_greedy: CUDA-graph replays, argmax fed back on the device"},
        "hbm": {"bytes_per_token": bytes_tok, "weight_bytes": st["weight_stream_bytes"],
                "kv_bytes_per_token": bytes_tok - st["weight_stream_bytes"],
                "achieved_gbs": bytes_tok * tok_s / world / 1e9,
                "frac_of_peak": bytes_tok * tok_s / world / 1e9 / peak, "peak_gbs": peak, "peak_kind": peak_kind},
        "roofline": roofline,
        "gemv_stream": {"kernel": "gemv_kernel: the step's 4-bit/bf16 GEMVs as separate launches, back to back",
                        "achieved": g_gbs, "unit": "GB/s", "frac": g_gbs / peak, "bytes_per_launch": g_bytes,
                        "ms_per_launch": g_ms},
        "kernel_share_eager": share,
        "regions": {"n": len(region_ms), "ms_per_step": [r / a.steps for r in region_ms],
                    "note": "each region decodes the same positions from a reset cache; value = the median"},
        "itl": itl,
        "e2e": e2e,
        "gpu_launches": st["kernels_per_step"] * a.steps,
        "clocks": clk,
    }
    line["sampling"] = sampled
    if prefill:
        line["prefill"] = prefill
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, w, prompt, a.cpu_seconds)
    m.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
