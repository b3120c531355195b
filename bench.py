#!/usr/bin/env python3
"""Decode-layer benchmark: 128K-context Llama-3.1-70B-shaped attention layer over a Q4_0 cache.

One step = one decode layer-call: append the new token's K and V (Q4_0 store, 1 launch) and run
the split-K decode attention over all 131072 cached tokens (phase 1 + LSE reduce). The metric
is the effective HBM bandwidth on packed KV (payload + fp16 scales) read per step, and the
microseconds per layer-call.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints exactly one JSON line on rank 0. Under torchrun every rank runs its own replica of the
workload (independent layers, no collective on the data path): weak scaling, the time is the
max over ranks.

Timing: W untimed warm-up steps (plus an untimed soak of --soak-s seconds so clock samples
exist), then exactly K steps bracketed by a barrier and a device synchronise, timed with CUDA
events on the launching stream. The K steps are captured once in a CUDA graph of the library's
own launches and replayed. Steps rotate over several cache replicas whose total size exceeds
L2, so no step reads a cache that is still L2-resident. Phase 1 (the streaming kernel) is
also timed per launch with CUDA events recorded around it inside the timed region.
"""
from __future__ import annotations

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")        # the CPU oracle baseline runs on one thread

import argparse
import hashlib
import json
import math
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "int4-KV decode attention µs/layer and effective HBM GB/s (% peak) at 128K"
WORKLOAD = "c5_q4_0_llama70b_128k"
VARIANT = "c5_asym4_g32_llama70b_128k"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    p.add_argument("--soak-s", type=float, default=1.0, help="untimed soak before timing (0 = none)")
    p.add_argument("--quick", action="store_true", help="device timing only (no e2e, variant, CPU baseline)")
    p.add_argument("--no-graph", action="store_true", help="plain stream launches instead of a CUDA graph")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU oracle sample budget")
    return p.parse_args()


# ------------------------------------------------------------------ helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_traffic(kernel_file: str, launches_per_unit=1.0):
    """dram bytes per launch from the committed ncu summary of `kernel_file`, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "attend_phase1_c5_q4_0_128k.md")
    src = os.path.join(ROOT, "sub_byte_quantized_gb300", "csrc", kernel_file)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    text = open(path).read()
    m_hash = re.search(r"source sha256:\s*([0-9a-f]{64})", text)
    m_bytes = re.search(r"dram bytes per launch:\s*([0-9]+)", text)
    if not (m_hash and m_bytes):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != m_hash.group(1):
        return None
    return int(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle baseline
def oracle_sample(w, inp, n_heads: int):
    """Prepare an oracle cache of the first `n_heads` kv heads (untimed) and return a step function:
    append the last token (oracle store) + oracle decode attention over the full cache."""
    from oracle import attention as OA
    S = inp["k"].shape[2]
    sub_k, sub_v = inp["k"][:, :n_heads], inp["v"][:, :n_heads]
    oc = OA.OracleCache(w.layout, w.batch, n_heads, w.head_dim, S)
    oc.store(sub_k[:, :, :S - 1], sub_v[:, :, :S - 1], 0)
    q = inp["q"][:, :n_heads * w.gqa]

    def step():
        oc.store(sub_k[:, :, S - 1:], sub_v[:, :, S - 1:], S - 1)
        return oc.attend(q, w.alpha, S)
    return step


def cpu_baseline(w, inp, budget_s: float):
    step = oracle_sample(w, inp, 1)
    S = inp["k"].shape[2]
    bytes_per = (S * 2 * (64 + 8)) * w.batch          # one kv head's packed K+V read by a step
    times = []
    t_all = time.perf_counter()
    while not times or (time.perf_counter() - t_all < budget_s and len(times) < 20):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    tm = statistics.median(times)
    return {"value": bytes_per / tm / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"oracle store of the appended token + float64 decode attention of 1 of 8 kv heads "
                      f"(8 query heads) over {S} tokens; median of {len(times)} runs, {tm * 1e3:.0f} ms each, "
                      f"{bytes_per} packed bytes per run",
            "us_per_layer_equiv": tm * 8 * 1e6}


# ------------------------------------------------------------------ reference arm (the oracle)
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from synth import WORKLOADS, make_inputs
    w = WORKLOADS[WORKLOAD]
    inp = make_inputs(w)
    # bound the run: each step is one kv head over a token sample sized so that W + K steps
    # take about two minutes in total
    S = inp["k"].shape[2]
    probe = oracle_sample(w, inp, 1)
    t0 = time.perf_counter()
    probe()
    t_full = time.perf_counter() - t0
    per_step = 120.0 / max(1, args.steps + args.warmup)
    frac = min(1.0, per_step / max(t_full, 1e-6))
    S_s = max(1024, int(S * frac) // 512 * 512)
    if S_s < S:
        from synth import Workload  # noqa: F401
        ws = w.scaled(kv_len=S_s, fill=S_s - 1)
        sub = {k: (v[:, :, :S_s] if k in ("k", "v") else v) for k, v in inp.items()}
        step = oracle_sample(ws, sub, 1)
    else:
        step = probe
    bytes_per = S_s * 2 * (64 + 8) * w.batch
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = bytes_per * args.steps / el / 1e9
    sample = (f"CPU oracle (numpy, 1 thread): per step, oracle store of 1 appended token + float64 decode "
              f"attention of 1 kv head (8 query heads) over {S_s} of {S} tokens ({bytes_per} packed bytes)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "Llama-3.1-70B layer, 128K context, Q4_0 KV (bf16 Student-t(4) K/V, "
                                   "4 outlier channels x10), B1 Hq64 Hkv8 D128",
                       "kv_len": S, "sampled_kv_len": S_s, "layout": "q4_0"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import torch.distributed as dist

    import sub_byte_quantized_gb300 as kvq
    from sub_byte_quantized_gb300 import _lib
    from synth import WORKLOADS, make_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    w = WORKLOADS[WORKLOAD]
    inp = make_inputs(w)
    B, H, S, D = inp["k"].shape

    def to_dev(name):
        return torch.from_numpy(np.ascontiguousarray(inp[name + "_bits"]).view(np.int16)).view(torch.bfloat16).to(dev)

    kd, vd, q = to_dev("k"), to_dev("v"), to_dev("q")
    k_new = kd[:, :, S - 1:].contiguous()
    v_new = vd[:, :, S - 1:].contiguous()

    def make_caches(layout, n):
        caches = []
        for _ in range(n):
            c = kvq.KVCache(layout, B, H, D, S, device=dev)
            kvq.store(c, kd[:, :, :S - 1].contiguous(), vd[:, :, :S - 1].contiguous(), 0)
            kvq.store(c, k_new, v_new, S - 1)
            caches.append(c)
        return caches

    n_rep = max(2, math.ceil(3 * L2_BYTES / (2 * B * H * S * 72)) + 1)
    caches = make_caches("q4_0", n_rep)
    read_bytes = caches[0].read_bytes(S)
    chunk = kvq.attend_chunk(caches[0], S, 0)          # automatic split: one chunk per resident warp
    ws = torch.empty(kvq.attend_workspace_bytes(caches[0], w.n_q_heads, 1, S, chunk), dtype=torch.uint8, device=dev)
    out = torch.empty((B, w.n_q_heads, 1, D), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    L = _lib.lib()

    def step(i, ev=None):
        c = caches[i % n_rep]
        kvq.store(c, k_new, v_new, S - 1, stream=stream)
        if ev is not None:
            L.kvq_profile_phase1_events(ev[0].cuda_event, ev[1].cuda_event)
        kvq.decode_attend(c, q, S, attn_scale=w.alpha, chunk=chunk, out=out, workspace=ws, stream=stream)
        if ev is not None:
            L.kvq_profile_phase1_events(None, None)

    K, W = args.steps, args.warmup
    use_graph = not args.no_graph
    ph_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(stream):
        for a, b in ph_ev:      # create the events (torch only times events it has recorded once)
            a.record(stream)
            b.record(stream)
        for i in range(max(W, 3)):
            step(i)
    torch.cuda.synchronize(dev)
    if use_graph:
        graph = torch.cuda.CUDAGraph()             # the timed steps, exactly as a caller runs them
        with torch.cuda.graph(graph, stream=stream):
            for i in range(K):
                step(i)
        ev_graph = torch.cuda.CUDAGraph()          # the same K steps with phase-1 events recorded
        with torch.cuda.graph(ev_graph, stream=stream):
            for i in range(K):
                step(i, ph_ev[i])
        soak_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(soak_graph, stream=stream):
            for i in range(64):
                step(i)
    torch.cuda.synchronize(dev)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # untimed soak so the clock record covers the GPU under this load
        t_end = time.perf_counter() + args.soak_s
        with torch.cuda.stream(stream):
            while time.perf_counter() < t_end:
                if use_graph:
                    soak_graph.replay()
                else:
                    for i in range(64):
                        step(i)
                torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            if use_graph:
                graph.replay()
            else:
                for i in range(K):
                    step(i, ph_ev[i])
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        elapsed_ms = ev0.elapsed_time(ev1)
        # phase-1 durations: the same K steps again, with CUDA events around every phase-1 launch
        # (an event between two kernels ends their launch overlap, so this pass is not the headline)
        if use_graph:
            with torch.cuda.stream(stream):
                ev0.record(stream)
                ev_graph.replay()
                ev1.record(stream)
            torch.cuda.synchronize(dev)
        ev_pass_ms = ev0.elapsed_time(ev1)
        time.sleep(0.25)
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    ph_ms = [a.elapsed_time(b) for a, b in ph_ev]
    ph_mean = statistics.fmean(ph_ms)
    ms_step = elapsed_ms / K
    value = world * read_bytes * K / (elapsed_ms / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    achieved = read_bytes / (ph_mean / 1e3) / 1e9
    traffic = kernel_traffic("attend_mma.cu")
    kinds = 3                                   # store + phase 1 + reduce per step

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_step, "us_per_layer": ms_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "Llama-3.1-70B layer, 128K context, Q4_0 KV (bf16 Student-t(4) K/V, 4 outlier "
                               "channels x10, N(0,1) Q), B1 Hq64 Hkv8 D128",
                   "chunk": chunk, "chunk_rule": "automatic: 4 warps per chunk, one 64-token-multiple slice per resident warp, one wave",
                   "kv_len": S, "layout": "q4_0", "step": "append 1 token (K,V) + split-K decode attention",
                   "read_bytes_per_step": read_bytes,
                   "l2": f"inputs larger than L2: {n_rep} cache replicas rotated "
                         f"({n_rep * read_bytes / 2**20:.0f} MiB > {L2_BYTES / 2**20:.0f} MiB L2)",
                   "timing": ("CUDA graph of the K library steps; phase 1 timed by events in a second pass "
                              "of the same K steps") if use_graph else "stream launches with phase-1 events",
                   "soak_s": args.soak_s, "parallelism": f"replicas x{world}"},
        "pct_of_peak": value / world / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": traffic, "kernel": "attend phase 1 (split-K chunk partials)",
                     "phase1_us_mean": ph_mean * 1e3, "phase1_us_p10": float(np.percentile(ph_ms, 10)) * 1e3,
                     "phase1_us_p90": float(np.percentile(ph_ms, 90)) * 1e3,
                     "phase1_pass_us_per_step": ev_pass_ms / K * 1e3},
        "clocks": clk.summary(),
        "gpu_launches": kinds * K,
    }

    if not args.quick and rank == 0:
        # end to end through the public API from pinned host buffers, one sync per step
        hk = k_new.cpu().pin_memory()
        hv = v_new.cpu().pin_memory()
        hq = q.cpu().pin_memory()
        hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        dk, dv, dq = torch.empty_like(k_new), torch.empty_like(v_new), torch.empty_like(q)
        n_e2e = min(K, 500)
        for i in range(n_e2e + 3):
            if i == 3:
                torch.cuda.synchronize(dev)
                t0 = time.perf_counter()
            with torch.cuda.stream(stream):
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
                dq.copy_(hq, non_blocking=True)
                c = caches[i % n_rep]
                kvq.store(c, dk, dv, S - 1, stream=stream)
                kvq.decode_attend(c, dq, S, attn_scale=w.alpha, chunk=chunk, out=out, workspace=ws, stream=stream)
                hout.copy_(out, non_blocking=True)
            stream.synchronize()
        t_e2e = (time.perf_counter() - t0) / n_e2e
        line["e2e"] = {"value": read_bytes / t_e2e / 1e9, "unit": "GB/s",
                       "h2d_bytes_per_step": hk.numel() * 2 + hv.numel() * 2 + hq.numel() * 2,
                       "d2h_bytes_per_step": hout.numel() * 4, "us_per_layer": t_e2e * 1e6, "steps": n_e2e}
        line["variants"] = {}

        def time_plain(cs, wsb, ch, n):
            with torch.cuda.stream(stream):
                for i in range(5):
                    kvq.store(cs[i % n_rep], k_new, v_new, S - 1, stream=stream)
                    kvq.decode_attend(cs[i % n_rep], q, S, attn_scale=w.alpha, chunk=ch, out=out, workspace=wsb,
                                      stream=stream)
                torch.cuda.synchronize(dev)
                ev0.record(stream)
                for i in range(n):
                    kvq.store(cs[i % n_rep], k_new, v_new, S - 1, stream=stream)
                    kvq.decode_attend(cs[i % n_rep], q, S, attn_scale=w.alpha, chunk=ch, out=out, workspace=wsb,
                                      stream=stream)
                ev1.record(stream)
            torch.cuda.synchronize(dev)
            return ev0.elapsed_time(ev1) / n
        ws512 = torch.empty(kvq.attend_workspace_bytes(caches[0], w.n_q_heads, 1, S, 512), dtype=torch.uint8,
                            device=dev)
        c_ms = time_plain(caches, ws512, 512, min(K, 1000))
        line["variants"]["q4_0_chunk512"] = {"us_per_layer": c_ms * 1e3, "gbs": read_bytes / (c_ms / 1e3) / 1e9,
                                             "timing": "stream launches", "chunk": 512}
        # asymmetric g=32 variant of the same layer (same device timing protocol, plain launches)
        del caches
        torch.cuda.empty_cache()
        acaches = make_caches("asym4_g32", n_rep)
        a_bytes = acaches[0].read_bytes(S)
        aws = torch.empty(kvq.attend_workspace_bytes(acaches[0], w.n_q_heads, 1, S, chunk), dtype=torch.uint8,
                          device=dev)
        a_ms = time_plain(acaches, aws, chunk, min(K, 1000))
        line["variants"]["asym4_g32"] = {"us_per_layer": a_ms * 1e3, "read_bytes_per_step": a_bytes,
                                         "gbs": a_bytes / (a_ms / 1e3) / 1e9, "timing": "stream launches",
                                         "chunk": chunk}
        if world == 1:
            line["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
