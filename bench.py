#!/usr/bin/env python3
"""Decode-layer benchmark of the packed sub-byte KV cache.

Default workload: a 128K-context Llama-3.1-70B-shaped attention layer over a Q4_0 cache. One step
= one decode layer-call: append the new token's K and V (one store launch) and run the split-K
decode attention over all 131072 cached tokens (phase 1 + LSE reduce). The metric is the
effective HBM bandwidth on packed KV (payload + fp16 scales) read per step; microseconds per
layer-call come with it. `--workload` selects another of the seeded workloads (the Llama-3-8B
layer, the Hadamard decode or causal prefill chunk, the Q6_0 Gemma-like layer, the asymmetric
128K layer); the default line is the 128K Q4_0 one.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

Prints exactly one JSON line on rank 0. Under torchrun every rank runs its own replica of the
workload (independent layer-calls, no collective on the data path): weak scaling, value = all
ranks' bytes over the max-over-ranks time.

Timing: W untimed warm-up steps (plus an untimed soak of --soak-s seconds so clock samples
exist), then exactly K steps bracketed by a barrier and a device synchronise, timed with CUDA
events on the launching stream. The K steps are captured once in a CUDA graph of the library's
own launches and replayed. Steps rotate over cache replicas whose total size exceeds L2 (for the
small workloads whose replicas would be too many, the config says the cache is L2-resident).
Phase 1 (the streaming kernel) is timed per launch with CUDA events in a second pass of the same
K steps (an event between two kernels ends their programmatic launch overlap, so that pass is
not the headline).
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

DEFAULT_WORKLOAD = "c5_q4_0_llama70b_128k"
METRIC = "int4-KV decode attention µs/layer and effective HBM GB/s (% peak) at 128K"
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
# vendor nominal figures of one GB300 (NVIDIA's published HBM3e bandwidth and dense bf16 tensor rate),
# reported beside the measured denominators
NOMINAL_HBM_GBS, NOMINAL_BF16_TFLOPS = 7900.0, 2250.0
# the other seeded workloads timed (compactly) inside the default run, so that one bench line carries
# every configuration
SUMMARY_WORKLOADS = ("c1_q4_0_tiny", "c2_q4_0_llama3_8b", "c3_had_int4_decode", "c3_had_int4_prefill",
                     "c4_q6_0_gemma", "c5_asym4_g32_llama70b_128k", "c5_q8_0_llama70b_128k",
                     "c5_q4_0_k_q8_0_v_llama70b_128k", "c3_had_int2_decode_w256", "paged_q4_0_llama3_8b_ragged")
L2_BYTES = 129 * 2 ** 20
DESCRIPTIONS = {
    "c1_q4_0_tiny": "Q4_0 tiny: B1 Hq8 Hkv2 D128 S512 decode, f32 N(0,1) K/V/Q, 2 K outlier channels x8",
    "c2_q4_0_llama3_8b": "Llama-3-8B layer: B4 Hq32 Hkv8 D128 S8192, Q4_0, bf16 Student-t(4) K/V, 4 outlier ch x10; "
                         "append 1 token then decode-attend",
    "c3_had_int4_decode": "Hadamard per-token int4, Qwen3-1.7B shape: B8 Hq16 Hkv8 D128 S4096, n_recent 64 f32 window",
    "c3_had_int4_prefill": "Hadamard per-token int4, Qwen3-1.7B shape: causal prefill chunk of 256 rows at 3840 "
                           "(B8 Hq16 Hkv8 D128, kv_len 4096, n_recent 64)",
    "c4_q6_0_gemma": "Q6_0 Gemma-like: B2 Hq16 Hkv8 D256 S32768, attention scale 1.0, unit-RMS Q/K rows, bf16 "
                     "Student-t(3) K/V",
    "c5_q4_0_llama70b_128k": "Llama-3.1-70B layer, 128K context, Q4_0 KV (bf16 Student-t(4) K/V, 4 outlier channels "
                             "x10, N(0,1) Q), B1 Hq64 Hkv8 D128",
    "c5_asym4_g32_llama70b_128k": "Llama-3.1-70B layer, 128K context, per-group asymmetric int4 g=32 KV, "
                                  "B1 Hq64 Hkv8 D128",
    "c5_q8_0_llama70b_128k": "Llama-3.1-70B layer, 128K context, Q8_0 KV (8-bit codes, fp16 scale per 32 values), "
                             "B1 Hq64 Hkv8 D128",
    "c5_q4_0_k_q8_0_v_llama70b_128k": "Llama-3.1-70B layer, 128K context, mixed K/V precision: Q4_0 keys, Q8_0 values, "
                                      "B1 Hq64 Hkv8 D128",
    "c3_had_int2_decode_w256": "Hadamard per-token int2 body + 256-token exact-f32 window, Qwen3-1.7B shape: B8 Hq16 "
                               "Hkv8 D128 S4096",
    "paged_q4_0_llama3_8b_ragged": "Paged Q4_0 pool, Llama-3-8B layer shapes (Hq32 Hkv8 D128): 16 sequences with seeded "
                                   "lengths 1024-16384 (116139 tokens), 64-token pages shuffled in the pool; append 1 "
                                   "token per sequence then attend over each sequence's own length",
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(DESCRIPTIONS))
    p.add_argument("--soak-s", type=float, default=1.0, help="untimed soak before timing (0 = none)")
    p.add_argument("--quick", action="store_true", help="device timing only (no e2e, variants, CPU baseline)")
    p.add_argument("--no-graph", action="store_true", help="plain stream launches instead of a CUDA graph")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU oracle sample budget")
    p.add_argument("--summary-steps", type=int, default=200,
                   help="steps per workload of the default run's per-configuration summary (0 = skip it)")
    return p.parse_args()


# ------------------------------------------------------------------ helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# committed ncu summaries of the phase-1 kernel per workload: (summary file, kernel source file)
PROFILES = {
    "c5_q4_0_llama70b_128k": ("attend_phase1_c5_q4_0_128k.md", "attend_mma.cu"),
    "c4_q6_0_gemma": ("attend_phase1_q6_0_c4_gemma.md", "attend_mma_q6.cu"),
    "c3_had_int4_prefill": ("attend_prefill_tc_c3_had_int4.md", "attend_prefill_tc.cu"),
    "c5_q8_0_llama70b_128k": ("attend_phase1_q8_0_128k.md", "attend_mma.cu"),
    "c5_q4_0_k_q8_0_v_llama70b_128k": ("attend_phase1_q4_0_k_q8_0_v_128k.md", "attend_mma.cu"),
    "c3_had_int2_decode_w256": ("attend_phase1_had_int2_w256.md", "attend_mma.cu"),
}


def kernel_traffic(profile: str, kernel_file: str):
    """DRAM bytes per launch from the committed ncu summary `profile`, or None when the kernel
    source changed since the counters were taken (the summary records the source's sha256)."""
    path = os.path.join(ROOT, "profiles", profile)
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


def chunk_rule(w, spec) -> str:
    """How the automatic split-K chunk of this workload is chosen (it follows the phase-1 kernel)."""
    rows = (w.n_q_heads // w.n_kv_heads) * spec.n_q
    if w.layout == "q6_0" and (w.head_dim == 256 or rows <= 8):
        return ("automatic: one 64-token-multiple chunk per resident CTA of the Q6_0 kernel (two per SM, one per "
                "group of four query rows), one wave")
    if w.layout == "asym4_g32" and w.head_dim == 128 and rows <= 8:
        return "automatic: one 64-token-multiple chunk per resident CTA of the warp-specialised kernel (two per SM), one wave"
    if w.layout in ("had_int4", "had_int2") and w.head_dim == 128 and rows > 64:
        return ("automatic: the tcgen05 kernel's body split (1..8 chunks per 128-row block, the fewest waves x "
                "stages); the f32 window is scored in 64-token chunks of its own")
    if w.head_dim == 128 and rows > 8:
        return "automatic: body split for about four waves of 64-query-row CTAs"
    return "automatic: 4 warps per chunk, one 32-token-multiple slice per resident warp, one wave"


def aggregate(world: int, units_per_rank: float, steps: int, elapsed_ms: float) -> float:
    """Whole-job throughput: all ranks' units over the (max-over-ranks) elapsed time, per second."""
    return world * units_per_rank * steps / (elapsed_ms / 1e3)


def max_over_ranks(value: float, dist, device) -> float:
    """The maximum of `value` over all ranks of the default process group (identity for one rank)."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


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


# ------------------------------------------------------------------ workload geometry
class Spec:
    """Shapes of one step of a workload: the cache holds S tokens; a step appends tokens
    [fill, S) and attends n_q query rows per head (causal from q_pos0 for the prefill chunk)."""

    def __init__(self, w, inp):
        self.w = w
        self.B, self.H, self.S, self.D = inp["k"].shape
        self.fill = w.n_fill
        self.n_q = inp["q"].shape[2]
        self.causal = w.causal
        self.q_pos0 = self.S - self.n_q if w.causal else 0
        kl, _, vl = w.layout.partition("+")
        planes = (kl, vl or kl)                           # each plane's layout (mixed K/V precision)
        self.n_win = min(w.n_recent, self.S) if kl.startswith("had") else 0
        nb = self.D // 32
        row = {"q4_0": 16 * nb + 2 * nb, "q6_0": 24 * nb + 2 * nb, "asym4_g32": 16 * nb + 4 * nb,
               "q8_0": 32 * nb + 2 * nb, "had_int4": self.D // 2 + 4, "had_int2": self.D // 4 + 4}
        # algorithmic bytes one attention call reads: every packed K/V row (+ scales) once; window
        # tokens as their exact f32 rows
        self.read_bytes = self.B * self.H * sum((self.S - self.n_win) * row[p] + self.n_win * self.D * 4
                                                for p in planes)
        # algorithmic flops of the attention call: QK and PV over every visible (row, token) pair
        vis = 0
        for i in range(self.n_q):
            vis += min(self.S, self.q_pos0 + i + 1) if self.causal else self.S
        self.flops = 4 * self.D * vis * w.n_q_heads * self.B


# ------------------------------------------------------------------ CPU oracle (baseline and reference arm)
def oracle_step(w, inp, n_heads: int, kv_len: int | None = None):
    """Prepare (untimed) an oracle cache of the first `n_heads` kv heads over the workload's tokens
    (or its first kv_len) and return a step: the oracle store of the appended tokens + the oracle
    attention of those heads' query rows."""
    from oracle import attention as OA
    S = inp["k"].shape[2] if kv_len is None else kv_len
    n_q = inp["q"].shape[2]
    fill = min(w.n_fill, S - 1)
    k, v = inp["k"][:, :n_heads, :S], inp["v"][:, :n_heads, :S]
    oc = OA.OracleCache(w.layout, w.batch, n_heads, w.head_dim, S, n_recent=w.n_recent)
    oc.store(k[:, :, :fill], v[:, :, :fill], 0)
    q = inp["q"][:, :n_heads * w.gqa]
    causal = w.causal and S - n_q >= 0
    q_pos0 = S - n_q if causal else 0

    def step():
        oc.store(k[:, :, fill:], v[:, :, fill:], fill)
        return oc.attend(q, w.alpha, S, causal=causal, q_pos0=q_pos0)
    return step


def paged_oracle_step(w, inp, n_heads: int, frac: float = 1.0):
    """The paged workload's oracle step over its first `n_heads` kv heads (and the first `frac` of
    every sequence): an oracle paged pool filled (untimed) with all but each sequence's last token;
    the step stores that token of every sequence and runs the paged oracle attention. Returns
    (step, packed bytes the step's attention reads)."""
    from oracle.paged import OraclePagedCache
    lens = np.maximum((inp["seq_lens"] * frac).astype(np.int64), 2)
    B, P = w.batch, w.page_size
    mpp = -(-int(lens.max()) // P)
    table = np.arange(B * mpp).reshape(B, mpp)
    pc = OraclePagedCache(w.layout, B, n_heads, w.head_dim, P, B * mpp, mpp, w.n_recent, table=table)
    D = w.head_dim
    k_all, v_all = inp["k"][:n_heads], inp["v"][:n_heads]
    pad = np.zeros((B, n_heads, int(lens.max()), D), np.float32)
    kp, vp = pad.copy(), pad.copy()
    for b in range(B):
        o, L = int(inp["offsets"][b]), int(lens[b])
        kp[b, :, :L] = k_all[:, o:o + L]
        vp[b, :, :L] = v_all[:, o:o + L]
    pc.store(kp[:, :, :-1], vp[:, :, :-1], np.zeros(B, np.int64))
    k_new = np.stack([kp[b, :, lens[b] - 1:lens[b]] for b in range(B)])
    v_new = np.stack([vp[b, :, lens[b] - 1:lens[b]] for b in range(B)])
    q = inp["q"][:, :n_heads * w.gqa]

    def step():
        pc.store(k_new, v_new, lens - 1)
        return pc.attend(q, w.alpha, lens, causal=False)
    row = {"q4_0": 18, "q6_0": 26, "asym4_g32": 20, "had_int4": 0}[w.layout] * (D // 32) if w.layout != "had_int4" \
        else D // 2 + 4
    return step, 2 * n_heads * int(lens.sum()) * row


def _oracle_all_cores_child(wname: str, budget_s: float, conn) -> None:
    """Spawned child: the same oracle step as cpu_baseline, with the BLAS threads of this process
    set to every host core by the parent (numpy loads after the environment is set)."""
    from synth import WORKLOADS, make_inputs, make_paged_inputs
    w = WORKLOADS[wname]
    if w.page_size:
        step = paged_oracle_step(w, make_paged_inputs(w), 1)[0]
    else:
        step = oracle_step(w, make_inputs(w), 1)
    times = []
    t_all = time.perf_counter()
    while not times or (time.perf_counter() - t_all < budget_s and len(times) < 20):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    conn.send(statistics.median(times))
    conn.close()


def oracle_all_cores(wname: str, budget_s: float):
    """Median step time of the oracle with BLAS threads = all host cores (None if it fails)."""
    import multiprocessing as mp
    n = os.cpu_count() or 1
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    try:
        for k in keys:
            os.environ[k] = str(n)
        ctx = mp.get_context("spawn")            # never fork a process that holds a CUDA context
        parent, child = ctx.Pipe(duplex=False)
        proc = ctx.Process(target=_oracle_all_cores_child, args=(wname, budget_s, child))
        proc.start()
        child.close()
        tm = parent.recv() if parent.poll(budget_s + 300) else None
        proc.join(30)
        return n, tm
    except Exception:
        return n, None
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def cpu_baseline(w, inp, spec, budget_s: float):
    step = oracle_step(w, inp, 1)
    per = spec.read_bytes / spec.H          # one kv head's share of the step's packed bytes
    times = []
    t_all = time.perf_counter()
    while not times or (time.perf_counter() - t_all < budget_s and len(times) < 20):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    tm = statistics.median(times)
    res = {"value": per / tm / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"oracle (numpy, one thread): store of the appended tokens + float64 attention of 1 of "
                     f"{spec.H} kv heads over {spec.S} tokens; median of {len(times)} runs of {tm * 1e3:.0f} ms, "
                     f"{per:.0f} packed bytes each",
           "us_per_layer_equiv": tm * spec.H * 1e6}
    n, ta = oracle_all_cores(w.name, min(budget_s, 15.0))
    if ta:
        res["all_cores"] = {"value": per / ta / 1e9, "unit": "GB/s", "cores": n,
                            "sample": "the same step with numpy's BLAS threads = every host core (spawned process)"}
    return res


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from synth import WORKLOADS, make_inputs
    w = WORKLOADS[args.workload]
    if w.page_size:
        return run_reference_paged(args, w)
    inp = make_inputs(w)
    spec = Spec(w, inp)
    # bound the run: each step is one kv head over a prefix of the tokens, sized so that the
    # W + K steps take about two minutes in total
    probe = oracle_step(w, inp, 1)
    t0 = time.perf_counter()
    probe()
    t_full = time.perf_counter() - t0
    per_step = 120.0 / max(1, args.steps + args.warmup)
    frac = min(1.0, per_step / max(t_full, 1e-6))
    S_s = spec.S if frac >= 1.0 else max(min(spec.S, 1024), int(spec.S * frac) // 64 * 64)
    step = probe if S_s == spec.S else oracle_step(w, inp, 1, kv_len=S_s)
    bytes_per = spec.read_bytes / spec.H * S_s / spec.S
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = bytes_per * args.steps / el / 1e9
    sample = (f"CPU oracle (numpy, one thread): per step, the oracle store of the appended tokens + float64 "
              f"attention of 1 of {spec.H} kv heads over {S_s} of {spec.S} tokens ({bytes_per:.0f} packed bytes)")
    line = {"impl": "reference", "metric": METRIC if args.workload == DEFAULT_WORKLOAD else
            f"{w.layout} KV attention µs/layer and effective HBM GB/s ({args.workload})",
            "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": DESCRIPTIONS[args.workload], "kv_len": spec.S, "sampled_kv_len": S_s,
                       "layout": w.layout},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_paged(args, w):
    """Reference arm of a paged workload: the paged oracle over one kv head and a prefix of every
    sequence, sized so that the W + K steps take about two minutes."""
    from synth import make_paged_inputs
    inp = make_paged_inputs(w)
    full_bytes = 2 * w.n_kv_heads * int(inp["seq_lens"].sum()) * 18 * (w.head_dim // 32)
    probe, _ = paged_oracle_step(w, inp, 1, 0.1)
    t0 = time.perf_counter()
    probe()
    t_probe = time.perf_counter() - t0
    frac = min(1.0, 0.1 * (120.0 / max(1, args.steps + args.warmup)) / max(t_probe, 1e-6))
    step, bytes_per = paged_oracle_step(w, inp, 1, frac)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = bytes_per * args.steps / el / 1e9
    sample = (f"paged CPU oracle (numpy, one thread): per step, the store of each sequence's new token + float64 "
              f"attention of 1 of {w.n_kv_heads} kv heads over {frac:.3f} of every sequence ({bytes_per:.0f} packed "
              f"bytes of {full_bytes} for the whole layer)")
    line = {"impl": "reference", "metric": f"paged {w.layout} KV attention µs/layer and effective HBM GB/s "
                                           f"({args.workload})",
            "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": DESCRIPTIONS[args.workload], "layout": w.layout, "sampled_fraction": frac},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    from synth import WORKLOADS
    if WORKLOADS[args.workload].page_size:
        return paged_main(args)
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

    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    spec = Spec(w, inp)
    B, H, S, D, fill = spec.B, spec.H, spec.S, spec.D, spec.fill

    def to_dev(name):
        if w.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(inp[name + "_bits"]).view(np.int16)).view(
                torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(inp[name])).to(dev)

    kd, vd, q = to_dev("k"), to_dev("v"), to_dev("q")
    k_new = kd[:, :, fill:].contiguous()               # the step's appended tokens
    v_new = vd[:, :, fill:].contiguous()

    def make_caches(layout, n):
        caches = []
        for _ in range(n):
            c = kvq.KVCache(layout, B, H, D, S, n_recent=w.n_recent, device=dev)
            kvq.store(c, kd[:, :, :fill].contiguous(), vd[:, :, :fill].contiguous(), 0)
            kvq.store(c, k_new, v_new, fill)
            caches.append(c)
        return caches

    cache_bytes = spec.read_bytes
    n_rep = min(64, max(2, math.ceil(3 * L2_BYTES / max(cache_bytes, 1)) + 1))
    l2_resident = n_rep * cache_bytes < 2 * L2_BYTES
    caches = make_caches(w.layout, n_rep)
    chunk = kvq.attend_chunk(caches[0], w.n_q_heads, spec.n_q, S, 0)
    ws = torch.empty(max(256, kvq.attend_workspace_bytes(caches[0], w.n_q_heads, spec.n_q, S, chunk)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((B, w.n_q_heads, spec.n_q, D), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    L = _lib.lib()

    def step(i, ev=None):
        c = caches[i % n_rep]
        if ev is not None:
            L.kvq_profile_phase1_events(ev[0].cuda_event, ev[1].cuda_event)
        kvq.append_decode_attend(c, k_new, v_new, fill, q, S, causal=spec.causal, q_pos0=spec.q_pos0,
                                 attn_scale=w.alpha, chunk=chunk, out=out, workspace=ws, stream=stream)
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
            for i in range(16):
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
                    for i in range(16):
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
        if use_graph:
            with torch.cuda.stream(stream):
                ev0.record(stream)
                ev_graph.replay()
                ev1.record(stream)
            torch.cuda.synchronize(dev)
        ev_pass_ms = ev0.elapsed_time(ev1)
        time.sleep(0.25)
    elapsed_ms = max_over_ranks(elapsed_ms, dist if world > 1 else None, dev)
    ph_ms = [a.elapsed_time(b) for a, b in ph_ev]
    ph_mean = statistics.fmean(ph_ms)
    ms_step = elapsed_ms / K
    value = aggregate(world, spec.read_bytes, K, elapsed_ms) / 1e9
    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    prefill = spec.causal and spec.n_q > 1
    if prefill:
        achieved = spec.flops / (ph_mean / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": achieved / bf16_peak, "flops_per_launch": spec.flops,
                "peak_note": "dense bf16 peak; f16 mma has the same nominal rate"}
    else:
        achieved = spec.read_bytes / (ph_mean / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak}
    traffic = kernel_traffic(*PROFILES[args.workload]) if args.workload in PROFILES else None
    roof["peak_nominal"] = NOMINAL_BF16_TFLOPS if prefill else NOMINAL_HBM_GBS
    roof["frac_nominal"] = achieved / roof["peak_nominal"]
    roof.update({"peak_kind": peak_kind, "traffic": traffic, "kernel": "attend phase 1 (split-K chunk partials)",
                 "phase1_us_mean": ph_mean * 1e3, "phase1_us_p10": float(np.percentile(ph_ms, 10)) * 1e3,
                 "phase1_us_p90": float(np.percentile(ph_ms, 90)) * 1e3,
                 "phase1_pass_us_per_step": ev_pass_ms / K * 1e3})
    # store (one launch per plane of a mixed cache), phase 1, reduce. Phase 1 is one launch, except:
    # many Hadamard rows (tcgen05 body) = query preparation + body + the window chunks' launch;
    # Hadamard on the CUDA cores (head_dim 256) = query preparation + attention
    kl, _, vl = w.layout.partition("+")
    mixed = bool(vl) and vl != kl
    had = kl.startswith("had")
    if had and not mixed and D == 128 and w.gqa * spec.n_q > 64:
        phase1_launches = 2 + (1 if spec.n_win > 0 else 0)
    elif had and D != 128:
        phase1_launches = 2
    else:
        phase1_launches = 1
    launches = (2 if mixed else 1) + phase1_launches + 1
    l2_note = (f"cache L2-resident ({n_rep} replicas x {cache_bytes / 2**20:.1f} MiB)" if l2_resident else
               f"inputs larger than L2: {n_rep} cache replicas rotated ({n_rep * cache_bytes / 2**20:.0f} MiB > "
               f"{L2_BYTES / 2**20:.0f} MiB L2)")
    line = {
        "metric": METRIC if args.workload == DEFAULT_WORKLOAD else
        f"{w.layout} KV attention µs/layer and effective HBM GB/s ({args.workload})",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_step, "us_per_layer": ms_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[args.workload], "name": args.workload, "layout": w.layout,
                   "kv_len": S, "n_q": spec.n_q, "causal": spec.causal, "chunk": chunk,
                   "chunk_rule": chunk_rule(w, spec),
                   "step": f"append {S - fill} token(s) (K,V) + split-K attention, one library call",
                   "read_bytes_per_step": spec.read_bytes, "flops_per_step": spec.flops, "l2": l2_note,
                   "timing": ("CUDA graph of the K library steps; phase 1 timed by events in a second pass "
                              "of the same K steps") if use_graph else "stream launches with phase-1 events",
                   "soak_s": args.soak_s, "parallelism": f"replicas x{world}"},
        "pct_of_peak": value / world / hbm_peak,
        "roofline": roof,
        "clocks": clk.summary(),
        "gpu_launches": launches * K,
    }

    if not args.quick and rank == 0:
        # end to end through the host-buffer C-ABI call: pinned host k_new, v_new and q in, the f32
        # result back in pinned host memory, one stream wait per step. The call copies q host ->
        # device; the store kernel reads k_new / v_new from the pinned buffers over the host link and
        # the reduce writes the result into the pinned output (every input and output byte crosses
        # the link inside the timed region)
        n_k, n_qe = k_new.numel(), q.numel()
        packed = torch.empty(2 * n_k + n_qe, dtype=k_new.dtype).pin_memory()
        hk, hv = packed[:n_k].view(k_new.shape), packed[n_k:2 * n_k].view(v_new.shape)
        hq = packed[2 * n_k:].view(q.shape)
        hk.copy_(k_new.cpu())
        hv.copy_(v_new.cpu())
        hq.copy_(q.cpu())
        hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        ws_h = torch.empty(kvq.append_decode_attend_host_workspace_bytes(caches[0], hk.dtype, hk.shape[2], hq.dtype,
                                                                         w.n_q_heads, spec.n_q, S, chunk),
                           dtype=torch.uint8, device=dev)
        n_e2e = min(K, 2000)
        # the C-ABI call itself, arguments prepared once (what a C caller pays per step)
        import ctypes
        dt = {torch.bfloat16: _lib.KVQ_BF16, torch.float16: _lib.KVQ_F16, torch.float32: _lib.KVQ_F32}
        fn = L.kvq_append_decode_attend_host
        argv = [(ctypes.byref(c.struct), hk.data_ptr(), hv.data_ptr(), dt[hk.dtype], hk.shape[2], fill, hq.data_ptr(),
                 dt[hq.dtype], w.n_q_heads, spec.n_q, S, int(spec.causal), spec.q_pos0, ctypes.c_float(w.alpha),
                 chunk, hout.data_ptr(), ws_h.data_ptr(), ws_h.numel(), stream.cuda_stream) for c in caches]
        for i in range(n_e2e + 3):
            if i == 3:
                t0 = time.perf_counter()
            st = fn(*argv[i % n_rep])
        t_e2e = (time.perf_counter() - t0) / n_e2e
        if st != 0:
            raise RuntimeError(f"host-buffer call failed: {L.kvq_last_error().decode()}")
        # the same through the Python binding (argument checks and marshalling on every call)
        for i in range(n_e2e + 3):
            if i == 3:
                t0 = time.perf_counter()
            kvq.append_decode_attend_host(caches[i % n_rep], hk, hv, fill, hq, S, causal=spec.causal,
                                          q_pos0=spec.q_pos0, attn_scale=w.alpha, chunk=chunk, out=hout,
                                          workspace=ws_h, stream=stream)
        t_py = (time.perf_counter() - t0) / n_e2e
        el = hk.element_size()
        line["e2e"] = {"value": spec.read_bytes / t_e2e / 1e9, "unit": "GB/s",
                       "h2d_bytes_per_step": (hk.numel() + hv.numel() + hq.numel()) * el,
                       "d2h_bytes_per_step": hout.numel() * 4, "us_per_layer": t_e2e * 1e6, "steps": n_e2e,
                       "call": "kvq_append_decode_attend_host through ctypes with prepared arguments (pinned "
                               "host buffers, one call and one stream wait per step; q copied host to device, "
                               "k_new / v_new read by the store kernel and the output written by the reduce "
                               "over the host link)",
                       "python_binding_us_per_layer": t_py * 1e6}
        line["store"] = store_timings(kvq, w, kd, vd, k_new, v_new, fill, stream, dev)
        if args.workload == DEFAULT_WORKLOAD:
            line["comparators"] = comparators(caches[0], kd, vd, q, out, w, spec, stream, dev)
            line["variants"] = variants(kvq, caches, n_rep, k_new, v_new, q, out, spec, stream, ev0, ev1,
                                        min(K, 1000), chunk, make_caches, dev)
        if world == 1:
            line["cpu_baseline"] = cpu_baseline(w, inp, spec, args.cpu_seconds)
        if args.workload == DEFAULT_WORKLOAD and args.summary_steps > 0:
            del caches, ws, kd, vd
            torch.cuda.empty_cache()
            line["workloads"] = workload_summaries(kvq, L, dev, stream, args.summary_steps, hbm_peak, bf16_peak)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def comparators(cache, kd, vd, q, out, w, spec, stream, dev, reps=20):
    """Optional comparators, for context only (not targets): torch's bf16 scaled_dot_product_attention
    over the unquantised K/V of the same layer, and a materialised path that first dequantises the Q4_0
    planes into bf16 K/V with plain torch tensor ops and then runs the same SDPA (the "dequantise, then
    attend" alternative to reading the packed cache in the attention kernel). Whole calls, CUDA events on
    the bench stream, K/V far larger than L2."""
    import torch
    import torch.nn.functional as F
    B, H, S, D = spec.B, spec.H, spec.S, spec.D
    qb = q.to(torch.bfloat16)
    res = {"note": "torch ops, not this library; context for the fused read, not a target. max_abs_diff: against this library's output of the same step (the unquantised SDPA differs by the Q4_0 quantisation error)"}

    def sdpa(k, v):
        return F.scaled_dot_product_attention(qb, k, v, scale=w.alpha, enable_gqa=True)

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps * 1e3

    ref = out.float()                          # this library's output of the same step (sanity check)
    res["library_max_abs_output"] = float(ref.abs().max())
    try:
        res["torch_sdpa_bf16_us"] = timed(lambda: sdpa(kd, vd))
        res["torch_sdpa_bf16_bytes_read"] = 2 * kd.numel() * kd.element_size()
        res["torch_sdpa_bf16_max_abs_diff"] = float((sdpa(kd, vd).float() - ref).abs().max())
    except Exception as e:   # a torch build without the GQA form of SDPA
        res["torch_sdpa_bf16_error"] = str(e)[:200]
    if w.layout == "q4_0":
        cap = cache.capacity

        def planes(t):
            return (cache.planes[t]["payload"].view(B, H, cap, D // 2)[:, :, :S],
                    cache.planes[t]["scale"].view(B, H, cap, D // 32)[:, :, :S])

        def deq(payload, scale):
            # byte j of a 32-value block: value 2j in the low nibble, 2j+1 in the high; code (n ^ 8) - 8
            n = torch.stack((payload & 15, payload >> 4), dim=-1).view(B, H, S, D).to(torch.int16)
            code = (n ^ 8) - 8
            return (code.to(torch.float32) * scale.to(torch.float32).repeat_interleave(32, dim=-1)).to(torch.bfloat16)

        (pk, sk), (pv, sv) = planes("k"), planes("v")
        try:
            res["dequant_then_sdpa_us"] = timed(lambda: sdpa(deq(pk, sk), deq(pv, sv)))
            res["dequant_then_sdpa_max_abs_diff"] = float((sdpa(deq(pk, sk), deq(pv, sv)).float() - ref).abs().max())
        except Exception as e:
            res["dequant_then_sdpa_error"] = str(e)[:200]
    return res


def workload_summaries(kvq, L, dev, stream, K, hbm_peak, bf16_peak):
    """Every other seeded workload, timed with the default line's protocol at a smaller step count:
    K library steps (append + attention, one call each) in a CUDA graph over cache replicas that
    exceed L2 (or the note says the cache is L2-resident), then the same steps with phase-1 events.
    Per workload: µs per layer-call, effective GB/s of the step, and phase 1 against its roofline
    (HBM for the decode shapes, the bf16 tensor peak for the causal prefill chunk)."""
    import torch
    from synth import WORKLOADS, make_inputs, make_paged_inputs
    out = {}
    for name in SUMMARY_WORKLOADS:
        w = WORKLOADS[name]
        if w.page_size:
            inp = make_paged_inputs(w)
            lens = inp["seq_lens"]
            B, H, D, P = w.batch, w.n_kv_heads, w.head_dim, w.page_size
            S_max, total = int(lens.max()), int(lens.sum())
            mpp = -(-S_max // P)
            kp = torch.zeros((B, H, S_max, D), dtype=torch.bfloat16, device=dev)
            vp = torch.zeros_like(kp)
            kf = torch.from_numpy(np.ascontiguousarray(inp["k_bits"]).view(np.int16)).view(torch.bfloat16)
            vf = torch.from_numpy(np.ascontiguousarray(inp["v_bits"]).view(np.int16)).view(torch.bfloat16)
            for b in range(B):
                o, Lb = int(inp["offsets"][b]), int(lens[b])
                kp[b, :, :Lb] = kf[:, o:o + Lb].to(dev)
                vp[b, :, :Lb] = vf[:, o:o + Lb].to(dev)
            k_new = torch.stack([kp[b, :, int(lens[b]) - 1:int(lens[b])] for b in range(B)]).contiguous()
            v_new = torch.stack([vp[b, :, int(lens[b]) - 1:int(lens[b])] for b in range(B)]).contiguous()
            q = torch.from_numpy(np.ascontiguousarray(inp["q_bits"]).view(np.int16)).view(torch.bfloat16).to(dev)
            lens_dev = torch.from_numpy(lens.astype(np.int32)).to(dev)
            read_bytes, flops = 2 * H * total * 18 * (D // 32), 4 * D * total * w.n_q_heads
            n_rep = min(64, max(2, math.ceil(3 * L2_BYTES / read_bytes) + 1))
            pools = []
            for r in range(n_rep):
                c = kvq.PagedKVCache(w.layout, B, H, D, P, B * mpp, mpp, device=dev)
                c.set_block_table(np.random.default_rng(w.seed + r).permutation(B * mpp).reshape(B, mpp))
                kvq.paged_store(c, kp[:, :, :S_max - 1].contiguous(), vp[:, :, :S_max - 1].contiguous(),
                                torch.zeros(B, dtype=torch.int32, device=dev))
                pools.append(c)
            del kp, vp
            chunk = kvq.paged_attend_plan_chunk(pools[0], w.n_q_heads, 1, lens)
            ws = torch.empty(max(256, kvq.paged_attend_workspace_bytes(pools[0], w.n_q_heads, 1, S_max, chunk)),
                             dtype=torch.uint8, device=dev)
            o_buf = torch.empty((B, w.n_q_heads, 1, D), dtype=torch.float32, device=dev)

            def call(i):
                kvq.paged_append_decode_attend(pools[i % n_rep], k_new, v_new, q, lens_dev, S_max,
                                               attn_scale=w.alpha, chunk=chunk, out=o_buf, workspace=ws,
                                               stream=stream)
            prefill, held = False, pools
        else:
            inp = make_inputs(w)
            spec = Spec(w, inp)
            B, H, S, D, fill = spec.B, spec.H, spec.S, spec.D, spec.fill

            def to_dev(n):
                if w.dtype == "bf16":
                    return torch.from_numpy(np.ascontiguousarray(inp[n + "_bits"]).view(np.int16)).view(
                        torch.bfloat16).to(dev)
                return torch.from_numpy(np.ascontiguousarray(inp[n])).to(dev)
            kd, vd, q = to_dev("k"), to_dev("v"), to_dev("q")
            k_new, v_new = kd[:, :, fill:].contiguous(), vd[:, :, fill:].contiguous()
            read_bytes, flops = spec.read_bytes, spec.flops
            n_rep = min(64, max(2, math.ceil(3 * L2_BYTES / max(read_bytes, 1)) + 1))
            caches = []
            for _ in range(n_rep):
                c = kvq.KVCache(w.layout, B, H, D, S, n_recent=w.n_recent, device=dev)
                kvq.store(c, kd[:, :, :fill].contiguous(), vd[:, :, :fill].contiguous(), 0)
                kvq.store(c, k_new, v_new, fill)
                caches.append(c)
            del kd, vd
            chunk = kvq.attend_chunk(caches[0], w.n_q_heads, spec.n_q, S, 0)
            ws = torch.empty(max(256, kvq.attend_workspace_bytes(caches[0], w.n_q_heads, spec.n_q, S, chunk)),
                             dtype=torch.uint8, device=dev)
            o_buf = torch.empty((B, w.n_q_heads, spec.n_q, D), dtype=torch.float32, device=dev)

            def call(i, spec=spec, caches=caches):
                kvq.append_decode_attend(caches[i % n_rep], k_new, v_new, fill, q, S, causal=spec.causal,
                                         q_pos0=spec.q_pos0, attn_scale=w.alpha, chunk=chunk, out=o_buf,
                                         workspace=ws, stream=stream)
            prefill, held = spec.causal and spec.n_q > 1, caches
        ph = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        with torch.cuda.stream(stream):
            for a, b in ph:
                a.record(stream)
                b.record(stream)
            for i in range(3):
                call(i)
        torch.cuda.synchronize(dev)
        g, g_ev = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(K):
                call(i)
        with torch.cuda.graph(g_ev, stream=stream):
            for i in range(K):
                L.kvq_profile_phase1_events(ph[i][0].cuda_event, ph[i][1].cuda_event)
                call(i)
                L.kvq_profile_phase1_events(None, None)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()                                   # warm
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        step_ms = e0.elapsed_time(e1) / K
        with torch.cuda.stream(stream):
            g_ev.replay()
        torch.cuda.synchronize(dev)
        # the median launch: one delayed event pair can dominate the mean (seen once: a mean of
        # 0.35 ms over 200 launches of a 0.05 ms kernel, i.e. one pair about 60 ms apart); the mean
        # is kept beside it
        ph_all = [a.elapsed_time(b) for a, b in ph]
        ph_ms, ph_mean = statistics.median(ph_all), statistics.fmean(ph_all)
        if prefill:
            ach = flops / (ph_ms / 1e3) / 1e12
            roof = {"bound": "tensor", "achieved": round(ach, 1), "unit": "TFLOP/s", "frac": round(ach / bf16_peak, 4),
                    "frac_nominal": round(ach / NOMINAL_BF16_TFLOPS, 4)}
        else:
            ach = read_bytes / (ph_ms / 1e3) / 1e9
            roof = {"bound": "hbm", "achieved": round(ach, 1), "unit": "GB/s", "frac": round(ach / hbm_peak, 4),
                    "frac_nominal": round(ach / NOMINAL_HBM_GBS, 4)}
        out[name] = {"us_per_layer": round(step_ms * 1e3, 2), "gbs": round(read_bytes / (step_ms / 1e3) / 1e9, 1),
                     "phase1_us": round(ph_ms * 1e3, 2), "phase1_us_mean": round(ph_mean * 1e3, 2),
                     "roofline": roof, "chunk": chunk,
                     "read_bytes_per_step": read_bytes, "flops_per_step": flops, "steps": K,
                     "l2": "cache L2-resident" if n_rep * read_bytes < 2 * L2_BYTES else
                     f"{n_rep} replicas rotated (> L2)"}
        del held, g, g_ev, ws, o_buf
        torch.cuda.empty_cache()
    return out


def store_timings(kvq, w, kd, vd, k_new, v_new, fill, stream, dev):
    """The store kernel timed on its own (CUDA events on the launching stream): the append of this
    workload's new rows (µs per call) and a bulk fill of the cache (input GB/s: bf16/f32 K and V
    bytes read per second; the packed bytes written are 0.28 of them for Q4_0 from bf16)."""
    import torch
    B, H, S, D = kd.shape
    c = kvq.KVCache(w.layout, B, H, D, S, n_recent=w.n_recent, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kf, vf = kd[:, :, :fill].contiguous(), vd[:, :, :fill].contiguous()

    def timed(fn, n):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n

    app_ms = timed(lambda: kvq.store(c, k_new, v_new, fill, stream=stream), 200)
    fill_ms = timed(lambda: kvq.store(c, kf, vf, 0, stream=stream), 10)
    in_bytes = 2 * kf.numel() * kf.element_size()
    out_bytes = c.read_bytes(fill)
    del c
    return {"append_tokens": S - fill, "append_us": app_ms * 1e3, "fill_tokens": fill, "fill_us": fill_ms * 1e3,
            "fill_input_gbs": in_bytes / (fill_ms / 1e3) / 1e9, "fill_output_gbs": out_bytes / (fill_ms / 1e3) / 1e9,
            "timing": "CUDA events around back-to-back store launches on one stream"}


def variants(kvq, caches, n_rep, k_new, v_new, q, out, spec, stream, ev0, ev1, n, chunk, make_caches, dev):
    """The 128K layer with the pages' fixed 512-token chunk, and with the asymmetric g=32 layout
    (plain stream launches, same replicas)."""
    import torch
    w, S, fill = spec.w, spec.S, spec.fill

    def time_plain(cs, wsb, ch):
        with torch.cuda.stream(stream):
            for i in range(5):
                kvq.append_decode_attend(cs[i % n_rep], k_new, v_new, fill, q, S, attn_scale=w.alpha, chunk=ch,
                                         out=out, workspace=wsb, stream=stream)
            torch.cuda.synchronize(dev)
            ev0.record(stream)
            for i in range(n):
                kvq.append_decode_attend(cs[i % n_rep], k_new, v_new, fill, q, S, attn_scale=w.alpha, chunk=ch,
                                         out=out, workspace=wsb, stream=stream)
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        return ev0.elapsed_time(ev1) / n

    res = {}
    ws512 = torch.empty(kvq.attend_workspace_bytes(caches[0], w.n_q_heads, 1, S, 512), dtype=torch.uint8, device=dev)
    c_ms = time_plain(caches, ws512, 512)
    res["q4_0_chunk512"] = {"us_per_layer": c_ms * 1e3, "gbs": spec.read_bytes / (c_ms / 1e3) / 1e9,
                            "timing": "stream launches", "chunk": 512}
    caches.clear()
    torch.cuda.empty_cache()
    acaches = make_caches("asym4_g32", n_rep)
    a_bytes = acaches[0].read_bytes(S)
    achunk = kvq.attend_chunk(acaches[0], w.n_q_heads, 1, S, 0)        # its own automatic chunk
    aws = torch.empty(kvq.attend_workspace_bytes(acaches[0], w.n_q_heads, 1, S, achunk), dtype=torch.uint8,
                      device=dev)
    a_ms = time_plain(acaches, aws, achunk)
    res["asym4_g32"] = {"us_per_layer": a_ms * 1e3, "read_bytes_per_step": a_bytes,
                        "gbs": a_bytes / (a_ms / 1e3) / 1e9, "timing": "stream launches", "chunk": achunk}
    return res


def paged_main(args):
    """GPU arm of a paged workload: the same protocol as main() (graph of K library steps, phase-1
    events in a second pass, clocks, e2e through the public API, CPU oracle baseline)."""
    import torch
    import torch.distributed as dist

    import sub_byte_quantized_gb300 as kvq
    from sub_byte_quantized_gb300 import _lib
    from synth import WORKLOADS, make_paged_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    w = WORKLOADS[args.workload]
    inp = make_paged_inputs(w)
    lens = inp["seq_lens"]
    B, H, D, P, Hq = w.batch, w.n_kv_heads, w.head_dim, w.page_size, w.n_q_heads
    S_max, total = int(lens.max()), int(lens.sum())
    mpp = -(-S_max // P)
    n_pages = B * mpp

    def bits(name):
        return torch.from_numpy(np.ascontiguousarray(inp[name + "_bits"]).view(np.int16)).view(torch.bfloat16)

    kf, vf, q = bits("k"), bits("v"), bits("q").to(dev)
    # every sequence's tokens padded to S_max ([B][H][S_max][D] on the device) for the bulk fill;
    # the new token of a step is each sequence's last one
    kp = torch.zeros((B, H, S_max, D), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    for b in range(B):
        o, L = int(inp["offsets"][b]), int(lens[b])
        kp[b, :, :L] = kf[:, o:o + L].to(dev)
        vp[b, :, :L] = vf[:, o:o + L].to(dev)
    idx = torch.from_numpy(lens - 1).to(dev)
    k_new = torch.stack([kp[b, :, int(lens[b]) - 1:int(lens[b])] for b in range(B)]).contiguous()
    v_new = torch.stack([vp[b, :, int(lens[b]) - 1:int(lens[b])] for b in range(B)]).contiguous()
    lens_dev = torch.from_numpy(lens.astype(np.int32)).to(dev)
    row = 18 * (D // 32)
    read_bytes = 2 * H * total * row
    flops = 4 * D * total * (Hq // H) * H

    def make_pool(seed):
        c = kvq.PagedKVCache(w.layout, B, H, D, P, n_pages, mpp, device=dev)
        c.set_block_table(np.random.default_rng(seed).permutation(n_pages).reshape(B, mpp))
        kvq.paged_store(c, kp[:, :, :S_max - 1].contiguous(), vp[:, :, :S_max - 1].contiguous(),
                        torch.zeros(B, dtype=torch.int32, device=dev))
        return c
    n_rep = min(64, max(2, math.ceil(3 * L2_BYTES / read_bytes) + 1))
    pools = [make_pool(w.seed + r) for r in range(n_rep)]
    del kp, vp
    torch.cuda.empty_cache()
    chunk = kvq.paged_attend_plan_chunk(pools[0], Hq, 1, lens)          # balanced from the host lengths
    chunk_tot = kvq.paged_attend_chunk(pools[0], Hq, 1, S_max, total)   # from the total length only
    chunk_max = kvq.paged_attend_chunk(pools[0], Hq, 1, S_max, 0)
    ws = torch.empty(max(256, kvq.paged_attend_workspace_bytes(pools[0], Hq, 1, S_max, chunk)), dtype=torch.uint8,
                     device=dev)
    out = torch.empty((B, Hq, 1, D), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    L = _lib.lib()

    def step(i, ev=None, c_chunk=None):
        if ev is not None:
            L.kvq_profile_phase1_events(ev[0].cuda_event, ev[1].cuda_event)
        kvq.paged_append_decode_attend(pools[i % n_rep], k_new, v_new, q, lens_dev, S_max, attn_scale=w.alpha,
                                       chunk=c_chunk or chunk, out=out, workspace=ws, stream=stream)
        if ev is not None:
            L.kvq_profile_phase1_events(None, None)

    K, W = args.steps, args.warmup
    ph_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(stream):
        for a, b in ph_ev:
            a.record(stream)
            b.record(stream)
        for i in range(max(W, 3)):
            step(i)
    torch.cuda.synchronize(dev)
    graph, ev_graph, soak_graph = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(K):
            step(i)
    with torch.cuda.graph(ev_graph, stream=stream):
        for i in range(K):
            step(i, ph_ev[i])
    with torch.cuda.graph(soak_graph, stream=stream):
        for i in range(16):
            step(i)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t_end = time.perf_counter() + args.soak_s
        with torch.cuda.stream(stream):
            while time.perf_counter() < t_end:
                soak_graph.replay()
                torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        elapsed_ms = ev0.elapsed_time(ev1)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            ev_graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        ev_pass_ms = ev0.elapsed_time(ev1)
        time.sleep(0.25)
    elapsed_ms = max_over_ranks(elapsed_ms, dist if world > 1 else None, dev)
    ph_ms = [a.elapsed_time(b) for a, b in ph_ev]
    ph_mean = statistics.fmean(ph_ms)
    ms_step = elapsed_ms / K
    value = aggregate(world, read_bytes, K, elapsed_ms) / 1e9
    hbm_peak, _, peak_kind = measured_peaks()
    achieved = read_bytes / (ph_mean / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
            "peak_kind": peak_kind, "traffic": kernel_traffic("attend_phase1_paged_q4_0_ragged.md", "attend_mma.cu"),
            "kernel": "attend phase 1 (split-K chunk partials), paged",
            "phase1_us_mean": ph_mean * 1e3, "phase1_us_p10": float(np.percentile(ph_ms, 10)) * 1e3,
            "phase1_us_p90": float(np.percentile(ph_ms, 90)) * 1e3, "phase1_pass_us_per_step": ev_pass_ms / K * 1e3}
    line = {
        "metric": f"paged {w.layout} KV attention µs/layer and effective HBM GB/s ({args.workload})",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_step, "us_per_layer": ms_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[args.workload], "name": args.workload, "layout": w.layout,
                   "sequences": B, "seq_lens": [int(x) for x in lens], "total_tokens": total, "page_size": P,
                   "pool_pages": n_pages, "chunk": chunk, "chunk_rule": "kvq_paged_attend_plan_chunk from the host "
                   "lengths: the shortest chunk whose equal per-sequence chunks fit one wave "
                   f"(total-length rule: {chunk_tot}, max-length rule: {chunk_max})",
                   "step": "append 1 token per sequence (K,V) + split-K attention over each sequence's length, "
                           "one library call",
                   "read_bytes_per_step": read_bytes, "flops_per_step": flops,
                   "l2": f"inputs larger than L2: {n_rep} pools rotated ({n_rep * read_bytes / 2**20:.0f} MiB read)",
                   "timing": "CUDA graph of the K library steps; phase 1 timed by events in a second pass",
                   "soak_s": args.soak_s, "parallelism": f"replicas x{world}"},
        "pct_of_peak": value / world / hbm_peak,
        "roofline": roof,
        "clocks": clk.summary(),
        "gpu_launches": 3 * K,
    }
    if not args.quick and rank == 0:
        # the max-length chunk rule on the same batch (stream launches)
        ws_m = torch.empty(max(256, kvq.paged_attend_workspace_bytes(pools[0], Hq, 1, S_max, chunk_max)),
                           dtype=torch.uint8, device=dev)

        def plain(ch, wsb, n=200):
            with torch.cuda.stream(stream):
                for i in range(5):
                    kvq.paged_append_decode_attend(pools[i % n_rep], k_new, v_new, q, lens_dev, S_max,
                                                   attn_scale=w.alpha, chunk=ch, out=out, workspace=wsb, stream=stream)
                ev0.record(stream)
                for i in range(n):
                    kvq.paged_append_decode_attend(pools[i % n_rep], k_new, v_new, q, lens_dev, S_max,
                                                   attn_scale=w.alpha, chunk=ch, out=out, workspace=wsb, stream=stream)
                ev1.record(stream)
            torch.cuda.synchronize(dev)
            return ev0.elapsed_time(ev1) / n
        ws_t = torch.empty(max(256, kvq.paged_attend_workspace_bytes(pools[0], Hq, 1, S_max, chunk_tot)),
                           dtype=torch.uint8, device=dev)
        t_plan, t_tot, t_max = plain(chunk, ws), plain(chunk_tot, ws_t), plain(chunk_max, ws_m)
        line["variants"] = {"planned_chunk": {"chunk": chunk, "us_per_layer": t_plan * 1e3, "timing": "stream launches"},
                            "total_length_chunk": {"chunk": chunk_tot, "us_per_layer": t_tot * 1e3,
                                                   "timing": "stream launches"},
                            "max_length_chunk": {"chunk": chunk_max, "us_per_layer": t_max * 1e3,
                                                 "gbs": read_bytes / (t_max / 1e3) / 1e9, "timing": "stream launches"}}
        # end to end through the host-buffer C-ABI call: new tokens, queries and the sequence lengths
        # from pinned host memory, the output back into pinned host memory, one stream wait per step
        hk, hv, hq = k_new.cpu().pin_memory(), v_new.cpu().pin_memory(), q.cpu().pin_memory()
        hl = lens_dev.cpu().pin_memory()
        hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        ws_h = torch.empty(kvq.paged_append_decode_attend_host_workspace_bytes(pools[0], hk.dtype, hk.shape[2],
                                                                               hq.dtype, Hq, 1, S_max, chunk),
                           dtype=torch.uint8, device=dev)
        n_e2e = min(K, 500)
        for i in range(n_e2e + 3):
            if i == 3:
                t0 = time.perf_counter()
            kvq.paged_append_decode_attend_host(pools[i % n_rep], hk, hv, hq, hl, S_max, attn_scale=w.alpha,
                                                chunk=chunk, out=hout, workspace=ws_h, stream=stream)
        t_e2e = (time.perf_counter() - t0) / n_e2e
        el = hk.element_size()
        line["e2e"] = {"value": read_bytes / t_e2e / 1e9, "unit": "GB/s",
                       "h2d_bytes_per_step": (hk.numel() + hv.numel() + hq.numel()) * el + hl.numel() * 4,
                       "d2h_bytes_per_step": hout.numel() * 4, "us_per_layer": t_e2e * 1e6, "steps": n_e2e,
                       "call": "kvq_paged_append_decode_attend_host (host buffers, one call and one stream wait "
                               "per step)"}
        if world == 1:
            step_o, per = paged_oracle_step(w, inp, 1)
            times = []
            t_all = time.perf_counter()
            while not times or (time.perf_counter() - t_all < args.cpu_seconds and len(times) < 20):
                t0 = time.perf_counter()
                step_o()
                times.append(time.perf_counter() - t0)
            tm = statistics.median(times)
            line["cpu_baseline"] = {"value": per / tm / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                    "sample": f"paged oracle (numpy, one thread): the store of every sequence's new "
                                              f"token + float64 attention of 1 of {H} kv heads over all {B} "
                                              f"sequences; median of {len(times)} runs of {tm * 1e3:.0f} ms, "
                                              f"{per} packed bytes each"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
