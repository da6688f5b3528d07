#!/usr/bin/env python3
"""Benchmark of the GB300 KV-cached decoder step.

Default workload: the GPT-2-XL-shaped bf16 decoder, batch 256, 960-token prompts in shuffled
paged blocks, decode positions 960..1023 (its 64 teacher-forced steps, the last one attending
over 1024 keys). One bench step = one batched decode step (every row of the hot path: embed,
norm+QKV(+RoPE)/kv_write, paged attention, O+residual, norm+FFN, final norm + tied head +
argmax), replayed as one CUDA graph. Decode positions cycle through the workload's steps, so
every `decode_steps` bench steps are exactly one pass of the workload.

The same JSON line carries a "prefill" object: prefill tok/s of the GPT-2-124M-shaped bf16
model on 16 x 1024-token prompts (one step = one llm_prefill of all 16 prompts), with its own
tensor-core roofline, CPU baseline and end-to-end figure.

--impl reference times the float64 CPU oracle on the host cores on a bounded sample of the same
workloads (test infrastructure, never the product path).

Prints one JSON line (rank 0). Multi-GPU: launched by torchrun, one replica per rank (the decode
batch shards by sequence; no data-path collective).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

try:
    import torch.distributed as dist
except Exception:   # the reference arm runs without torch
    dist = None

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "decode tok/s at batch B and prefill tok/s; % of GB300 HBM BW / bf16 TC peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------------------------
# algorithmic work per unit (decode step)
# ------------------------------------------------------------------------------------------------

# DRAM traffic per launch of each workload's dominant kernel family, from one single-pass ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum summed over one decode step's or one
# prefill's launches of that family, divided by the launch count). It holds for the kernel
# build the capture was taken on; the bench reports it when its dominant family matches, and
# the commands and per-launch figures sit with the other profile summaries.
TRAFFIC = {
    "gpt2-124m-fp32-b32-teacher": ("proj (gemm_tcs)", 10.392e6),
    "gpt2-124m-fp32-b1-greedy": ("proj (gemv)", 10.17e6),
    "smollm2-360m-bf16-b64-ctx64to2048": ("proj (gemm_tcs)", 6.155e6),
    "gpt2-xl-bf16-b256-ctx1024": ("attn_decode", 3175.5e6),
    "gpt2-124m-bf16-prefill-16x1024": ("gemm_tc2 (tcgen05 projections on SM pairs)", 184.6e6),
}


def traffic_for(workload: str, kernel: str):
    t = TRAFFIC.get(workload)
    return t[1] if t and t[0] == kernel else None


def job_rate(ms_local: float, units_per_rank: float, world: int, device: str = "cuda"):
    """Whole-job rate of N replicas: the job takes as long as its slowest rank (max over ranks of
    the timed milliseconds) and processes every rank's units. Returns (ms, units, units per s).
    Call on every rank (it is a collective when world > 1)."""
    ms = ms_local
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    units = units_per_rank * world
    return ms, units, units / (ms / 1000.0)


WEIGHTS_LABEL = {wl.DTYPE_F32: "fp32 weights", wl.DTYPE_BF16: "bf16 weights",
                 wl.DTYPE_Q8: "Q8_0 weights (int8 quants, fp16 block scales)"}


def dtype_label(s: wl.ModelShape) -> str:
    """The arithmetic type of the path: the weights' type for fp32 / bf16 models; Q8_0 weights are
    dequantised into fp32 arithmetic."""
    return {wl.DTYPE_F32: "f32", wl.DTYPE_BF16: "bf16", wl.DTYPE_Q8: "q8_0 weights, f32 arithmetic"}[s.dtype]


def weight_bytes(s: wl.ModelShape) -> int:
    """Projection weights read once per step, including the tied head (vocab x d)."""
    return int(round((s.n_layers * s.layer_params() + s.vocab * s.d_model) * s.elt_bytes))


def gemv_bytes(s: wl.ModelShape, B: int) -> int:
    """Projection kernels: weights once, plus activations in and outputs out (4 bytes a value:
    fp32, or a bf16 pair for bf16 weights)."""
    a = 4
    d, F, qkv, hq = s.d_model, s.d_ff, s.qkv_dim, s.n_heads * s.head_dim
    per_layer = B * (d * a + qkv * 4)             # qkv: x in, q (fp32) / k,v out
    per_layer += B * (hq * a + 2 * d * 4)         # o: x in, residual read+write
    per_layer += B * (d * a + F * a)              # up
    per_layer += B * (F * a + 2 * d * 4)          # down
    return weight_bytes(s) + s.n_layers * per_layer + B * d * a


def attn_bytes(s: wl.ModelShape, ctx: np.ndarray, kv_elt: int = 4) -> int:
    """Decode attention: K and V of every cached position (incl. the new one) once per layer
    (kv_elt bytes an element: 4 for the fp32 cache, 2 for bf16)."""
    kv = int(ctx.sum()) * s.n_kv_heads * s.head_dim * kv_elt * 2 * s.n_layers
    qo = len(ctx) * s.n_heads * s.head_dim * (4 + 4) * s.n_layers
    return kv + qo


def step_bytes(s: wl.ModelShape, ctx: np.ndarray, kv_elt: int = 4) -> int:
    return gemv_bytes(s, len(ctx)) + attn_bytes(s, ctx, kv_elt)


def prefill_gemm_flops(s: wl.ModelShape, lengths: np.ndarray) -> float:
    """Projection flops of one prefill: 2 * rows * (layer params) plus the head on the last rows."""
    rows = float(lengths.sum())
    return 2.0 * rows * s.n_layers * s.layer_params() + 2.0 * len(lengths) * s.vocab * s.d_model


def prefill_attn_flops(s: wl.ModelShape, lengths: np.ndarray) -> float:
    """Causal attention flops: q.k and p.v over the (T+1)T/2 visible pairs of every head."""
    pairs = float(sum(int(L) * (int(L) + 1) // 2 for L in lengths))
    return 4.0 * pairs * s.head_dim * s.n_heads * s.n_layers


# ------------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# ------------------------------------------------------------------------------------------------

def oracle_decode_rate(W: wl.Workload, steps: int, warmup: int = 0, n_seq: int = 1, weights=None):
    """Time the float64 oracle, as it stands, on `steps` decode steps of `n_seq` sequences.

    Prefill is untimed; positions cycle through the workload's decode positions exactly
    as the GPU bench does. Returns (tok/s, seconds, description).
    """
    import oracle
    w = weights or wl.make_weights(W.model, scale=W.weight_scale)
    model = oracle.OracleModel(w, kv_dtype=W.kv_dtype)
    prompts = wl.draw_prompts(W.lengths(), W.model.vocab)
    stream = wl.draw_stream(W.batch, max(W.decode_steps, 1), W.model.vocab)
    period = max(W.decode_steps, 1)
    seqs = []
    for b in range(n_seq):
        s = oracle.Sequence(model)
        s.prefill(prompts[b])
        seqs.append((s, list(s.k), list(s.v), s.length))
    done = 0
    t0 = None
    for i in range(warmup + steps):
        if i == warmup:
            t0 = time.perf_counter()
        j = i % period
        for b, (s, k0, v0, L0) in enumerate(seqs):
            if j == 0:
                s.k, s.v, s.length = list(k0), list(v0), L0
            s.step(int(stream[j, b]))
        if i >= warmup:
            done += n_seq
    dt = time.perf_counter() - t0
    desc = (f"float64 NumPy oracle, KV-cached mode, {n_seq} of {W.batch} sequences, {steps} decode steps "
            f"(positions {int(W.lengths()[0])}..{int(W.lengths()[0]) + period - 1} cycled), prefill untimed")
    return done / dt, dt, desc


def gpu_id_for_smi(local: int) -> str:
    """nvidia-smi --id of this process's GPU (its UUID when torch reports one)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(local)


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# Bounded CPU sample of each decode workload for the oracle: (sequences, decode steps). The
# prefill that fills each sampled sequence's cache is untimed.
CPU_SAMPLE = {
    wl.W_GPT2XL_B256.name: (2, 2),
    wl.W_SMOLLM2_B64.name: (2, 1),
    wl.W_GPT2_F32_B32.name: (1, 256),
    wl.W_GPT2_F32_B32_X8.name: (1, 256),
    wl.W_GPT2_F32_B1.name: (1, 16),
}


def oracle_prefill_rate(W: wl.Workload, n: int = 1, weights=None):
    """Time the float64 oracle's stateless forward over one prompt of a prefill workload, n times.
    Returns (tok/s, seconds, description)."""
    import oracle
    w = weights or wl.make_weights(W.model, scale=W.weight_scale)
    model = oracle.OracleModel(w)
    prompt = wl.draw_prompts(W.lengths(), W.model.vocab)[0]
    t0 = time.perf_counter()
    for _ in range(n):
        oracle.forward_full(model, prompt, last_only=True)
    dt = time.perf_counter() - t0
    desc = (f"float64 NumPy oracle, stateless forward of 1 of {W.batch} prompts ({len(prompt)} tokens), "
            f"{n} time(s)")
    return n * len(prompt) / dt, dt, desc


def reference_prefill_object(W: wl.Workload, n: int):
    rate, dt, desc = oracle_prefill_rate(W, n)
    return {"metric_detail": f"prefill tok/s, {W.batch} x {int(W.lengths()[0])} tokens", "value": rate,
            "unit": "tok/s", "ms_per_step": 1000.0 * dt / n, "steps": n, "dtype": "f64",
            "config": {"workload": W.name, "batch": W.batch, "prompt_len": int(W.lengths()[0])},
            "cpu_baseline": {"value": rate, "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle", "sample": desc},
            "e2e": {"value": rate, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_reference(args, W, PW):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    if W.mode == "prefill" or W.decode_steps == 0:
        n = max(1, min(args.steps, 3))
        obj = reference_prefill_object(W, n)
        line = {"impl": "reference", "metric": METRIC, "n_gpus": args.gpus, "warmup": 0,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "data": "synthetic", **obj}
        print(json.dumps(line), flush=True)
        return 0
    rate, dt, desc = oracle_decode_rate(W, args.steps, args.warmup, n_seq=1)
    line = {"impl": "reference", "metric": METRIC, "metric_detail": f"decode tok/s at batch {W.batch}",
            "value": rate, "unit": "tok/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": W.name, "batch": W.batch, "prompt_len": int(W.lengths()[0]),
                       "decode_steps_cycled": W.decode_steps},
            "cpu_baseline": {"value": rate, "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle", "sample": desc},
            "e2e": {"value": rate, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    if PW is not None:
        line["prefill"] = reference_prefill_object(PW, 1)
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------

def family_roofline(fams: dict, dom: str, steps_profiled: int, ms_step: float, alg_total: float, unit: str,
                    peak: float, peak_source: str, label: str, traffic):
    launches, dom_ms = fams[dom]
    total_ms = sum(v[1] for v in fams.values())
    share = dom_ms / total_ms
    per_step_events = dom_ms / steps_profiled
    if per_step_events <= ms_step:
        per_step, method = per_step_events, "CUDA events around every launch (profiled graph replay)"
    else:
        per_step, method = share * ms_step, "share of the event-timed launches x the timed step"
    assert per_step <= ms_step * (1 + 1e-9), "dominant family's time per step exceeds the step"
    avg_launch_s = per_step * steps_profiled / launches / 1000.0
    per_launch = alg_total / launches
    scale = 1e9 if unit == "GB/s" else 1e12
    achieved = per_launch / avg_launch_s / scale
    return {"bound": "hbm" if unit == "GB/s" else "tensor", "kernel": label, "launches": launches,
            "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak, "traffic": traffic,
            "peak_source": peak_source,
            ("alg_bytes_per_launch" if unit == "GB/s" else "alg_flops_per_launch"): per_launch,
            "avg_launch_us": avg_launch_s * 1e6, "duration_method": method,
            "family_ms_per_step": per_step, "family_share": share,
            "event_ms_per_step": per_step_events}


def decode_part(args, W, world: int, rank: int, local: int) -> dict:
    import torch
    from transformer_decoder_forward_gb300.runner import WorkloadRun

    s = W.model
    kv_elt = 2 if W.kv_dtype == wl.DTYPE_BF16 else 4
    host_w = wl.make_weights(s, scale=W.weight_scale)
    period = W.decode_steps
    run = WorkloadRun(W, host_weights=host_w)
    B = run.B
    stream_np = wl.draw_stream(B, period, s.vocab)
    toks = torch.from_numpy(stream_np).cuda()
    run.prefill()
    torch.cuda.synchronize()

    def step(i):
        run.decode(toks[i % period], i % period)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    launches_per_step = run.dec.last_launch_count()

    # ---- timed region: K graph replays, barrier + synchronize on both sides
    st = run.stream
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id_for_smi(local)) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ev0.record(st)
        for i in range(args.steps):
            step(i)
        ev1.record(st)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    ms, tokens, value = job_rate(ev0.elapsed_time(ev1), B * args.steps, world)
    ms_step = ms / args.steps
    assert run.dec.error_flags() == 0, "device error flags set during the bench"

    # ---- per-kernel durations: the timed steps' positions once more, CUDA events around every launch
    n_prof = min(args.steps, period)
    run.dec.set_profiling(True)
    run.dec.kernel_stats(reset=True)
    for i in range(n_prof):
        step(i)
    stats = run.dec.kernel_stats(reset=True)
    run.dec.set_profiling(False)
    fam, kinds = {}, {}
    for name, (n, t) in stats.items():
        # every projection kernel (CUDA-core GEMV or tcgen05) is one family: they share the
        # weight-stream roofline
        f = "proj" if name.startswith(("gemv", "gemm")) else name
        if f == "proj":
            kinds[name.split("_")[0] + ("_" + name.split("_")[1] if name.startswith("gemm") else "")] = 1
        a = fam.setdefault(f, [0, 0.0])
        a[0] += n
        a[1] += t
    dom = max(fam, key=lambda k: fam[k][1])
    pk, pk_kind = peaks()
    ctx_of = lambda i: run.lengths + (i % period) + 1        # keys read by step i
    if dom == "proj":
        alg = float(gemv_bytes(s, B)) * n_prof
    elif dom == "attn_decode":
        alg = float(sum(attn_bytes(s, ctx_of(i), kv_elt) for i in range(n_prof)))
    else:
        alg = None
    label = dom if dom != "proj" else "proj (" + "+".join(sorted(kinds)) + ")"
    roof = None
    if alg is not None:
        roof = family_roofline(fam, dom, n_prof, ms_step, alg, "GB/s", pk["hbm_gbs"], f"hbm_gbs of {pk_kind}",
                               label, traffic_for(W.name, label) if kv_elt == 4 else None)
    step_alg = float(np.mean([step_bytes(s, ctx_of(i), kv_elt) for i in range(args.steps)]))
    step_gbs = step_alg / (ms_step / 1000.0) / 1e9
    kernel_share = {k: round(v[1] / sum(x[1] for x in fam.values()), 4) for k, v in sorted(fam.items())}

    # ---- end to end through the C ABI with host buffers (H2D inputs, D2H ids, every step)
    n_e2e = min(args.steps, 2 * period)
    tok_h = [np.ascontiguousarray(stream_np[j]) for j in range(period)]
    pos_h = [np.ascontiguousarray((run.lengths + j).astype(np.int32)) for j in range(period)]
    tables_h = None if W.contiguous_kv else np.ascontiguousarray(run.tables_np, dtype=np.int32)
    ids_h = np.zeros(B, np.int32)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        j = i % period
        run.dec.decode_step_host(tok_h[j], pos_h[j], tables_h, ids_h)
    e2e_s = time.perf_counter() - t0
    h2d = B * 4 * 2 + (0 if tables_h is None else tables_h.nbytes)
    e2e = {"value": B * n_e2e / e2e_s * world, "unit": "tok/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": B * 4,
           "steps": n_e2e, "api": "llm_decode_step_host"}
    ctx_lo, ctx_hi = int(run.lengths.min()) + 1, int(run.lengths.max()) + min(args.steps, period)
    line = {"metric": METRIC, "metric_detail": f"decode tok/s at batch {B}", "value": value,
            "unit": "tok/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dtype_label(s), "data": "synthetic",
            "config": {"workload": W.name, "batch": B, "prompt_len": int(run.lengths[0]),
                       "decode_positions": f"{int(run.lengths.min())}..{int(run.lengths.max()) + period - 1} cycled",
                       "context_timed": f"{ctx_lo}..{ctx_hi} keys",
                       "kv": ("contiguous" if W.contiguous_kv else "paged16, shuffled tables")
                       + (", bf16" if kv_elt == 2 else ", fp32"),
                       "precision": WEIGHTS_LABEL[s.dtype]
                       + (", bf16 KV cache" if kv_elt == 2 else ", fp32 KV cache")
                       + ", fp32 residual, fp32 accumulation"
                       + (", activations as bf16 (hi, lo) pairs" if s.dtype == wl.DTYPE_BF16 else ""),
                       "l2": "inputs larger than L2: %.0f MB weights + %.0f MB KV per step" % (
                           weight_bytes(s) / 1e6, attn_bytes(s, ctx_of(0), kv_elt) / 1e6),
                       "graph": "one CUDA graph per step"},
            "roofline": roof,
            "step_roofline": {"alg_bytes_per_step": step_alg, "achieved_gbs": step_gbs,
                              "frac": step_gbs / pk["hbm_gbs"], "peak_source": f"hbm_gbs of {pk_kind}",
                              "positions": "the timed steps' positions"},
            "kernel_share": kernel_share,
            "gpu_launches": launches_per_step * args.steps,
            "launches_per_step": launches_per_step,
            "e2e": e2e,
            "clocks": clk.summary()}
    run.close()
    del run, toks
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_seq, n_steps = CPU_SAMPLE.get(W.name, (1, 4))
        if args.cpu_steps:
            n_steps = args.cpu_steps
        rate, dt, desc = oracle_decode_rate(W, n_steps, 0, n_seq=n_seq, weights=host_w)
        line["cpu_baseline"] = {"value": rate, "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": desc, "seconds": dt}
    return line


def prefill_part(args, W, world: int, rank: int, local: int, steps: int, warmup: int) -> dict:
    """One step = one prefill of the whole batch (every row of the hot path, attention over the
    full causal prompt, K/V written into the paged pool, last-position argmax)."""
    import torch
    from transformer_decoder_forward_gb300.runner import WorkloadRun

    s = W.model
    host_w = wl.make_weights(s, scale=W.weight_scale)
    run = WorkloadRun(W, host_weights=host_w)
    B = run.B
    tokens_total = int(run.lengths.sum())
    for _ in range(warmup):
        run.prefill()
    torch.cuda.synchronize()
    launches_per_step = run.dec.last_launch_count()
    st = run.stream
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id_for_smi(local)) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ev0.record(st)
        for _ in range(steps):
            run.prefill()
        ev1.record(st)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    ms, _, value = job_rate(ev0.elapsed_time(ev1), tokens_total * steps, world)
    ms_step = ms / steps
    assert run.dec.error_flags() == 0, "device error flags set during the bench"
    # per-kernel durations over one more prefill (eager launches, a CUDA event around each)
    run.dec.set_profiling(True)
    run.dec.kernel_stats(reset=True)
    run.prefill()
    stats = run.dec.kernel_stats(reset=True)
    run.dec.set_profiling(False)
    fam = {}
    for name, (n, t) in stats.items():
        f = "gemm_tc" if name.startswith("gemm_tc") else ("proj" if name.startswith(("gemv", "gemm")) else name)
        a = fam.setdefault(f, [0, 0.0])
        a[0] += n
        a[1] += t
    pk, pk_kind = peaks()
    gflops = prefill_gemm_flops(s, run.lengths)
    # the SM-pair kernel (default for prefill) or the one-SM kernel; the stored DRAM traffic
    # belongs to the kernel it was captured on
    pair = any(name.startswith("gemm_tc2") for name in stats)
    label = "gemm_tc2 (tcgen05 projections on SM pairs)" if pair else "gemm_tc (tcgen05 projections)"
    roof = None
    if "gemm_tc" in fam:
        roof = family_roofline(fam, "gemm_tc", 1, ms_step, gflops, "TFLOP/s", pk["bf16_tflops"],
                               f"bf16_tflops (burst) of {pk_kind}", label, traffic_for(W.name, label))
    attn_roof = None
    if "attn_prefill" in fam:
        attn_roof = family_roofline(fam, "attn_prefill", 1, ms_step, prefill_attn_flops(s, run.lengths), "TFLOP/s",
                                    pk["bf16_tflops"], f"bf16_tflops (burst) of {pk_kind}",
                                    "attn_prefill (causal attention, algorithmic flops)", None)
    total = sum(v[1] for v in fam.values())
    kernel_share = {k: round(v[1] / total, 4) for k, v in sorted(fam.items())}
    # end to end: host token ids in, next ids out, through the C ABI
    tok_h = torch.from_numpy(np.concatenate(run.prompts).astype(np.int32)).pin_memory()
    ids_h = torch.zeros(B, dtype=torch.int32).pin_memory()
    n_e2e = max(1, min(steps, 10))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        with torch.cuda.stream(st):
            run.tokens.copy_(tok_h, non_blocking=True)
            run.dec.prefill(run.tokens, [int(x) for x in run.lengths], run.tables, run.next_ids)
            ids_h.copy_(run.next_ids, non_blocking=True)
        st.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e = {"value": tokens_total * n_e2e / e2e_s * world, "unit": "tok/s", "h2d_bytes_per_step": int(tok_h.numel() * 4),
           "d2h_bytes_per_step": B * 4, "steps": n_e2e, "api": "llm_prefill (pinned host ids in, ids out)"}
    line = {"metric": METRIC, "metric_detail": f"prefill tok/s, {B} x {int(run.lengths[0])} tokens",
            "value": value, "unit": "tok/s", "n_gpus": world, "steps": steps, "warmup": warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dtype_label(s), "data": "synthetic",
            "config": {"workload": W.name, "batch": B, "prompt_len": int(run.lengths[0]),
                       "kv": "paged16, " + ("bf16" if W.kv_dtype == wl.DTYPE_BF16 else "fp32"),
                       "l2": "inputs larger than L2: %.0f MB activations per step" % (tokens_total * s.d_model * 4 / 1e6)},
            "roofline": roof,
            "attention_roofline": attn_roof,
            "attention_flops_per_step": prefill_attn_flops(s, run.lengths),
            "gemm_flops_per_step": gflops,
            "kernel_share": kernel_share, "gpu_launches": launches_per_step * steps,
            "launches_per_step": launches_per_step, "e2e": e2e, "clocks": clk.summary()}
    run.close()
    del run
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, dt, desc = oracle_prefill_rate(W, 1, weights=host_w)
        line["cpu_baseline"] = {"value": rate, "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": desc, "seconds": dt}
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=wl.W_GPT2XL_B256.name, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--prefill-workload", default=wl.W_GPT2_BF16_PREFILL.name,
                    choices=sorted(n for n, w in wl.WORKLOADS.items() if w.mode == "prefill") + ["none"],
                    help="prefill workload reported in the decode line's 'prefill' object")
    ap.add_argument("--prefill-steps", type=int, default=20, help="timed prefills of the prefill object (0: none)")
    ap.add_argument("--cpu-steps", type=int, default=0, help="oracle decode steps of the CPU sample (0: per workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv-dtype", default="f32", choices=["f32", "bf16"], help="element type of the KV cache")
    args = ap.parse_args()
    if args.warmup < 3:
        # the timing rules' minimum; the JSON line reports the count actually run
        print(f"bench: --warmup {args.warmup} raised to 3", file=sys.stderr)
        args.warmup = 3
    W = wl.WORKLOADS[args.workload]
    if args.kv_dtype == "bf16":
        from dataclasses import replace
        W = replace(W, kv_dtype=wl.DTYPE_BF16)
    is_prefill = W.mode == "prefill" or W.decode_steps == 0
    PW = None if (is_prefill or args.prefill_workload == "none") else wl.WORKLOADS[args.prefill_workload]
    if args.impl == "reference":
        return run_reference(args, W, PW)

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    if is_prefill:
        line = prefill_part(args, W, world, rank, local, args.steps, args.warmup)
    else:
        line = decode_part(args, W, world, rank, local)
        if PW is not None and args.prefill_steps > 0:   # --prefill-steps 0: decode only
            line["prefill"] = prefill_part(args, PW, world, rank, local, args.prefill_steps, max(3, args.warmup))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
