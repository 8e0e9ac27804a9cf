#!/usr/bin/env python
"""Benchmark of the routed-expert forward of a Kimi K2 MoE block on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload k2_decode] [--impl ours|reference]

One step = one pass of the whole path on one batch of synthetic input:
routing plan (histogram + stable permutation), sorted-row gather, gate/up
grouped GEMM with SwiGLU, down grouped GEMM with router weighting and
scatter, ordered combine (plus RMSNorm, shared expert and residual for the
full-block workload).  Inputs and all 384 experts' FP8 weights are resident
in HBM before the timed region; the touched weights of one step (>= 4.8 GB)
are far larger than L2, so no flush is needed.

Multi-GPU: the path is data-parallel over tokens (replicated weights, no
exchange), so each rank runs its own batch (weak scaling) and the job value is
all ranks' tokens / the slowest rank's time.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "K2 MoE-layer tokens/s; % of HBM (decode) / FP8 tensor (prefill) roofline"


def _peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        return None


def _hbm_peak():
    p = _peaks()
    if p and p.get("hbm_gbs"):
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _bf16_peak(sustained):
    p = _peaks()
    if p:
        k = "bf16_tflops_sustained" if sustained else "bf16_tflops"
        if p.get(k):
            return float(p[k]), "measured"
    return (1700.0 if sustained else 1900.0), "fallback"


# dense e4m3 / bf16 tensor throughput of the part (4.5 / 2.25 PFLOP/s nominal); f16 runs at the bf16 rate
FP8_PER_BF16 = 2.0

# what the tensor cores compute in, per activation scheme and tile width
DTYPE_EXACT = "e4m3 weights x e4m3 split-term activations (exact scheme, 16-token tiles), fp32 accumulation"
DTYPE_EXACT_WIDE = ("f16 x f16: e4m3 weights widened on chip with their block scale folded in, f16 activations "
                    "with a power-of-two factor per row (exact scheme, 128-token tiles), fp32 accumulation")
DTYPE_FP8 = "e4m3 weights x e4m3 dynamic activations (amax/448 per 128), fp32 accumulation"


def wide_tiles(n_tokens, top_k, num_experts):
    """The library's tile width rule: 128-token tiles once the batch averages 24 or more rows per expert."""
    return n_tokens * top_k >= 24 * num_experts


def kernel_roofline(kernel, alg_bytes, alg_flops, ms, hbm_gbs, hbm_src, tensor_tflops, tensor_src, traffic):
    """A kernel's algorithmic work against the roof that bounds it: HBM when its bytes take longer at the
    copy bandwidth than its flops at the tensor peak of its MMAs' operand type, else the tensor cores.
    `achieved` is algorithmic bytes (or flops) over the measured duration."""
    t_hbm = alg_bytes / (hbm_gbs * 1e9)
    t_tensor = alg_flops / (tensor_tflops * 1e12)
    r = {"kernel": kernel, "alg_bytes_per_launch": alg_bytes, "alg_flops_per_launch": alg_flops, "kernel_ms": ms,
         "traffic": traffic, "t_roof_ms": max(t_hbm, t_tensor) * 1e3}
    if t_tensor > t_hbm:
        achieved = alg_flops / (ms / 1e3) / 1e12 if ms else None
        r.update(bound="tensor", achieved=achieved, peak=tensor_tflops, unit="TFLOP/s", peak_source=tensor_src)
    else:
        achieved = alg_bytes / (ms / 1e3) / 1e9 if ms else None
        r.update(bound="hbm", achieved=achieved, peak=hbm_gbs, unit="GB/s", peak_source=hbm_src)
    r["frac"] = achieved / r["peak"] if achieved else None
    return r


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _traffic(workload, kernel, fp8=False):
    """DRAM bytes per launch from the committed ncu summary of this workload and activation scheme,
    or None when there is none or the kernel's source file has changed since its counters were taken."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", f"traffic_{workload}{'_fp8' if fp8 else ''}.json")
    try:
        rec = json.load(open(prof))
        src = os.path.join(ROOT, "mixture_experts_ffn_infer_gb300", "csrc", rec["source"])
        if rec.get("source_sha256") != hashlib.sha256(open(src, "rb").read()).hexdigest():
            return None
        return rec.get(kernel)
    except (OSError, ValueError, KeyError):
        return None


# ---------------------------------------------------------------------------- algorithmic cost

def algorithmic(wl, ids_list, n_tokens):
    """Bytes and flops one step must move / do (touched experts only; intermediates excluded)."""
    import torch
    d, dff = wl.d, wl.d_ff
    per_proj = d * dff + (d // 128) * (dff // 128) * 4          # e4m3 codes + fp32 block scales
    touched = sum(int(torch.unique(ids).numel()) for ids in ids_list)
    R = n_tokens * wl.top_k
    gateup_bytes = touched * 2 * per_proj + R * d * 2 + R * dff * 2   # weights + sorted rows in + h out
    down_bytes = touched * per_proj + R * dff * 2 + R * d * 2           # weights + h in + weighted rows out
    gateup_flops = 4 * d * dff * R                                      # gate and up: 2 flops per product
    down_flops = 2 * d * dff * R
    step_bytes = touched * 3 * per_proj + n_tokens * d * 2 * (2 if not wl.full_block else 3) + n_tokens * 8 * wl.top_k
    flops = 6 * d * dff * R
    if wl.full_block:
        step_bytes += 3 * (d * wl.d_ff_shared + (d // 128) * (wl.d_ff_shared // 128) * 4)
        flops += 6 * d * wl.d_ff_shared * n_tokens
    return {"touched_experts": touched, "gateup_bytes": gateup_bytes, "down_bytes": down_bytes,
            "gateup_flops": gateup_flops, "down_flops": down_flops, "step_bytes": step_bytes, "step_flops": flops}


# ---------------------------------------------------------------------------- multi-rank host logic

def rank_workload(wl, rank):
    """Each rank draws its own batch (weak scaling): the seed moves by 1000 per rank; the
    expert bank (bank_seed) is the same on every rank."""
    from mixture_experts_ffn_infer_gb300 import synthetic as syn
    return syn.Workload(**{**wl.__dict__, "seed": wl.seed + 1000 * rank,
                           "bank_seed": syn.bank_seed_of(wl)})


def max_over_ranks(value, world, device="cpu"):
    """The slowest rank's time: all-reduce MAX (no-op on one rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, steps, ms_total_max):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world * steps / (ms_total_max / 1e3)


# ---------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import torch

    import mixture_experts_ffn_infer_gb300 as mx
    from mixture_experts_ffn_infer_gb300 import synthetic as syn

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = syn.WORKLOADS[args.workload]
    if args.num_experts:
        wl = syn.Workload(**{**wl.__dict__, "num_experts": args.num_experts})
    if args.n_tokens:
        wl = syn.Workload(**{**wl.__dict__, "n_tokens": args.n_tokens})
    mx.load_library()
    # all 384 experts' weights resident in HBM, prepared once at load time into the tiled streaming layout;
    # the row-major bank stays for the CPU baseline, which reads the model's layout
    bank = syn.expert_bank(wl.num_experts, wl.d, wl.d_ff, syn.bank_seed_of(wl), dev)
    bank_t = mx.pack_bank(bank)
    torch.cuda.synchronize(dev)
    result = measure(args, wl, args.workload, bank, bank_t, rank, world, local_rank, dev)
    # the default run also measures the prefill batch on the same resident bank: the metric names both
    # the decode (HBM) and the prefill roofline
    pre = syn.WORKLOADS["k2_prefill"]
    if (args.workload == "k2_decode" and not args.no_prefill and not args.num_experts and not args.n_tokens
            and syn.bank_seed_of(pre) == syn.bank_seed_of(wl)):
        result["prefill"] = measure(args, pre, "k2_prefill", bank, bank_t, rank, world, local_rank, dev)
    return result


L2_BYTES = 129e6  # GB300 L2


def run_config(wl, wl_name, n, fp8, alg, world):
    """The workload a line measures; both arms report it alike."""
    return {"workload": wl_name, "n_tokens_per_gpu": n, "d": wl.d, "d_ff": wl.d_ff,
            "num_experts": wl.num_experts, "top_k": wl.top_k, "routing": wl.routing,
            "full_block": wl.full_block, "weights": "e4m3, fp32 scale per 128x128 block, tiled layout",
            "act_scheme": "fp8_dynamic" if fp8 else "exact",
            "touched_experts": alg["touched_experts"],
            "l2": ("inputs larger than L2: %.2f GB of touched expert weights per step" if alg["step_bytes"] > L2_BYTES
                   else "inputs fit in L2 (%.3f GB per step): no flush between steps, a latency figure") % (
                       alg["step_bytes"] / 1e9),
            "parallelism": f"replicas{world}" if world > 1 else "single"}


def measure(args, wl, wl_name, bank, bank_t, rank, world, local_rank, dev):
    """One workload: W warm-up steps, K untimed-event steps timed as a whole (the headline), then a
    separate sample of steps with events around the GEMMs (per-kernel times), the host-buffer end-to-end
    leg and the CPU oracle baseline."""
    import torch
    import torch.distributed as dist

    import mixture_experts_ffn_infer_gb300 as mx
    from mixture_experts_ffn_infer_gb300 import synthetic as syn

    # each rank its own batch (seed offset by rank), the same resident weights
    rank_wl = rank_workload(wl, rank)
    x, ids, w, gain = syn.make_host_inputs(rank_wl)
    shared = syn.expert_bank(1, wl.d, wl.d_ff_shared, wl.seed + 1_000_003, dev) if wl.full_block else None
    n = x.shape[0]
    xd, idsd, wd = x.to(dev), ids.to(dev), w.to(dev)
    gaind = gain.to(dev) if gain is not None else None
    fp8 = args.act == "fp8"
    dm = mx.dims(wl.d, wl.d_ff, wl.num_experts, wl.top_k, mx.MOE_ACT_FP8_DYNAMIC if fp8 else mx.MOE_ACT_EXACT)
    dff_sh = wl.d_ff_shared if wl.full_block else 0
    ws = mx.workspace(dm, n, dff_sh, dev)
    out = torch.empty(n, wl.d, dtype=torch.bfloat16, device=dev)
    shared_t = mx.pack_bank(shared) if shared is not None else None
    torch.cuda.synchronize(dev)
    W = mx.weights(bank_t)
    WS = mx.weights(shared_t) if shared_t is not None else None
    stream = torch.cuda.current_stream(dev)

    def step(trace=None, xin=xd, idin=idsd, win=wd, o=out):
        if wl.full_block:
            mx.moe_layer_forward(dm, n, xin, gaind, 1e-6, idin, win, W, WS, dff_sh, o, ws, stream=stream,
                                 trace=trace)
        else:
            mx.moe_infer(dm, n, xin, idin, win, W, o, ws, stream=stream, trace=trace)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = mx.moe_get_error(ws, stream)
    if st != mx.MOE_OK:
        raise RuntimeError(f"device error after warm-up: {mx.STATUS.get(st)}")

    # The headline: K steps as a caller runs them, no events between kernels.  A trace without events
    # only counts the kernels each call launched.
    counters = [mx.moe_trace() for _ in range(args.steps)]
    for t in counters:
        t.n_events = 0
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        step(counters[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1), world, dev)
    launches = sum(t.n_launched for t in counters)

    # Per-kernel durations: a separate sample of steps, each with events on the launching stream just before
    # the first grouped GEMM and after each (an event between two kernels costs the stream about a launch
    # gap, so these steps stay out of the headline).
    n_traced = min(args.steps, 30)
    n_ev = 12
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(n_traced)]
    traces = []
    for k in range(n_traced):
        t = mx.moe_trace()
        for i, e in enumerate(evs[k]):
            e.record(stream)  # materialise the event handle
            t.events[i] = e.cuda_event
        t.n_events = n_ev
        t.gemms_only = 1
        traces.append(t)
    torch.cuda.synchronize(dev)
    for k in range(n_traced):
        step(traces[k])
    torch.cuda.synchronize(dev)
    per_kernel = {}
    for k in range(n_traced):
        t = traces[k]
        for i in range(t.n_recorded - 1):
            per_kernel.setdefault(t.labels[i].decode(), []).append(evs[k][i].elapsed_time(evs[k][i + 1]))
    kern_ms = {k: statistics.mean(v) for k, v in per_kernel.items()}

    # end to end through the same C ABI with host buffers: every step copies its inputs from pinned
    # host memory and reads its result back, all inside the timed region.  As a serving loop would,
    # uploads and downloads run on streams of their own with two buffer sets, so step i + 1's upload
    # and step i - 1's download overlap step i's compute (and each other).
    xh, idh, wh = x.pin_memory(), ids.pin_memory(), w.pin_memory()
    oh = torch.empty(n, wl.d, dtype=torch.bfloat16).pin_memory()
    sets = [(torch.empty_like(xd), torch.empty_like(idsd), torch.empty_like(wd), torch.empty_like(out))
            for _ in range(2)]
    up_stream, down_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    downloaded = [torch.cuda.Event() for _ in range(2)]

    def upload(b):
        xe, ide, we, _ = sets[b]
        with torch.cuda.stream(up_stream):
            xe.copy_(xh, non_blocking=True)
            ide.copy_(idh, non_blocking=True)
            we.copy_(wh, non_blocking=True)
            uploaded[b].record(up_stream)

    def e2e_run(steps):
        up_stream.wait_stream(stream)
        down_stream.wait_stream(stream)
        upload(0)
        for i in range(steps):
            b = i % 2
            stream.wait_event(uploaded[b])
            if i >= 2:
                stream.wait_event(downloaded[b])      # step i - 2's result has left this set
            step(None, *sets[b])
            computed[b].record(stream)
            if i + 1 < steps:
                up_stream.wait_event(computed[1 - b])   # step i - 1 is done with the other set's inputs
                upload(1 - b)
            down_stream.wait_event(computed[b])
            with torch.cuda.stream(down_stream):
                oh.copy_(sets[b][3], non_blocking=True)
                downloaded[b].record(down_stream)
        stream.wait_stream(up_stream)
        stream.wait_stream(down_stream)

    e2e_ms = float("nan")
    if not args.no_e2e:
        e2e_run(args.warmup)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(args.steps)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    st = mx.moe_get_error(ws, stream)
    if st != mx.MOE_OK:
        raise RuntimeError(f"device error in the timed region: {mx.STATUS.get(st)}")

    alg = algorithmic(wl, [ids], n)
    ms_step = ms_total / args.steps
    tokens = n * world
    value = job_tokens_per_s(n, world, args.steps, ms_total)
    hbm, hbm_src = _hbm_peak()
    dominant = "gateup_swiglu"
    step_roof_ms = alg["step_bytes"] / (hbm * 1e9) * 1e3
    bf16, bf16_src = _bf16_peak(sustained=True)
    # kernels timed inside a long step: the sustained tensor peak of their MMAs' operand type
    e4m3_peak = bf16 * FP8_PER_BF16
    f16_mma = not fp8 and wide_tiles(n, wl.top_k, wl.num_experts)
    if f16_mma:
        tensor_peak, tensor_src = bf16, f"{bf16_src} bf16_tflops_sustained (f16 operands, the bf16 rate)"
    else:
        tensor_peak = e4m3_peak
        tensor_src = (f"{bf16_src} bf16_tflops_sustained x {FP8_PER_BF16:g} (e4m3 operands: nominal e4m3 / bf16 "
                      "dense ratio)")
    hbm_label = hbm_src + " (MEASURED_PEAKS.json hbm_gbs)" if hbm_src == "measured" else hbm_src
    tflops = alg["step_flops"] / (ms_step / 1e3) / 1e12
    traffic = _traffic(wl_name, dominant, fp8)
    result = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": DTYPE_FP8 if fp8 else (DTYPE_EXACT_WIDE if f16_mma else DTYPE_EXACT),
        "data": "synthetic",
        "config": run_config(wl, wl_name, n, fp8, alg, world),
        "roofline": kernel_roofline(dominant, alg["gateup_bytes"], alg["gateup_flops"], kern_ms.get(dominant),
                                    hbm, hbm_label, tensor_peak, tensor_src, traffic),
        "down_roofline": kernel_roofline("down_scatter", alg["down_bytes"], alg["down_flops"],
                                         kern_ms.get("down_scatter"), hbm, hbm_label, tensor_peak, tensor_src,
                                         _traffic(wl_name, "down_scatter", fp8)),
        "step_roofline": {"bytes": alg["step_bytes"], "flops": alg["step_flops"], "t_roof_ms_hbm": step_roof_ms,
                          "frac_hbm": step_roof_ms / ms_step, "tflops": tflops,
                          "frac_bf16_sustained": tflops / bf16,
                          "frac_e4m3_sustained": tflops / e4m3_peak, "bf16_peak_source": bf16_src},
        "kernel_ms": kern_ms,
        "kernel_ms_steps": n_traced,   # separate steps with events around the GEMMs, after the timed region
        "e2e": None if args.no_e2e else {"value": tokens * args.steps / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(x.numel() * 2 + ids.numel() * 4 + w.numel() * 4),
                "d2h_bytes_per_step": int(n * wl.d * 2), "ms_per_step": e2e_ms / args.steps,
                "copies": "pinned host buffers; uploads and downloads on streams of their own, overlapping "
                          "the neighbouring steps' compute and each other (two buffer sets)"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, x, ids, w, gain, bank, shared, budget_s=args.cpu_budget,
                                              fp8=fp8)
    del ws, shared_t
    return result


def _oracle_rate(wl, x, ids, w, gain, bank, shared, n_tok, budget_s, fp8=False):
    """Time the oracle on a token sample; returns (tokens/s, tokens, seconds, threads)."""
    import oracle
    import torch
    tokens = [i % x.shape[0] for i in range(n_tok)]
    used = torch.unique(ids[tokens]).tolist()
    bank_h = _HostBank(bank, used)          # experts the sample touches, copied to host before timing
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    if wl.full_block:
        oracle.layer_forward(x, gain, 1e-6, ids, w, bank_h, _HostBank(shared, [0]), tokens=tokens, threads=threads,
                             fp8_act=fp8)
    else:
        oracle.moe_infer(x, ids, w, bank_h, tokens=tokens, threads=threads, fp8_act=fp8)
    dt = time.perf_counter() - t0
    return n_tok / dt, n_tok, dt, threads


class _HostBank:
    """Host copies of the listed experts, indexable like the device bank (others absent)."""

    def __init__(self, bank, experts):
        for nm in ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down"):
            full = getattr(bank, nm)
            setattr(self, nm, _Sparse(full, experts))


class _Sparse:
    def __init__(self, full, experts):
        self.shape = tuple(full.shape)
        self.rows = {int(e): full[int(e)].to("cpu") for e in experts}

    def __getitem__(self, e):
        return self.rows[int(e)]


def cpu_baseline(wl, x, ids, w, gain, bank, shared, budget_s=20.0, fp8=False):
    # sample: the first tokens of the batch; one probe token sizes the sample to the budget
    rate1, _, dt1, threads = _oracle_rate(wl, x, ids, w, gain, bank, shared, 1, budget_s, fp8)
    n_tok = max(1, min(4096, int(budget_s / max(dt1, 1e-3) * max(1, threads))))
    rate, n_tok, dt, threads = _oracle_rate(wl, x, ids, w, gain, bank, shared, n_tok, budget_s, fp8)
    return {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_tok} token evaluations cycling over the {x.shape[0]}-token {wl.name} batch "
                      f"(fp64 C oracle, one thread per token), {dt:.1f} s"}


# ---------------------------------------------------------------------------- reference arm (CPU oracle)

def run_reference(args):
    import torch

    from mixture_experts_ffn_infer_gb300 import synthetic as syn
    wl = syn.WORKLOADS[args.workload]
    x, ids, w, gain = syn.make_host_inputs(wl)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    bank = syn.expert_bank(wl.num_experts, wl.d, wl.d_ff, syn.bank_seed_of(wl), dev)
    shared = syn.expert_bank(1, wl.d, wl.d_ff_shared, wl.seed + 1_000_003, dev) if wl.full_block else None
    import oracle
    threads = oracle.default_threads()
    per_step = max(1, min(x.shape[0], args.ref_tokens_per_step))
    times = []
    for s in range(args.warmup + args.steps):
        lo = (s * per_step) % x.shape[0]
        tok = [(lo + i) % x.shape[0] for i in range(per_step)]
        used = torch.unique(ids[tok]).tolist()
        hb = _HostBank(bank, used)
        t0 = time.perf_counter()
        fp8 = args.act == "fp8"
        if wl.full_block:
            oracle.layer_forward(x, gain, 1e-6, ids, w, hb, _HostBank(shared, [0]), tokens=tok, threads=threads,
                                 fp8_act=fp8)
        else:
            oracle.moe_infer(x, ids, w, hb, tokens=tok, threads=threads, fp8_act=fp8)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = per_step * len(times) / total
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total / len(times) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": run_config(wl, args.workload, x.shape[0], args.act == "fp8", algorithmic(wl, [ids], x.shape[0]),
                             int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{per_step} tokens of the {wl.name} batch per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="k2_decode",
                    choices=["tiny", "k2_decode", "k2_prefill", "k2_skewed", "k2_block"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-tokens-per-step", type=int, default=2)
    ap.add_argument("--num-experts", type=int, default=0,
                    help="override E (a smaller bank for profiling captures; routing redrawn over E)")
    ap.add_argument("--n-tokens", type=int, default=0,
                    help="override N (with --num-experts: a small case of the same rows per expert)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-prefill", action="store_true",
                    help="default decode run only: skip the prefill sub-record")
    ap.add_argument("--act", default="exact", choices=["exact", "fp8"],
                    help="activation scheme: exact split terms (default) or dynamic FP8 (per-128 e4m3, amax/448)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
