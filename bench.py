#!/usr/bin/env python
"""Benchmark of the routed-expert hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the whole hot path over one batch: forward with saved
activations (dispatch, gather, W13 GEMM + SwiGLU, W2 GEMM x score, combine) and
backward (dY gather, DGRAD-W2 + SwiGLU backward, DGRAD-W13, dX/dscores combine,
WGRAD-W2, WGRAD-W13) of the training workload T=8192, d=2048, I=768, E=128,
k=8 with uniform routing, on synthetic seeded inputs (moe_inputs).

Throughput is routed-expert TFLOP/s counted as 18*T*k*d*I per forward+backward
(6*T*k*d*I forward), the whole job over all ranks.  Under torchrun each rank
runs an independent replica on its own GPU and its own batch (weak scaling; the
only collectives are the barrier and the max over ranks of the timed region).

--impl reference times the CPU oracle (on all host cores) on a bounded sample of
the same workload: it is the reference arm of this benchmark.

Prints ONE JSON line on rank 0.
"""

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "routed-expert TFLOP/s (fwd; fwd+bwd) at T=8192 E=128 k=8; % of GB300 tensor peak"
WORKLOAD = "train_e128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0    # nominal dense E4M3 / bf16 tensor throughput ratio (4.5 / 2.25 PFLOP/s)
FP4_OVER_BF16 = 6.0    # nominal dense E2M1 / bf16 tensor throughput ratio (13.5 / 2.25 PFLOP/s)
WGRAD_SMS = 0          # default split of the backward (set from measurements)
NOMINAL_HBM_GBS = 8000.0   # nominal HBM3e bandwidth of the part (~8 TB/s), beside the measured copy rate

FWD_STAGES = ["dispatch", "gather_x", "w13_swiglu", "w2_score", "combine_y"]
BWD_STAGES = ["gather_dy", "dgrad_w2_swiglu", "dgrad_w13", "combine_dx", "wgrad_w2", "wgrad_w13"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--mx-steps", type=int, default=50,
                    help="timed MXFP8 forward steps on the same inputs (0: skip)")
    ap.add_argument("--fwd-steps", type=int, default=50,
                    help="timed bf16 forward steps that save nothing (inference; 0: skip)")
    # smaller cases of the same workload (profiling captures); defaults = the full workload
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--E", type=int, default=None)
    ap.add_argument("--graph", action="store_true",
                    help="time the steps as one CUDA graph replay (stage events as graph nodes)")
    ap.add_argument("--cta-pairs", action="store_true",
                    help="W13, W2 and DGRAD-W13 on CTA pairs (moe_plan_set_cta_pairs)")
    ap.add_argument("--wgrad-sms", type=int, default=WGRAD_SMS,
                    help="SMs of the weight-gradient GEMMs running beside DGRAD-W13 in the "
                         "backward (moe_plan_set_backward_split; 0: one stream)")
    ap.add_argument("--dp-allreduce", action="store_true",
                    help="with --gpus N > 1: sum the weight gradients over the ranks after "
                         "every backward (one data-parallel training step instead of N "
                         "independent replicas)")
    ap.add_argument("--extra-workloads", default="infer_e16,skew_pad",
                    help="comma list of the other workloads to time (infer_e16, skew_pad)")
    ap.add_argument("--extra-steps", type=int, default=30,
                    help="timed steps of the inference (E=16) and skewed-routing workloads "
                         "(0: skip)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# algorithmic work per stage (routed rows R = T*k; padding rows not counted)


def stage_model(c, n_nonempty=None):
    """n_nonempty: experts with routed rows (default E); the weight-gradient
    read-modify-write touches only theirs."""
    T, d, I, E, k = c["T"], c["d"], c["I"], c["E"], c["k"]
    R = T * k
    Ew = E if n_nonempty is None else n_nonempty
    return {
        # bound, algorithmic flops, algorithmic bytes
        "dispatch": ("hbm", 0, 8 * R + 4 * R * 3),
        "gather_x": ("hbm", 0, 2 * T * d + 2 * R * d),
        "w13_swiglu": ("tensor", 4 * R * d * I, 2 * R * d + E * 2 * I * d * 2 + 2 * R * I + 4 * R * I),
        "w2_score": ("tensor", 2 * R * d * I, 2 * R * I + E * d * I * 2 + 2 * R * d),
        "combine_y": ("hbm", 0, 2 * R * d + 2 * T * d + 4 * T * k),
        "gather_dy": ("hbm", 0, 2 * T * d + 2 * R * d),
        # dY, W2, a (h is recomputed from a, not read), dA and hs written
        "dgrad_w2_swiglu": ("hbm", 2 * R * d * I, 2 * R * d + E * d * I * 2 + 4 * R * I
                            + 4 * R * I + 2 * R * I),
        "dgrad_w13": ("tensor", 4 * R * d * I, 4 * R * I + E * 2 * I * d * 2 + 2 * R * d),
        "combine_dx": ("hbm", 0, 2 * R * d + 2 * T * d + 8 * T * k),
        "wgrad_w2": ("hbm", 2 * R * d * I, 2 * R * d + 2 * R * I + 8 * Ew * d * I),
        "wgrad_w13": ("hbm", 4 * R * d * I, 4 * R * I + 2 * R * d + 8 * Ew * 2 * I * d),
    }


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            m = json.load(f)
        return {k: float(m[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak(pk, clk):
    """bf16 tensor peak for kernels timed here: the burst figure while the clock
    record shows no power capping, the sustained (power-capped) one otherwise."""
    capped = clk is None or "sw_power_cap" in (clk.get("reasons") or [])
    if capped:
        return pk["bf16_tflops_sustained"], "sustained bf16 (%s)" % (
            "power cap active" if clk else "no clock record")
    return pk["bf16_tflops"], "burst bf16 (no power cap in the clock record)"


def stage_table(model, stage_ms, tpeak, hbm_peak):
    """Per stage: time, roofline bound, achieved rate and fraction of its peak
    (and, for HBM-bound stages, of the nominal HBM bandwidth)."""
    out = {}
    for name, t_ms in stage_ms.items():
        bound, fl, by = model[name]
        if bound == "tensor":
            ach, peak, unit = fl / (t_ms * 1e-3) / 1e12, tpeak, "TFLOP/s"
        else:
            ach, peak, unit = by / (t_ms * 1e-3) / 1e9, hbm_peak, "GB/s"
        ent = {"ms": round(t_ms, 5), "bound": bound, "achieved": round(ach, 1), "peak": peak,
               "unit": unit, "frac": round(ach / peak, 4),
               "tflops": round(fl / (t_ms * 1e-3) / 1e12, 1) if fl else None}
        if bound == "hbm":
            ent["frac_nominal_hbm"] = round(ach / NOMINAL_HBM_GBS, 4)
        out[name] = ent
    return out


_TOKEN = re.compile(r'"(?:\\.|[^"\\])*"' r"|'(?:\\.|[^'\\])*'" r"|//[^\n]*|/\*.*?\*/", re.S)


def _code_only(src):
    """C/C++ source without its comments and blank space: what the compiler sees
    (string and character literals are kept as they are)."""
    out = _TOKEN.sub(lambda m: " " if m.group(0)[0] == "/" else m.group(0), src)
    return " ".join(out.split())


def kernel_source_hash():
    """Hash of the CUDA sources' code (comments and layout excluded), so that a
    committed counter taken on the same kernels stays valid across comment edits."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "routed_mixture_experts_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_for(stage):
    """DRAM bytes per launch of `stage` from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == stage:
                return float(parts[1]) if parts[2] == cur else None
    return None


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        if not sm:
            return None
        mx = max(float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed helpers (timing only; no data-path collective)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, device=None):
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def allreduce_grads(tensors):
    """Data-parallel split of the training step: after the backward each rank holds
    the weight-gradient increments of its own tokens; summing the fp32 gradient
    buffers over the ranks gives every rank the step's full gradient.  Works on
    any backend (NCCL for device tensors, gloo for CPU tensors); a no-op on one
    rank."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return
    for t in tensors:
        dist.all_reduce(t, op=dist.ReduceOp.SUM)


# ---------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)


def oracle_sample(inp, n_tokens, seconds, max_experts=None, threads=0):
    """Time the oracle on forward+backward (with weight gradients) of the routed
    rows of experts 0, 1, ... among the first n_tokens tokens, until `seconds`
    have passed, on `threads` host threads (0: all cores).  Returns (flops,
    seconds, experts, threads used)."""
    from oracle import load_oracle

    orc = load_oracle("float")
    n_all = orc.threads() if not hasattr(oracle_sample, "n_all") else oracle_sample.n_all
    oracle_sample.n_all = n_all
    used = orc.set_threads(threads if threads > 0 else n_all)
    c = inp["cfg"]
    sub = {k: inp[k][:n_tokens].copy() for k in ("x", "ids", "scores", "dy")}
    flops = 0.0
    t0 = time.perf_counter()
    e = 0
    while True:
        _, _, rows = orc.wgrad_expert(sub["x"], sub["ids"], sub["scores"], inp["w13"], inp["w2"],
                                      sub["dy"], e % c["E"], clamp=c["clamp"])
        flops += 18.0 * c["d"] * c["I"] * rows
        e += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_experts and e >= max_experts):
            orc.set_threads(n_all)
            return flops, el, e, used


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import moe_inputs as mi

    inp = mi.make_inputs(WORKLOAD, seed=args.seed,
                         need=("x", "ids", "scores", "w13", "w2", "dy"))
    c = inp["cfg"]
    n_tok = 1024
    # warm-up samples, then K timed samples (one expert's rows per step)
    oracle_sample(inp, n_tok, 0.0, max_experts=max(args.warmup, 1))
    flops, el, ne, cores = oracle_sample(inp, n_tok, 1e9, max_experts=args.steps)
    value = flops / el / 1e12
    sample = ("per step: forward+backward incl. weight gradients of the routed rows of one expert "
              "among tokens 0..%d (%d steps, %.1f GFLOP, %.1f s, %d host threads)"
              % (n_tok - 1, ne, flops / 1e9, el, cores))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / ne * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "%s (T=%d, d=%d, I=%d, E=%d, k=%d, uniform routing, forward+backward)"
                   % (WORKLOAD, c["T"], c["d"], c["I"], c["E"], c["k"])},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm


def run_ours(args):
    import numpy as np
    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from routed_mixture_experts_gb300 import build as _build

    _build.build()
    import moe_inputs as mi
    import routed_mixture_experts_gb300 as moe

    need = ("x", "ids", "scores", "w13", "w2", "dy", "dw13", "dw2")
    over = {key: v for key, v in (("T", args.T), ("E", args.E)) if v is not None}
    inp = mi.make_inputs(WORKLOAD, seed=args.seed + rank, need=need, **over)
    c = inp["cfg"]
    T, d, I, E, k = c["T"], c["d"], c["I"], c["E"], c["k"]

    def to_dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.to(dev)

    D = {key: to_dev(inp[key]) for key in need}
    plan = moe.MoePlan(T, d, I, E, k, clamp=c["clamp"],
                       flags=moe.MOE_WS_TRAINING | moe.MOE_WS_HOST_STAGING, device=dev,
                       cta_pairs=args.cta_pairs)
    if args.wgrad_sms:
        plan.set_backward_split(args.wgrad_sms)
    y = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    dx = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    dsc = torch.empty(T, k, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    dp = args.dp_allreduce and ws > 1

    def step():
        plan.forward(D["x"], D["ids"], D["scores"], D["w13"], D["w2"], y=y, save=True)
        plan.backward(D["dy"], D["w13"], D["w2"], D["dw13"], D["dw2"], dx=dx, dscores=dsc)
        if dp:
            allreduce_grads((D["dw13"], D["dw2"]))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    rc, det = plan.check()
    if rc != 0:
        raise RuntimeError("device error %d (%d) during warm-up" % (rc, det))

    # stage breakdown: a separate pass with an event at every stage boundary (an
    # event between two kernels keeps the second from being scheduled before the
    # first ends, so the timed loop below records only the dominant stage's two)
    K = args.steps
    KB = min(K, 50)
    evf = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(KB)]
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(KB)]
    for ev in [e for s_ in evf + evb for e in s_]:
        ev.record(stream)                       # materialise the handles
    # (one kernel at a time here, so that every stage has its own time)
    plan.set_backward_split(0)
    for i in range(KB):
        plan.set_timing_events(0, evf[i])
        plan.set_timing_events(1, evb[i])
        step()
    torch.cuda.synchronize()
    plan.set_timing_events(0, None)
    plan.set_timing_events(1, None)
    plan.set_backward_split(args.wgrad_sms)
    stage_ms = {}
    for j, name in enumerate(FWD_STAGES):
        stage_ms[name] = sum(evf[i][j].elapsed_time(evf[i][j + 1]) for i in range(KB)) / KB
    for j, name in enumerate(BWD_STAGES):
        stage_ms[name] = sum(evb[i][j].elapsed_time(evb[i][j + 1]) for i in range(KB)) / KB
    fwd_ms = sum(stage_ms[s] for s in FWD_STAGES)
    dom = max(stage_ms, key=stage_ms.get)
    dwhich, dj = (0, FWD_STAGES.index(dom)) if dom in FWD_STAGES else (1, BWD_STAGES.index(dom))

    # the timed region: K steps, events only around the dominant stage's kernel
    ed = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for a_, b_ in ed:
        a_.record(stream)
        b_.record(stream)                       # materialise the handles
    empty = [None] * (6 if dwhich == 0 else 7)

    def dom_events(i):
        ev = list(empty)
        ev[dj], ev[dj + 1] = ed[i]
        return ev

    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.25 if clocks else 0)
    n0 = plan.launch_count()
    if args.graph:
        # the K timed steps as one CUDA graph: the plan allocates nothing and
        # never synchronises, so the step captures
        cs = torch.cuda.Stream()
        cs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cs):
            for i in range(K):
                plan.set_timing_events(dwhich, dom_events(i))
                step()
        torch.cuda.synchronize()
        t_start.record(stream)
        graph.replay()
        t_end.record(stream)
    else:
        t_start.record(stream)
        for i in range(K):
            plan.set_timing_events(dwhich, dom_events(i))
            step()
        t_end.record(stream)
    n1 = plan.launch_count()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    plan.set_timing_events(dwhich, None)
    rc, det = plan.check()
    if rc != 0:
        raise RuntimeError("device error %d (%d) in the timed region" % (rc, det))

    ms = t_start.elapsed_time(t_end)
    ms = max_over_ranks(ms, dev)
    ms_step = ms / K
    flops_step = 18.0 * T * k * d * I
    value = flops_step * ws / (ms_step * 1e-3) / 1e12
    dom_timed_ms = sum(a_.elapsed_time(b_) for a_, b_ in ed) / K

    # roofline of every stage; the dominant one is reported as "roofline".  Tensor
    # peak: burst unless the clock record of the timed region shows power capping
    pk, pk_src = peaks()
    tpeak, tpeak_src = tensor_peak(pk, clk)
    model = stage_model(c)
    stages = stage_table(model, stage_ms, tpeak, pk["hbm_gbs"])
    # the dominant kernel's roofline from its events in the timed region
    bound, fl, by = model[dom]
    if bound == "tensor":
        d_ach, d_peak = fl / (dom_timed_ms * 1e-3) / 1e12, tpeak
        d_unit = "TFLOP/s"
    else:
        d_ach, d_peak, d_unit = by / (dom_timed_ms * 1e-3) / 1e9, pk["hbm_gbs"], "GB/s"
    roofline = {"kernel": dom, "bound": bound, "achieved": round(d_ach, 1), "peak": d_peak,
                "unit": d_unit, "frac": round(d_ach / d_peak, 4), "ms": round(dom_timed_ms, 5),
                "traffic": traffic_for(dom),
                "peak_source": "%s (%s)" % (pk_src, tpeak_src if bound == "tensor"
                                            else "copy bandwidth")}
    if bound == "hbm":
        roofline["frac_nominal_hbm"] = round(d_ach / NOMINAL_HBM_GBS, 4)
    peak_note = {"tensor": tpeak_src, "tensor_peak": tpeak, "hbm": "measured copy bandwidth",
                 "hbm_peak": pk["hbm_gbs"], "nominal_hbm": NOMINAL_HBM_GBS, "source": pk_src}

    # end to end through the C ABI with pinned host buffers (copies in the timed region)
    e2e = None
    if args.e2e_steps > 0:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        xh, dyh = pin(inp["x"]).view(torch.bfloat16), pin(inp["dy"]).view(torch.bfloat16)
        idh, sch = pin(inp["ids"]), pin(inp["scores"])
        yh = torch.empty(T, d, dtype=torch.bfloat16).pin_memory()
        dxh = torch.empty(T, d, dtype=torch.bfloat16).pin_memory()
        dsh = torch.empty(T, k, dtype=torch.float32).pin_memory()

        def hstep():
            plan.step_host(xh, idh, sch, D["w13"], D["w2"], yh, dyh, D["dw13"], D["dw2"], dxh, dsh)

        for _ in range(2):
            hstep()
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            hstep()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), dev) / args.e2e_steps
        h2d = 2 * T * d * 2 + 4 * T * k * 2
        d2h = 2 * T * d * 2 + 4 * T * k
        e2e = {"value": flops_step * ws / (ems * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ems}

    # bf16 forward that saves nothing (inference) on the same inputs
    fwd_inf = None
    if args.fwd_steps > 0:
        iplan = moe.MoePlan(T, d, I, E, k, clamp=c["clamp"], flags=0, device=dev)
        yi = torch.empty(T, d, dtype=torch.bfloat16, device=dev)

        def istep():
            iplan.forward(D["x"], D["ids"], D["scores"], D["w13"], D["w2"], y=yi)

        for _ in range(args.warmup):
            istep()
        iev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)]
               for _ in range(args.fwd_steps)]
        for ev in [e for st_ in iev for e in st_]:
            ev.record(stream)
        torch.cuda.synchronize()
        i0 = torch.cuda.Event(enable_timing=True)
        i1 = torch.cuda.Event(enable_timing=True)
        i0.record(stream)
        for i in range(args.fwd_steps):
            iplan.set_timing_events(0, iev[i])
            istep()
        i1.record(stream)
        torch.cuda.synchronize()
        iplan.set_timing_events(0, None)
        rc, det = iplan.check()
        if rc != 0:
            raise RuntimeError("device error %d (%d) in the bf16 forward" % (rc, det))
        ims = max_over_ranks(i0.elapsed_time(i1), dev) / args.fwd_steps
        ist = {}
        for j, name in enumerate(FWD_STAGES):
            ist[name] = {"ms": round(sum(iev[i][j].elapsed_time(iev[i][j + 1])
                                         for i in range(args.fwd_steps)) / args.fwd_steps, 5)}
        fwd_inf = {"workload": "train_e128 sizes and inputs, bf16 forward that saves nothing "
                               "(inference)",
                   "value": 6.0 * T * k * d * I * ws / (ims * 1e-3) / 1e12, "unit": "TFLOP/s",
                   "ms_per_step": ims, "steps": args.fwd_steps, "stages": ist}
        del iplan

    # MXFP8 E4M3 forward on the same inputs (its workload differs only in precision)
    mx = None
    mx_train = None
    if args.mx_steps > 0:
        w13q, w13s, w2q, w2s = moe.prepare_weights_mxfp8(D["w13"], D["w2"])
        mplan = moe.MoePlan(T, d, I, E, k, precision=moe.MOE_PREC_MXFP8, clamp=c["clamp"], flags=0,
                            device=dev)
        ym = torch.empty(T, d, dtype=torch.bfloat16, device=dev)

        def mstep():
            mplan.forward(D["x"], D["ids"], D["scores"], w13q, w2q, y=ym, w13_sf=w13s, w2_sf=w2s)

        for _ in range(args.warmup):
            mstep()
        mev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.mx_steps)]
        for ev in [e for st_ in mev for e in st_]:
            ev.record(stream)
        torch.cuda.synchronize()
        m0 = torch.cuda.Event(enable_timing=True)
        m1 = torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        for i in range(args.mx_steps):
            mplan.set_timing_events(0, mev[i])
            mstep()
        m1.record(stream)
        torch.cuda.synchronize()
        mplan.set_timing_events(0, None)
        rc, det = mplan.check()
        if rc != 0:
            raise RuntimeError("device error %d (%d) in the MXFP8 forward" % (rc, det))
        mms = max_over_ranks(m0.elapsed_time(m1), dev) / args.mx_steps
        fp8_peak = tpeak * FP8_OVER_BF16
        mst = {}
        for j, name in enumerate(FWD_STAGES):
            t_ms = sum(mev[i][j].elapsed_time(mev[i][j + 1]) for i in range(args.mx_steps)) / args.mx_steps
            bound, fl, by = model[name]
            ent = {"ms": round(t_ms, 5)}
            if fl:
                ach = fl / (t_ms * 1e-3) / 1e12
                ent.update(achieved=round(ach, 1), unit="TFLOP/s", peak=fp8_peak,
                           frac=round(ach / fp8_peak, 4))
            mst[name] = ent
        mx = {"workload": "mxfp8_e128 (same sizes and inputs, E4M3 block-scaled forward)",
              "value": 6.0 * T * k * d * I * ws / (mms * 1e-3) / 1e12, "unit": "TFLOP/s",
              "ms_per_step": mms, "steps": args.mx_steps,
              "peak_note": "fp8 peak = %s x 2 (nominal ratio)" % tpeak_src, "stages": mst}
        del mplan

        # MXFP8 training step: saving forward + block-scaled backward
        w13t, w13ts, w2t, w2ts = moe.prepare_weights_mxfp8_backward(D["w13"], D["w2"])
        tplan = moe.MoePlan(T, d, I, E, k, precision=moe.MOE_PREC_MXFP8, clamp=c["clamp"],
                            flags=moe.MOE_WS_TRAINING, device=dev)
        dxm = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
        dsm = torch.empty(T, k, dtype=torch.float32, device=dev)

        def tstep():
            tplan.forward(D["x"], D["ids"], D["scores"], w13q, w2q, y=ym, w13_sf=w13s,
                          w2_sf=w2s, save=True)
            tplan.backward_mxfp8(D["dy"], w13t, w13ts, w2t, w2ts, D["dw13"], D["dw2"], dx=dxm,
                                 dscores=dsm)

        for _ in range(args.warmup):
            tstep()
        tf = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.mx_steps)]
        tb = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.mx_steps)]
        for ev in [e for st_ in tf + tb for e in st_]:
            ev.record(stream)
        torch.cuda.synchronize()
        m0.record(stream)
        for i in range(args.mx_steps):
            tplan.set_timing_events(0, tf[i])
            tplan.set_timing_events(1, tb[i])
            tstep()
        m1.record(stream)
        torch.cuda.synchronize()
        tplan.set_timing_events(0, None)
        tplan.set_timing_events(1, None)
        rc, det = tplan.check()
        if rc != 0:
            raise RuntimeError("device error %d (%d) in the MXFP8 training step" % (rc, det))
        tms = max_over_ranks(m0.elapsed_time(m1), dev) / args.mx_steps
        tst = {}
        for evs, names in ((tf, FWD_STAGES), (tb, BWD_STAGES)):
            for j, name in enumerate(names):
                t_ms = sum(evs[i][j].elapsed_time(evs[i][j + 1])
                           for i in range(args.mx_steps)) / args.mx_steps
                tst[name] = {"ms": round(t_ms, 5)}
        mx_train = {"workload": "mxfp8_e128 training (same sizes and inputs; forward with saved "
                                "activations + block-scaled DGRAD and WGRAD)",
                    "value": 18.0 * T * k * d * I * ws / (tms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "ms_per_step": tms, "steps": args.mx_steps, "stages": tst}
        del tplan

    extra = {}
    if args.extra_steps > 0:
        wanted = [w for w in args.extra_workloads.split(",") if w]
        for name, train in (("infer_e16", False), ("skew_pad", True)):
            if name in wanted:
                extra[name] = run_extra(moe, name, train, args, dev, ws, tpeak, pk)

    if rank != 0:
        return
    cpu = None
    if args.cpu_seconds > 0 and (ws == 1 or rank == 0):
        # all host cores (the parallel oracle; same sums, same order), then one core
        flops, el, ne, cores = oracle_sample(inp, 1024, 0.7 * args.cpu_seconds)
        cpu = {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": "forward+backward incl. weight gradients of the routed rows of one "
                         "expert at a time (%d expert passes, experts taken in order 0, 1, ... "
                         "mod E) among tokens 0..1023 (%.2f GFLOP in %.1f s, %d host threads)"
                         % (ne, flops / 1e9, el, cores)}
        f1, e1, n1c, _ = oracle_sample(inp, 1024, 0.3 * args.cpu_seconds, threads=1)
        cpu["single_core"] = {"value": f1 / e1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                              "sample": "%d expert passes, same tokens (%.2f GFLOP in %.1f s)"
                                        % (n1c, f1 / 1e9, e1)}
    ws_bytes = plan.workspace.numel() + sum(t.numel() * t.element_size() for t in D.values())
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s (T=%d, d=%d, I=%d, E=%d, k=%d, uniform routing, "
                               "forward+backward)" % (WORKLOAD, T, d, I, E, k),
                   "tokens_per_gpu": T, "l2": "inputs larger than L2 (%.1f GB resident per GPU)"
                   % (ws_bytes / 1e9),
                   "parallelism": ("data parallel, weight gradients summed over ranks (NCCL "
                                   "all-reduce) every step" if dp else "replicas")
                   if ws > 1 else "single GPU",
                   "launch": "CUDA graph replay of the timed steps" if args.graph
                             else "eager launches",
                   "backward": ("weight gradients on %d SMs beside DGRAD-W13 (own stream)"
                                % args.wgrad_sms) if args.wgrad_sms else "one stream"},
        "fwd_tflops": 6.0 * T * k * d * I / (fwd_ms * 1e-3) / 1e12,
        "bf16_forward": fwd_inf,
        "fwd_ms": fwd_ms,
        "e2e": e2e, "gpu_launches": int(n1 - n0), "roofline": roofline, "stages": stages,
        "stages_note": "%d untimed steps with an event at every stage boundary, one kernel at "
                       "a time; the timed steps record only the dominant stage's events" % KB,
        "cpu_baseline": cpu, "clocks": clk, "peaks": peak_note, "mxfp8_forward": mx,
        "mxfp8_training": mx_train, "infer_e16": extra.get("infer_e16"),
        "skew_pad": extra.get("skew_pad"),
    }
    print(json.dumps(line), flush=True)


def run_extra(moe, name, train, args, dev, ws, tpeak, pk):
    """Throughput of another workload of the method: the bf16 inference forward at
    E = 16 (forward only) or the skewed-routing training step (Zipf routing,
    zero-score padding tokens, clamped SwiGLU).  A timed loop without stage events
    gives the value; a separate pass with an event at every stage boundary gives
    the stage table."""
    import numpy as np
    import torch

    import moe_inputs as mi

    _, rank, _ = dist_env()
    need = ("x", "ids", "scores", "w13", "w2") + (("dy", "dw13", "dw2") if train else ())
    inp = mi.make_inputs(name, seed=args.seed + rank, need=need)
    c = inp["cfg"]
    T, d, I, E, k = c["T"], c["d"], c["I"], c["E"], c["k"]

    def to_dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.to(dev)

    D = {key: to_dev(inp[key]) for key in need}
    del inp
    plan = moe.MoePlan(T, d, I, E, k, clamp=c["clamp"],
                       flags=moe.MOE_WS_TRAINING if train else 0, device=dev)
    y = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    if train:
        dx = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
        dsc = torch.empty(T, k, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        plan.forward(D["x"], D["ids"], D["scores"], D["w13"], D["w2"], y=y, save=train)
        if train:
            plan.backward(D["dy"], D["w13"], D["w2"], D["dw13"], D["dw2"], dx=dx, dscores=dsc)

    for _ in range(args.warmup):
        step()
    K = args.extra_steps
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), dev) / K
    evf = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(K)]
    for ev in [e for s_ in evf + evb for e in s_]:
        ev.record(stream)
    torch.cuda.synchronize()
    for i in range(K):
        plan.set_timing_events(0, evf[i])
        if train:
            plan.set_timing_events(1, evb[i])
        step()
    torch.cuda.synchronize()
    plan.set_timing_events(0, None)
    plan.set_timing_events(1, None)
    rc, det = plan.check()
    if rc != 0:
        raise RuntimeError("device error %d (%d) in %s" % (rc, det, name))
    stage_ms = {}
    for j, st_ in enumerate(FWD_STAGES):
        stage_ms[st_] = sum(evf[i][j].elapsed_time(evf[i][j + 1]) for i in range(K)) / K
    if train:
        for j, st_ in enumerate(BWD_STAGES):
            stage_ms[st_] = sum(evb[i][j].elapsed_time(evb[i][j + 1]) for i in range(K)) / K
    counts = np.bincount(D["ids"].cpu().numpy().reshape(-1), minlength=E)
    model = stage_model(c, n_nonempty=int((counts > 0).sum()))
    if not train:
        # an inference forward does not store a
        b, fl, by = model["w13_swiglu"]
        model["w13_swiglu"] = (b, fl, by - 4 * T * k * I)
    stages = stage_table(model, stage_ms, tpeak, pk["hbm_gbs"])
    flops = (18.0 if train else 6.0) * T * k * d * I
    desc = ("%s (T=%d, d=%d, I=%d, E=%d, k=%d, %s routing%s%s, %s)"
            % (name, T, d, I, E, k, c["routing"],
               ", last %d tokens zero-score padding" % c["pad"] if c["pad"] else "",
               ", SwiGLU clamped to +-%g" % c["clamp"] if c["clamp"] else "",
               "forward+backward" if train else "forward"))
    out = {"workload": desc, "value": flops * ws / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "ms_per_step": ms, "steps": K, "stages": stages,
           "rows_per_expert": {"max": int(counts.max()), "median": float(np.median(counts)),
                               "empty": int((counts == 0).sum())}}
    if not train and d % 256 == 0 and I % 256 == 0:
        out["nvfp4"] = run_nvfp4(moe, plan, D, c, args, dev, ws, tpeak, model, stage_ms)
    del plan, D
    torch.cuda.empty_cache()
    return out


def run_nvfp4(moe, bplan, D, c, args, dev, ws, tpeak, model, bf16_stage_ms):
    """NVFP4 inference forward on the same inputs: static activation scales from a
    calibration on them (amax / (6 * 448) of x and of the bf16 forward's h, device
    amax), prepared weights, then the timed loop and the stage table."""
    import torch

    T, d, I, E, k = c["T"], c["d"], c["I"], c["E"], c["k"]
    n = int(bplan.buffer("off_pad", torch.int32)[-1].item())
    x_amax = float(moe.amax_bf16(D["x"]).item())
    h_amax = float(moe.amax_bf16(bplan.buffer("h", torch.bfloat16)[: n * I]).item())
    prep = moe.prepare_weights_nvfp4(D["w13"], D["w2"])
    plan = moe.MoePlan(T, d, I, E, k, precision=moe.MOE_PREC_NVFP4, clamp=c["clamp"], flags=0,
                       device=dev)
    plan.set_activation_scales(x_amax / 2688.0, h_amax / 2688.0)
    y = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        plan.forward_nvfp4(D["x"], D["ids"], D["scores"], prep, y=y)

    for _ in range(args.warmup):
        step()
    K = args.extra_steps
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), dev) / K
    evf = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for ev in [e for s_ in evf for e in s_]:
        ev.record(stream)
    torch.cuda.synchronize()
    for i in range(K):
        plan.set_timing_events(0, evf[i])
        step()
    torch.cuda.synchronize()
    plan.set_timing_events(0, None)
    rc, det = plan.check()
    if rc != 0:
        raise RuntimeError("device error %d (%d) in the NVFP4 forward" % (rc, det))
    fp4_peak = tpeak * FP4_OVER_BF16
    stages = {}
    for j, name in enumerate(FWD_STAGES):
        t_ms = sum(evf[i][j].elapsed_time(evf[i][j + 1]) for i in range(K)) / K
        bound, fl, by = model[name]
        ent = {"ms": round(t_ms, 5)}
        if fl:
            ach = fl / (t_ms * 1e-3) / 1e12
            ent.update(achieved=round(ach, 1), unit="TFLOP/s", peak=fp4_peak,
                       frac=round(ach / fp4_peak, 4))
        stages[name] = ent
    return {"workload": "infer_e16 sizes and inputs, NVFP4 (E2M1, E4M3 scales per 16, "
                        "per-tensor scales) inference forward, static activation scales "
                        "calibrated on the same inputs",
            "value": 6.0 * T * k * d * I * ws / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": ms, "steps": K,
            "peak_note": "fp4 peak = bf16 tensor peak x %g (nominal ratio)" % FP4_OVER_BF16,
            "stages": stages}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    ws, _, _ = dist_env()
    if ws > 1:
        import torch.distributed as dist

        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
