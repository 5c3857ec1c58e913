#!/usr/bin/env python
"""Throughput of the KDA mixer on GB300: chunked prefill and decode tokens/s.

One step = one pass of the whole mixer hot path on synthetic inputs:
  * a fused-mixer prefill, B=1, T=65536, H=32, dk=dv=128, chunk 64: width-4
    causal SiLU convs on q, k, v, in-kernel q/k L2 norm, chunked KDA with an
    FP32 state, sigmoid output gate, bf16 activations in and out;
  * one decode step for 256 independent sequences, H=32, d=128: conv window
    update, L2 norm, FP32 state read-modify-write ([256,32,128,128] = 512 MiB),
    gate.
value = (prefill tokens + decode tokens) per step / step time, device-resident
inputs; the "prefill" and "decode" objects give each part on its own with its
roofline.  Beside the step, not in value: "e2e" (the same step from pinned host
buffers), "configs" (the other synthetic workloads timed on their own: the fp32
core's latency, the chunked prefill T=8192 and the packed varlen prefill with
initial states, each with its roofline), "parity" (each workload's max-abs and
RMS-relative error on one small seeded case against the oracle), "backward"
(gradients of the recurrence, T=8192, H=32) and "mla_decode" (one decode token of
the hybrid's attention layers, 256 sequences with bf16 caches of 8192 rows).  With --gpus N under torchrun every rank runs its own replica of the
step (heads and sequences never interact, so there is no collective): weak
scaling, max time over ranks.

--impl reference times the CPU oracle (the reference arm for this method) on a
bounded sample of the same workload on the host cores.  The CPU-baseline leg (rank 0,
N=1, before any GPU work) times the FP64 oracle and the FP32 per-token loop on a
sample of the step, and runs the oracle on the small parity cases whose GPU results
are compared after the timed arm.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s & decode tokens/s at 1 GB300; % of tensor/HBM roofline"
PREFILL = dict(T=65536, H=32, d=128, chunk=64, W=4)
DECODE = dict(N=256, H=32, d=128, W=4)
BACKWARD = dict(T=8192, H=32, d=128)      # gradients of the recurrence: the chunked-prefill shape
CORE = dict(T=64, H=2, d=16, chunk=16)    # the fp32 core workload (latency)
CHUNKED = dict(T=8192, H=32, d=128, chunk=64)                        # chunked prefill, bf16, S0 = 0
VARLEN = dict(n_seqs=16, lo=256, hi=16384, H=32, d=128, chunk=64)    # packed, lengths from seed 0, S0 != 0
MLA = dict(N=256, H=32, d=128, L_max=8192)   # the attention layers' decode token: the decode batch
MLA_TRAFFIC_PER_KEY_HEAD = 1.388077e9 / ((84420 + 16) * 32)   # DRAM bytes per attended (key, head), measured


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=8)
    p.add_argument("--cpu-sample-tokens", type=int, default=16384,
                   help="prefill tokens (all heads) the CPU baseline runs; scaled to the full workload")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-backward", action="store_true")
    p.add_argument("--no-mla", action="store_true")
    p.add_argument("--no-configs", action="store_true", help="skip the other workloads' lines")
    p.add_argument("--mla-seqs", type=int, default=None,
                   help="override the attention decode batch (profiling captures on a smaller case)")
    p.add_argument("--backward-tokens", type=int, default=None,
                   help="override the backward's length (profiling captures on a smaller case)")
    p.add_argument("--prefill-tokens", type=int, default=None,
                   help="override the prefill length (profiling captures on a smaller case; "
                        "the JSON config records the length used)")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return dict(hbm=float(m["hbm_gbs"]), bf16=float(m["bf16_tflops"]),
                    bf16_sustained=float(m.get("bf16_tflops_sustained", m["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


# ---- algorithmic work (bytes that must cross HBM, flops of the chunked form) ----

def prefill_work(T, H, d, chunk, W, N=1, gate=True, initial_state=False):
    """Bytes: q, k, v (bf16), g (fp32), beta, the gate (bf16) when gated, the bf16 output, the fp32
    final state (and the initial state when given), the conv state in and out and the conv weights
    when W > 0.  Flops: the chunked form, 10 C d + 6 d^2 per (token, head), plus the conv."""
    dk = dv = d
    per_tok_head = 2 * (2 * dk + dv) + 4 * dk + 4 + (2 * dv if gate else 0) + 2 * dv
    D = 2 * H * dk + H * dv
    conv = 2 * N * (W - 1) * D * 4 + D * W * 4 if W > 0 else 0     # conv state in and out, weights
    bytes_ = T * H * per_tok_head + N * H * dk * dv * 4 * (2 if initial_state else 1) + conv
    flops = T * H * (10 * chunk * d + 6 * d * d) + T * D * 2 * W
    return bytes_, flops


def backward_work(T, H, d):
    """Bytes: q, k, v (bf16), g, dO (fp32), beta in; dq, dk, dg, dv (fp32), dbeta out.
    Flops: one forward pass of the recurrence (5 d^2 per token and head) plus the reverse
    sweep (18 d^2), the minimal work of the method; the chunked kernels do more (the WY tiles and
    the chunk products)."""
    per_tok_head = 3 * 2 * d + 4 * d + 4 * d + 4 + 4 * (3 * d + d) + 4
    return T * H * per_tok_head, T * H * 23 * d * d


def mla_work(lens, H, d):
    """Bytes of one attention decode token with bf16 caches: every cached key and value row read
    once (the appended one included), the new rows written, q, k, v, gate read and the bf16
    output written, the lengths read and written.  Flops: 4 d per attended key (score and
    weighted value)."""
    keys = int(np.sum(np.asarray(lens, dtype=np.int64) + 1))
    N = len(lens)
    bytes_ = keys * H * d * 2 * 2 + N * H * d * 2 * 2 + N * H * d * 2 * 5 + N * 8
    return bytes_, keys * H * 4 * d


def decode_work(N, H, d, W):
    dk = dv = d
    D = 2 * H * dk + H * dv
    per_nh = 2 * 4 * dk * dv + 2 * (2 * dk + dv) + 4 * dk + 4 + 2 * dv + 2 * dv
    bytes_ = N * H * per_nh + 2 * N * (W - 1) * D * 4 + D * W * 4
    flops = N * H * (7 * dk * dv + 2 * W * (2 * dk + dv))
    return bytes_, flops


# ---- clocks during the timed region ----

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---- replicas: the slowest rank's time is the job's time ----

def max_over_ranks(values, world, device):
    """Elementwise max of a list of floats over all ranks (identity at world == 1)."""
    if world <= 1:
        return [float(x) for x in values]
    import torch
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_value(units_per_rank, world, seconds):
    """Whole-job throughput of `world` replicas that each process `units_per_rank` units."""
    return world * units_per_rank / seconds


# ---- the GPU arm ----

def make_inputs(torch, dev, seed):
    """Seeded synthetic inputs drawn on the device with the workload recipe
    (q,k,v,gate ~ N(0,1) bf16; g = -softplus(N(0,1)); beta = sigmoid(N(0,1));
    conv weights ~ N(0, 0.5); decode state ~ N(0, 0.02); conv windows ~ N(0,1))."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    f32, bf16 = torch.float32, torch.bfloat16

    def n(shape, std=1.0, dt=f32):
        return (torch.randn(shape, generator=gen, device=dev, dtype=f32) * std).to(dt)

    T, H, d, W = PREFILL["T"], PREFILL["H"], PREFILL["d"], PREFILL["W"]
    D = 3 * H * d
    P = dict(q=n((T, H, d), dt=bf16), k=n((T, H, d), dt=bf16), v=n((T, H, d), dt=bf16),
             g=-torch.nn.functional.softplus(n((T, H, d))), beta=torch.sigmoid(n((T, H))),
             gate=n((T, H, d), dt=bf16), conv_w=n((D, W), 0.5), conv_state=torch.zeros((1, W - 1, D), device=dev))
    N, Hd, dd, Wd = DECODE["N"], DECODE["H"], DECODE["d"], DECODE["W"]
    Dd = 3 * Hd * dd
    Dc = dict(q=n((N, Hd, dd), dt=bf16), k=n((N, Hd, dd), dt=bf16), v=n((N, Hd, dd), dt=bf16),
              g=-torch.nn.functional.softplus(n((N, Hd, dd))), beta=torch.sigmoid(n((N, Hd))),
              gate=n((N, Hd, dd), dt=bf16), conv_w=n((Dd, Wd), 0.5),
              conv_state=n((N, Wd - 1, Dd)).to(bf16).to(f32), state=n((N, Hd, dd, dd), 0.02))
    return P, Dc


def run_ours(args, rank, world, dev, torch):
    import hybrid_linear_attention_rule_gb300 as K
    K.load_library()
    pk = peaks()
    P, Dc = make_inputs(torch, dev, seed=1000 + rank)
    T, H, d, C, W = PREFILL["T"], PREFILL["H"], PREFILL["d"], PREFILL["chunk"], PREFILL["W"]
    N, Hd, dd, Wd = DECODE["N"], DECODE["H"], DECODE["d"], DECODE["W"]
    cu_h = torch.tensor([0, T], dtype=torch.int32)
    cu_d = cu_h.to(dev)
    out_p = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    fs = torch.empty((1, H, d, d), dtype=torch.float32, device=dev)
    out_d = torch.empty((N, Hd, dd), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(K.k3kda_prefill_workspace_size(1, T, H, d, d, C, K.BF16, True), dtype=torch.uint8, device=dev)
    scale = d ** -0.5
    stream = torch.cuda.current_stream()

    def prefill_call(p, out, f):
        K.k3kda_prefill(p["q"], p["k"], p["v"], p["g"], p["beta"], None, cu_d, cu_h, 1, T, H, d, d, C, scale, True,
                        p["conv_w"], p["conv_state"], W, p["gate"], out, f, ws, stream)

    def decode_call(c, out):
        K.k3kda_decode_step(c["q"], c["k"], c["v"], c["g"], c["beta"], c["gate"], c["conv_w"], c["conv_state"],
                            c["state"], N, Hd, dd, dd, Wd, scale, True, out, stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        prefill_call(P, out_p, fs)
        decode_call(Dc, out_d)
    torch.cuda.synchronize()
    st = K.k3kda_workspace_status(ws)
    if st != 0:
        raise RuntimeError(f"prefill workspace status {st}")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    n0 = K.k3kda_launch_count()
    gpu_id = os.environ.get("LOCAL_RANK", "0")
    with ClockSampler(gpu_id) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s in range(args.steps):
            ev[s][0].record(stream)
            prefill_call(P, out_p, fs)
            ev[s][1].record(stream)
            decode_call(Dc, out_d)
            ev[s][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    launches = K.k3kda_launch_count() - n0
    barrier()
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    total_ms, pre_ms, dec_ms = max_over_ranks([total_ms, pre_ms, dec_ms], world, dev)
    ms_per_step = total_ms / args.steps
    tokens_per_step = T + N

    pb, pf = prefill_work(T, H, d, C, W)
    db, df = decode_work(N, Hd, dd, Wd)
    pre_tok_s = T / (pre_ms / 1e3)
    dec_tok_s = N / (dec_ms / 1e3)
    roof_p = {"bound": "hbm", "achieved": pb / (pre_ms / 1e3) / 1e9, "peak": pk["hbm"], "unit": "GB/s",
              "traffic": PREFILL_TRAFFIC_PER_LAUNCH}
    roof_p["frac"] = roof_p["achieved"] / roof_p["peak"]
    roof_p["tensor"] = {"achieved_tflops": pf / (pre_ms / 1e3) / 1e12, "peak": pk["bf16"],
                        "frac": pf / (pre_ms / 1e3) / 1e12 / pk["bf16"]}
    roof_d = {"bound": "hbm", "achieved": db / (dec_ms / 1e3) / 1e9, "peak": pk["hbm"], "unit": "GB/s",
              "traffic": DECODE_TRAFFIC_PER_LAUNCH}
    roof_d["frac"] = roof_d["achieved"] / roof_d["peak"]

    res = {
        "metric": METRIC, "value": job_value(tokens_per_step, world, ms_per_step / 1e3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "io_dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"KDA mixer step: fused prefill T={T} H=32 d=128 chunk64 conv4 gate + "
                               "decode step N=256 H=32 d=128 conv4 gate",
                   "prefill": dict(PREFILL, B=1, l2norm=True, gate=True, out="bf16"),
                   "decode": dict(DECODE, l2norm=True, gate=True, state="fp32", out="bf16"),
                   "l2_flush": "inputs larger than L2 (prefill 3.8 GB, decode 1.2 GB per step)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "prefill": {"tokens_per_s": world * pre_tok_s, "ms": pre_ms, "algorithmic_bytes": pb,
                    "algorithmic_flops": pf, "roofline": roof_p},
        "decode": {"tokens_per_s": world * dec_tok_s, "ms": dec_ms, "algorithmic_bytes": db,
                   "algorithmic_flops": df, "roofline": roof_d},
        "roofline": roof_p,
        "peaks_source": pk["src"],
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, K, torch, dev, P, Dc, prefill_call, decode_call, out_p, fs, out_d, world, barrier)
    if not args.no_configs:
        res["configs"] = run_configs(args, K, torch, dev, rank, world)
    if not args.no_backward:
        res["backward"] = run_backward(args, K, torch, dev, rank, world, clk_mhz=res["clocks"].get("sm_mhz"))
    if not args.no_mla:
        res["mla_decode"] = run_mla(args, K, torch, dev, rank, world)
    return res


def _time_calls(torch, call, steps, warmup, stream):
    """Average CUDA-event time (ms) of `steps` calls after `warmup` untimed ones."""
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def _prefill_roofline(pk, by, fl, ms, traffic):
    ach = by / (ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": pk["hbm"], "unit": "GB/s", "frac": ach / pk["hbm"],
            "traffic": traffic,
            "tensor": {"achieved_tflops": fl / (ms / 1e3) / 1e12, "peak": pk["bf16"],
                       "frac": fl / (ms / 1e3) / 1e12 / pk["bf16"]}}


def run_configs(args, K, torch, dev, rank, world):
    """The other synthetic workloads, each timed on its own with CUDA events on the launching
    stream (inputs drawn on the device with the workload recipe, larger than L2 except the fp32
    core): the fp32 core (T=64, H=2, d=16, chunk 16; a latency), the chunked prefill (B=1, T=8192,
    H=32, d=128, bf16 q/k/v, zero initial state, bf16 outputs, fp32 final state) and the packed
    varlen prefill (16 sequences, lengths uniform in [256, 16384] from seed 0, initial states
    ~ N(0, 0.02), bf16 outputs, fp32 final states)."""
    import kda_inputs as KI
    pk = peaks()
    gen = torch.Generator(device=dev)
    gen.manual_seed(4000 + rank)
    f32, bf16 = torch.float32, torch.bfloat16
    stream = torch.cuda.current_stream()

    def n(shape, std=1.0, dt=f32):
        return (torch.randn(shape, generator=gen, device=dev, dtype=f32) * std).to(dt)

    def prefill_inputs(T, H, d, dt):
        return dict(q=n((T, H, d), dt=dt), k=n((T, H, d), dt=dt), v=n((T, H, d), dt=dt),
                    g=-torch.nn.functional.softplus(n((T, H, d))), beta=torch.sigmoid(n((T, H))))

    out = {}
    steps = max(1, args.steps)
    # ---- fp32 core: latency of one call ----
    T, H, d, C = CORE["T"], CORE["H"], CORE["d"], CORE["chunk"]
    x = prefill_inputs(T, H, d, f32)
    cu_h = torch.tensor([0, T], dtype=torch.int32)
    cu_d = cu_h.to(dev)
    o = torch.empty((T, H, d), device=dev)
    fs = torch.empty((1, H, d, d), device=dev)
    ws = torch.zeros(K.k3kda_prefill_workspace_size(1, T, H, d, d, C, K.F32, False), dtype=torch.uint8, device=dev)
    call = lambda: K.k3kda_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], None, cu_d, cu_h, 1, T, H, d, d, C,
                                   d ** -0.5, True, None, None, 0, None, o, fs, ws, stream)
    ms = _time_calls(torch, call, max(steps, 200), args.warmup, stream)
    ms = max_over_ranks([ms], world, dev)[0]
    out["core_fp32"] = {"workload": f"KDA core fp32, T={T} H={H} d={d} chunk {C}, no conv or gate", "us": ms * 1e3,
                        "tokens_per_s": world * T / (ms / 1e3), "bound": "latency"}
    # ---- chunked prefill ----
    T, H, d, C = CHUNKED["T"], CHUNKED["H"], CHUNKED["d"], CHUNKED["chunk"]
    x = prefill_inputs(T, H, d, bf16)
    cu_h = torch.tensor([0, T], dtype=torch.int32)
    cu_d = cu_h.to(dev)
    o = torch.empty((T, H, d), dtype=bf16, device=dev)
    fs = torch.empty((1, H, d, d), device=dev)
    ws = torch.zeros(K.k3kda_prefill_workspace_size(1, T, H, d, d, C, K.BF16, False), dtype=torch.uint8, device=dev)
    call = lambda: K.k3kda_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], None, cu_d, cu_h, 1, T, H, d, d, C,
                                   d ** -0.5, True, None, None, 0, None, o, fs, ws, stream)
    ms = _time_calls(torch, call, steps, args.warmup, stream)
    ms = max_over_ranks([ms], world, dev)[0]
    by, fl = prefill_work(T, H, d, C, 0, gate=False)
    out["chunked_prefill"] = {"workload": f"chunked prefill B=1 T={T} H={H} d={d} chunk {C}, bf16 in/out, S0=0",
                              "ms": ms, "tokens_per_s": world * T / (ms / 1e3), "algorithmic_bytes": by,
                              "algorithmic_flops": fl, "workspace_bytes": ws.numel(),
                              "roofline": _prefill_roofline(pk, by, fl, ms, CHUNKED_TRAFFIC_PER_LAUNCH)}
    del x, o, ws
    # ---- packed varlen prefill with initial states ----
    lengths = KI.varlen_lengths(VARLEN["n_seqs"], VARLEN["lo"], VARLEN["hi"], 0)
    N, H, d, C = len(lengths), VARLEN["H"], VARLEN["d"], VARLEN["chunk"]
    cu_np = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu_np[-1])
    x = prefill_inputs(T, H, d, bf16)
    S0 = n((N, H, d, d), 0.02)
    cu_h = torch.from_numpy(cu_np)
    cu_d = cu_h.to(dev)
    o = torch.empty((T, H, d), dtype=bf16, device=dev)
    fs = torch.empty((N, H, d, d), device=dev)
    ws = torch.zeros(K.k3kda_prefill_workspace_size(N, T, H, d, d, C, K.BF16, False), dtype=torch.uint8, device=dev)
    call = lambda: K.k3kda_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], S0, cu_d, cu_h, N, T, H, d, d, C,
                                   d ** -0.5, True, None, None, 0, None, o, fs, ws, stream)
    ms = _time_calls(torch, call, steps, args.warmup, stream)
    ms = max_over_ranks([ms], world, dev)[0]
    by, fl = prefill_work(T, H, d, C, 0, N=N, gate=False, initial_state=True)
    out["varlen_prefill"] = {"workload": f"packed varlen prefill, {N} sequences (lengths uniform in "
                                         f"[{VARLEN['lo']}, {VARLEN['hi']}] from seed 0: {T} tokens), H={H} d={d} "
                                         f"chunk {C}, bf16 in/out, fp32 initial and final states",
                             "ms": ms, "tokens_per_s": world * T / (ms / 1e3), "algorithmic_bytes": by,
                             "algorithmic_flops": fl, "workspace_bytes": ws.numel(),
                             "longest_sequence": int(lengths.max()),
                             "roofline": _prefill_roofline(pk, by, fl, ms, VARLEN_TRAFFIC_PER_LAUNCH)}
    del x, o, ws, fs, S0
    torch.cuda.empty_cache()
    return out


def run_parity(K, torch, refs):
    """Each workload's error on its small seeded case: the GPU through the public binding against
    the oracle's outputs computed in the CPU-baseline leg (bf16-input workloads store fp32 outputs,
    the comparison the 5e-3 x RMS bar is stated on)."""
    out = {}
    for name, r in refs.items():
        c = r["case"]
        dev = lambda a, bf=False: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(
            torch.bfloat16 if bf else torch.float32).cuda()
        bf = c.in_dtype == "bf16"
        if name == "decode":
            st, cs = dev(c.state), dev(c.conv_state)
            o = K.decode_step(dev(c.q, bf), dev(c.k, bf), dev(c.v, bf), dev(c.g), dev(c.beta), st,
                              gate=dev(c.gate, bf), conv_weight=dev(c.conv_w), conv_state=cs,
                              out_dtype=torch.float32)
            got = [o, st]
        else:
            cs = None
            if c.conv_w is not None:
                cs = torch.zeros((c.N, c.W - 1, 2 * c.H * c.dk + c.H * c.dv), device="cuda")
            o, fs = K.prefill(dev(c.q, bf), dev(c.k, bf), dev(c.v, bf), dev(c.g), dev(c.beta),
                              initial_state=dev(c.S0), cu_seqlens=torch.from_numpy(c.cu_seqlens.copy()),
                              chunk=c.chunk, scale=c.scale, use_qk_l2norm=c.use_qk_l2norm,
                              conv_weight=dev(c.conv_w), conv_state=cs, gate=dev(c.gate, bf),
                              out_dtype=torch.float32)
            got = [o, fs]
        torch.cuda.synchronize()
        entry = {"case": r["desc"], "bar": r["bar"]}
        for what, g, w in zip(("out", "final_state"), got, r["want"]):
            gv = g.detach().double().cpu().numpy()
            err = float(np.abs(gv - w).max())
            rms = float(np.sqrt(np.mean(w * w)))
            entry[what] = {"max_abs": err, "rms_rel": err / rms if rms > 0 else None}
        out[name] = entry
    return out


def run_mla(args, K, torch, dev, rank, world):
    """One decode token of the attention layers (k3mla_decode_step): 256 sequences x 32 heads,
    d = 128, bf16 key/value caches of 8192 rows per (sequence, head), cached lengths uniform in
    [1, 8191], no RoPE, sigmoid gate, bf16 output.  The lengths are reset before every step (outside
    the events), so each timed step attends over the same keys; reported beside the main step."""
    N, H, d, L = args.mla_seqs or MLA["N"], MLA["H"], MLA["d"], MLA["L_max"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(3000 + rank)
    bf = dict(device=dev, dtype=torch.bfloat16)
    kc = torch.randn(N, H, L, d, generator=gen, **bf)
    vc = torch.randn(N, H, L, d, generator=gen, **bf)
    q, k, v, g = (torch.randn(N, H, d, generator=gen, **bf) for _ in range(4))
    lens_np = np.random.default_rng(99 + rank).integers(1, L, size=N).astype(np.int32)
    lens0 = torch.from_numpy(lens_np).to(dev)
    lens = lens0.clone()
    out = torch.empty(N, H, d, **bf)
    ws = torch.empty(K.k3mla_decode_workspace_size(N, H, d, d, L), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        K.k3mla_decode_step(q, k, v, g, kc, vc, lens, N, H, d, d, L, 0, 10000.0, d ** -0.5, out, ws, stream)

    for _ in range(args.warmup):
        lens.copy_(lens0)
        call()
    torch.cuda.synchronize()
    steps = max(1, args.steps)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in ev:
        lens.copy_(lens0)
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
    ms = max_over_ranks([ms], world, dev)[0]
    by, fl = mla_work(lens_np, H, d)
    pk = peaks()
    ach = by / (ms / 1e3) / 1e9
    # DRAM bytes of the attention kernel from one ncu capture of the 16-sequence case (1.3860 GB for
    # 84420 cached keys per head), scaled by the keys attended: traffic grows in proportion to them
    traffic = MLA_TRAFFIC_PER_KEY_HEAD * float(np.sum(lens_np.astype(np.int64) + 1)) * H
    del kc, vc
    return {"workload": f"attention decode token, N={N} H={H} d={d}, bf16 caches L_max={L}, lengths uniform in "
                        f"[1, {L - 1}] ({int(lens_np.sum())} cached keys per head), NoPE, gate",
            "ms": ms, "tokens_per_s": world * N / (ms / 1e3), "algorithmic_bytes": by, "algorithmic_flops": fl,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": pk["hbm"], "unit": "GB/s", "frac": ach / pk["hbm"],
                         "traffic": traffic}}


def run_backward(args, K, torch, dev, rank, world, clk_mhz=None):
    """Gradients of the recurrence (k3kda_backward) on the chunked-prefill shape, timed with CUDA
    events over the same steps and warm-up as the main step; reported beside it, not in value."""
    T, H, d = args.backward_tokens or BACKWARD["T"], BACKWARD["H"], BACKWARD["d"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(2000 + rank)
    n = lambda *s: torch.randn(s, generator=gen, device=dev)
    unit = lambda x: (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    q, k, v = unit(n(T, H, d)), unit(n(T, H, d)), n(T, H, d).to(torch.bfloat16)
    g, beta, dO = -torch.nn.functional.softplus(n(T, H, d)), torch.sigmoid(n(T, H)), n(T, H, d)
    cu_h = torch.tensor([0, T], dtype=torch.int32)
    cu_d = cu_h.to(dev)
    f32 = dict(dtype=torch.float32, device=dev)
    outs = [torch.empty(T, H, d, **f32) for _ in range(4)] + [torch.empty(T, H, **f32), torch.empty(1, H, d, d, **f32)]
    ws = torch.empty(K.k3kda_backward_workspace_size(1, T, H, d, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        K.k3kda_backward(q, k, v, g, beta, None, cu_d, cu_h, 1, T, H, d, d, d ** -0.5, dO, None, outs[0], outs[1],
                         outs[2], outs[3], outs[4], outs[5], ws, stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(1, args.steps)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    ms = max_over_ranks([ms], world, dev)[0]
    by, fl = backward_work(T, H, d)
    pk = peaks()
    mhz = clk_mhz or 2070.0
    fp32_peak = 152 * 128 * 2 * mhz * 1e6 / 1e12          # FP32 FMA lanes x 2 flop x SM clock, TFLOP/s
    ach = fl / (ms / 1e3) / 1e12
    return {"workload": f"gradients of the recurrence, T={T} H={H} d={d}, bf16 q/k/v, fp32 dO", "ms": ms,
            "tokens_per_s": world * T / (ms / 1e3), "algorithmic_bytes": by, "algorithmic_flops": fl,
            "roofline": {"bound": "alu", "achieved": ach, "peak": fp32_peak, "unit": "TFLOP/s", "frac": ach / fp32_peak,
                         "hbm_achieved_gbs": by / (ms / 1e3) / 1e9, "hbm_peak_gbs": pk["hbm"]}}


# Layer parameters and caches that a serving loop keeps in HBM between steps: the conv weights of
# both calls, and the decode's recurrent state and conv window (the per-sequence KDA cache).
RESIDENT_P = ("conv_w",)
RESIDENT_D = ("conv_w", "state", "conv_state")


def run_e2e(args, K, torch, dev, P, Dc, prefill_call, decode_call, out_p, fs, out_d, world, barrier):
    """Same step through the C ABI, starting from pinned HOST buffers: every step copies its
    inputs host->device -- the prompt's q, k, v, g, beta, gate and initial conv window for the
    prefill, the new token's q, k, v, g, beta, gate for the decode -- and reads both outputs back
    to the host, inside the timed region.  The conv weights and the decode's recurrent state and
    conv window are the layers' parameters and cache: uploaded once, then resident, the decode
    updating its cache in place every step.  The inputs are double-buffered, as a serving loop
    would run it: step i+1's inputs go up on a copy stream while step i computes and its outputs
    come back on the compute stream (the host link carries the two directions at once).  The
    time is taken over all steps, from the first upload to the last read-back."""
    hostP = {k: v.cpu().pin_memory() for k, v in P.items() if k not in RESIDENT_P}
    hostD = {k: v.cpu().pin_memory() for k, v in Dc.items() if k not in RESIDENT_D}
    resP = {k: P[k].clone() for k in RESIDENT_P}
    resD = {k: Dc[k].clone() for k in RESIDENT_D}
    sets = [(dict(resP, **{k: torch.empty_like(P[k]) for k in hostP}),
             dict(resD, **{k: torch.empty_like(Dc[k]) for k in hostD})) for _ in range(2)]
    res_p = torch.empty(out_p.shape, dtype=out_p.dtype).pin_memory()
    res_d = torch.empty(out_d.shape, dtype=out_d.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in list(hostP.values()) + list(hostD.values()))
    d2h = sum(v.numel() * v.element_size() for v in (res_p, res_d))
    comp = torch.cuda.current_stream()
    up = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]      # inputs of a buffer set are on the device
    free = [torch.cuda.Event() for _ in range(2)]       # a buffer set's step has computed and read back

    def upload(i):
        b = i % 2
        up.wait_event(free[b])
        with torch.cuda.stream(up):
            for k, v in hostP.items():
                sets[b][0][k].copy_(v, non_blocking=True)
            for k, v in hostD.items():
                sets[b][1][k].copy_(v, non_blocking=True)
        ready[b].record(up)

    def compute(i):
        b = i % 2
        comp.wait_event(ready[b])
        prefill_call(sets[b][0], out_p, fs)
        decode_call(sets[b][1], out_d)
        res_p.copy_(out_p, non_blocking=True)
        res_d.copy_(out_d, non_blocking=True)
        free[b].record(comp)

    def run(n):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute(i)

    run(2)
    torch.cuda.synchronize()
    # the host link's rate on this machine: one step's uploads alone, timed on the copy stream
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    upload(0)
    e1.record(up)
    torch.cuda.synchronize()
    h2d_gbs = h2d / (e0.elapsed_time(e1) * 1e-3) / 1e9
    n = max(1, args.e2e_steps)
    barrier()
    t0 = time.perf_counter()
    run(n)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / n
    dt = max_over_ranks([dt], world, dev)[0]
    return {"value": job_value(PREFILL["T"] + DECODE["N"], world, dt), "unit": "tokens/s", "ms_per_step": dt * 1e3,
            "steps": n, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_gbs": h2d_gbs, "h2d_floor_ms": h2d / h2d_gbs / 1e6,
            "pipelining": "inputs double-buffered: step i+1 uploads during step i's compute and read-back",
            "resident": "conv weights; the decode's recurrent state and conv window (its cache)"}


# Measured DRAM bytes per call (ncu dram__bytes_read.sum + dram__bytes_write.sum, summed over the
# call's kernels) of the current kernel versions, or None when not yet captured for a kernel
# version.  The prefill figure is a T=8192 capture scaled by the tokens processed to T=65536.
PREFILL_TRAFFIC_PER_LAUNCH = 13.02e9     # segment 0 prep + the cooperative segments launch, 1.628 GB at T=8192 x 8
CHUNKED_TRAFFIC_PER_LAUNCH = None
VARLEN_TRAFFIC_PER_LAUNCH = None
DECODE_TRAFFIC_PER_LAUNCH = 1.1028e9


# ---- the CPU oracle (baseline leg and the reference arm) ----

def cpu_oracle_sample(prefill_tokens, decode_seqs, seed=0):
    """Time the oracle on the first `prefill_tokens` tokens of the fused-mixer workload
    (all 32 heads) and on `decode_seqs` sequences of the decode workload; return the
    seconds each took and the threads used."""
    import kda_inputs as KI
    import oracle as O
    O.load()
    c = KI.fused_mixer(seed=seed, T=prefill_tokens, H=PREFILL["H"], d=PREFILL["d"], W=PREFILL["W"])
    t0 = time.perf_counter()
    O.mixer(c.q, c.k, c.v, c.g, c.beta, gate=c.gate, conv_w=c.conv_w, use_qk_l2norm=True)
    tp = time.perf_counter() - t0
    dc = KI.decode_case(seed=seed, N=decode_seqs, H=DECODE["H"], d=DECODE["d"], W=DECODE["W"])
    t0 = time.perf_counter()
    O.decode_step(dc.q, dc.k, dc.v, dc.g, dc.beta, dc.state, gate=dc.gate, conv_w=dc.conv_w,
                  conv_state=dc.conv_state)
    td = time.perf_counter() - t0
    return tp, td, O.num_threads()


def cpu_f32_sample(prefill_tokens, seed=0):
    """Time the FP32 per-token CPU baseline on the first `prefill_tokens` tokens of the fused-mixer
    workload (all 32 heads); return the seconds and the threads used."""
    import kda_inputs as KI
    import oracle as O
    O.load_cpu_f32()
    c = KI.fused_mixer(seed=seed, T=prefill_tokens, H=PREFILL["H"], d=PREFILL["d"], W=PREFILL["W"])
    t0 = time.perf_counter()
    O.cpu_f32_mixer(c.q, c.k, c.v, c.g, c.beta, gate=c.gate, conv_w=c.conv_w)
    return time.perf_counter() - t0, O.cpu_f32_threads()


def parity_refs():
    """The oracle's results on one small seeded case of each workload (run in the CPU leg)."""
    import kda_inputs as KI
    import oracle as O
    cases = {
        "core_fp32": (KI.core_fp32(seed=0), "T=64 H=2 d=16 chunk 16 fp32, q/k unit rows, seed 0", "1e-5 max-abs"),
        "chunked_prefill": (KI.chunked_prefill(seed=0, T=1000, H=4), "T=1000 H=4 d=128 chunk 64 bf16, seed 0",
                            "5e-3 x RMS"),
        "varlen_prefill": (KI.prefill_case("varlen_parity", [300, 65, 1, 700], 4, 128, 128, 64, "bf16", seed=0,
                                           s0_std=0.02),
                           "4 sequences (300, 65, 1, 700 tokens) H=4 d=128 bf16, S0 ~ N(0, 0.02), seed 0",
                           "5e-3 x RMS"),
        "fused_mixer": (KI.fused_mixer(seed=0, T=777, H=4), "T=777 H=4 d=128 conv 4 gate bf16, seed 0", "5e-3 x RMS"),
    }
    refs = {}
    for name, (c, desc, bar) in cases.items():
        o, S, _ = O.mixer(c.q, c.k, c.v, c.g, c.beta, initial_state=c.S0, gate=c.gate, conv_w=c.conv_w,
                          cu_seqlens=c.cu_seqlens, scale=c.scale, use_qk_l2norm=c.use_qk_l2norm)
        refs[name] = {"case": c, "desc": desc, "bar": bar, "want": [o, S]}
    d = KI.decode_case(seed=0, N=16, H=4, d=128)
    o, S, _ = O.decode_step(d.q, d.k, d.v, d.g, d.beta, d.state, gate=d.gate, conv_w=d.conv_w,
                            conv_state=d.conv_state)
    d.in_dtype = "bf16"
    refs["decode"] = {"case": d, "desc": "N=16 H=4 d=128 conv 4 gate bf16, fp32 state, seed 0", "bar": "5e-3 x RMS",
                      "want": [o, S]}
    return refs


def cpu_value(tp, td, prefill_tokens, decode_seqs):
    """Composite tokens/s of the oracle, scaled to the full step's token counts."""
    t_step = tp * PREFILL["T"] / prefill_tokens + td * DECODE["N"] / decode_seqs
    return (PREFILL["T"] + DECODE["N"]) / t_step, t_step


def run_reference(args):
    tok, seqs = max(256, args.cpu_sample_tokens // 4), 64
    cpu_oracle_sample(64, 4)                                # load + warm the library
    for _ in range(args.warmup):
        cpu_oracle_sample(256, 8)
    times = []
    for s in range(args.steps):
        tp, td, th = cpu_oracle_sample(tok, seqs, seed=s)
        times.append(cpu_value(tp, td, tok, seqs)[1])
    t_step = float(np.mean(times))
    v = (PREFILL["T"] + DECODE["N"]) / t_step
    sample = (f"each step: oracle fused mixer on the first {tok} of {PREFILL['T']} tokens (all 32 heads) and "
              f"decode on {seqs} of {DECODE['N']} sequences, times scaled to the full step")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "KDA mixer step: fused prefill T=65536 H=32 d=128 chunk64 conv4 gate + "
                                   "decode step N=256 H=32 d=128 conv4 gate", "prefill": PREFILL, "decode": DECODE},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": th, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.prefill_tokens:
        PREFILL["T"] = int(args.prefill_tokens)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    # the CPU baseline leg runs before any CUDA work of the timed arm, on rank 0 at N=1 only: the
    # oracle (FP64) and the FP32 per-token loop timed on a sample of the step, and the oracle's
    # results on the small parity cases
    cpu = cpu32 = refs = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok, seqs = args.cpu_sample_tokens, 64
        tp, td, th = cpu_oracle_sample(tok, seqs)
        v, _ = cpu_value(tp, td, tok, seqs)
        cpu = {"value": v, "unit": "tokens/s", "cores": th, "kind": "oracle",
               "sample": f"oracle fused mixer on the first {tok} of {PREFILL['T']} tokens (all 32 heads, "
                         f"{tp:.1f} s) + decode on {seqs} of {DECODE['N']} sequences ({td:.1f} s), "
                         f"scaled to the full step"}
        t32, th32 = cpu_f32_sample(tok)
        cpu32 = {"value": PREFILL["T"] / (t32 * PREFILL["T"] / tok), "unit": "tokens/s", "cores": th32,
                 "kind": "CPU baseline: FP32 per-token loop, the oracle's threading",
                 "sample": f"fused mixer prefill on the first {tok} of {PREFILL['T']} tokens (all 32 heads, "
                           f"{t32:.1f} s), scaled to the full prefill; prefill tokens/s"}
        refs = parity_refs()
    res = run_ours(args, rank, world, dev, torch)
    res["cpu_baseline"] = cpu
    res["cpu_baseline_f32"] = cpu32
    if refs is not None:
        import hybrid_linear_attention_rule_gb300 as K
        res["parity"] = run_parity(K, torch, refs)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
