"""Shared helpers for the GPU parity tests: move a seeded case to the device,
run the CUDA path through the C ABI, run the oracle on the same values
(optionally on a subset of heads, which are independent), and compare.

Tolerances (written here, used by every parity test):
  fp32 workloads      max |gpu - oracle| <= 1e-5 on outputs and final states
  bf16-input workloads max |gpu - oracle| <= 5e-3 * RMS(oracle) per tensor, on
                      fp32-stored outputs and fp32 final states;
                      bf16-stored outputs: |err_i| <= 5e-3 * RMS + 2^-8 |ref_i|
                      (the second term is the bf16 store's own rounding)
The oracle consumes the exact values the GPU receives (bf16 inputs widened),
so input rounding is not counted as error.
"""
from __future__ import annotations

import numpy as np
import torch

import hybrid_linear_attention_rule_gb300 as K
import kda_inputs as KI
import oracle as O

FP32_TOL = 1e-5
BF16_REL = 5e-3


def dev_tensor(x, bf16, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(x))
    t = t.to(torch.bfloat16) if bf16 else t
    return t.to(device)


def case_to_device(c: KI.KdaCase):
    bf = c.in_dtype == "bf16"
    d = dict(q=dev_tensor(c.q, bf), k=dev_tensor(c.k, bf), v=dev_tensor(c.v, bf),
             g=dev_tensor(c.g, False), beta=dev_tensor(c.beta, False),
             cu=torch.from_numpy(c.cu_seqlens.copy()))
    d["S0"] = None if c.S0 is None else dev_tensor(c.S0, False)
    d["gate"] = None if c.gate is None else dev_tensor(c.gate, bf)
    d["conv_w"] = None if c.conv_w is None else dev_tensor(c.conv_w, False)
    d["conv_state"] = None
    if c.conv_w is not None:
        if c.conv_state is not None:
            d["conv_state"] = dev_tensor(c.conv_state, False)
        else:
            d["conv_state"] = torch.zeros((c.N, c.W - 1, 2 * c.H * c.dk + c.H * c.dv), dtype=torch.float32,
                                          device="cuda")
    return d


def run_prefill(c: KI.KdaCase, out_dtype=torch.float32, d=None, min_workspace=False):
    """min_workspace=True gives the prefill the smallest workspace it accepts, which selects
    the single-pass tensor-core kernel instead of the two-pass one for bf16 d = 128 shapes."""
    d = d or case_to_device(c)
    out, fs = K.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["S0"], cu_seqlens=d["cu"],
                        chunk=c.chunk, scale=c.scale, use_qk_l2norm=c.use_qk_l2norm, conv_weight=d["conv_w"],
                        conv_state=d["conv_state"], gate=d["gate"], out_dtype=out_dtype,
                        min_workspace=min_workspace)
    torch.cuda.synchronize()
    return out, fs, d


def head_subset(c: KI.KdaCase, heads):
    """The same workload restricted to some heads (heads never interact)."""
    heads = list(heads)
    H, dk, dv = c.H, c.dk, c.dv
    sub = KI.KdaCase(name=c.name + "_heads", T=c.T, H=len(heads), dk=dk, dv=dv, chunk=c.chunk,
                     in_dtype=c.in_dtype, cu_seqlens=c.cu_seqlens, q=c.q[:, heads], k=c.k[:, heads],
                     v=c.v[:, heads], g=c.g[:, heads], beta=c.beta[:, heads], scale=c.scale,
                     use_qk_l2norm=c.use_qk_l2norm)
    if c.S0 is not None:
        sub.S0 = c.S0[:, heads]
    if c.gate is not None:
        sub.gate = c.gate[:, heads]
    if c.conv_w is not None:
        idx = _conv_channels(H, dk, dv, heads)
        sub.conv_w = c.conv_w[idx]
        if c.conv_state is not None:
            sub.conv_state = c.conv_state[:, :, idx]
    return sub


def _conv_channels(H, dk, dv, heads):
    q = [h * dk + i for h in heads for i in range(dk)]
    k = [H * dk + h * dk + i for h in heads for i in range(dk)]
    v = [2 * H * dk + h * dv + i for h in heads for i in range(dv)]
    return np.array(q + k + v)


def oracle_prefill(c: KI.KdaCase):
    o, S, cs = O.mixer(c.q, c.k, c.v, c.g, c.beta, initial_state=c.S0, gate=c.gate, conv_w=c.conv_w,
                       conv_state=c.conv_state, cu_seqlens=c.cu_seqlens, scale=c.scale,
                       use_qk_l2norm=c.use_qk_l2norm)
    return o, S, cs


def max_err(a, b):
    return float(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)).max()) if np.size(a) else 0.0


def rms(x):
    x = np.asarray(x, np.float64)
    return float(np.sqrt((x * x).mean())) if x.size else 0.0


def assert_close(gpu, ref, fp32, what, store_bf16=False):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite values"
    if gpu.size == 0:
        return 0.0
    err = np.abs(gpu - ref)
    if fp32:
        tol = FP32_TOL
        bad = err > tol
    else:
        r = rms(ref)
        tol = BF16_REL * r
        bad = err > (np.maximum(tol, (2.0 ** -8) * np.abs(ref)) if store_bf16 else tol)
    assert not bad.any(), (f"{what}: max err {err.max():.3e} (tol {tol:.3e}, rms {rms(ref):.3e}); "
                           f"{int(bad.sum())} of {err.size} elements out of tolerance")
    return float(err.max())


def to_np(t):
    return t.detach().float().cpu().numpy()
