"""Seeded synthetic inputs for the KDA mixer workloads and the attention layers' decode token.

This module only draws random numbers and shapes them; it holds none of the
mixer's arithmetic, so the CPU oracle and the CUDA path can both take their
inputs from it.  Every tensor comes from its own numpy PCG64 stream keyed by
(seed, stream id), so any tensor can be regenerated alone and the draw does
not depend on which other tensors were drawn first.

Distributions (the workloads of the KDA mixer):
  q, k, v      ~ N(0, 1), rounded to bf16 for the bf16 workloads
  g (log-decay) = -softplus(N(0, 1))          so alpha = exp(g) is in (0, 1)
  beta          = sigmoid(N(0, 1))
  gate logits   ~ N(0, 1) (bf16 for the bf16 workloads)
  conv weights  ~ N(0, 0.5)  (0.5 is the standard deviation)
  initial state ~ N(0, 0.02) (0.02 is the standard deviation), fp32
  conv state    ~ N(0, 1) rounded to bf16 values (it holds past pre-conv inputs)
  varlen lengths uniform integers in [256, 16384]
softplus and sigmoid here shape the input distribution; the mixer itself
receives g and beta as given.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

STREAMS = {"q": 1, "k": 2, "v": 3, "g": 4, "beta": 5, "gate": 6, "conv_w": 7, "S0": 8,
           "lengths": 9, "conv_state": 10, "mla_q": 11, "mla_k": 12, "mla_v": 13, "mla_gate": 14,
           "mla_k_cache": 15, "mla_v_cache": 16, "mla_lengths": 17}


def _rng(seed: int, name: str) -> np.random.Generator:
    return np.random.default_rng([int(seed), STREAMS[name]])


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) & np.uint32(0xFFFF0000)).view(np.float32)


def normal(shape, std, seed, name, bf16=False):
    x = _rng(seed, name).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return round_bf16(x) if bf16 else x


def log_decay(shape, seed):
    z = _rng(seed, "g").standard_normal(size=shape, dtype=np.float32)
    return -np.logaddexp(np.float32(0.0), z)


def stronger_decay(g, factor=1.0, pinned=()):
    """The log-decay g scaled by factor, with some channels pinned to a fixed log-decay for every
    token and head ((channel, value) pairs): inputs on which a channel forgets by hundreds to
    thousands of nats within one 64-token chunk (factor 4 gives ~200 nats, 16 ~800)."""
    out = (np.asarray(g, dtype=np.float32) * np.float32(factor)).astype(np.float32)
    for c, val in pinned:
        out[..., c] = np.float32(val)
    return out


def beta_values(shape, seed):
    z = _rng(seed, "beta").standard_normal(size=shape, dtype=np.float32)
    return (np.float32(1.0) / (np.float32(1.0) + np.exp(-z))).astype(np.float32)


def varlen_lengths(n, lo, hi, seed):
    return _rng(seed, "lengths").integers(lo, hi + 1, size=n).astype(np.int64)


@dataclass
class KdaCase:
    """One prefill workload: packed tokens [T] split by cu_seqlens into N sequences."""
    name: str
    T: int
    H: int
    dk: int
    dv: int
    chunk: int
    in_dtype: str                      # "f32" or "bf16": storage type of q, k, v, gate
    cu_seqlens: np.ndarray             # int32 [N+1]
    q: np.ndarray                      # float32 [T, H, dk] (bf16-exact when in_dtype == "bf16")
    k: np.ndarray
    v: np.ndarray                      # float32 [T, H, dv]
    g: np.ndarray                      # float32 [T, H, dk]
    beta: np.ndarray                   # float32 [T, H]
    scale: float
    use_qk_l2norm: bool = True
    S0: np.ndarray | None = None       # float32 [N, H, dk, dv]
    gate: np.ndarray | None = None     # float32 [T, H, dv]
    conv_w: np.ndarray | None = None   # float32 [2*H*dk + H*dv, W]
    conv_state: np.ndarray | None = None  # float32 [N, W-1, 2*H*dk + H*dv]
    meta: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def W(self) -> int:
        return 0 if self.conv_w is None else int(self.conv_w.shape[1])


@dataclass
class DecodeCase:
    """One decode step: one new token for each of N sequences."""
    name: str
    N: int
    H: int
    dk: int
    dv: int
    in_dtype: str
    q: np.ndarray                      # float32 [N, H, dk] pre-conv
    k: np.ndarray
    v: np.ndarray                      # [N, H, dv]
    g: np.ndarray                      # [N, H, dk]
    beta: np.ndarray                   # [N, H]
    state: np.ndarray                  # float32 [N, H, dk, dv]
    scale: float
    use_qk_l2norm: bool = True
    gate: np.ndarray | None = None
    conv_w: np.ndarray | None = None   # [2*H*dk + H*dv, W]
    conv_state: np.ndarray | None = None  # [N, W-1, 2*H*dk + H*dv]

    @property
    def W(self) -> int:
        return 0 if self.conv_w is None else int(self.conv_w.shape[1])


def _cu_from_lengths(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    return cu.astype(np.int32)


def prefill_case(name, lengths, H, dk, dv, chunk, in_dtype="bf16", seed=0, s0_std=None,
                 gate=False, conv_width=0, conv_state=False, use_qk_l2norm=True) -> KdaCase:
    """Generic prefill workload over packed sequences of the given lengths."""
    bf = in_dtype == "bf16"
    cu = _cu_from_lengths(lengths)
    T = int(cu[-1])
    N = len(lengths)
    D = 2 * H * dk + H * dv
    case = KdaCase(
        name=name, T=T, H=H, dk=dk, dv=dv, chunk=chunk, in_dtype=in_dtype, cu_seqlens=cu,
        q=normal((T, H, dk), 1.0, seed, "q", bf), k=normal((T, H, dk), 1.0, seed, "k", bf),
        v=normal((T, H, dv), 1.0, seed, "v", bf), g=log_decay((T, H, dk), seed),
        beta=beta_values((T, H), seed), scale=float(dk) ** -0.5, use_qk_l2norm=use_qk_l2norm)
    if s0_std:
        case.S0 = normal((N, H, dk, dv), s0_std, seed, "S0")
    if gate:
        case.gate = normal((T, H, dv), 1.0, seed, "gate", bf)
    if conv_width:
        case.conv_w = normal((D, conv_width), 0.5, seed, "conv_w")
        if conv_state:
            case.conv_state = normal((N, conv_width - 1, D), 1.0, seed, "conv_state", True)
    return case


# ---- the five workloads (sizes may be scaled down for fast parity runs) ----

def core_fp32(seed=0, T=64, H=2, d=16, chunk=16) -> KdaCase:
    """KDA core in fp32: B=1, T=64, H=2, dk=dv=16, chunk 16; q, k L2-normalised by the
    mixer's norm step; no conv, no gate, zero initial state."""
    return prefill_case("core_fp32_T%d_H%d_d%d" % (T, H, d), [T], H, d, d, chunk, "f32", seed)


def decode_case(seed=0, N=256, H=32, d=128, W=4) -> DecodeCase:
    """Decode step: N independent sequences, H heads, dk=dv=d, fp32 state ~ N(0, 0.02),
    bf16 pre-conv q, k, v, width-W conv with state, sigmoid gate."""
    D = 2 * H * d + H * d
    return DecodeCase(
        name="decode_N%d_H%d_d%d_W%d" % (N, H, d, W), N=N, H=H, dk=d, dv=d, in_dtype="bf16",
        q=normal((N, H, d), 1.0, seed, "q", True), k=normal((N, H, d), 1.0, seed, "k", True),
        v=normal((N, H, d), 1.0, seed, "v", True), g=log_decay((N, H, d), seed),
        beta=beta_values((N, H), seed), state=normal((N, H, d, d), 0.02, seed, "S0"),
        scale=float(d) ** -0.5, gate=normal((N, H, d), 1.0, seed, "gate", True),
        conv_w=normal((D, W), 0.5, seed, "conv_w") if W else None,
        conv_state=normal((N, W - 1, D), 1.0, seed, "conv_state", True) if W else None)


def chunked_prefill(seed=0, T=8192, H=32, d=128, chunk=64) -> KdaCase:
    """Chunked prefill: B=1, bf16 q, k, v (L2 in the mixer), fp32 g and beta, zero S0."""
    return prefill_case("prefill_T%d_H%d_d%d" % (T, H, d), [T], H, d, d, chunk, "bf16", seed)


def varlen_prefill(seed=0, n_seqs=16, lo=256, hi=16384, H=32, d=128, chunk=64) -> KdaCase:
    """Packed varlen prefill: lengths uniform in [lo, hi], nonzero fp32 S0 ~ N(0, 0.02)."""
    lengths = varlen_lengths(n_seqs, lo, hi, seed)
    c = prefill_case("varlen_N%d_%d-%d_H%d_d%d" % (n_seqs, lo, hi, H, d), lengths, H, d, d,
                     chunk, "bf16", seed, s0_std=0.02)
    c.meta["lengths"] = lengths
    return c


def fused_mixer(seed=0, T=65536, H=32, d=128, chunk=64, W=4) -> KdaCase:
    """Full mixer: width-W causal SiLU convs on q, k, v (weights ~ N(0, 0.5)), L2 norm,
    chunked KDA, output * sigmoid(gate); bf16 activations, fp32 state from zero."""
    return prefill_case("mixer_T%d_H%d_d%d_W%d" % (T, H, d, W), [T], H, d, d, chunk, "bf16",
                        seed, gate=True, conv_width=W)


# ---- the gated attention (MLA) layers' decode token ----

@dataclass
class MlaDecodeCase:
    """One decode token of the hybrid's attention layers for N sequences: projected q, k, v of the
    new token, the per-head key/value caches [N, H, L_max, d] (every row filled, so that a read past
    a sequence's length shows), and the cached lengths."""
    name: str
    N: int
    H: int
    d: int
    L_max: int
    in_dtype: str                      # storage type of q, k_new, v_new, gate
    cache_dtype: str                   # storage type of the caches
    q: np.ndarray                      # float32 [N, H, d]
    k_new: np.ndarray                  # [N, H, d]
    v_new: np.ndarray                  # [N, H, dv]
    k_cache: np.ndarray                # float32 [N, H, L_max, d]
    v_cache: np.ndarray                # [N, H, L_max, dv]
    cache_len: np.ndarray              # int32 [N]
    scale: float
    rope_dim: int = 0
    theta: float = 10000.0
    gate: np.ndarray | None = None


def mla_decode_case(name, N, H, d, L_max, lengths, seed=0, in_dtype="bf16", cache_dtype="bf16",
                    rope_dim=0, theta=10000.0, gate=True, dv=None) -> MlaDecodeCase:
    """q, k_new, v_new, gate and the cached rows ~ N(0, 1) (bf16-exact for bf16 storage); lengths
    given explicitly, or as (lo, hi) for uniform integers in [lo, hi]; d is the query/key width,
    dv the value width (default d); scale = d^-1/2."""
    dv = d if dv is None else dv
    bi, bc = in_dtype == "bf16", cache_dtype == "bf16"
    if isinstance(lengths, tuple):
        lens = _rng(seed, "mla_lengths").integers(lengths[0], lengths[1] + 1, size=N)
    else:
        lens = np.asarray(lengths)
    return MlaDecodeCase(
        name=name, N=N, H=H, d=d, L_max=L_max, in_dtype=in_dtype, cache_dtype=cache_dtype,
        q=normal((N, H, d), 1.0, seed, "mla_q", bi), k_new=normal((N, H, d), 1.0, seed, "mla_k", bi),
        v_new=normal((N, H, dv), 1.0, seed, "mla_v", bi),
        k_cache=normal((N, H, L_max, d), 1.0, seed, "mla_k_cache", bc),
        v_cache=normal((N, H, L_max, dv), 1.0, seed, "mla_v_cache", bc),
        cache_len=lens.astype(np.int32), scale=float(d) ** -0.5, rope_dim=rope_dim, theta=theta,
        gate=normal((N, H, dv), 1.0, seed, "mla_gate", bi) if gate else None)
