"""The FP32 CPU baseline that the benchmark times beside the oracle computes the mixer: it agrees
with the FP64 oracle to float32 rounding (no GPU)."""
import numpy as np

import kda_inputs as KI
import oracle as O


def _rel(a, b):
    return float(np.abs(a - b).max() / np.sqrt(np.mean(b * b)))


def test_cpu_f32_baseline_matches_the_oracle_on_the_fused_mixer():
    c = KI.fused_mixer(seed=3, T=300, H=2)
    o, S = O.cpu_f32_mixer(c.q, c.k, c.v, c.g, c.beta, gate=c.gate, conv_w=c.conv_w)
    ro, rs, _ = O.mixer(c.q, c.k, c.v, c.g, c.beta, gate=c.gate, conv_w=c.conv_w)
    assert _rel(o, ro) < 1e-4 and _rel(S, rs) < 1e-4


def test_cpu_f32_baseline_without_conv_or_gate():
    c = KI.chunked_prefill(seed=4, T=200, H=2)
    o, S = O.cpu_f32_mixer(c.q, c.k, c.v, c.g, c.beta)
    ro, rs, _ = O.mixer(c.q, c.k, c.v, c.g, c.beta)
    assert _rel(o, ro) < 1e-4 and _rel(S, rs) < 1e-4
