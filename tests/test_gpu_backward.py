"""Parity of k3kda_backward (through the C ABI) with the FP64 reverse-mode oracle.

The gradients of the ungated recurrence with respect to q, k, v, g, beta and the initial
state, for seeded output and final-state gradients, compared element by element per tensor:
max |gpu - oracle| <= 5e-5 * RMS(oracle) + 1e-6 (FP32 arithmetic on 16-token chunks, whose
rescalings by e^(+-G') bound the cancellation in dg: a numpy restatement of the chunk formulas in
fp32 stays under 1.7e-5 RMS at this chunk length; the oracle receives the exact values the GPU
reads, bf16 inputs widened).  The full-size case is checked on the last tokens of sampled heads:
the oracle runs the forward over the whole
sequence without keeping states, then the reverse sweep over the window from the state it
reached (gradients of tokens in the window depend on earlier tokens only through that state).
"""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_rule_gb300 as K
import kda_inputs as KI
import oracle as O

pytestmark = pytest.mark.gpu

REL = 5e-5


def _case(lengths, H, seed, bf16, s0=True):
    c = KI.prefill_case("bwd", lengths, H, 128, 128, 64, "bf16" if bf16 else "f32", seed=seed,
                        s0_std=0.05 if s0 else None)
    # the recurrence reads q, k as given: unit rows (as after the mixer's L2 norm), exact in bf16
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    c.q, c.k = (KI.round_bf16(unit(x)) if bf16 else unit(x) for x in (c.q, c.k))
    rng = np.random.default_rng(seed + 1000)
    dO = rng.standard_normal((c.T, H, 128))
    dSf = rng.standard_normal((c.N, H, 128, 128)) * 0.1
    return c, dO, dSf


def _run_gpu(c, dO, dSf):
    bf = c.in_dtype == "bf16"
    dev = lambda x, low=False: None if x is None else (torch.from_numpy(np.ascontiguousarray(x)).to(
        torch.bfloat16 if low else torch.float32).cuda())
    q, k, v = dev(c.q, bf), dev(c.k, bf), dev(c.v, bf)
    res = K.backward(q, k, v, dev(c.g), dev(c.beta), dev(dO), initial_state=dev(c.S0), dS_final=dev(dSf),
                     cu_seqlens=torch.from_numpy(c.cu_seqlens.copy()), scale=c.scale)
    torch.cuda.synchronize()
    return {kk: vv.cpu().double().numpy() for kk, vv in res.items()}


def _compare(got, want, what):
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dS0"):
        if key not in want:
            continue
        g, w = got[key], want[key]
        assert g.shape == w.shape, (what, key, g.shape, w.shape)
        assert np.isfinite(g).all(), f"{what} {key}: non-finite"
        if w.size == 0:
            continue
        rms = float(np.sqrt((w * w).mean()))
        err = float(np.abs(g - w).max())
        tol = REL * rms + 1e-6
        assert err <= tol, f"{what} {key}: max err {err:.3e} > tol {tol:.3e} (rms {rms:.3e})"
        print(f"{what} {key}: max err {err:.3e} = {err / max(rms, 1e-30):.2e} rms")


@pytest.mark.parametrize("bf16", [False, True])
def test_backward_varlen_edges(bf16):
    """Empty, one-token, 16-token-chunk -1 / exact / +1, and multi-chunk sequences (with an empty
    one between them), with initial and final-state gradients; an empty sequence passes dS_final
    straight to dS0."""
    c, dO, dSf = _case([0, 1, 15, 16, 17, 0, 63, 64, 65, 130], 2, seed=60, bf16=bf16)
    got = _run_gpu(c, dO, dSf)
    want = O.recurrent_backward(c.q, c.k, c.v, c.g, c.beta, dO, initial_state=c.S0, dS_final=dSf,
                                cu_seqlens=c.cu_seqlens, scale=c.scale)
    _compare(got, want, f"varlen bf16={bf16}")
    assert np.array_equal(got["dS0"][0], dSf[0].astype(np.float32).astype(np.float64))


def test_backward_long_sequence_zero_state():
    """1000 tokens of one head (62 full 16-token chunks and a ragged one), no initial state and
    no final-state gradient."""
    c, dO, _ = _case([1000], 1, seed=61, bf16=True, s0=False)
    got = _run_gpu(c, dO, None)
    want = O.recurrent_backward(c.q, c.k, c.v, c.g, c.beta, dO, cu_seqlens=c.cu_seqlens, scale=c.scale)
    _compare(got, want, "long")


def test_backward_many_chains_in_several_waves():
    """60 sequences of mixed lengths x 4 heads: 240 (sequence, head) pairs, so the chains' launch
    (one CTA per pair and chain, one CTA an SM) runs in several waves; bf16 inputs."""
    lengths = [1 + (37 * i) % 90 for i in range(60)]
    c, dO, dSf = _case(lengths, 4, seed=63, bf16=True, s0=True)
    got = _run_gpu(c, dO, dSf)
    want = O.recurrent_backward(c.q, c.k, c.v, c.g, c.beta, dO, initial_state=c.S0, dS_final=dSf,
                                cu_seqlens=c.cu_seqlens, scale=c.scale)
    _compare(got, want, "many chains")


@pytest.mark.slow
def test_backward_full_size_sampled_window():
    """B=1, T=8192, H=32, bf16 inputs: the last 384 tokens of three sampled heads."""
    c, dO, dSf = _case([8192], 32, seed=62, bf16=True, s0=True)
    got = _run_gpu(c, dO, dSf)
    t0 = c.T - 384
    for h in (0, 17, 31):
        sl = lambda x: np.ascontiguousarray(x[:, h:h + 1])
        _, S_t0 = O.recurrent(sl(c.q)[:t0], sl(c.k)[:t0], sl(c.v)[:t0], sl(c.g)[:t0], sl(c.beta)[:t0],
                              initial_state=c.S0[:, h:h + 1], scale=c.scale)
        want = O.recurrent_backward(sl(c.q)[t0:], sl(c.k)[t0:], sl(c.v)[t0:], sl(c.g)[t0:], sl(c.beta)[t0:],
                                    sl(dO)[t0:], initial_state=S_t0, dS_final=dSf[:, h:h + 1], scale=c.scale)
        want.pop("dS0")
        gw = {kk: got[kk][t0:, h:h + 1] for kk in ("dq", "dk", "dv", "dg", "dbeta")}
        _compare(gw, want, f"full T=8192 head {h}")


def test_backward_rejects_unsupported_head_dim():
    q = torch.zeros(4, 1, 64, device="cuda")
    v = torch.zeros(4, 1, 64, device="cuda")
    with pytest.raises(K.K3KDAError):
        K.backward(q, q, v, q, torch.zeros(4, 1, device="cuda"), v)
