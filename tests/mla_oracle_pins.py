"""Pins that tie the MLA decode oracle to facts other than itself.

Each pin runs the oracle (through a given ctypes library handle, so that the
same pins can run against deliberately mutated builds) on a small input whose
answer is fixed by mathematics or by a library routine, and returns
(max_abs_error, tolerance).  The operation pinned is one decode token of the
hybrid's gated attention layers (metrale kimi_k3 docs, mla_decode_token:
optional RoPE, append K/V, scaled dot-product attention, optional output gate).
"""
from __future__ import annotations

import numpy as np
import scipy.special
import torch

import oracle.mla as M


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _rope_complex(x, pos, rd, theta):
    """RoPE written as complex rotation: z_i = x_i + 1j x_{i+rd/2} turned by pos * theta^(-2i/rd)."""
    x = np.array(x, dtype=np.float64)
    if rd == 0:
        return x
    half = rd // 2
    i = np.arange(half)
    z = x[..., :half] + 1j * x[..., half:rd]
    z = z * np.exp(1j * np.asarray(pos, dtype=np.float64)[..., None] * theta ** (-2.0 * i / rd))
    x[..., :half], x[..., half:rd] = z.real, z.imag
    return x


def _torch_bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def pin_round_bf16_matches_torch(lib):
    """Nearest-bf16 rounding against torch's float32 -> bfloat16 conversion on float32 values,
    including exact ties, subnormals and values that overflow to infinity."""
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(3.0),
        np.float32(1.0) + np.arange(0, 64, dtype=np.float32) * np.float32(2.0 ** -8),   # ties and halves
        -(np.float32(1.0) + np.arange(0, 64, dtype=np.float32) * np.float32(2.0 ** -8)),
        np.array([3.38e38, 3.3961e38, 3.3963e38, -3.4e38, 1e-39, 3e-40, 1.2e-38, 0.0], dtype=np.float32),
    ])
    got = M.round_bf16(x, lib=lib)
    ref = _torch_bf16(x)
    inf_ok = np.array_equal(np.isinf(got), np.isinf(ref)) and np.array_equal(np.sign(got[np.isinf(got)]),
                                                                               np.sign(ref[np.isinf(ref)]))
    fin = np.isfinite(ref)
    err = float(np.max(np.abs(got[fin] - ref[fin]))) if inf_ok else np.inf
    return err, 0.0


def pin_rope_complex_form(lib):
    """Rotate-half RoPE equals the complex rotation z_i * exp(i pos theta^(-2i/rd)) on the first rd
    dims and leaves the rest alone; position 0 is the identity."""
    rng = np.random.default_rng(2)
    err = 0.0
    for d, rd, theta in ((16, 16, 10000.0), (24, 8, 500.0), (8, 0, 1.0)):
        x = _rand(rng, 5, d)
        pos = np.array([0, 1, 7, 1000, 123456])
        got = M.rope(x, pos, rd, theta, lib=lib)
        err = max(err, float(np.max(np.abs(got - _rope_complex(x, pos, rd, theta)))))
        err = max(err, float(np.max(np.abs(got[0] - x[0]))))
    return err, 1e-12


def pin_rope_relative_position(lib):
    """RoPE scores depend on positions only through their difference and rotation keeps norms."""
    rng = np.random.default_rng(3)
    d, rd, th = 32, 32, 10000.0
    q, k = _rand(rng, d), _rand(rng, d)
    err = 0.0
    for p, pk, delta in ((5, 2, 11), (100, 100, 3), (40, 0, 997)):
        a = M.rope(q, p, rd, th, lib=lib) @ M.rope(k, pk, rd, th, lib=lib)
        b = M.rope(q, p + delta, rd, th, lib=lib) @ M.rope(k, pk + delta, rd, th, lib=lib)
        err = max(err, abs(a - b), abs(np.linalg.norm(M.rope(q, p, rd, th, lib=lib)) - np.linalg.norm(q)))
    return err, 1e-11


def pin_empty_cache_returns_value(lib):
    """A first token attends only to itself: out = v * sigmoid(gate), the key lands in row 0 and the
    length becomes 1 (bf16 cache: the value as stored, i.e. rounded to bf16)."""
    rng = np.random.default_rng(4)
    N, H, d, L = 2, 3, 16, 5
    q, k, v, gate = (_rand(rng, N, H, d) for _ in range(4))
    kc, vc = np.zeros((N, H, L, d)), np.zeros((N, H, L, d))
    err = 0.0
    for bf in (False, True):
        out, kc2, vc2, lens = M.decode_step(q, k, v, kc, vc, [0, 0], 0.25, gate=gate, rope_dim=8,
                                            theta=100.0, cache_bf16=bf, lib=lib)
        vs = _torch_bf16(v.astype(np.float32)) if bf else v
        ks = _torch_bf16(k.astype(np.float32)) if bf else k
        err = max(err, float(np.max(np.abs(out - vs * scipy.special.expit(gate)))))
        err = max(err, float(np.max(np.abs(kc2[:, :, 0] - ks))), float(np.max(np.abs(vc2[:, :, 0] - vs))))
        err = max(err, float(np.max(np.abs(kc2[:, :, 1:]))), float(np.abs(lens - 1).max()))
    return err, 1e-14


def pin_attention_matches_scipy_softmax(lib):
    """NoPE, f32 cache: the output is softmax(scale K q) V over the cached rows plus the new one,
    computed here with scipy's softmax and a matrix product, times sigmoid(gate)."""
    rng = np.random.default_rng(5)
    N, H, dqk, dv, L = 3, 2, 12, 10, 9
    q, k = _rand(rng, N, H, dqk), _rand(rng, N, H, dqk)
    v, gate = _rand(rng, N, H, dv), _rand(rng, N, H, dv)
    kc, vc = _rand(rng, N, H, L, dqk), _rand(rng, N, H, L, dv)
    lens = np.array([0, 4, L - 1])
    scale = 0.3
    out, _, _, _ = M.decode_step(q, k, v, kc, vc, lens, scale, gate=gate, lib=lib)
    err = 0.0
    for n in range(N):
        for h in range(H):
            K = np.vstack([kc[n, h, :lens[n]], k[n, h]])
            V = np.vstack([vc[n, h, :lens[n]], v[n, h]])
            w = scipy.special.softmax(scale * (K @ q[n, h]))
            ref = (w @ V) * scipy.special.expit(gate[n, h])
            err = max(err, float(np.max(np.abs(out[n, h] - ref))))
    return err, 1e-12


def pin_equal_keys_average_values(lib):
    """When every key (cached and new) is the same row, the weights are uniform and the output is the
    mean of the value rows, whatever q and the scale."""
    rng = np.random.default_rng(6)
    N, H, d, L, pos = 1, 2, 8, 7, 6
    row = _rand(rng, d)
    kc = np.broadcast_to(row, (N, H, L, d)).copy()
    k = np.broadcast_to(row, (N, H, d)).copy()
    q, v = 5 * _rand(rng, N, H, d), _rand(rng, N, H, d)
    vc = _rand(rng, N, H, L, d)
    out, _, _, _ = M.decode_step(q, k, v, kc, vc, [pos], 2.0, lib=lib)
    ref = (vc[:, :, :pos].sum(axis=2) + v) / (pos + 1)
    return float(np.max(np.abs(out - ref))), 1e-12


def pin_dominant_key_selects_its_value(lib):
    """A key that scores 60 above all others takes all the weight: the others add under 30 e^-60,
    far below double rounding."""
    rng = np.random.default_rng(7)
    d, L, pos, j = 8, 6, 5, 2
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 1.0
    kc = np.zeros((1, 1, L, d)); kc[0, 0, j, 0] = 60.0
    k = np.zeros((1, 1, d))
    vc, v = _rand(rng, 1, 1, L, d), _rand(rng, 1, 1, d)
    out, _, _, _ = M.decode_step(q, k, v, kc, vc, [pos], 1.0, lib=lib)
    return float(np.max(np.abs(out[0, 0] - vc[0, 0, j]))), 1e-14


def pin_append_and_full_cache(lib):
    """The step writes only row pos of each (sequence, head) and adds one to the length; a sequence
    whose cache is full (or whose length is negative) gets NaN outputs and keeps cache and length."""
    rng = np.random.default_rng(8)
    N, H, d, L = 4, 2, 6, 5
    q, k, v = (_rand(rng, N, H, d) for _ in range(3))
    kc, vc = _rand(rng, N, H, L, d), _rand(rng, N, H, L, d)
    lens = np.array([2, L, L - 1, -1])
    out, kc2, vc2, lens2 = M.decode_step(q, k, v, kc, vc, lens, 0.5, rope_dim=4, theta=50.0, lib=lib)
    err = float(np.abs(lens2 - np.array([3, L, L, -1])).max())
    for n in range(N):
        touched = [lens[n]] if 0 <= lens[n] < L else []
        for t in range(L):
            if t in touched:
                kr = _rope_complex(k[n], np.full(H, lens[n]), 4, 50.0)
                err = max(err, float(np.max(np.abs(kc2[n, :, t] - kr))), float(np.max(np.abs(vc2[n, :, t] - v[n]))))
            else:
                err = max(err, float(np.max(np.abs(kc2[n, :, t] - kc[n, :, t]))),
                          float(np.max(np.abs(vc2[n, :, t] - vc[n, :, t]))))
        nan_expected = not touched
        if bool(np.all(np.isnan(out[n]))) != nan_expected or (not nan_expected and np.any(np.isnan(out[n]))):
            err = np.inf
    return err, 1e-12


def pin_permutation_invariance(lib):
    """Without RoPE, attention does not depend on the order of the cached rows."""
    rng = np.random.default_rng(9)
    N, H, d, L, pos = 1, 3, 8, 10, 9
    q, k, v = (_rand(rng, N, H, d) for _ in range(3))
    kc, vc = _rand(rng, N, H, L, d), _rand(rng, N, H, L, d)
    perm = np.concatenate([rng.permutation(pos), np.arange(pos, L)])
    a, _, _, _ = M.decode_step(q, k, v, kc, vc, [pos], 0.7, lib=lib)
    b, _, _, _ = M.decode_step(q, k, v, kc[:, :, perm], vc[:, :, perm], [pos], 0.7, lib=lib)
    return float(np.max(np.abs(a - b))), 1e-12


def pin_token_by_token_equals_causal_attention(lib):
    """T decode steps from an empty cache give causal attention over the whole sequence with RoPE
    at each token's own position: out_t = softmax_j<=t(scale R_t q_t . R_j k_j) v_j, built here
    from the complex form of the rotation and scipy's softmax."""
    rng = np.random.default_rng(10)
    T, H, d, rd, th, scale = 7, 2, 8, 6, 30.0, 0.45
    Q, K, V, G = (_rand(rng, T, H, d) for _ in range(4))
    kc, vc = np.zeros((1, H, T, d)), np.zeros((1, H, T, d))
    lens = np.array([0])
    err = 0.0
    Kr = _rope_complex(K, np.arange(T)[:, None].repeat(H, 1), rd, th)
    Qr = _rope_complex(Q, np.arange(T)[:, None].repeat(H, 1), rd, th)
    for t in range(T):
        out, kc, vc, lens = M.decode_step(Q[t][None], K[t][None], V[t][None], kc, vc, lens, scale, gate=G[t][None],
                                          rope_dim=rd, theta=th, lib=lib)
        for h in range(H):
            w = scipy.special.softmax(scale * (Kr[:t + 1, h] @ Qr[t, h]))
            ref = (w @ V[:t + 1, h]) * scipy.special.expit(G[t, h])
            err = max(err, float(np.max(np.abs(out[0, h] - ref))))
    return err, 1e-12


ALL_PINS = [pin_round_bf16_matches_torch, pin_rope_complex_form, pin_rope_relative_position,
            pin_empty_cache_returns_value, pin_attention_matches_scipy_softmax, pin_equal_keys_average_values,
            pin_dominant_key_selects_its_value, pin_append_and_full_cache, pin_permutation_invariance,
            pin_token_by_token_equals_causal_attention]


def failing_pins(lib):
    """Names of the pins a given oracle build fails (an exception counts as a failure)."""
    bad = []
    for p in ALL_PINS:
        try:
            err, tol = p(lib)
            if not (err <= tol):
                bad.append(p.__name__)
        except Exception:                      # noqa: BLE001 - a crash is a failed pin
            bad.append(p.__name__)
    return bad
