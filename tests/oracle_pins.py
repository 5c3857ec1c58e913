"""Pins that tie the CPU oracle to facts other than itself.

Each pin runs the oracle (through a given ctypes library handle, so the same
pins can be run against deliberately mutated builds of the oracle) on a small
input whose answer is fixed by mathematics or by a library routine, and returns
(max_abs_error, tolerance).  The KDA gated delta rule being pinned:
    S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale * S_t^T q_t,  alpha_t = exp(g_t),
with causal Q/K/V short convolutions (+SiLU), q/k L2 norm and a sigmoid output
gate ("Experimental Native Vulkan Backend for Kimi K3", feature list; metrale
kimi_k3 docs, KdaState / kda_decode_token).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import scipy.special

import oracle as O


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def pin_single_token_closed_form(lib):
    """T=1 from a zero state: S_1 = beta k v^T, o_1 = scale * beta (k.q) v."""
    rng = np.random.default_rng(11)
    H, dk, dv = 3, 5, 7
    q, k = _rand(rng, 1, H, dk), _rand(rng, 1, H, dk)
    v, g = _rand(rng, 1, H, dv), -np.abs(_rand(rng, 1, H, dk))
    beta = rng.uniform(0.1, 0.9, (1, H))
    o, S = O.recurrent(q, k, v, g, beta, scale=0.37, lib=lib)
    err = 0.0
    for h in range(H):
        S_ref = beta[0, h] * np.outer(k[0, h], v[0, h])
        o_ref = 0.37 * beta[0, h] * np.dot(k[0, h], q[0, h]) * v[0, h]
        err = max(err, np.abs(S[0, h] - S_ref).max(), np.abs(o[0, h] - o_ref).max())
    return err, 1e-13


def pin_pure_decay(lib):
    """beta = 0: nothing is written or erased, S_t = Diag(prod_{s<=t} alpha_s) S_0."""
    rng = np.random.default_rng(12)
    T, H, dk, dv = 9, 2, 6, 4
    q, k, v = _rand(rng, T, H, dk), _rand(rng, T, H, dk), _rand(rng, T, H, dv)
    g = -np.abs(_rand(rng, T, H, dk)) * 0.3
    S0 = _rand(rng, 1, H, dk, dv)
    o, S = O.recurrent(q, k, v, g, np.zeros((T, H)), initial_state=S0, scale=0.5, lib=lib)
    err = 0.0
    for h in range(H):
        cum = np.cumsum(g[:, h, :], axis=0)          # [T, dk]
        for t in range(T):
            St = np.exp(cum[t])[:, None] * S0[0, h]
            err = max(err, np.abs(o[t, h] - 0.5 * St.T @ q[t, h]).max())
        err = max(err, np.abs(S[0, h] - np.exp(cum[-1])[:, None] * S0[0, h]).max())
    o0, S0out = O.recurrent(q, k, v, g, np.zeros((T, H)), scale=0.5, lib=lib)
    err = max(err, np.abs(o0).max(), np.abs(S0out).max())
    return err, 1e-13


def pin_orthonormal_delta_rule(lib):
    """alpha = 1, beta = 1, orthonormal keys: the delta rule stores each pair exactly,
    S_T = (I - K^T K) S_0 + K^T V, so S_T^T k_s = v_s + ... and a query equal to a stored
    key reads back scale * v_s (plus the part of S_0 orthogonal to nothing stored)."""
    rng = np.random.default_rng(13)
    H, dk, dv, T = 2, 8, 5, 6
    err = 0.0
    for h_seed in range(2):
        Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
        K = Qm[:T]                                   # T orthonormal rows
        V = rng.standard_normal((T, dv))
        S0 = rng.standard_normal((dk, dv)) if h_seed else np.zeros((dk, dv))
        k = np.repeat(K[:, None, :], H, axis=1)
        v = np.repeat(V[:, None, :], H, axis=1)
        q = k.copy()
        q[-1] = K[2]                                 # last query asks for the third key
        g = np.zeros((T, H, dk))
        beta = np.ones((T, H))
        S0b = np.repeat(S0[None, None], H, axis=1)
        o, S = O.recurrent(q, k, v, g, beta, initial_state=S0b, scale=1.0, lib=lib)
        S_ref = (np.eye(dk) - K.T @ K) @ S0 + K.T @ V
        err = max(err, np.abs(S[0, 0] - S_ref).max())
        err = max(err, np.abs(o[-1, 0] - V[2]).max())     # exact retrieval
        for t in range(T):                                # each step reads back its own value
            err = max(err, np.abs(o[t, 1] - V[t]).max() if t < T - 1 else 0.0)
    return err, 1e-12


def pin_repeated_key_overwrites(lib):
    """alpha = 1, beta = 1, the same unit key twice: the newer value replaces the older."""
    rng = np.random.default_rng(14)
    dk, dv = 6, 3
    kvec = _unit_rows(rng.standard_normal(dk))
    k = np.stack([kvec, kvec])[:, None, :]
    v = rng.standard_normal((2, 1, dv))
    S0 = rng.standard_normal((1, 1, dk, dv))
    o, S = O.recurrent(k.copy(), k, v, np.zeros((2, 1, dk)), np.ones((2, 1)), initial_state=S0,
                       scale=1.0, lib=lib)
    err = max(np.abs(S[0, 0].T @ kvec - v[1, 0]).max(), np.abs(o[1, 0] - v[1, 0]).max(),
              np.abs(o[0, 0] - v[0, 0]).max())
    return err, 1e-13


def pin_linearity(lib):
    """Outputs and final state are jointly linear in (v, S_0) when the gate is off."""
    rng = np.random.default_rng(15)
    T, H, dk, dv = 13, 2, 5, 4
    q, k = _rand(rng, T, H, dk), _rand(rng, T, H, dk)
    g = -np.abs(_rand(rng, T, H, dk)) * 0.5
    beta = rng.uniform(0, 1, (T, H))
    v1, v2 = _rand(rng, T, H, dv), _rand(rng, T, H, dv)
    Sa, Sb = _rand(rng, 1, H, dk, dv), _rand(rng, 1, H, dk, dv)
    c = -1.7
    oa, Fa = O.recurrent(q, k, v1, g, beta, initial_state=Sa, lib=lib)
    ob, Fb = O.recurrent(q, k, v2, g, beta, initial_state=Sb, lib=lib)
    oc, Fc = O.recurrent(q, k, v1 + c * v2, g, beta, initial_state=Sa + c * Sb, lib=lib)
    return max(np.abs(oc - (oa + c * ob)).max(), np.abs(Fc - (Fa + c * Fb)).max()), 1e-12


def pin_exact_rational(lib):
    """dk = dv = 2, three tokens, rational alpha/beta/k/v/q: the matrix form of the rule
    evaluated in exact rational arithmetic (Fractions) against the oracle."""
    F = Fraction
    alphas = [[F(1, 2), F(3, 4)], [F(2, 3), F(1, 5)], [F(9, 10), F(1, 3)]]
    betas = [F(1, 3), F(3, 4), F(1, 2)]
    ks = [[F(1), F(2)], [F(-3, 2), F(1, 2)], [F(1, 4), F(-1)]]
    vs = [[F(2), F(-1)], [F(1, 2), F(3)], [F(-2), F(5, 4)]]
    qs = [[F(1), F(-1)], [F(2), F(1, 3)], [F(-1, 2), F(3, 2)]]
    S0 = [[F(1, 7), F(-2, 5)], [F(3, 8), F(1, 9)]]
    scale = F(1, 2)

    def mm(A, B):
        return [[sum(A[i][t] * B[t][j] for t in range(len(B))) for j in range(len(B[0]))]
                for i in range(len(A))]

    S = S0
    outs = []
    for t in range(3):
        k_, a_, b_ = ks[t], alphas[t], betas[t]
        M = [[((1 if i == j else 0) - b_ * k_[i] * k_[j]) * a_[j] for j in range(2)] for i in range(2)]
        S = mm(M, S)
        S = [[S[i][j] + b_ * k_[i] * vs[t][j] for j in range(2)] for i in range(2)]
        outs.append([scale * sum(S[c][j] * qs[t][c] for c in range(2)) for j in range(2)])
    f = lambda x: np.array(x, dtype=np.float64)
    o, Sf = O.recurrent(f(qs)[:, None], f(ks)[:, None], f(vs)[:, None],
                        np.log(f(alphas))[:, None], f(betas)[:, None],
                        initial_state=f(S0)[None, None], scale=0.5, lib=lib)
    err = max(np.abs(o[:, 0] - f(outs)).max(), np.abs(Sf[0, 0] - f(S)).max())
    return err, 1e-14


def pin_bruteforce_agrees(lib):
    """Rank-1 per-token loop vs the dense transition-matrix product, random tiny inputs
    with varlen, initial state and gate."""
    rng = np.random.default_rng(16)
    cu = np.array([0, 5, 5, 17, 20], dtype=np.int32)
    T, H, dk, dv = 20, 2, 6, 5
    args = (_rand(rng, T, H, dk), _unit_rows(_rand(rng, T, H, dk)), _rand(rng, T, H, dv),
            -np.abs(_rand(rng, T, H, dk)), rng.uniform(0, 1, (T, H)))
    S0 = _rand(rng, 4, H, dk, dv)
    gate = _rand(rng, T, H, dv)
    o1, S1 = O.recurrent(*args, initial_state=S0, gate=gate, cu_seqlens=cu, lib=lib)
    o2, S2 = O.bruteforce(*args, initial_state=S0, gate=gate, cu_seqlens=cu, lib=lib)
    return max(np.abs(o1 - o2).max(), np.abs(S1 - S2).max()), 1e-12


def pin_gate_is_sigmoid(lib):
    """The gated output equals the ungated one times scipy's logistic function."""
    rng = np.random.default_rng(17)
    T, H, dk, dv = 7, 2, 4, 3
    args = (_rand(rng, T, H, dk), _rand(rng, T, H, dk), _rand(rng, T, H, dv),
            -np.abs(_rand(rng, T, H, dk)), rng.uniform(0, 1, (T, H)))
    gate = 3 * _rand(rng, T, H, dv)
    o, _ = O.recurrent(*args, lib=lib)
    og, _ = O.recurrent(*args, gate=gate, lib=lib)
    return np.abs(og - o * scipy.special.expit(gate)).max(), 1e-13


def pin_state_chaining(lib):
    """Running T tokens at once equals running T1 then T-T1 from the carried state."""
    rng = np.random.default_rng(18)
    T, T1, H, dk, dv = 23, 9, 2, 5, 6
    q, k, v = _rand(rng, T, H, dk), _unit_rows(_rand(rng, T, H, dk)), _rand(rng, T, H, dv)
    g, beta = -np.abs(_rand(rng, T, H, dk)), rng.uniform(0, 1, (T, H))
    S0 = _rand(rng, 1, H, dk, dv)
    o, S = O.recurrent(q, k, v, g, beta, initial_state=S0, lib=lib)
    oa, Sa = O.recurrent(q[:T1], k[:T1], v[:T1], g[:T1], beta[:T1], initial_state=S0, lib=lib)
    ob, Sb = O.recurrent(q[T1:], k[T1:], v[T1:], g[T1:], beta[T1:], initial_state=Sa, lib=lib)
    return max(np.abs(o - np.concatenate([oa, ob])).max(), np.abs(S - Sb).max()), 1e-13


def pin_varlen_is_independent(lib):
    """A packed varlen run equals separate runs, bit for bit, including empty sequences."""
    rng = np.random.default_rng(19)
    lens = [4, 0, 11, 1, 6]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, H, dk, dv = int(cu[-1]), 2, 4, 5
    q, k, v = _rand(rng, T, H, dk), _rand(rng, T, H, dk), _rand(rng, T, H, dv)
    g, beta = -np.abs(_rand(rng, T, H, dk)), rng.uniform(0, 1, (T, H))
    S0 = _rand(rng, len(lens), H, dk, dv)
    o, S = O.recurrent(q, k, v, g, beta, initial_state=S0, cu_seqlens=cu, lib=lib)
    err = 0.0
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        on, Sn = O.recurrent(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], initial_state=S0[n:n + 1],
                             lib=lib)
        err = max(err, np.abs(o[a:b] - on).max() if b > a else 0.0, np.abs(S[n] - Sn[0]).max())
    err = max(err, np.abs(S[1] - S0[1]).max())     # empty sequence keeps its state
    return err, 0.0


def pin_chunked_equals_recurrent(lib):
    """The chunked (WY/UT) algebra reaches the per-token result for every chunk size."""
    rng = np.random.default_rng(20)
    cu = np.array([0, 37, 38, 101], dtype=np.int32)
    T, H, dk, dv = 101, 2, 8, 6
    args = (_unit_rows(_rand(rng, T, H, dk)), _unit_rows(_rand(rng, T, H, dk)), _rand(rng, T, H, dv),
            -np.logaddexp(0, _rand(rng, T, H, dk)), scipy.special.expit(_rand(rng, T, H)))
    S0 = 0.1 * _rand(rng, 3, H, dk, dv)
    gate = _rand(rng, T, H, dv)
    o, S = O.recurrent(*args, initial_state=S0, gate=gate, cu_seqlens=cu, lib=lib)
    err = 0.0
    for C in (1, 4, 16, 64, 128):
        oc, Sc = O.chunked(*args, initial_state=S0, gate=gate, cu_seqlens=cu, chunk=C, lib=lib)
        err = max(err, np.abs(o - oc).max(), np.abs(S - Sc).max())
    return err, 1e-12


def pin_conv_matches_numpy(lib):
    """Causal depthwise conv = numpy.convolve per channel (full mode, first L outputs,
    taps reversed), with the history rows prepended; SiLU = z * expit(z)."""
    rng = np.random.default_rng(21)
    lens = [7, 2, 12]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, D, W = int(cu[-1]), 5, 4
    x, w = _rand(rng, T, D), _rand(rng, D, W)
    cs = _rand(rng, len(lens), W - 1, D)
    y, cs_out = O.short_conv(x, w, conv_state=cs, cu_seqlens=cu, apply_silu=True, return_state=True,
                             lib=lib)
    err = 0.0
    for n in range(len(lens)):
        xs = np.concatenate([cs[n], x[cu[n]:cu[n + 1]]])          # [W-1+L, D]
        for c in range(D):
            full = np.convolve(xs[:, c], w[c, ::-1])               # y[t] = sum_i w[i] xs[t-(W-1)+i]
            pre = full[W - 1:W - 1 + lens[n]]
            err = max(err, np.abs(y[cu[n]:cu[n + 1], c] - pre * scipy.special.expit(pre)).max())
        err = max(err, np.abs(cs_out[n] - xs[-(W - 1):]).max())
    # impulse: a unit input at t=0 of an empty-history sequence gives back the taps (no SiLU)
    imp = np.zeros((W, D))
    imp[0] = 1.0
    yi = O.short_conv(imp, w, apply_silu=False, lib=lib)
    err = max(err, np.abs(yi - w[:, ::-1].T).max())
    return err, 1e-13


def pin_conv_chaining(lib):
    """Conv over a whole sequence = conv over its first part, then over the rest from the
    carried conv state (including a part shorter than W-1)."""
    rng = np.random.default_rng(22)
    D, W = 6, 4
    x, w = _rand(rng, 15, D), _rand(rng, D, W)
    cs = _rand(rng, 1, W - 1, D)
    y, cs1 = O.short_conv(x, w, conv_state=cs, return_state=True, lib=lib)
    err = 0.0
    for split in (1, 2, 9):
        ya, csa = O.short_conv(x[:split], w, conv_state=cs, return_state=True, lib=lib)
        yb, csb = O.short_conv(x[split:], w, conv_state=csa, return_state=True, lib=lib)
        err = max(err, np.abs(y - np.concatenate([ya, yb])).max(), np.abs(cs1 - csb).max())
    return err, 0.0


def pin_l2norm(lib):
    """Rows divided by numpy's norm (eps aside); scale invariance; eps placement."""
    rng = np.random.default_rng(23)
    x = _rand(rng, 40, 16)
    y = O.l2norm(x, eps=0.0, lib=lib)
    err = np.abs(y - x / np.linalg.norm(x, axis=1, keepdims=True)).max()
    err = max(err, np.abs(O.l2norm(1e3 * x, eps=0.0, lib=lib) - y).max())
    z = np.zeros((1, 16))
    z[0, 3] = 0.5                                   # sum x^2 = 0.25: 0.5 / sqrt(0.25 + 0.75) = 0.5
    err = max(err, abs(O.l2norm(z, eps=0.75, lib=lib)[0, 3] - 0.5))
    return err, 1e-14


def pin_decode_is_one_more_token(lib):
    """A decode step from the state and conv state after L-1 tokens gives the L-th token's
    output, state and conv state of a single L-token mixer run (conv, L2, gate on)."""
    rng = np.random.default_rng(24)
    L, H, dk, dv, W = 10, 2, 4, 3, 4
    D = 2 * H * dk + H * dv
    q, k, v = _rand(rng, L, H, dk), _rand(rng, L, H, dk), _rand(rng, L, H, dv)
    g, beta = -np.abs(_rand(rng, L, H, dk)), rng.uniform(0, 1, (L, H))
    gate, cw = _rand(rng, L, H, dv), _rand(rng, D, W)
    cs0 = _rand(rng, 1, W - 1, D)
    o, S, cs = O.mixer(q, k, v, g, beta, gate=gate, conv_w=cw, conv_state=cs0, lib=lib)
    oa, Sa, csa = O.mixer(q[:-1], k[:-1], v[:-1], g[:-1], beta[:-1], gate=gate[:-1], conv_w=cw,
                          conv_state=cs0, lib=lib)
    od, Sd, csd = O.decode_step(q[-1:], k[-1:], v[-1:], g[-1:], beta[-1:], Sa, gate=gate[-1:],
                                conv_w=cw, conv_state=csa, lib=lib)
    return max(np.abs(od[0] - o[-1]).max(), np.abs(Sd - S).max(), np.abs(csd - cs).max()), 1e-13


def pin_mixer_composition(lib):
    """The mixer equals conv+SiLU on [q|k|v], then numpy-normalised q and k, then the rule."""
    rng = np.random.default_rng(25)
    T, H, dk, dv, W = 9, 2, 4, 3, 3
    D = 2 * H * dk + H * dv
    q, k, v = _rand(rng, T, H, dk), _rand(rng, T, H, dk), _rand(rng, T, H, dv)
    g, beta = -np.abs(_rand(rng, T, H, dk)), rng.uniform(0, 1, (T, H))
    cw = _rand(rng, D, W)
    o, S, _ = O.mixer(q, k, v, g, beta, conv_w=cw, eps=0.0, lib=lib)
    x = np.concatenate([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], axis=1)
    y = O.short_conv(x, cw, lib=lib)
    qc = y[:, :H * dk].reshape(T, H, dk)
    kc = y[:, H * dk:2 * H * dk].reshape(T, H, dk)
    vc = y[:, 2 * H * dk:].reshape(T, H, dv)
    qc = qc / np.linalg.norm(qc, axis=-1, keepdims=True)
    kc = kc / np.linalg.norm(kc, axis=-1, keepdims=True)
    o2, S2 = O.recurrent(qc, kc, vc, g, beta, lib=lib)
    return max(np.abs(o - o2).max(), np.abs(S - S2).max()), 1e-13


def pin_backward_finite_differences(lib):
    """The reverse-mode gradients equal central differences of the forward oracle's loss
    sum(dO * o) + sum(dS_final * S_final), for every element of q, k, v, g, beta and S_0
    (varlen, two heads, decaying, non-unit keys)."""
    rng = np.random.default_rng(31)
    cu = np.array([0, 3, 3, 7], dtype=np.int32)
    T, H, dk, dv = 7, 2, 3, 4
    args = dict(q=_rand(rng, T, H, dk), k=0.5 * _rand(rng, T, H, dk), v=_rand(rng, T, H, dv),
                g=-0.3 * np.abs(_rand(rng, T, H, dk)), beta=rng.uniform(0.1, 0.9, (T, H)),
                S0=0.3 * _rand(rng, 3, H, dk, dv))
    dO, dSf, scale = _rand(rng, T, H, dv), _rand(rng, 3, H, dk, dv), 0.7

    def loss(a):
        o, S = O.recurrent(a["q"], a["k"], a["v"], a["g"], a["beta"], initial_state=a["S0"], cu_seqlens=cu,
                           scale=scale, lib=lib)
        return float((o * dO).sum() + (S * dSf).sum())

    gr = O.recurrent_backward(args["q"], args["k"], args["v"], args["g"], args["beta"], dO, initial_state=args["S0"],
                              dS_final=dSf, cu_seqlens=cu, scale=scale, lib=lib)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", S0="dS0")
    err, eps = 0.0, 1e-6
    for nm, arr in args.items():
        for idx in np.ndindex(arr.shape):
            a1 = {kk: vv.copy() for kk, vv in args.items()}
            a2 = {kk: vv.copy() for kk, vv in args.items()}
            a1[nm][idx] += eps
            a2[nm][idx] -= eps
            fd = (loss(a1) - loss(a2)) / (2 * eps)
            err = max(err, abs(fd - gr[names[nm]][idx]) / max(1.0, abs(fd)))
    return err, 1e-7


def pin_backward_single_token_closed_form(lib):
    """T=1 from a zero state (S_1 = beta k v^T, o = scale beta (k.q) v), by hand: with
    G = dS_final + scale q dO^T and h = G^T k: dq = scale beta k (v.dO), dv = beta h,
    dbeta = h.v, dk = beta G v, dg = 0, dS0 = Diag(alpha) (G - beta k h^T)."""
    rng = np.random.default_rng(32)
    H, dk, dv = 2, 5, 3
    q, k, v = _rand(rng, 1, H, dk), _rand(rng, 1, H, dk), _rand(rng, 1, H, dv)
    g, beta = -np.abs(_rand(rng, 1, H, dk)), rng.uniform(0.1, 0.9, (1, H))
    dO, dSf, scale = _rand(rng, 1, H, dv), _rand(rng, 1, H, dk, dv), 0.45
    gr = O.recurrent_backward(q, k, v, g, beta, dO, dS_final=dSf, scale=scale, lib=lib)
    err = 0.0
    for h in range(H):
        qh, kh, vh, dOh, b = q[0, h], k[0, h], v[0, h], dO[0, h], beta[0, h]
        G = dSf[0, h] + scale * np.outer(qh, dOh)
        hv = G.T @ kh
        want = dict(dq=scale * b * kh * (vh @ dOh), dv=b * hv, dbeta=hv @ vh, dk=b * G @ vh, dg=np.zeros(dk),
                    dS0=np.exp(g[0, h])[:, None] * (G - b * np.outer(kh, hv)))
        got = dict(dq=gr["dq"][0, h], dv=gr["dv"][0, h], dbeta=gr["dbeta"][0, h], dk=gr["dk"][0, h],
                   dg=gr["dg"][0, h], dS0=gr["dS0"][0, h])
        for key in want:
            err = max(err, float(np.abs(np.asarray(want[key]) - np.asarray(got[key])).max()))
    return err, 1e-13


def pin_backward_autograd(lib):
    """The reverse-mode gradients equal torch autograd (float64) through a plain token-by-token
    forward of the gated delta rule, to rounding: an exact check, independent of the oracle's
    hand-written reverse sweep (varlen, two heads, initial state, final-state gradient)."""
    import torch
    rng = np.random.default_rng(33)
    cu = [0, 5, 5, 12]
    T, H, dk, dv = 12, 2, 3, 4
    arrs = dict(q=_rand(rng, T, H, dk), k=0.6 * _rand(rng, T, H, dk), v=_rand(rng, T, H, dv),
                g=-0.4 * np.abs(_rand(rng, T, H, dk)), beta=rng.uniform(0.1, 0.9, (T, H)),
                S0=0.3 * _rand(rng, 3, H, dk, dv))
    dO, dSf, scale = _rand(rng, T, H, dv), _rand(rng, 3, H, dk, dv), 0.55
    ts = {kk: torch.tensor(vv, dtype=torch.float64, requires_grad=True) for kk, vv in arrs.items()}
    loss = torch.zeros((), dtype=torch.float64)
    for n in range(3):
        for h in range(H):
            S = ts["S0"][n, h]
            for t in range(cu[n], cu[n + 1]):
                kt, vt, qt = ts["k"][t, h], ts["v"][t, h], ts["q"][t, h]
                P = torch.exp(ts["g"][t, h])[:, None] * S
                S = P + ts["beta"][t, h] * torch.outer(kt, vt - P.T @ kt)
                loss = loss + (scale * (S.T @ qt) * torch.from_numpy(dO[t, h])).sum()
            loss = loss + (S * torch.from_numpy(dSf[n, h])).sum()
    loss.backward()
    gr = O.recurrent_backward(arrs["q"], arrs["k"], arrs["v"], arrs["g"], arrs["beta"], dO, initial_state=arrs["S0"],
                              dS_final=dSf, cu_seqlens=np.array(cu, dtype=np.int32), scale=scale, lib=lib)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", S0="dS0")
    err = max(float(np.abs(ts[nm].grad.numpy() - gr[names[nm]]).max()) for nm in names)
    return err, 1e-12


ALL_PINS = [pin_single_token_closed_form, pin_pure_decay, pin_orthonormal_delta_rule,
            pin_repeated_key_overwrites, pin_linearity, pin_exact_rational, pin_bruteforce_agrees,
            pin_gate_is_sigmoid, pin_state_chaining, pin_varlen_is_independent,
            pin_chunked_equals_recurrent, pin_conv_matches_numpy, pin_conv_chaining, pin_l2norm,
            pin_decode_is_one_more_token, pin_mixer_composition, pin_backward_finite_differences,
            pin_backward_single_token_closed_form, pin_backward_autograd]


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
