"""The chunk algebra of the tensor-core prefill, restated in numpy, against the oracle's
token-by-token recurrence (no GPU).

Per 64-token chunk, with G the in-chunk cumulative log decay (per channel), G_L its last row and D =
G_0 - G_L the channel's decay across the chunk:
    rho = (G_0 + G_L) / 2 where D <= 160 nats, rho = G_0 for the other ("strong") channels;
    E = e^(G - rho), Kh = k E, Qh = q E, Kb = k / E (zero for strong channels), Kd = k e^(G_L - G);
    Akk = diag(beta) strict_lower(Kh Kb^T + Sk), Aqk = lower(Qh Kb^T + Sq), where Sk, Sq are the strong
        channels' exact share sum_c x_ic k_jc e^(G_ic - G_jc);
    Tb = (I + Akk)^-1 diag(beta), W = Tb Kh, U = Tb v, S' = e^rho S,
    V' = U - W S', O = scale (Qh S' + Aqk V'), S_next = e^G_L S + Kd^T V'.
In float64 this must equal the recurrence to rounding, at the workloads' decays and at decays far
beyond the fp32 exponent range.  In float32 no factor and no kept product may overflow (each factor
is within e^(+-80); only the discarded upper triangle of Kh Kb^T may) and the result must stay well
inside the 5e-3 x RMS bar.
"""
import numpy as np
import pytest

import oracle as O

STRONG = 160.0


def chunk_forward(q, k, v, g, beta, S0, scale, C=64):
    dt = q.dtype
    T, d = k.shape
    S = S0.copy()
    out = np.zeros_like(v)
    for c0 in range(0, T, C):
        sl = slice(c0, min(T, c0 + C))
        n = sl.stop - sl.start
        G = np.cumsum(g[sl], axis=0)
        G0, GL = G[0], G[-1]
        strong = (G0 - GL) > STRONG
        rho = np.where(strong, G0, 0.5 * (G0 + GL)).astype(dt)
        E = np.exp(G - rho)
        Eb = np.where(strong, 0.0, np.exp(np.where(strong, 0.0, rho - G))).astype(dt)
        kk, qq = k[sl], q[sl]
        Kh, Qh, Kb, Kd = kk * E, qq * E, kk * Eb, kk * np.exp(GL - G)
        for x in (Kh, Qh, Kb, Kd):
            assert np.isfinite(x).all()
        # above the diagonal (discarded) the factorised product may overflow, as on the GPU; the
        # entries kept are sums of terms <= |x_ic k_jc|
        with np.errstate(over="ignore", invalid="ignore"):
            Ak, Aq = Kh @ Kb.T, Qh @ Kb.T
        low = np.tril(np.ones((n, n), dtype=bool))
        assert np.isfinite(Ak[low]).all() and np.isfinite(Aq[low]).all()
        Ak, Aq = np.where(low, Ak, 0.0).astype(dt), np.where(low, Aq, 0.0).astype(dt)
        if strong.any():
            Gs = G[:, strong]
            P = np.exp(np.minimum(Gs[:, None, :] - Gs[None, :, :], 0.0)).astype(dt)
            Ak = Ak + np.einsum("ic,jc,ijc->ij", kk[:, strong], kk[:, strong], P)
            Aq = Aq + np.einsum("ic,jc,ijc->ij", qq[:, strong], kk[:, strong], P)
        b = beta[sl]
        Akk = b[:, None] * np.tril(Ak, -1)
        Aqk = np.tril(Aq)
        Tb = np.linalg.inv(np.eye(n, dtype=dt) + Akk) * b[None, :]
        W, U = Tb @ Kh, Tb @ v[sl]
        Sp = np.exp(rho)[:, None] * S
        Vp = U - W @ Sp
        out[sl] = scale * (Qh @ Sp + Aqk @ Vp)
        S = np.exp(GL)[:, None] * S + Kd.T @ Vp
    return out, S


def _case(T, d, seed, decay=1.0, pinned=()):
    rng = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    q, k = unit(rng.standard_normal((T, 1, d))), unit(rng.standard_normal((T, 1, d)))
    v = rng.standard_normal((T, 1, d))
    g = -decay * np.logaddexp(0.0, rng.standard_normal((T, 1, d)))
    for c, gv in pinned:
        g[:, :, c] = gv
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, 1))))
    S0 = 0.02 * rng.standard_normal((1, 1, d, d))
    return q, k, v, g, beta, S0


CASES = [(1.0, ()), (4.0, ()), (16.0, ()), (1.0, ((0, -30.0), (3, -80.0), (7, -2.9)))]


@pytest.mark.parametrize("decay,pinned", CASES)
def test_chunk_forward_equals_recurrence_in_float64(decay, pinned):
    q, k, v, g, beta, S0 = _case(200, 16, seed=3, decay=decay, pinned=pinned)
    scale = 0.25
    ro, rs = O.recurrent(q, k, v, g, beta, initial_state=S0, scale=scale)
    o, S = chunk_forward(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0[0, 0], scale)
    err_o = np.abs(o - ro[:, 0]).max() / np.sqrt(np.mean(ro ** 2))
    err_s = np.abs(S - rs[0, 0]).max() / np.sqrt(np.mean(rs ** 2))
    assert max(err_o, err_s) < 1e-11


def test_strong_channels_take_the_exact_share():
    """The workloads' decays leave every channel on the factorised product; 4x those decays and the
    pinned channels put channels past the 160-nat threshold in every chunk."""
    for (decay, pinned), expect in zip(CASES, (False, True, True, True)):
        _, _, _, g, _, _ = _case(200, 16, seed=3, decay=decay, pinned=pinned)
        D = -g[:64, 0].sum(axis=0)
        assert bool((D > STRONG).any()) == expect


@pytest.mark.parametrize("decay,pinned", CASES)
def test_chunk_forward_float32_stays_finite_and_accurate(decay, pinned):
    q, k, v, g, beta, S0 = _case(300, 128, seed=4, decay=decay, pinned=pinned)
    scale = 128 ** -0.5
    ro, rs = O.recurrent(q, k, v, g, beta, initial_state=S0, scale=scale)
    f32 = [x.astype(np.float32) for x in (q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0[0, 0])]
    with np.errstate(over="raise", invalid="raise"):
        o, S = chunk_forward(*f32, np.float32(scale))
    err = max(np.abs(o - ro[:, 0]).max() / np.sqrt(np.mean(ro ** 2)), np.abs(S - rs[0, 0]).max() / np.sqrt(np.mean(rs ** 2)))
    assert err < 5e-5
