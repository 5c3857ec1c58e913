"""The chunk-algebra derivative that the GPU backward evaluates, restated in numpy, against the
oracle's token-by-token reverse mode (no GPU).

Per chunk, with Gamma the in-chunk cumulative log decay, r = (Gamma_0 + Gamma_L) / 2, G' = Gamma - r:
    Qt = q e^G', Kt = k e^G', Kh = k e^-G', B = strict_lower(Kt Kh^T), Aqk = lower(Qt Kh^T),
    Tm = (I + diag(beta) B)^-1, W = Tm diag(beta) Kt, U = Tm diag(beta) V,
    S' = e^r S, Delta = U - W S', O = scale (Qt S' + Aqk Delta), S_next = e^(Gamma_L - r) (S' + Kh^T Delta),
and its reverse mode (dX = e^(Gamma_L - r) Dout, dDelta = Kh dX + Aqk^T dOs, dR = Tm^T dDelta, ...).
In float64 the restatement must agree with the oracle to rounding for any chunk length; in float32
its error grows with the chunk (the e^(+-G') rescalings), which is why the kernels use 16 tokens.
"""
import numpy as np
import pytest

import oracle as O


def _prep(q, k, v, g, beta, C):
    T = k.shape[0]
    out = []
    for c0 in range(0, T, C):
        sl = slice(c0, min(T, c0 + C))
        G = np.cumsum(g[sl], axis=0)
        r = 0.5 * (G[0] + G[-1])
        Gp = G - r
        Qt, Kt, Kh = q[sl] * np.exp(Gp), k[sl] * np.exp(Gp), k[sl] * np.exp(-Gp)
        n = Kt.shape[0]
        B = np.tril(Kt @ Kh.T, -1)
        b = beta[sl][:, None]
        # Tm by forward substitution, column by column (as the kernels do)
        A = b * B
        Tm = np.zeros((n, n), dtype=q.dtype)
        for col in range(n):
            x = np.zeros(n, dtype=q.dtype)
            for i in range(n):
                x[i] = 1.0 if i == col else (0.0 if i < col else -(A[i, :i] @ x[:i]))
            Tm[:, col] = x
        out.append(dict(sl=sl, G=G, r=r, Gp=Gp, Qt=Qt, Kt=Kt, Kh=Kh, B=B, Tm=Tm, Aqk=np.tril(Qt @ Kh.T),
                        W=Tm @ (b * Kt), U=Tm @ (b * v[sl]), b=b, v=v[sl]))
    return out


def chunk_backward(q, k, v, g, beta, S0, scale, dO, dSf, C):
    P = _prep(q, k, v, g, beta, C)
    S = S0.copy()
    for p in P:                                          # forward: chunk-start states and Delta
        p["Sp"] = np.exp(p["r"])[:, None] * S
        p["D"] = p["U"] - p["W"] @ p["Sp"]
        S = np.exp(p["G"][-1] - p["r"])[:, None] * (p["Sp"] + p["Kh"].T @ p["D"])
        p["Snext"] = S
    res = {n: np.zeros_like(x) for n, x in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta))}
    Dout = dSf.copy()
    for p in reversed(P):
        sl = p["sl"]
        dOs = scale * dO[sl]
        dX = np.exp(p["G"][-1] - p["r"])[:, None] * Dout
        dGL = np.sum(p["Snext"] * Dout, axis=1)
        dD = p["Kh"] @ dX + p["Aqk"].T @ dOs
        dR = p["Tm"].T @ dD
        Dout = np.exp(p["r"])[:, None] * (dX + p["Qt"].T @ dOs - p["Kt"].T @ (p["b"] * dR))
        dA = -np.tril(dR @ p["D"].T, -1)
        dAqk = np.tril(dOs @ p["D"].T)
        Y = dR @ p["Sp"].T
        dQt = dOs @ p["Sp"].T + dAqk @ p["Kh"]
        dKt = p["b"] * (dA @ p["Kh"] - Y)
        dKh = p["D"] @ dX.T + dAqk.T @ p["Qt"] + dA.T @ (p["b"] * p["Kt"])
        res["dv"][sl] = p["b"] * dR
        res["dbeta"][sl] = np.sum(p["v"] * dR, axis=1) - np.sum(p["Kt"] * Y, axis=1) + np.sum(dA * p["B"], axis=1)
        E = np.exp(p["Gp"])
        res["dq"][sl] = dQt * E
        res["dk"][sl] = dKt * E + dKh / E
        dGam = dQt * p["Qt"] + dKt * p["Kt"] - dKh * p["Kh"]
        dGam[-1] += dGL
        res["dg"][sl] = np.cumsum(dGam[::-1], axis=0)[::-1]
    res["dS0"] = Dout
    return res


def _case(T, d, seed):
    rng = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    q, k = unit(rng.standard_normal((T, 1, d))), unit(rng.standard_normal((T, 1, d)))
    v, dO = rng.standard_normal((T, 1, d)), rng.standard_normal((T, 1, d))
    g = -np.logaddexp(0.0, rng.standard_normal((T, 1, d)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, 1))))
    S0, dSf = 0.05 * rng.standard_normal((1, 1, d, d)), 0.1 * rng.standard_normal((1, 1, d, d))
    return q, k, v, g, beta, S0, dO, dSf


def _errors(got, ref):
    out = {}
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dS0"):
        r = ref[n][0, 0] if n == "dS0" else ref[n][:, 0]
        out[n] = float(np.abs(got[n] - r).max() / np.sqrt(np.mean(r * r)))
    return out


@pytest.mark.parametrize("C", [16, 32, 64])
def test_chunk_derivative_equals_reverse_mode_in_float64(C):
    q, k, v, g, beta, S0, dO, dSf = _case(150, 8, seed=C)
    scale = 0.3
    ref = O.recurrent_backward(q, k, v, g, beta, dO, initial_state=S0, dS_final=dSf, scale=scale)
    got = chunk_backward(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0[0, 0], scale, dO[:, 0], dSf[0, 0], C)
    assert max(_errors(got, ref).values()) < 1e-12


def test_float32_error_of_16_token_chunks_is_within_the_backward_bar():
    """At the real head size, fp32 arithmetic on 16-token chunks stays well inside the GPU backward's
    5e-5 x RMS bar, and 64-token chunks do not keep that margin."""
    q, k, v, g, beta, S0, dO, dSf = _case(400, 128, seed=1)
    scale = 128 ** -0.5
    ref = O.recurrent_backward(q, k, v, g, beta, dO, initial_state=S0, dS_final=dSf, scale=scale)
    f32 = [x.astype(np.float32) for x in (q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0[0, 0])]
    err = {}
    for C in (16, 64):
        got = chunk_backward(*f32, np.float32(scale), dO[:, 0].astype(np.float32), dSf[0, 0].astype(np.float32), C)
        err[C] = max(_errors(got, ref).values())
    assert err[16] < 2.5e-5
    assert err[64] > err[16]
