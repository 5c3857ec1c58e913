"""Property-based checks of the CPU oracles over random shapes, lengths and chunk sizes (no GPU):
the fixed-seed pins of oracle_pins.py and mla_oracle_pins.py, swept by hypothesis."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle as O  # noqa: E402
import oracle.mla as OM  # noqa: E402

SETTINGS = settings(max_examples=25, deadline=None)


def _inputs(seed, T, H, dk, dv, decay=1.0):
    rng = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    q, k = unit(rng.standard_normal((T, H, dk))), unit(rng.standard_normal((T, H, dk)))
    v = rng.standard_normal((T, H, dv))
    g = -decay * np.logaddexp(0.0, rng.standard_normal((T, H, dk)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, g, beta


@SETTINGS
@given(seed=st.integers(0, 10**6), lens=st.lists(st.integers(0, 40), min_size=1, max_size=4),
       H=st.integers(1, 3), dk=st.sampled_from([2, 4, 8]), dv=st.sampled_from([2, 3, 8]),
       chunk=st.sampled_from([1, 2, 4, 16, 64]))
def test_chunked_equals_recurrent_over_varlen(seed, lens, H, dk, dv, chunk):
    T = sum(lens)
    q, k, v, g, beta = _inputs(seed, T, H, dk, dv)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    S0 = 0.1 * np.random.default_rng(seed + 1).standard_normal((len(lens), H, dk, dv))
    o1, s1 = O.recurrent(q, k, v, g, beta, initial_state=S0, cu_seqlens=cu, scale=0.5)
    o2, s2 = O.chunked(q, k, v, g, beta, initial_state=S0, cu_seqlens=cu, scale=0.5, chunk=chunk)
    assert np.abs(o1 - o2).max(initial=0.0) < 1e-10 and np.abs(s1 - s2).max() < 1e-10


@SETTINGS
@given(seed=st.integers(0, 10**6), lens=st.lists(st.integers(1, 30), min_size=2, max_size=4))
def test_packed_sequences_equal_separate_runs(seed, lens):
    H, dk, dv = 2, 4, 3
    T = sum(lens)
    q, k, v, g, beta = _inputs(seed, T, H, dk, dv)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, s = O.recurrent(q, k, v, g, beta, cu_seqlens=cu, scale=0.7)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        on, sn = O.recurrent(q[sl], k[sl], v[sl], g[sl], beta[sl], scale=0.7)
        assert np.array_equal(o[sl], on) and np.array_equal(s[n], sn[0])


@SETTINGS
@given(seed=st.integers(0, 10**6), T=st.integers(1, 24), c=st.floats(-3, 3))
def test_linear_in_values_and_initial_state(seed, T, c):
    H, dk, dv = 2, 3, 4
    q, k, v1, g, beta = _inputs(seed, T, H, dk, dv)
    rng = np.random.default_rng(seed + 7)
    v2 = rng.standard_normal(v1.shape)
    Sa, Sb = rng.standard_normal((1, H, dk, dv)), rng.standard_normal((1, H, dk, dv))
    oa, sa = O.recurrent(q, k, v1, g, beta, initial_state=Sa)
    ob, sb = O.recurrent(q, k, v2, g, beta, initial_state=Sb)
    oc, sc = O.recurrent(q, k, v1 + c * v2, g, beta, initial_state=Sa + c * Sb)
    assert np.abs(oc - (oa + c * ob)).max() < 1e-10 and np.abs(sc - (sa + c * sb)).max() < 1e-10


@SETTINGS
@given(seed=st.integers(0, 10**6), T=st.integers(2, 20), cut=st.integers(1, 19))
def test_prefill_splits_at_any_token(seed, T, cut):
    cut = min(cut, T - 1)
    H, dk, dv = 2, 4, 4
    q, k, v, g, beta = _inputs(seed, T, H, dk, dv)
    o, s = O.recurrent(q, k, v, g, beta, scale=0.9)
    o1, s1 = O.recurrent(q[:cut], k[:cut], v[:cut], g[:cut], beta[:cut], scale=0.9)
    o2, s2 = O.recurrent(q[cut:], k[cut:], v[cut:], g[cut:], beta[cut:], initial_state=s1, scale=0.9)
    assert np.abs(np.concatenate([o1, o2]) - o).max() < 1e-12 and np.abs(s2 - s).max() < 1e-12


@SETTINGS
@given(seed=st.integers(0, 10**6), L=st.integers(2, 40), pos=st.integers(0, 39), rd=st.sampled_from([0, 2, 8]))
def test_attention_token_equals_softmax_attention(seed, L, pos, rd):
    pos = min(pos, L - 1)
    rng = np.random.default_rng(seed)
    H, d = 2, 8
    q, k, v, gate = (rng.standard_normal((1, H, d)) for _ in range(4))
    kc, vc = rng.standard_normal((1, H, L, d)), rng.standard_normal((1, H, L, d))
    out, kc2, vc2, lens = OM.decode_step(q, k, v, kc, vc, [pos], 0.4, gate=gate, rope_dim=rd, theta=50.0)
    qr = OM.rope(q, pos, rd, 50.0)
    for h in range(H):
        s = 0.4 * (kc2[0, h, :pos + 1] @ qr[0, h])
        w = np.exp(s - s.max())
        w /= w.sum()
        ref = (w @ vc2[0, h, :pos + 1]) / (1.0 + np.exp(-gate[0, h]))
        assert np.abs(out[0, h] - ref).max() < 1e-12
    assert lens[0] == pos + 1
