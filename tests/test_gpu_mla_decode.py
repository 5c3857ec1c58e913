"""Parity of k3mla_decode_step (through the C ABI) with the MLA oracle's decode token.

Tolerances: outputs within 1e-5 absolute whenever both sides attend over identical stored
values (fp32 caches, or no RoPE: the appended row is then an exact copy); with RoPE into a
bf16 cache the GPU rounds its fp32 rotation and the oracle its double one, so one element of
the new key may differ by a bf16 step, and the bf16 bar 5e-3 * RMS applies.  bf16-stored
outputs add the store's own rounding (2^-8 relative).  Cache rows other than the appended one
must be bit-identical; the appended row exact without RoPE, within 1e-6 (fp32) or one bf16 step
with it.
"""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_rule_gb300 as K
import kda_inputs as KI
import oracle.mla as OM
from parity_utils import dev_tensor, to_np

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def _to_dev(c: KI.MlaDecodeCase):
    bi, bc = c.in_dtype == "bf16", c.cache_dtype == "bf16"
    return dict(q=dev_tensor(c.q, bi), k=dev_tensor(c.k_new, bi), v=dev_tensor(c.v_new, bi),
                gate=None if c.gate is None else dev_tensor(c.gate, bi),
                kc=dev_tensor(c.k_cache, bc), vc=dev_tensor(c.v_cache, bc),
                lens=torch.from_numpy(c.cache_len.copy()).cuda())


def _oracle(c: KI.MlaDecodeCase, q=None, k=None, v=None, gate=None, kc=None, vc=None, lens=None):
    return OM.decode_step(c.q if q is None else q, c.k_new if k is None else k, c.v_new if v is None else v,
                          c.k_cache if kc is None else kc, c.v_cache if vc is None else vc,
                          c.cache_len if lens is None else lens, c.scale,
                          gate=c.gate if gate is None else gate, rope_dim=c.rope_dim, theta=c.theta,
                          cache_bf16=c.cache_dtype == "bf16")


def _check_out(got, ref, tight, bf16_store, what):
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref), f"{what}: NaN rows differ"
    g, r = got[~nan_ref], ref[~nan_ref]
    if r.size == 0:
        return 0.0
    err = np.abs(g - r)
    bound = 1e-5 if tight else 5e-3 * float(np.sqrt(np.mean(r * r)))
    if bf16_store:
        bound = np.maximum(bound, 2.0 ** -8 * np.abs(r))   # one bf16 ulp of the value, if larger
    assert np.all(err <= bound), f"{what}: max err {err.max():.3e} over bound"
    return float(err.max())


def _check_rows(c, kc_dev, vc_dev, kc_ref, vc_ref, lens_before):
    """Cache rows: appended ones against the oracle, all others unchanged (the oracle's returned
    caches are the inputs with the appended rows written)."""
    kc, vc = to_np(kc_dev).astype(np.float64), to_np(vc_dev).astype(np.float64)
    app = np.zeros(kc.shape[:3], dtype=bool)
    for n, p in enumerate(lens_before):
        if 0 <= p < c.L_max:
            app[n, :, p] = True
    assert np.array_equal(kc[~app], kc_ref[~app]), "key rows outside the appended one changed"
    assert np.array_equal(vc[~app], vc_ref[~app]), "value rows outside the appended one changed"
    assert np.array_equal(vc[app], vc_ref[app]), "appended value row"
    ka, kr = kc[app], kc_ref[app]
    if c.rope_dim == 0:
        assert np.array_equal(ka, kr), "appended key row (no RoPE) must be exact"
    elif c.cache_dtype == "bf16":
        assert np.all(np.abs(ka - kr) <= 2.0 ** -8 * np.abs(kr) + 1e-30), "appended key row beyond one bf16 step"
    else:
        assert np.all(np.abs(ka - kr) <= 1e-6 * (1 + np.abs(kr))), "appended key row (fp32)"


CONFIGS = [  # dqk, dv, in, cache, out, rope_dim, gate
    (128, 128, "bf16", "bf16", "f32", 0, True),
    (128, 128, "bf16", "bf16", "bf16", 64, True),
    (128, 128, "f32", "f32", "f32", 128, False),
    (128, 128, "bf16", "f32", "f32", 0, True),
    (64, 64, "bf16", "bf16", "f32", 0, True),
    (64, 64, "f32", "f32", "f32", 32, True),
    (256, 256, "bf16", "bf16", "f32", 0, False),
    (256, 256, "f32", "f32", "f32", 64, True),
    (192, 128, "bf16", "bf16", "f32", 64, True),     # 128 rotation-free dims + a 64-dim RoPE part
    (192, 128, "f32", "f32", "f32", 64, True),
    (192, 256, "bf16", "bf16", "bf16", 0, True),
    (128, 64, "f32", "bf16", "f32", 32, False),
    (64, 256, "bf16", "f32", "f32", 0, True),
]


@pytest.mark.parametrize("d,dv,ind,cad,outd,rd,gate", CONFIGS,
                         ids=lambda x: str(x) if not isinstance(x, bool) else ("gate" if x else "nogate"))
def test_mla_decode_small_parity(d, dv, ind, cad, outd, rd, gate):
    """12 sequences x 3 heads, L_max = 1100 (three 512-key splits, the last ragged); cached lengths
    0, 1, 15, 16, 17, 511, 512, 513, 1000, L_max - 1 (fills the cache), L_max (full: NaN) and -1;
    query/key width d, value width dv."""
    L = 1100
    lens = [0, 1, 15, 16, 17, 511, 512, 513, 1000, L - 1, L, -1]
    c = KI.mla_decode_case("mla_small", len(lens), 3, d, L, lens, seed=d + dv + rd, in_dtype=ind, cache_dtype=cad,
                           rope_dim=rd, theta=10000.0 if rd != 32 else 500.0, gate=gate, dv=dv)
    t = _to_dev(c)
    out = K.mla_decode_step(t["q"], t["k"], t["v"], t["kc"], t["vc"], t["lens"], gate=t["gate"], scale=c.scale,
                            rope_dim=rd, rope_theta=c.theta, out_dtype=TORCH_DT[outd])
    torch.cuda.synchronize()
    ref, kc_ref, vc_ref, lens_ref = _oracle(c)
    tight = rd == 0 or cad == "f32"
    _check_out(to_np(out).astype(np.float64), ref, tight, outd == "bf16", "out")
    assert np.array_equal(to_np(t["lens"]), lens_ref)
    _check_rows(c, t["kc"], t["vc"], kc_ref, vc_ref, lens)


def test_mla_decode_consecutive_tokens():
    """40 tokens in a row (RoPE, bf16 cache) from lengths 0, 500, 1000 and 1030 with L_max = 1060:
    the appends cross the 512- and 1024-key split edges, the last sequence fills its cache after 30
    tokens and returns NaN from then on; every step is checked against the oracle stepping its own
    copy of the caches."""
    L, H, d, rd = 1060, 2, 128, 64
    c = KI.mla_decode_case("mla_steps", 4, H, d, L, [0, 500, 1000, 1030], seed=3, rope_dim=rd)
    t = _to_dev(c)
    kc_o, vc_o, lens_o = c.k_cache.astype(np.float64), c.v_cache.astype(np.float64), c.cache_len.copy()
    rng = np.random.default_rng(17)
    ws = torch.empty(K.k3mla_decode_workspace_size(4, H, d, d, L), dtype=torch.uint8, device="cuda")
    worst = 0.0
    for step in range(40):
        q, k, v, g = (KI.round_bf16(rng.standard_normal((4, H, d)).astype(np.float32)) for _ in range(4))
        out = K.mla_decode_step(dev_tensor(q, True), dev_tensor(k, True), dev_tensor(v, True), t["kc"], t["vc"],
                                t["lens"], gate=dev_tensor(g, True), scale=c.scale, rope_dim=rd,
                                out_dtype=torch.float32, workspace=ws)
        ref, kc_o, vc_o, lens_o = OM.decode_step(q, k, v, kc_o, vc_o, lens_o, c.scale, gate=g, rope_dim=rd,
                                                 theta=c.theta, cache_bf16=True)
        torch.cuda.synchronize()
        worst = max(worst, _check_out(to_np(out).astype(np.float64), ref, False, False, f"step {step}"))
        assert np.array_equal(to_np(t["lens"]), lens_o)
    assert lens_o.tolist() == [40, 540, 1040, L]


def test_mla_decode_no_sequences():
    e = torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.empty(0, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    lens = torch.empty(0, dtype=torch.int32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    out = K.mla_decode_step(e, e, e, kc, kc.clone(), lens, workspace=ws)
    assert out.shape == (0, 2, 128)


def test_mla_decode_full_size_sampled():
    """The full decode token of the attention layers: 256 sequences x 32 heads, d = 128, bf16 caches
    of L_max = 8192 rows (2 x 17.2 GB), cached lengths uniform in [1, 8191], NoPE with the sigmoid
    gate, in the launch configuration the benchmark times.  Eight seeded (sequence, head) pairs,
    including the longest and the shortest sequence, are checked against the oracle; every
    length must advance by one."""
    N, H, d, L = 256, 32, 128, 8192
    gen = torch.Generator(device="cuda").manual_seed(1234)
    kc = torch.randn(N, H, L, d, generator=gen, device="cuda", dtype=torch.bfloat16)
    vc = torch.randn(N, H, L, d, generator=gen, device="cuda", dtype=torch.bfloat16)
    q, k, v, g = (torch.randn(N, H, d, generator=gen, device="cuda", dtype=torch.bfloat16) for _ in range(4))
    lens_np = np.random.default_rng(99).integers(1, L, size=N).astype(np.int32)
    lens = torch.from_numpy(lens_np).cuda()
    rng = np.random.default_rng(7)
    pairs = [(int(np.argmax(lens_np)), 0), (int(np.argmin(lens_np)), H - 1)] + \
        [(int(n), int(h)) for n, h in zip(rng.integers(0, N, 6), rng.integers(0, H, 6))]
    before = {(n, h): (to_np(kc[n, h, :lens_np[n] + 1]).astype(np.float64),
                       to_np(vc[n, h, :lens_np[n] + 1]).astype(np.float64)) for n, h in pairs}
    out = K.mla_decode_step(q, k, v, kc, vc, lens, gate=g, scale=d ** -0.5, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(lens), lens_np + 1)
    f64 = lambda x: to_np(x).astype(np.float64)
    for n, h in pairs:
        p = int(lens_np[n])
        kh, vh = before[(n, h)]
        kcs = np.zeros((1, 1, p + 1, d)); kcs[0, 0, :p] = kh[:p]
        vcs = np.zeros((1, 1, p + 1, d)); vcs[0, 0, :p] = vh[:p]
        ref, kc_r, vc_r, _ = OM.decode_step(f64(q[n, h])[None, None], f64(k[n, h])[None, None],
                                            f64(v[n, h])[None, None], kcs, vcs, [p], d ** -0.5,
                                            gate=f64(g[n, h])[None, None], cache_bf16=True)
        _check_out(f64(out[n, h]), ref[0, 0], True, False, f"pair {(n, h)}")
        assert np.array_equal(f64(kc[n, h, p]), kc_r[0, 0, p]) and np.array_equal(f64(vc[n, h, p]), vc_r[0, 0, p])
        assert np.array_equal(f64(kc[n, h, :p]), kh[:p]), "cached rows changed"
    del kc, vc
    torch.cuda.empty_cache()


def test_mla_decode_slot_pool():
    """Continuous batching: 4 sequences over a pool of 7 cache slots.  Mapped slots match the oracle
    run on the gathered caches (outputs, appended rows, lengths); unmapped slots stay bit for bit;
    entries outside the pool give NaN outputs and write nothing."""
    P, H, d, dv, L = 7, 2, 192, 128, 700
    pool = KI.mla_decode_case("mla_pool", P, H, d, L, (0, 650), seed=21, rope_dim=64, dv=dv)
    tok = KI.mla_decode_case("mla_tok", 4, H, d, 8, [0, 0, 0, 0], seed=22, rope_dim=64, dv=dv)
    t = _to_dev(pool)
    q, k, v, g = (dev_tensor(x, True) for x in (tok.q, tok.k_new, tok.v_new, tok.gate))
    for idx, checked in (([5, 0, 3, 6], True), ([5, 9, 3, -2], False)):
        kc0, vc0, len0 = to_np(t["kc"]).copy(), to_np(t["vc"]).copy(), to_np(t["lens"]).copy()
        cache_idx = torch.tensor(idx, dtype=torch.int32)
        out = torch.empty(4, H, dv, dtype=torch.float32, device="cuda")
        ws = torch.empty(K.k3mla_decode_workspace_size(4, H, d, dv, L), dtype=torch.uint8, device="cuda")
        K.k3mla_decode_step_slots(q, k, v, g, t["kc"], t["vc"], t["lens"], cache_idx.cuda(),
                                  cache_idx if checked else None, P, 4, H, d, dv, L, 64, pool.theta, d ** -0.5, out, ws)
        torch.cuda.synchronize()
        good = [j for j, sidx in enumerate(idx) if 0 <= sidx < P]
        sl = [idx[j] for j in good]
        ref, kr, vr, lr = OM.decode_step(tok.q[good], tok.k_new[good], tok.v_new[good], kc0[sl], vc0[sl], len0[sl],
                                         d ** -0.5, gate=tok.gate[good], rope_dim=64, theta=pool.theta,
                                         cache_bf16=True)
        got = to_np(out).astype(np.float64)
        _check_out(got[good], ref, False, False, "slots")
        assert np.all(np.isnan(got[[j for j in range(4) if j not in good]]))
        kc, vc, ln = to_np(t["kc"]), to_np(t["vc"]), to_np(t["lens"])
        assert np.array_equal(ln[sl], lr)
        assert np.array_equal(vc[sl].astype(np.float64), vr)
        assert np.all(np.abs(kc[sl].astype(np.float64) - kr) <= 2.0 ** -8 * np.abs(kr) + 1e-30)
        rest = [x for x in range(P) if x not in sl]
        assert np.array_equal(kc[rest], kc0[rest]) and np.array_equal(vc[rest], vc0[rest])
        assert np.array_equal(ln[rest], len0[rest])
