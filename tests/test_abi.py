"""The C-ABI library loads, exports every symbol include/k3kda.h declares, and
rejects bad arguments on the host before launching anything (no GPU needed:
every call here returns from argument validation)."""
import ctypes
import os
import re

import pytest

import hybrid_linear_attention_rule_gb300 as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "k3kda.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(k3(?:kda|mla)_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return K.load_library()


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("k3kda_short_conv", "k3kda_prefill", "k3kda_decode_step", "k3mla_decode_step"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_wait_timeout_hook_takes_the_four_kinds(lib):
    """The internal test hook (exported for the GPU timeout tests, not in the public header) arms
    the chunk scan, the single-pass prefill, the decode and the backward's chains, and rejects
    any other kind; arming with zero tries disarms."""
    for which in range(4):
        assert lib.k3kda_test_arm_wait_timeout(which, 0) == 0
    assert lib.k3kda_test_arm_wait_timeout(4, 1) == -1
    assert lib.k3kda_test_arm_wait_timeout(-1, 1) == -1


def test_version_and_status_strings(lib):
    assert K.k3kda_version() == 1
    assert K.k3kda_status_string(0) == "K3KDA_OK"
    assert K.k3kda_status_string(-6) == "K3KDA_ERR_TIMEOUT"
    assert K.k3kda_status_string(123) == "K3KDA_UNKNOWN_STATUS"


def test_workspace_size_is_aligned_and_grows_with_conv(lib):
    # tensor-core shape (bf16, d = 128, chunk 64): the conv is fused; the full workspace holds one
    # 148,480-byte record per (chunk, head) for the two-pass path, the minimum only the status word
    a = K.k3kda_prefill_workspace_size(1, 1024, 4, 128, 128, 64, K.BF16, False)
    b = K.k3kda_prefill_workspace_size(1, 1024, 4, 128, 128, 64, K.BF16, True)
    assert a == b and a % 256 == 0
    assert a == 256 + 256 + 16 * 4 * 148480          # status, chunk offsets, 16 chunks x 4 heads
    assert K.k3kda_prefill_workspace_min(1, 1024, 4, 128, 128, 64, K.BF16, True) == 256
    # packed sequences: at most (T + 63 N) / 64 chunks in all
    e = K.k3kda_prefill_workspace_size(3, 1000, 2, 128, 128, 64, K.BF16, True)
    assert e == 256 + 256 + ((1000 + 63 * 3) // 64) * 2 * 148480
    # long sequences with few (sequence, head) pairs: the segments' record tables (int32 [N + 1] for
    # each of at most ceil(chunks / 48) segments), the segment counters (int32: two per segment and
    # an abort word), the scan's state carry (65,536 B per sequence and head) and a ring of three
    # segments' records (80 chunks, or chunks / 64 beyond 64 segments), independent of T; all
    # records when they take less room than the ring
    carry = 32 * 65536
    r256 = lambda b: (b + 255) // 256 * 256
    ring = lambda chunks: min(chunks, 3 * max(80, -(-chunks // 64))) * 32 * 148480
    for T in (8192, 65536, 1 << 18, 1 << 21):
        chunks = T // 64
        nseg = -(-chunks // 48)
        tables, counters = r256(nseg * 2 * 4), r256((2 * nseg + 1) * 4)
        want = 256 + tables + counters + carry + ring(chunks)
        assert K.k3kda_prefill_workspace_size(1, T, 32, 128, 128, 64, K.BF16, True) == want
    # many (sequence, head) chains whose records would exceed 1.25 GiB: a ring of two buffers of
    # `per` local chunks of every sequence, per = 1.25 GiB / (2 N H 148480 B); the 16-sequence varlen
    # workload (135,937 tokens) fits in 1.3 GB instead of 10.2 GB
    N, T, H = 16, 135937, 32
    per = (5 << 28) // (2 * N * H * 148480)
    nseg = -(-((T + 63) // 64) // per)
    tables, counters = r256(nseg * (N + 1) * 4), r256((2 * nseg + 1) * 4)
    want = 256 + tables + counters + N * H * 65536 + 2 * min(N * per, (T + 63 * N) // 64) * H * 148480
    got = K.k3kda_prefill_workspace_size(N, T, H, 128, 128, 64, K.BF16, True)
    assert got == want and got < 1.5e9
    c = K.k3kda_prefill_workspace_size(1, 1024, 4, 64, 128, 64, K.BF16, False)
    d = K.k3kda_prefill_workspace_size(1, 1024, 4, 64, 128, 64, K.BF16, True)
    assert c >= 256 and c % 256 == 0 and d % 256 == 0
    assert d >= c + 1024 * (2 * 4 * 64 + 4 * 128) * 4
    assert K.k3kda_prefill_workspace_min(1, 1024, 4, 64, 128, 64, K.BF16, True) == d


# Fake, never-dereferenced device addresses: validation must reject before use.
A16 = ctypes.c_void_p(0x10000)
MIS = ctypes.c_void_p(0x10004)


def _prefill(lib, **kw):
    args = dict(q=A16, k=A16, v=A16, in_dtype=1, g=A16, beta=A16, S0=None, cu=None, cu_h=None, N=1, T=64,
                H=2, dk=128, dv=128, chunk=64, scale=1.0, l2=1, conv=None, gate=None, out=A16, out_dtype=0,
                fs=None, ws=None, ws_bytes=0, stream=None)
    args.update(kw)
    return lib.k3kda_prefill(*args.values())


def test_prefill_rejects_bad_arguments(lib):
    assert _prefill(lib, N=0) == -1
    assert _prefill(lib, q=None) == -1
    assert _prefill(lib, N=2) == -1                      # two sequences but no cu_seqlens
    assert _prefill(lib, dk=200) == -2
    assert _prefill(lib, dk=24) == -2
    assert _prefill(lib, chunk=48) == -2
    assert _prefill(lib, in_dtype=7) == -1
    assert _prefill(lib, g=MIS) == -3
    assert _prefill(lib, ws=None) == -4                  # no workspace
    assert _prefill(lib, ws=A16, ws_bytes=16) == -4      # too small


def _backward(lib, **kw):
    args = dict(q=A16, k=A16, v=A16, in_dtype=1, g=A16, beta=A16, S0=None, cu=None, cu_h=None, N=1, T=64, H=2,
                dk=128, dv=128, scale=1.0, dO=A16, dSf=None, dq=A16, dk_out=A16, dv_out=A16, dg=A16, dbeta=A16,
                dS0=A16, ws=None, ws_bytes=0, stream=None)
    args.update(kw)
    return lib.k3kda_backward(*args.values())


def test_backward_rejects_bad_arguments(lib):
    assert _backward(lib, N=0) == -1
    assert _backward(lib, dO=None) == -1
    assert _backward(lib, dS0=None) == -1
    assert _backward(lib, N=2) == -1                     # two sequences but no cu_seqlens
    assert _backward(lib, dk=64, dv=64) == -2            # only dk = dv = 128
    assert _backward(lib, in_dtype=5) == -1
    assert _backward(lib, dq=MIS) == -3
    assert _backward(lib, ws=None) == -4
    assert _backward(lib, ws=A16, ws_bytes=16) == -4
    bad = (ctypes.c_int32 * 3)(0, 40, 30)
    assert _backward(lib, N=2, cu=A16, cu_h=ctypes.cast(bad, ctypes.c_void_p), T=30) == -1


def test_backward_workspace_size(lib):
    """The chunked backward's scratch: per (16-token chunk, head) item its fp32 tiles (Q0, K0, Kd,
    Gamma, W, U, Delta, dR: 16 x 128 each; Tm, Aqk, B: 16 x 16; Gamma_L: 128; Dout: 128 x 128),
    the state at every chunk start and each sequence's end, the chunk tables (offsets; first
    token, length and sequence of each chunk) and a readiness flag per item plus an abort word;
    each array starts on a 256-byte boundary after a 256-byte status word."""
    r = lambda b: (b + 255) // 256 * 256
    for N, T, H in ((1, 8192, 32), (3, 1000, 4)):
        Q = (T + 15 * N) // 16 + 1
        NI = Q * H
        want = 256 + r(4 * (N + 1)) + 3 * r(4 * Q) + r(4 * (NI + 1)) + 8 * r(NI * 16 * 128 * 4) + \
            3 * r(NI * 256 * 4) + r(NI * 128 * 4) + r(NI * 128 * 128 * 4) + r((Q + N) * H * 128 * 128 * 4)
        assert K.k3kda_backward_workspace_size(N, T, H, 128, 128) == want
    assert K.k3kda_backward_workspace_size(1, 8192, 32, 64, 64) == 256


def test_prefill_validates_host_cu_seqlens(lib):
    bad = (ctypes.c_int32 * 3)(0, 40, 30)                # decreasing
    assert _prefill(lib, N=2, cu=A16, cu_h=ctypes.cast(bad, ctypes.c_void_p), T=30) == -1
    bad_end = (ctypes.c_int32 * 3)(0, 10, 20)            # last != T
    assert _prefill(lib, N=2, cu=A16, cu_h=ctypes.cast(bad_end, ctypes.c_void_p), T=30) == -1


def test_decode_rejects_bad_arguments(lib):
    def dec(**kw):
        a = dict(q=A16, k=A16, v=A16, in_dtype=1, g=A16, beta=A16, gate=None, cw=None, cs=None, state=A16,
                 N=4, H=2, dk=128, dv=128, W=4, scale=1.0, l2=1, out=A16, out_dtype=0, stream=None)
        a.update(kw)
        return lib.k3kda_decode_step(*a.values())
    assert dec(state=None) == -1
    assert dec(dv=130) == -2
    assert dec(cw=A16, cs=None) == -1                    # conv weights without conv state
    assert dec(cw=A16, cs=A16, W=5) == -1
    assert dec(out=MIS) == -3


def _i32(*vals):
    arr = (ctypes.c_int32 * len(vals))(*vals)
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def test_slot_pool_calls_validate_the_slot_map(lib):
    def pre(**kw):
        a = dict(q=A16, k=A16, v=A16, in_dtype=1, g=A16, beta=A16, pool=A16, idx=A16, idx_h=None, slots=8,
                 cu=A16, cu_h=None, N=3, T=96, H=2, dk=128, dv=128, chunk=64, scale=1.0, l2=1, conv=None, gate=None,
                 out=A16, out_dtype=0, ws=None, ws_bytes=0, stream=None)
        a.update(kw)
        return lib.k3kda_prefill_slots(*a.values())

    def dec(**kw):
        a = dict(q=A16, k=A16, v=A16, in_dtype=1, g=A16, beta=A16, gate=None, cw=None, cs=None, pool=A16,
                 idx=A16, idx_h=None, slots=8, N=3, H=2, dk=128, dv=128, W=4, scale=1.0, l2=1, out=A16,
                 out_dtype=0, stream=None)
        a.update(kw)
        return lib.k3kda_decode_step_slots(*a.values())

    ok_keep, ok = _i32(5, 0, 7)
    oob_keep, oob = _i32(5, 8, 1)                        # 8 is past the pool
    neg_keep, neg = _i32(-1, 2, 3)
    dup_keep, dup = _i32(2, 4, 2)                        # two sequences on one slot would race
    for call in (pre, dec):
        assert call(slots=0) == -1
        assert call(idx=None) == -1
        assert call(idx=ctypes.c_void_p(0x10002)) == -3     # state_idx must be 4-byte aligned
        for bad in (oob, neg, dup):
            assert call(idx_h=bad) == -1
    assert pre(pool=None) == -1
    assert pre(idx_h=ok, ws=None) == -4                  # a good map reaches the workspace check
    assert dec(idx_h=ok, dv=130) == -2                   # ... and the shape checks


def test_short_conv_rejects_bad_arguments(lib):
    def conv(**kw):
        a = dict(x=A16, xt=1, w=A16, cs=None, cu=None, N=1, T=10, D=64, W=4, silu=1, out=ctypes.c_void_p(0x20000),
                 ot=1, stream=None)
        a.update(kw)
        return lib.k3kda_short_conv(*a.values())
    assert conv(W=0) == -1
    assert conv(W=5) == -1
    assert conv(out=A16) == -1                           # out aliases x
    assert conv(N=3) == -1                               # no cu_seqlens
    assert conv(w=MIS) == -3


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 8)
    with pytest.raises(ValueError):
        K.k3kda_short_conv(x, torch.zeros(8, 4), None, None, 1, 4, 8, 4, True, torch.zeros(4, 8))


def _mla(lib, **kw):
    a = dict(q=A16, k=A16, v=A16, in_dtype=1, gate=None, kc=A16, vc=A16, cache_dtype=1, lens=A16, N=4, H=2, dq=128,
             dv=128, L_max=1024, rope_dim=0, theta=10000.0, scale=1.0, out=A16, out_dtype=1, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.k3mla_decode_step(*a.values())


def test_mla_decode_rejects_bad_arguments(lib):
    big = 1 << 30
    assert _mla(lib, N=0) == 0                           # nothing to do: no launch, no workspace needed
    assert _mla(lib, N=-1) == -1
    assert _mla(lib, L_max=0) == -1
    assert _mla(lib, kc=None) == -1
    assert _mla(lib, lens=None) == -1
    assert _mla(lib, rope_dim=3) == -1                   # odd
    assert _mla(lib, rope_dim=130) == -1                 # above d
    assert _mla(lib, rope_dim=64, theta=0.0) == -1
    assert _mla(lib, cache_dtype=7) == -1
    assert _mla(lib, dq=96) == -2
    assert _mla(lib, dv=192) == -2                       # only the key width may be 192
    assert _mla(lib, dq=192, dv=128, rope_dim=200) == -1
    assert _mla(lib, N=4096, H=64, L_max=big) == -2      # grid above 2^31 - 1 blocks
    assert _mla(lib, vc=MIS) == -3
    assert _mla(lib, ws=None) == -4
    assert _mla(lib, ws=A16, ws_bytes=16) == -4


def test_mla_workspace_size(lib):
    r = lambda b: (b + 255) // 256 * 256
    N, H, d, L = 256, 32, 128, 8192
    S = L // 512
    # per sequence: keys to attend and cache slot; per (sequence, head): the query, and per split the
    # (max, sum) pair and the weighted value row
    assert K.k3mla_decode_workspace_size(N, H, d, d, L) == 2 * r(N * 4) + r(N * H * d * 4) + r(N * H * S * 8) + \
        r(N * H * S * d * 4)
    assert K.k3mla_decode_workspace_size(3, 2, 192, 64, 513) == 2 * r(12) + r(3 * 2 * 192 * 4) + r(3 * 2 * 2 * 8) + \
        r(3 * 2 * 2 * 64 * 4)


def test_mla_slot_call_validates_the_map(lib):
    def call(**kw):
        a = dict(q=A16, k=A16, v=A16, in_dtype=1, gate=None, kc=A16, vc=A16, cache_dtype=1, lens=A16, idx=A16,
                 idx_h=None, slots=8, N=3, H=2, dq=128, dv=128, L_max=1024, rope_dim=0, theta=10000.0, scale=1.0,
                 out=A16, out_dtype=1, ws=None, ws_bytes=0, stream=None)
        a.update(kw)
        return lib.k3mla_decode_step_slots(*a.values())
    assert call(idx=None) == -1
    assert call(slots=0) == -1
    assert call(idx=ctypes.c_void_p(0x10002)) == -3      # int32 map off a 4-byte boundary
    dup, dup_p = _i32(1, 1, 2)
    assert call(idx_h=dup_p) == -1                       # a slot twice
    far, far_p = _i32(1, 8, 2)
    assert call(idx_h=far_p) == -1                       # outside the pool
    ok, ok_p = _i32(7, 0, 2)
    assert call(idx_h=ok_p) == -4                        # the map passes; the missing workspace does not
