"""Parity of k3kda_prefill (through the C ABI) with the oracle on the five workload
families: fp32 core, chunked bf16 prefill, varlen with initial states, the fused
mixer (conv + L2 + gate), plus edge cases.  Small cases are compared element by
element; the full-size workloads run in the bench's launch configuration and are
checked on seeded samples of heads (heads never interact)."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_rule_gb300 as K
import kda_inputs as KI
import oracle as O
from parity_utils import (assert_close, case_to_device, head_subset, oracle_prefill, run_prefill,
                          to_np)

pytestmark = pytest.mark.gpu


# The tensor-core shapes (bf16, d = 128, chunk 64) have two paths: the two-pass one (chunk-prep
# kernel over all (chunk, head) items, then a scan kernel per sequence and head), selected by the
# full workspace, and the single-pass kernel, selected by the minimum workspace.
PATHS = pytest.mark.parametrize("path", ["two_pass", "single_pass"])


def _check(c, out_dtype=torch.float32, heads=None, path="two_pass"):
    out, fs, d = run_prefill(c, out_dtype, min_workspace=path == "single_pass")
    sub = c if heads is None else head_subset(c, heads)
    ro, rs, rcs = oracle_prefill(sub)
    o = to_np(out) if heads is None else to_np(out[:, heads])
    s = to_np(fs) if heads is None else to_np(fs[:, heads])
    fp32 = c.in_dtype == "f32"
    eo = assert_close(o, ro, fp32, f"{c.name} out", store_bf16=out_dtype == torch.bfloat16)
    es = assert_close(s, rs, fp32, f"{c.name} final state")
    if c.conv_w is not None and heads is None:
        assert np.array_equal(to_np(d["conv_state"]), rcs), "conv state must be the last inputs exactly"
    print(f"{c.name}: max err out {eo:.3e} state {es:.3e}")
    return out, fs, d


# ---- fp32 core (the 1e-5 workload) ----

def test_core_fp32_workload():
    _check(KI.core_fp32(seed=0))


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_core_fp32_chunk_sizes_and_ragged_tail(chunk):
    c = KI.prefill_case("fp32_ragged", [203], 2, 32, 48, chunk, "f32", seed=1, s0_std=0.02, gate=True)
    _check(c)


# ---- bf16 chunked prefill ----

@PATHS
def test_prefill_bf16_small_ragged(path):
    """15 full chunks plus a 40-token tail, 4 heads, d = 128, chunk 64."""
    _check(KI.chunked_prefill(seed=1, T=1000, H=4), path=path)


@PATHS
def test_prefill_shorter_than_one_chunk(path):
    """T < 64: the staged token tile is shorter than a chunk."""
    _check(KI.fused_mixer(seed=12, T=37, H=2), path=path)


def test_prefill_bf16_output_store():
    _check(KI.chunked_prefill(seed=2, T=300, H=2), out_dtype=torch.bfloat16)


@PATHS
def test_prefill_bf16_output_varlen_ragged(path):
    """bf16 outputs of whole chunks leave through a TMA tile store; a ragged chunk at a sequence
    end inside the batch is stored row by row (a tile would cross into the next sequence), a
    ragged chunk at the end of the batch by a tile clipped at the tensor's end."""
    c = KI.prefill_case("bf16_out_varlen", [70, 3, 190, 64, 1, 129], 2, 128, 128, 64, "bf16", seed=30,
                        s0_std=0.02, gate=True, conv_width=4, conv_state=True)
    _check(c, out_dtype=torch.bfloat16, path=path)


def test_prefill_bf16_output_shorter_than_one_chunk_varlen():
    """T < 64: the tile box is T rows; the second sequence's tile starts inside it and is clipped."""
    c = KI.prefill_case("bf16_out_short", [10, 27], 2, 128, 128, 64, "bf16", seed=31, s0_std=0.02, gate=True)
    _check(c, out_dtype=torch.bfloat16)


@PATHS
def test_prefill_without_l2norm(path):
    c = KI.chunked_prefill(seed=3, T=200, H=2)
    c.use_qk_l2norm = False
    c.q = KI.round_bf16(c.q * 0.08)
    c.k = KI.round_bf16(c.k * 0.08)
    _check(c, path=path)


# ---- varlen with initial states ----

@PATHS
def test_varlen_small_with_edge_lengths(path):
    """Empty, one-token, chunk-1, chunk, chunk+1 and multi-chunk sequences packed together."""
    c = KI.prefill_case("varlen_edges", [0, 1, 63, 64, 65, 200, 0, 7], 3, 128, 128, 64, "bf16", seed=4,
                        s0_std=0.02, gate=True)
    _check(c, path=path)


def test_varlen_mixed_head_dims_f32_path():
    c = KI.prefill_case("varlen_dk64_dv128", [5, 90, 33], 2, 64, 128, 64, "bf16", seed=5, s0_std=0.02)
    _check(c)


def test_final_state_may_alias_initial_state():
    c = KI.prefill_case("alias", [100, 30], 2, 128, 128, 64, "bf16", seed=6, s0_std=0.02)
    d = case_to_device(c)
    T, H, dk, dv, N = c.T, c.H, c.dk, c.dv, c.N
    out = torch.empty((T, H, dv), device="cuda")
    ws = torch.zeros(K.k3kda_prefill_workspace_size(N, T, H, dk, dv, 64, K.BF16, False), dtype=torch.uint8,
                     device="cuda")
    S = d["S0"].clone()
    K.k3kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], S, d["cu"].cuda(), d["cu"], N, T, H, dk, dv, 64,
                    c.scale, True, None, None, 0, None, out, S, ws)
    torch.cuda.synchronize()
    ro, rs, _ = oracle_prefill(c)
    assert_close(to_np(out), ro, False, "alias out")
    assert_close(to_np(S), rs, False, "alias state")


# ---- fused mixer: conv + SiLU + L2 + chunked KDA + gate ----

@PATHS
def test_fused_mixer_small(path):
    _check(KI.fused_mixer(seed=1, T=777, H=2), path=path)


@PATHS
def test_fused_mixer_varlen_with_conv_state(path):
    c = KI.prefill_case("mixer_varlen", [2, 130, 1, 64], 2, 128, 128, 64, "bf16", seed=7, s0_std=0.02,
                        gate=True, conv_width=4, conv_state=True)
    _check(c, path=path)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_two_pass_segmented_varlen_with_states(out_dtype):
    """Few (sequence, head) pairs and a sequence of >= 128 chunks: the two passes run as a pipeline of
    segments of local chunks, all sequences advancing together through a ring of record buffers, the
    scan handing each chain's state between segment launches; the sequences end in different
    segments (130, 66 and 2 chunks)."""
    c = KI.prefill_case("segmented_varlen", [8300, 4200, 70], 2, 128, 128, 64, "bf16", seed=40, s0_std=0.02,
                        gate=True, conv_width=4, conv_state=True)
    _check(c, out_dtype=out_dtype)


def test_two_pass_segmented_single_long_sequence():
    _check(KI.fused_mixer(seed=41, T=8300, H=1))


def test_two_pass_pipeline_from_two_host_threads():
    """Two host threads, each on its own stream, run the segmented call (one cooperative launch
    that takes every SM, so two of them run one after the other) repeatedly; every result must
    equal a run made alone, bit for bit."""
    import threading
    cases = [KI.fused_mixer(seed=50 + i, T=8300, H=1) for i in range(2)]
    devs = [case_to_device(c) for c in cases]

    def once(i):
        d = dict(devs[i])
        d["conv_state"] = devs[i]["conv_state"].clone()
        out, fs, _ = run_prefill(cases[i], d=d)
        return out, fs

    refs = [once(i) for i in range(2)]
    results, errors = [[], []], []

    def work(i):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(4):
                    results[i].append(once(i))
        except Exception as exc:          # surfaced below
            errors.append(exc)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        for out, fs in results[i]:
            assert torch.equal(out, refs[i][0]) and torch.equal(fs, refs[i][1])


def test_two_pass_segment_ring_wraps():
    """300 chunks of one head: four segments through a ring of three record buffers, so a
    prep launch rewrites the buffer of a segment whose scan has finished."""
    _check(KI.fused_mixer(seed=42, T=19200, H=1))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_one_launch_segments_many_chains_ring_wraps(out_dtype):
    """Three sequences of 313, 141 and 3 chunks over 8 heads (24 chains, 458 chunks in all): the
    segmented call is one cooperative launch whose 24 chains run beside the prep CTAs through
    a ring of three segment buffers that wraps, the sequences ending in different segments, with
    initial states, conv state and gate.  Checked on three heads (heads never interact)."""
    c = KI.prefill_case("one_launch_ring", [20000, 9000, 130], 8, 128, 128, 64, "bf16", seed=43, s0_std=0.02,
                        gate=True, conv_width=4, conv_state=True)
    _check(c, out_dtype=out_dtype, heads=[0, 3, 7])


@pytest.mark.parametrize("host_lengths", [True, False], ids=["host_cu_seqlens", "device_only"])
def test_two_pass_bounded_segments_many_chains(host_lengths):
    """Many (sequence, head) chains whose records would exceed the record budget (4 sequences x 32
    heads, 322 chunks: 1.53 GB): the call runs in segments of 35 local chunks of every sequence, all
    sequences advancing together through a ring of two record buffers; the scan hands each chain's
    state from segment to segment.  Without a host copy of cu_seqlens the segments run to the bound
    ceil(T / 64), the ones past the longest sequence empty.  Checked on sampled heads."""
    c = KI.prefill_case("bounded_segments", [9000, 300, 64, 11000], 32, 128, 128, 64, "bf16", seed=43,
                        s0_std=0.02, gate=True, conv_width=4, conv_state=True)
    ws_bytes = K.k3kda_prefill_workspace_size(c.N, c.T, c.H, 128, 128, 64, K.BF16, True)
    assert ws_bytes < 1.5e9                               # the ring, not 322 x 32 records
    d = case_to_device(c)
    out = torch.empty((c.T, c.H, 128), device="cuda")
    fs = torch.empty((c.N, c.H, 128, 128), device="cuda")
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    cs = d["conv_state"].clone()
    K.k3kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["cu"].cuda(),
                    d["cu"] if host_lengths else None, c.N, c.T, c.H, 128, 128, 64, c.scale, True, d["conv_w"], cs,
                    4, d["gate"], out, fs, ws)
    torch.cuda.synchronize()
    assert K.k3kda_workspace_status(ws) == 0
    heads = [3, 30]
    sub = head_subset(c, heads)
    ro, rs, _ = oracle_prefill(sub)
    assert_close(to_np(out[:, heads]), ro, False, "bounded segments out")
    assert_close(to_np(fs[:, heads]), rs, False, "bounded segments final state")


@pytest.mark.parametrize("W", [1, 2, 3])
def test_fused_mixer_narrow_conv_two_pass(W):
    """Conv widths below 4: the conv history before each chunk comes from the inputs (or, before
    the sequence start, from the right-aligned conv state) with taps right-aligned."""
    c = KI.prefill_case(f"mixer_w{W}", [70, 3, 190], 2, 128, 128, 64, "bf16", seed=20 + W, s0_std=0.02,
                        gate=True, conv_width=W, conv_state=True)
    _check(c)


def test_state_and_conv_state_chaining():
    """prefill(T) == prefill(T1) then prefill(T - T1) from the carried state and conv state."""
    c = KI.fused_mixer(seed=8, T=300, H=2)
    d = case_to_device(c)
    out, fs = K.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], conv_weight=d["conv_w"],
                        conv_state=d["conv_state"].clone(), gate=d["gate"], out_dtype=torch.float32)
    T1 = 129
    cs = d["conv_state"].clone()
    sl = lambda x, a, b: x[a:b].contiguous()
    o1, f1 = K.prefill(*(sl(d[n], 0, T1) for n in ("q", "k", "v", "g", "beta")), conv_weight=d["conv_w"],
                       conv_state=cs, gate=sl(d["gate"], 0, T1), out_dtype=torch.float32)
    o2, f2 = K.prefill(*(sl(d[n], T1, c.T) for n in ("q", "k", "v", "g", "beta")), initial_state=f1,
                       conv_weight=d["conv_w"], conv_state=cs, gate=sl(d["gate"], T1, c.T), out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rs, _ = oracle_prefill(c)
    assert_close(to_np(torch.cat([o1, o2])), ro, False, "chained out")
    assert_close(to_np(f2), rs, False, "chained state")
    assert_close(to_np(out), ro, False, "whole out")


def test_prefill_then_decode_continues_the_sequence():
    """A decode step after prefill(L-1) reproduces token L of the mixer."""
    c = KI.fused_mixer(seed=9, T=70, H=2)
    d = case_to_device(c)
    L = c.T
    cs = d["conv_state"].clone()
    sl = lambda x: x[:L - 1].contiguous()
    _, f1 = K.prefill(*(sl(d[n]) for n in ("q", "k", "v", "g", "beta")), conv_weight=d["conv_w"], conv_state=cs,
                      gate=sl(d["gate"]), out_dtype=torch.float32)
    last = lambda x: x[L - 1:].contiguous()
    o = K.decode_step(*(last(d[n]) for n in ("q", "k", "v", "g", "beta")), f1, gate=last(d["gate"]),
                      conv_weight=d["conv_w"], conv_state=cs, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rs, _ = oracle_prefill(c)
    assert_close(to_np(o)[0], ro[-1], False, "decode after prefill")
    assert_close(to_np(f1), rs, False, "state after decode")


def test_empty_batch_copies_initial_state():
    c = KI.prefill_case("empty", [0, 0], 2, 64, 64, 64, "bf16", seed=10, s0_std=0.02)
    d = case_to_device(c)
    out, fs = K.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["S0"], cu_seqlens=d["cu"])
    torch.cuda.synchronize()
    assert np.array_equal(to_np(fs), c.S0)


# ---- the full-size workloads (bench launch configuration), sampled heads ----

@pytest.mark.slow
def test_full_chunked_prefill_sampled_heads():
    c = KI.chunked_prefill(seed=0)
    _check(c, heads=[0, 13, 31])


@pytest.mark.slow
def test_full_varlen_prefill_sampled_heads():
    c = KI.varlen_prefill(seed=0)
    _check(c, heads=[7])


@pytest.mark.slow
@PATHS
def test_full_fused_mixer_sampled_heads(path):
    c = KI.fused_mixer(seed=0)
    _check(c, out_dtype=torch.bfloat16, heads=[5, 26], path=path)
