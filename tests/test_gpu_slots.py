"""Slot-indexed state pools (continuous batching): k3kda_decode_step_slots and
k3kda_prefill_slots read and update pool slot state_idx[n] for sequence n.

Each case runs the pool call and, on copies of the same slots gathered into a plain
batch, the plain call (whose parity with the oracle the other GPU tests establish):
outputs and updated slots must agree bit for bit, slots outside the map must not change,
and one case is also compared with the oracle directly.  The wrong-slot mutant (a
permuted map) must change the results, which shows the kernels follow the map."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_rule_gb300 as K
import kda_inputs as KI
import oracle as O
from parity_utils import assert_close, case_to_device, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(x, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return (t.to(torch.bfloat16) if bf16 else t).to(DEV)


# ---------------- decode ----------------

def _decode_pools(c, num_slots, idx, seed=0):
    """Pools whose slots idx[n] hold the case's state n; the other slots hold unrelated values."""
    g = torch.Generator().manual_seed(seed)
    N, H, d = c.N, c.H, c.dk
    D = 3 * H * d
    pool = torch.randn((num_slots, H, d, d), generator=g) * 0.02
    cpool = torch.randn((num_slots, c.conv_state.shape[1], D), generator=g)
    for n, s in enumerate(idx):
        pool[s] = torch.from_numpy(c.state[n])
        cpool[s] = torch.from_numpy(c.conv_state[n])
    return pool.to(DEV), cpool.to(DEV)


def _decode_slots(c, pool, cpool, idx, idx_host=True):
    N, H, d = c.N, c.H, c.dk
    out = torch.empty((N, H, d), device=DEV)
    idx_d = torch.tensor(idx, dtype=torch.int32, device=DEV)
    idx_h = torch.tensor(idx, dtype=torch.int32) if idx_host else None
    K.k3kda_decode_step_slots(_t(c.q, True), _t(c.k, True), _t(c.v, True), _t(c.g), _t(c.beta), _t(c.gate, True),
                              _t(c.conv_w), cpool, pool, idx_d, idx_h, pool.shape[0], N, H, d, d,
                              c.conv_w.shape[1], c.scale, True, out)
    torch.cuda.synchronize()
    return out


def test_decode_slots_match_the_plain_call_and_leave_other_slots():
    c = KI.decode_case(seed=21, N=5, H=4, d=128, W=4)
    idx = [7, 2, 0, 5, 8]
    pool, cpool = _decode_pools(c, 9, idx)
    pool0, cpool0 = pool.clone(), cpool.clone()
    out = _decode_slots(c, pool, cpool, idx)
    # the plain call on the gathered slots
    st, cs = pool0[idx].clone(), cpool0[idx].clone()
    ref = K.decode_step(_t(c.q, True), _t(c.k, True), _t(c.v, True), _t(c.g), _t(c.beta), st, gate=_t(c.gate, True),
                        conv_weight=_t(c.conv_w), conv_state=cs, scale=c.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.equal(pool[idx], st) and torch.equal(cpool[idx], cs)
    other = [s for s in range(9) if s not in idx]
    assert torch.equal(pool[other], pool0[other]) and torch.equal(cpool[other], cpool0[other])
    # and the oracle, on the case's own (gathered) values
    ro, rs, rc = O.decode_step(c.q, c.k, c.v, c.g, c.beta, c.state, gate=c.gate, conv_w=c.conv_w,
                               conv_state=c.conv_state, scale=c.scale)
    assert_close(to_np(out), ro, False, "slot decode out")
    assert_close(to_np(pool[idx]), rs, False, "slot decode state")
    assert np.array_equal(to_np(cpool[idx]), rc)


def test_decode_wrong_slot_mutant_changes_the_result():
    c = KI.decode_case(seed=22, N=4, H=2, d=128, W=4)
    idx = [3, 1, 4, 0]
    pool, cpool = _decode_pools(c, 6, idx)
    good = _decode_slots(c, pool.clone(), cpool.clone(), idx)
    wrong = _decode_slots(c, pool.clone(), cpool.clone(), [1, 3, 4, 0])   # two sequences swapped
    assert not torch.allclose(good[:2], wrong[:2])
    assert torch.equal(good[2:], wrong[2:])


def test_decode_out_of_range_slot_touches_no_pool_row():
    c = KI.decode_case(seed=23, N=3, H=2, d=128, W=4)
    idx = [2, -1, 0]                                     # no host copy: the kernel must skip sequence 1
    pool, cpool = _decode_pools(c, 4, [2, 3, 0])
    pool0, cpool0 = pool.clone(), cpool.clone()
    out = _decode_slots(c, pool, cpool, idx, idx_host=False)
    assert torch.count_nonzero(out[1]) == 0
    assert torch.equal(pool[[1, 3]], pool0[[1, 3]]) and torch.equal(cpool[[1, 3]], cpool0[[1, 3]])
    assert not torch.equal(pool[2], pool0[2])            # the others were updated


# ---------------- prefill ----------------

def _prefill_pools(c, num_slots, idx, seed=0):
    g = torch.Generator().manual_seed(seed)
    pool = torch.randn((num_slots, c.H, c.dk, c.dv), generator=g) * 0.02
    D = 2 * c.H * c.dk + c.H * c.dv
    cpool = torch.randn((num_slots, c.W - 1, D), generator=g)
    for n, s in enumerate(idx):
        pool[s] = torch.from_numpy(c.S0[n])
        cpool[s] = torch.from_numpy(c.conv_state[n])
    return pool.to(DEV), cpool.to(DEV)


def _prefill_slots(c, d, pool, cpool, idx, min_ws, idx_host=True):
    T, H, dk, dv, N = c.T, c.H, c.dk, c.dv, c.N
    size_fn = K.k3kda_prefill_workspace_min if min_ws else K.k3kda_prefill_workspace_size
    ws = torch.zeros(size_fn(N, T, H, dk, dv, c.chunk, K.BF16, True), dtype=torch.uint8, device=DEV)
    out = torch.empty((T, H, dv), device=DEV)
    idx_d = torch.tensor(idx, dtype=torch.int32, device=DEV)
    idx_h = torch.tensor(idx, dtype=torch.int32) if idx_host else None
    K.k3kda_prefill_slots(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, idx_d, idx_h, pool.shape[0],
                          d["cu"].to(DEV), d["cu"], N, T, H, dk, dv, c.chunk, c.scale, True, d["conv_w"], cpool, c.W,
                          d["gate"], out, ws)
    torch.cuda.synchronize()
    return out


CASES = {
    "tensor_core_two_pass": dict(lengths=[100, 7, 190], dk=128, min_ws=False),
    "tensor_core_single_pass": dict(lengths=[100, 7, 190], dk=128, min_ws=True),
    "tensor_core_segmented": dict(lengths=[4100, 4200, 70], dk=128, min_ws=False),
    # 250, 66 and 2 chunks: the one-launch segmented path with its record ring wrapping
    "tensor_core_one_launch": dict(lengths=[16000, 4200, 70], dk=128, min_ws=False),
    "fp32_path": dict(lengths=[77, 3, 123], dk=64, min_ws=False),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_slots_match_the_plain_call_and_leave_other_slots(name):
    cfg = CASES[name]
    c = KI.prefill_case("slots_" + name, cfg["lengths"], 2, cfg["dk"], 128, 64, "bf16", seed=30, s0_std=0.02,
                        gate=True, conv_width=4, conv_state=True)
    d = case_to_device(c)
    idx = [4, 1, 3]
    pool, cpool = _prefill_pools(c, 6, idx)
    pool0, cpool0 = pool.clone(), cpool.clone()
    out = _prefill_slots(c, d, pool, cpool, idx, cfg["min_ws"])
    S, cs = pool0[idx].clone(), cpool0[idx].clone()
    ref, _ = K.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=S, cu_seqlens=d["cu"],
                       conv_weight=d["conv_w"], conv_state=cs, gate=d["gate"], out_dtype=torch.float32,
                       min_workspace=cfg["min_ws"], return_final_state=False)
    # the plain call writes its final state to a fresh tensor; run it again in place for the state
    S2, cs2 = pool0[idx].clone(), cpool0[idx].clone()
    _, fs = K.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=S2, cu_seqlens=d["cu"],
                      conv_weight=d["conv_w"], conv_state=cs2, gate=d["gate"], out_dtype=torch.float32,
                      min_workspace=cfg["min_ws"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.equal(pool[idx], fs)
    assert torch.equal(cpool[idx], cs2)
    other = [s for s in range(6) if s not in idx]
    assert torch.equal(pool[other], pool0[other]) and torch.equal(cpool[other], cpool0[other])


def test_prefill_slots_against_the_oracle_and_the_wrong_slot_mutant():
    c = KI.prefill_case("slots_oracle", [90, 130], 2, 128, 128, 64, "bf16", seed=31, s0_std=0.02, gate=True,
                        conv_width=4, conv_state=True)
    d = case_to_device(c)
    idx = [2, 0]
    pool, cpool = _prefill_pools(c, 3, idx)
    out = _prefill_slots(c, d, pool.clone(), cpool.clone(), idx, False)
    ro, rs, rc = O.mixer(c.q, c.k, c.v, c.g, c.beta, initial_state=c.S0, gate=c.gate, conv_w=c.conv_w,
                         conv_state=c.conv_state, cu_seqlens=c.cu_seqlens, scale=c.scale)
    assert_close(to_np(out), ro, False, "slot prefill out")
    p2, c2 = pool.clone(), cpool.clone()
    _prefill_slots(c, d, p2, c2, idx, False)
    assert_close(to_np(p2[idx]), rs, False, "slot prefill state")
    assert np.array_equal(to_np(c2[idx]), rc)
    wrong = _prefill_slots(c, d, pool.clone(), cpool.clone(), [0, 2], False)
    assert not torch.allclose(out, wrong)


def test_prefill_out_of_range_slot_starts_from_zero_and_writes_nothing():
    c = KI.prefill_case("slots_oob", [70, 50], 2, 128, 128, 64, "bf16", seed=32, s0_std=0.02, gate=True,
                        conv_width=4, conv_state=True)
    d = case_to_device(c)
    pool, cpool = _prefill_pools(c, 2, [0, 1])
    pool0, cpool0 = pool.clone(), cpool.clone()
    out = _prefill_slots(c, d, pool, cpool, [0, 5], False, idx_host=False)
    assert torch.equal(pool[1], pool0[1]) and torch.equal(cpool[1], cpool0[1])
    # sequence 1 ran from zero state and conv history
    zero = KI.prefill_case("slots_oob", [70, 50], 2, 128, 128, 64, "bf16", seed=32, s0_std=0.02, gate=True,
                           conv_width=4, conv_state=True)
    zero.S0[1] = 0.0
    zero.conv_state[1] = 0.0
    ro, _, _ = O.mixer(zero.q, zero.k, zero.v, zero.g, zero.beta, initial_state=zero.S0, gate=zero.gate,
                       conv_w=zero.conv_w, conv_state=zero.conv_state, cu_seqlens=zero.cu_seqlens, scale=zero.scale)
    assert_close(to_np(out), ro, False, "out-of-range slot out")
