"""Failure detection on the GPU: a bounded in-kernel wait that runs out is reported, and the library
keeps working afterwards.

Every wait of the kernels on an mbarrier (a bulk copy or an MMA landing) polls a bounded number of
times and, when that runs out, records K3KDA_ERR_TIMEOUT, lets whatever it issued land, frees its
tensor memory and returns.  The internal hook k3kda_test_arm_wait_timeout (exported for these tests,
not part of the public header) makes the next launch of one kernel starve its first wait on a
working GPU: CTA 0 requests none of the copies that wait is for and gives up after a few hundred
polls.  Nothing faults and nothing hangs: the other copies it issued land before it exits.  Each
test checks that the status reader reports the timeout once, then that a normal call on the same
workspace reports K3KDA_OK and matches the oracle.
"""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_rule_gb300 as K
import kda_inputs as KI
import oracle as O
from parity_utils import assert_close, case_to_device, oracle_prefill, to_np

pytestmark = pytest.mark.gpu

SCAN, SINGLE_PASS, DECODE, BACKWARD = 0, 1, 2, 3
TIMEOUT = -6
TRIES = 256


def _arm(which):
    assert K.load_library().k3kda_test_arm_wait_timeout(which, TRIES) == 0


def _prefill(c, d, ws, out):
    T, H, dk, dv, N = c.T, c.H, c.dk, c.dv, c.N
    fs = torch.empty((N, H, dk, dv), device="cuda")
    K.k3kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["cu"].cuda(), d["cu"], N, T, H, dk, dv,
                    c.chunk, c.scale, True, None, None, 0, d["gate"], out, fs, ws)
    return fs


@pytest.mark.parametrize("which", [SCAN, SINGLE_PASS], ids=["two_pass_scan", "single_pass"])
def test_prefill_wait_runs_out_then_recovers(which):
    c = KI.prefill_case("timeout", [200, 90], 2, 128, 128, 64, "bf16", seed=80, s0_std=0.02, gate=True)
    d = case_to_device(c)
    size = (K.k3kda_prefill_workspace_size if which == SCAN else K.k3kda_prefill_workspace_min)(
        c.N, c.T, c.H, 128, 128, 64, K.BF16, False)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    out = torch.zeros((c.T, c.H, 128), device="cuda")
    _arm(which)
    _prefill(c, d, ws, out)
    assert K.k3kda_workspace_status(ws) == TIMEOUT
    assert K.k3kda_workspace_status(ws) == 0                  # read once, then cleared
    fs = _prefill(c, d, ws, out)
    assert K.k3kda_workspace_status(ws) == 0
    ro, rs, _ = oracle_prefill(c)
    assert_close(to_np(out), ro, False, "out after a timed-out call")
    assert_close(to_np(fs), rs, False, "final state after a timed-out call")


def test_segmented_launch_wait_runs_out_then_recovers():
    """One long sequence in segments (320 chunks: four segments of 80 in a ring of three), all in
    one launch in which the scan chains and the prep CTAs wait on one another's counters.  The
    chain's first tile is starved: it gives up, raises the abort word, and the prep CTAs waiting
    for that chain to free a ring buffer stop too; the call reports the timeout once and the next
    call is exact."""
    c = KI.prefill_case("timeout_seg", [20480], 1, 128, 128, 64, "bf16", seed=82, s0_std=0.02, gate=True)
    d = case_to_device(c)
    size = K.k3kda_prefill_workspace_size(c.N, c.T, c.H, 128, 128, 64, K.BF16, False)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    out = torch.zeros((c.T, c.H, 128), device="cuda")
    _arm(SCAN)
    _prefill(c, d, ws, out)
    assert K.k3kda_workspace_status(ws) == TIMEOUT
    assert K.k3kda_workspace_status(ws) == 0
    fs = _prefill(c, d, ws, out)
    assert K.k3kda_workspace_status(ws) == 0
    ro, rs, _ = oracle_prefill(c)
    assert_close(to_np(out), ro, False, "out after a timed-out segmented call")
    assert_close(to_np(fs), rs, False, "final state after a timed-out segmented call")


def test_decode_wait_runs_out_then_recovers():
    dc = KI.decode_case(seed=81, N=2, H=2, d=128)
    dev = lambda x, bf=False: torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16 if bf else torch.float32).cuda()
    args = lambda st, cs: (dev(dc.q, 1), dev(dc.k, 1), dev(dc.v, 1), dev(dc.g), dev(dc.beta), st)
    assert K.k3kda_decode_status() == 0
    _arm(DECODE)
    st, cs = dev(dc.state), dev(dc.conv_state)
    K.decode_step(*args(st, cs), gate=dev(dc.gate, 1), conv_weight=dev(dc.conv_w), conv_state=cs,
                  out_dtype=torch.float32)
    assert K.k3kda_decode_status() == TIMEOUT
    assert K.k3kda_decode_status() == 0
    st, cs = dev(dc.state), dev(dc.conv_state)
    o = K.decode_step(*args(st, cs), gate=dev(dc.gate, 1), conv_weight=dev(dc.conv_w), conv_state=cs,
                      out_dtype=torch.float32)
    assert K.k3kda_decode_status() == 0
    ro, rs, rcs = O.decode_step(dc.q, dc.k, dc.v, dc.g, dc.beta, dc.state, gate=dc.gate, conv_w=dc.conv_w,
                                conv_state=dc.conv_state)
    assert_close(to_np(o), ro, False, "decode out after a timed-out call")
    assert_close(to_np(st), rs, False, "decode state after a timed-out call")
    assert np.array_equal(to_np(cs), rcs)


def test_backward_chain_wait_runs_out_then_recovers():
    """The backward's chains: the first forward chain issues no MMA for its first chunk, gives up
    that wait, and stops; the call reports the timeout through the workspace's status word once,
    and the next call on the same workspace matches the reverse-mode oracle."""
    c = KI.prefill_case("timeout_bwd", [150, 40], 2, 128, 128, 64, "bf16", seed=83, s0_std=0.05)
    unit = lambda x: KI.round_bf16(x / np.linalg.norm(x, axis=-1, keepdims=True))
    c.q, c.k = unit(c.q), unit(c.k)
    rng = np.random.default_rng(84)
    dO = rng.standard_normal((c.T, c.H, 128))
    dev = lambda x, low=False: torch.from_numpy(np.ascontiguousarray(x)).to(
        torch.bfloat16 if low else torch.float32).cuda()
    q, k, v, g, beta, S0, dOd = dev(c.q, 1), dev(c.k, 1), dev(c.v, 1), dev(c.g), dev(c.beta), dev(c.S0), dev(dO)
    cu_h = torch.from_numpy(c.cu_seqlens.copy())
    N, T, H = c.N, c.T, c.H
    ws = torch.zeros(K.k3kda_backward_workspace_size(N, T, H, 128, 128), dtype=torch.uint8, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    outs = [torch.empty(T, H, 128, **f32) for _ in range(4)] + [torch.empty(T, H, **f32), torch.empty(N, H, 128, 128, **f32)]

    def call():
        K.k3kda_backward(q, k, v, g, beta, S0, cu_h.cuda(), cu_h, N, T, H, 128, 128, c.scale, dOd, None, *outs, ws)

    _arm(BACKWARD)
    call()
    assert K.k3kda_workspace_status(ws) == TIMEOUT
    assert K.k3kda_workspace_status(ws) == 0
    call()
    assert K.k3kda_workspace_status(ws) == 0
    want = O.recurrent_backward(c.q, c.k, c.v, c.g, c.beta, dO, initial_state=c.S0, scale=c.scale,
                                cu_seqlens=c.cu_seqlens)
    for name, got in zip(("dq", "dk", "dv", "dg", "dbeta", "dS0"), outs):
        w = want[name]
        err = float(np.abs(got.cpu().double().numpy() - w).max())
        assert err <= 5e-5 * float(np.sqrt((w * w).mean())) + 1e-6, (name, err)


def test_disarmed_hook_changes_nothing():
    assert K.load_library().k3kda_test_arm_wait_timeout(SCAN, 0) == 0
    assert K.load_library().k3kda_test_arm_wait_timeout(7, 1) == -1
