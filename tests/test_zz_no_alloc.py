"""k3kda_prefill_noalloc, the prefill for callers that cannot allocate device
memory where they run the mixer (inside an allocator or memory pool, runtimes
that forbid cudaMalloc after start-up, plug-ins handed only their buffers).

It must give the same results as k3kda_prefill with a caller workspace, call
after call (its scratch is one library-held array whose contents persist
between calls), must not take device memory from the process (free memory as
the driver reports it does not drop over a call), must report a bounded wait
that ran out through k3kda_prefill_noalloc_status, and must refuse work whose
scratch exceeds the array.  This file is collected last so that a run stopping
at the first failure has run every other test first; it also passes alone in a
fresh process."""
import pytest
import torch

import hybrid_linear_attention_rule_gb300 as K
import kda_inputs as KI
from parity_utils import assert_close, case_to_device, to_np

pytestmark = pytest.mark.gpu


def _noalloc(c, d, conv_state, out=None, fs=None):
    T, H, dk, dv, N = c.T, c.H, c.dk, c.dv, c.N
    if out is None:
        out = torch.full((T, H, dv), float("nan"), dtype=torch.float32, device="cuda")
    if fs is None:
        fs = torch.full((N, H, dk, dv), float("nan"), dtype=torch.float32, device="cuda")
    K.k3kda_prefill_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S0"], d["cu"].cuda(), d["cu"], N, T, H,
                            dk, dv, c.chunk, c.scale, c.use_qk_l2norm, d["conv_w"], conv_state, c.W, d["gate"], out,
                            fs)
    torch.cuda.synchronize()
    return out, fs


@pytest.mark.parametrize("shape", ["tensor_core_d128", "fp32_path_conv_staging"])
def test_noalloc_matches_workspace_prefill_twice(shape):
    if shape == "tensor_core_d128":
        c = KI.prefill_case("noalloc_tc", [130, 170], 2, 128, 128, 64, "bf16", seed=31, s0_std=0.02,
                            gate=True, conv_width=4, conv_state=True)
    else:   # dk = 64 runs the fp32 kernel, whose fused conv stages its output in the scratch
        c = KI.prefill_case("noalloc_f32", [77, 123], 2, 64, 128, 64, "bf16", seed=32, s0_std=0.02,
                            gate=True, conv_width=4, conv_state=True)
    d = case_to_device(c)
    cs_ref = d["conv_state"].clone()
    ref_out, ref_fs = K.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["S0"],
                                cu_seqlens=d["cu"], chunk=c.chunk, scale=c.scale, conv_weight=d["conv_w"],
                                conv_state=cs_ref, gate=d["gate"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    for call in range(2):
        cs = d["conv_state"].clone()
        out, fs = _noalloc(c, d, cs)
        assert K.k3kda_prefill_noalloc_status() == 0
        assert_close(to_np(out), to_np(ref_out), False, f"{shape} out, call {call}")
        assert_close(to_np(fs), to_np(ref_fs), False, f"{shape} final state, call {call}")
        assert torch.equal(cs, cs_ref), "conv state"


def test_noalloc_call_takes_no_device_memory():
    """After a first call (which loads the kernels), a call leaves the device's free memory as it was:
    nothing in its call tree allocates, through cudaMalloc or any library."""
    c = KI.prefill_case("noalloc_mem", [300], 2, 128, 128, 64, "bf16", seed=33, gate=True, conv_width=4)
    d = case_to_device(c)
    cs = torch.zeros((1, 3, 3 * 2 * 128), device="cuda")
    out = torch.empty((c.T, c.H, 128), device="cuda")
    fs = torch.empty((1, c.H, 128, 128), device="cuda")
    _noalloc(c, d, cs, out, fs)
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc(c, d, cs, out, fs)
    free1, _ = torch.cuda.mem_get_info()
    assert free1 >= free0, f"free device memory dropped by {free0 - free1} bytes over the calls"


@pytest.mark.parametrize("T", [300, 8192], ids=["two_pass", "single_pass"])
def test_noalloc_status_reports_a_wait_that_ran_out(T):
    """Small work runs the two-pass kernels in the array, long work (more chunk records than the
    array holds) the single-pass kernel; the internal test hook starves one wait of the call."""
    c = KI.prefill_case("noalloc_status", [T], 1, 128, 128, 64, "bf16", seed=34, gate=True)
    d = case_to_device(c)
    assert K.load_library().k3kda_test_arm_wait_timeout(0 if T == 300 else 1, 256) == 0
    _noalloc(c, d, None)
    assert K.k3kda_prefill_noalloc_status() == -6
    assert K.k3kda_prefill_noalloc_status() == 0
    out, fs = _noalloc(c, d, None)
    assert K.k3kda_prefill_noalloc_status() == 0
    ref_out, ref_fs = K.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], gate=d["gate"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_close(to_np(out), to_np(ref_out), False, "noalloc out after a timed-out call")
    assert_close(to_np(fs), to_np(ref_fs), False, "noalloc final state after a timed-out call")


def test_noalloc_refuses_work_larger_than_its_scratch():
    # fp32 path with a conv: the staging buffer is T * (2*H*dk + H*dv) * 4 bytes = 32 MiB here
    T, H, dk, dv = 8192, 4, 64, 128
    dev = "cuda"
    q = torch.zeros((T, H, dk), dtype=torch.bfloat16, device=dev)
    v = torch.zeros((T, H, dv), dtype=torch.bfloat16, device=dev)
    g = torch.zeros((T, H, dk), device=dev)
    beta = torch.zeros((T, H), device=dev)
    cw = torch.zeros((2 * H * dk + H * dv, 4), device=dev)
    out = torch.zeros((T, H, dv), device=dev)
    with pytest.raises(K.K3KDAError) as ei:
        K.k3kda_prefill_noalloc(q, q, v, g, beta, None, None, None, 1, T, H, dk, dv, 64, dk ** -0.5, True, cw, None,
                                4, None, out, None)
    assert ei.value.status == -4
