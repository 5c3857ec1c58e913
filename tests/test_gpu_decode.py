"""Parity of k3kda_decode_step (through the C ABI) with the oracle's decode step."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_rule_gb300 as K
import kda_inputs as KI
import oracle as O
from parity_utils import assert_close, dev_tensor, to_np

pytestmark = pytest.mark.gpu


def _run(c: KI.DecodeCase, out_dtype=torch.float32, rows=None):
    bf = c.in_dtype == "bf16"
    q, k, v = dev_tensor(c.q, bf), dev_tensor(c.k, bf), dev_tensor(c.v, bf)
    g, beta = dev_tensor(c.g, False), dev_tensor(c.beta, False)
    gate = None if c.gate is None else dev_tensor(c.gate, bf)
    cw = None if c.conv_w is None else dev_tensor(c.conv_w, False)
    cs = None if c.conv_state is None else dev_tensor(c.conv_state, False)
    st = dev_tensor(c.state, False)
    out = K.decode_step(q, k, v, g, beta, st, gate=gate, conv_weight=cw, conv_state=cs, scale=c.scale,
                        use_qk_l2norm=c.use_qk_l2norm, out_dtype=out_dtype)
    torch.cuda.synchronize()
    sel = slice(None) if rows is None else torch.as_tensor(rows, device=out.device)
    return to_np(out[sel]), to_np(st[sel]), None if cs is None else to_np(cs[sel])


def _oracle(c: KI.DecodeCase, rows=None):
    sel = slice(None) if rows is None else rows
    pick = lambda x: None if x is None else x[sel]
    return O.decode_step(pick(c.q), pick(c.k), pick(c.v), pick(c.g), pick(c.beta), pick(c.state),
                         gate=pick(c.gate), conv_w=c.conv_w, conv_state=pick(c.conv_state), scale=c.scale,
                         use_qk_l2norm=c.use_qk_l2norm)


def _check(c, out_dtype=torch.float32, rows=None):
    o, s, cs = _run(c, out_dtype, rows)
    ro, rs, rcs = _oracle(c, rows)
    fp32 = c.in_dtype == "f32"
    e1 = assert_close(o, ro, fp32, "decode out", store_bf16=out_dtype == torch.bfloat16)
    e2 = assert_close(s, rs, fp32, "decode state")
    if cs is not None:
        assert np.array_equal(cs, rcs), "conv state must shift exactly"
    return e1, e2


def test_decode_small_bf16_conv_gate():
    _check(KI.decode_case(seed=1, N=8, H=4, d=128))


def test_decode_full_size_sampled_sequences():
    """The full workload (256 sequences x 32 heads, 512 MiB fp32 state) in the bench's
    launch configuration; a seeded sample of 12 sequences checked against the oracle."""
    c = KI.decode_case(seed=0)
    rows = np.sort(np.random.default_rng(5).choice(c.N, 12, replace=False))
    _check(c, rows=rows)


def test_decode_bf16_output():
    _check(KI.decode_case(seed=2, N=4, H=2, d=128), out_dtype=torch.bfloat16)


@pytest.mark.parametrize("d", [16, 64, 128])
def test_decode_fp32_inputs_no_conv(d):
    c = KI.decode_case(seed=3, N=5, H=3, d=d, W=0)
    c.in_dtype = "f32"
    c.q, c.k, c.v = (KI.normal(x.shape, 1.0, 3, n) for x, n in ((c.q, "q"), (c.k, "k"), (c.v, "v")))
    c.gate = None
    _check(c)


@pytest.mark.parametrize("W", [1, 2, 3])
def test_decode_conv_widths(W):
    _check(KI.decode_case(seed=4, N=3, H=2, d=32, W=W))


def test_decode_without_l2norm():
    c = KI.decode_case(seed=6, N=3, H=2, d=64)
    c.use_qk_l2norm = False
    c.q = KI.round_bf16(c.q * 0.1)
    c.k = KI.round_bf16(c.k * 0.1)
    _check(c)


def test_decode_two_steps_chain():
    c = KI.decode_case(seed=7, N=4, H=2, d=128)
    bf = True
    q, k, v = dev_tensor(c.q, bf), dev_tensor(c.k, bf), dev_tensor(c.v, bf)
    g, beta, gate = dev_tensor(c.g, False), dev_tensor(c.beta, False), dev_tensor(c.gate, bf)
    cw, cs, st = dev_tensor(c.conv_w, False), dev_tensor(c.conv_state, False), dev_tensor(c.state, False)
    for _ in range(2):
        out = K.decode_step(q, k, v, g, beta, st, gate=gate, conv_weight=cw, conv_state=cs, out_dtype=torch.float32)
    torch.cuda.synchronize()
    o1, s1, c1 = O.decode_step(c.q, c.k, c.v, c.g, c.beta, c.state, gate=c.gate, conv_w=c.conv_w,
                               conv_state=c.conv_state)
    o2, s2, c2 = O.decode_step(c.q, c.k, c.v, c.g, c.beta, s1, gate=c.gate, conv_w=c.conv_w, conv_state=c1)
    assert_close(to_np(out), o2, False, "second step out")
    assert_close(to_np(st), s2, False, "second step state")
    assert np.array_equal(to_np(cs), c2)


def test_decode_zero_sequences_is_a_no_op():
    z = torch.zeros((0, 2, 16), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros((0, 2, 16, 16), device="cuda")
    out = K.decode_step(z, z, z, torch.zeros((0, 2, 16), device="cuda"), torch.zeros((0, 2), device="cuda"), st)
    torch.cuda.synchronize()
    assert out.shape == (0, 2, 16)
