"""Parity of k3kda_short_conv (through the C ABI) with the oracle's causal conv."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_rule_gb300 as K
import kda_inputs as KI
import oracle as O
from parity_utils import FP32_TOL, assert_close, dev_tensor, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("bf16", [False, True])
def test_short_conv_varlen_with_state(W, bf16):
    lens = [0, 1, 2, 37, 70, 3]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, D = int(cu[-1]), 300
    x = KI.normal((T, D), 1.0, W, "q", bf16)
    w = KI.normal((D, W), 0.5, W, "conv_w")
    cs = KI.normal((len(lens), W - 1, D), 1.0, W, "conv_state", True)
    xd, wd, csd = dev_tensor(x, bf16), dev_tensor(w, False), dev_tensor(cs, False)
    out = K.short_conv(xd, wd, conv_state=csd, cu_seqlens=torch.from_numpy(cu), out_dtype=torch.float32)
    torch.cuda.synchronize()
    ry, rcs = O.short_conv(x, w, conv_state=cs, cu_seqlens=cu, apply_silu=True, return_state=True)
    assert_close(to_np(out), ry, True, "conv out")
    assert np.array_equal(to_np(csd), rcs)


def test_short_conv_no_state_no_silu_bf16_out():
    T, D, W = 513, 128, 4
    x = KI.normal((T, D), 1.0, 11, "k", True)
    w = KI.normal((D, W), 0.5, 11, "conv_w")
    out = K.short_conv(dev_tensor(x, True), dev_tensor(w, False), apply_silu=False, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ry = O.short_conv(x, w, apply_silu=False)
    err = np.abs(to_np(out) - ry)
    assert (err <= np.maximum(FP32_TOL, 2.0 ** -8 * np.abs(ry))).all()   # one bf16 ulp of the value, if larger
