"""The bench's algorithmic accounting matches the per-unit figures the roofline is stated in
(no GPU): bytes that must cross HBM and flops of the method, per (token, head) or per item."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_prefill_bytes_and_flops_per_token_head():
    T, H, d, C, W = 65536, 32, 128, 64, 4
    by, fl = bench.prefill_work(T, H, d, C, W)
    D = 3 * H * d
    # q, k, v 768 + g 512 + beta 4 + gate 256 + out 256 = 1796 B per (token, head); one final state
    # per head; the conv state in and out and the conv weights
    assert by == T * H * 1796 + H * d * d * 4 + 2 * (W - 1) * D * 4 + D * W * 4
    assert fl == T * H * (10 * C * d + 6 * d * d) + T * D * 2 * W
    assert abs(by - 3.769e9) < 1e6                        # the 3.77 GB of the fused-mixer call


def test_chunked_and_varlen_prefill_bytes():
    """No conv, no gate: 1540 B per (token, head) and the fp32 states (406 MB for T=8192, H=32)."""
    by, fl = bench.prefill_work(8192, 32, 128, 64, 0, gate=False)
    assert by == 8192 * 32 * 1540 + 32 * 128 * 128 * 4
    assert abs(by - 406e6) < 1e6
    assert fl == 8192 * 32 * (10 * 64 * 128 + 6 * 128 * 128)
    by3, _ = bench.prefill_work(135937, 32, 128, 64, 0, N=16, gate=False, initial_state=True)
    assert by3 == 135937 * 32 * 1540 + 2 * 16 * 32 * 128 * 128 * 4


def test_decode_bytes_per_sequence_head():
    N, H, d, W = 256, 32, 128, 4
    by, _ = bench.decode_work(N, H, d, W)
    D = 3 * H * d
    per_nh = 2 * 4 * d * d + 768 + 512 + 4 + 256 + 256     # state in and out, the token's vectors
    assert by == N * H * per_nh + 2 * N * (W - 1) * D * 4 + D * W * 4
    assert by == 1164148736                                # 1.164 GB per step


def test_attention_decode_bytes_per_attended_key():
    lens = np.array([0, 5, 511, 8191])
    H, d = 32, 128
    by, fl = bench.mla_work(lens, H, d)
    keys = int((lens + 1).sum())
    # key and value rows (bf16) of every attended key, the appended rows, five vectors a head, lengths
    assert by == keys * H * d * 4 + len(lens) * H * d * 4 + len(lens) * H * d * 10 + len(lens) * 8
    assert fl == keys * H * 4 * d


def test_backward_flops_per_token_head():
    T, H, d = 8192, 32, 128
    by, fl = bench.backward_work(T, H, d)
    assert fl == T * H * 23 * d * d                        # forward 5 d^2 + reverse sweep 18 d^2
    assert by == T * H * (6 * d + 4 * d + 4 * d + 4 + 4 * 4 * d + 4)
