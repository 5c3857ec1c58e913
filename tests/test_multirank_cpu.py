"""The multi-GPU story of this path is replicas: sequences and heads never interact, so N
ranks each run their own share with no collective inside the mixer, and the job's time is
the slowest rank's.  These tests run that logic as world_size-2 gloo process groups on the
CPU: the bench's max-over-ranks timing and job throughput, sharding a packed batch by
sequence (each rank runs the oracle on its sequences; the gathered result equals one
process running them all), and the reference arm printing one line under torchrun."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(world, fn, *args):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_entry, args=(r, world, port, fn, args, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    for _ in procs:
        r, res = q.get(timeout=300)
        results[r] = res
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0, f"rank process exited with {p.exitcode}"
    return results


def _entry(rank, world, port, fn, args, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, fn(rank, world, *args)))
    finally:
        dist.destroy_process_group()


def _bench_reduce(rank, world):
    import bench
    times = [10.0 + rank, 2.0 - rank, 1.5 * (rank + 1)]       # each rank's (total, prefill, decode) ms
    mx = bench.max_over_ranks(times, world, "cpu")
    return mx, bench.job_value(1000, world, mx[0] / 1e3)


def test_bench_takes_the_slowest_rank_and_counts_all_replicas():
    res = _run(2, _bench_reduce)
    for r in (0, 1):
        mx, value = res[r]
        assert mx == [11.0, 2.0, 3.0]
        assert value == pytest.approx(2 * 1000 / 0.011)


def _shard_oracle(rank, world, lengths, seed):
    import kda_inputs as KI
    import oracle as O
    c = KI.prefill_case("shard", lengths, 2, 16, 16, 16, "f32", seed=seed, s0_std=0.02, gate=True)
    cu = c.cu_seqlens
    mine = list(range(rank, len(lengths), world))          # sequences of this rank
    outs = {}
    for n in mine:
        a, b = int(cu[n]), int(cu[n + 1])
        o, S, _ = O.mixer(c.q[a:b], c.k[a:b], c.v[a:b], c.g[a:b], c.beta[a:b], initial_state=c.S0[n:n + 1],
                          gate=c.gate[a:b], scale=c.scale)
        outs[n] = (o, S[0])
    gathered = [None] * world
    dist.all_gather_object(gathered, outs)
    return {n: v for part in gathered for n, v in part.items()}


def test_sequence_sharding_over_two_ranks_matches_one_process():
    import kda_inputs as KI
    import oracle as O
    lengths, seed = [37, 64, 5, 90, 0, 17], 3
    res = _run(2, _shard_oracle, lengths, seed)
    c = KI.prefill_case("shard", lengths, 2, 16, 16, 16, "f32", seed=seed, s0_std=0.02, gate=True)
    o_full, S_full, _ = O.mixer(c.q, c.k, c.v, c.g, c.beta, initial_state=c.S0, gate=c.gate,
                                cu_seqlens=c.cu_seqlens, scale=c.scale)
    for r in (0, 1):
        parts = res[r]
        assert sorted(parts) == list(range(len(lengths)))
        for n in range(len(lengths)):
            a, b = int(c.cu_seqlens[n]), int(c.cu_seqlens[n + 1])
            assert np.array_equal(parts[n][0], o_full[a:b]), f"sequence {n} output"
            assert np.array_equal(parts[n][1], S_full[n]), f"sequence {n} state"


def test_reference_arm_prints_one_line_from_rank_zero_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-sample-tokens", "256"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
