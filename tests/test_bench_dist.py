"""Multi-rank host logic of bench.py on CPU: two gloo ranks (replicas), the
barrier, the max-over-ranks timing and the summed token count that make the
whole-job value, and the reference arm's rank-0-only rule."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_env()
    bench.maybe_init_dist(w)
    bench.barrier(w)
    ms = 10.0 * (r + 1)                 # rank 1 is the slow one
    tokens = 800.0 + r                  # per-rank tokens
    mx = bench.max_over_ranks(ms, w)
    tot = bench.sum_over_ranks(tokens, w)
    q.put((r, w, mx, tot, tot / (mx / 1e3)))
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, mx, tot, value in out:
        assert w == 2
        assert mx == 20.0               # whole-job time = the slowest rank
        assert tot == 1601.0            # all ranks' tokens
        assert value == pytest.approx(1601.0 / 0.020)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    from bloom_decoder_token_gb300 import synth
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        warmup = 3
        steps = 1
        ref_decode_steps = 1
    bench.run_reference(A(), synth.PRESETS["block"])   # returns at once: no work, no line
    assert capsys.readouterr().out == ""
