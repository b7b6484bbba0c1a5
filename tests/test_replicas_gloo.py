"""The multi-GPU path is replicas only: every rank builds the trees of its own batch, and the job takes as long as its
slowest rank. Its host side on the CPU, two ranks over gloo: the maximum over ranks, the whole-job throughput, one
batch of inputs per replica, and the reference arm that rank 0 alone runs."""
import os
import socket
import types

import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from speculative_decoding_tree_top_gb300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, seconds, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), GLOO_SOCKET_IFNAME="lo")  # loopback: no hostname lookup needed
    w, r, _ = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        t = bench.max_over_ranks(seconds[r], w, "cpu")
        queue.put((r, w, t, bench.job_throughput(w, 4, 10, t)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    world, seconds = 2, [1.25, 2.5]
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica, args=(r, world, port, seconds, queue)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        got = sorted(queue.get(timeout=120) for _ in range(world))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    assert [g[0] for g in got] == [0, 1]
    for _, w, t, v in got:  # every rank: the slowest rank's time, and both ranks' trees over it
        assert w == 2 and t == 2.5 and v == 2 * 4 * 10 / 2.5


def test_one_rank_needs_no_process_group():
    assert not (dist.is_available() and dist.is_initialized())
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_throughput(1, 1, 500, 0.038) == 500 / 0.038


def test_replicas_draw_their_own_batches():
    # rank 0 reproduces the one-GPU workload; the other ranks' batches differ from it and from each other
    for cfg in range(5):
        assert bench.replica_seed(cfg, 0) == synth._resolve(cfg, None, {})[1]
        assert len({bench.replica_seed(cfg, r) for r in range(8)}) == 8
    a = synth.make_inputs(0, device="cpu", seed=bench.replica_seed(0, 0))
    b = synth.make_inputs(0, device="cpu", seed=bench.replica_seed(0, 1))
    assert not a.logits.equal(b.logits)


def test_reference_arm_runs_on_rank_zero_only():
    args = types.SimpleNamespace(config=0, steps=1, warmup=0, reference_budget=1.0)
    assert bench.run_reference(args, 2, 1) is None   # the other ranks leave at once, without work
