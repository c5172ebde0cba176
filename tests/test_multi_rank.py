"""Host logic of the N > 1 bench path on CPU: two gloo ranks, each with its own
replica inputs, no collective on the data path, and whole-job aggregation as the
slowest rank's time over the bytes of all ranks."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    import kvq_synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = kvq_synth.WORKLOADS["tiny_kivi"]
    K, V = kvq_synth.prefill_kv(wl, 64, replica=rank)
    q = kvq_synth.queries(wl, 2, replica=rank)
    ms = 10.0 + 5.0 * rank                   # rank 1 is the slow one
    nbytes = 1000.0 * (rank + 1)
    ms_max, b_all = bench.reduce_over_ranks(ms, nbytes, world)
    out[rank] = (ms_max, b_all, float(K.astype(np.float32).sum()), float(q.astype(np.float32).sum()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_and_replicas():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    r0, r1 = out[0], out[1]
    assert r0[0] == r1[0] == 15.0            # max over ranks
    assert r0[1] == r1[1] == 3000.0          # bytes summed over ranks
    assert r0[2] != r1[2] and r0[3] != r1[3]  # each rank draws its own replica


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(3.5, 7.0, 1) == (3.5, 7.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    import kvq_synth

    class A:
        steps, warmup = 3, 3
    called = []
    monkeypatch.setattr(bench, "print", lambda *a, **k: called.append(a), raising=False)
    assert bench.reference_arm(A(), kvq_synth.WORKLOADS["tiny_kivi"], {"metric": "m"}, 1, 2) == 0
    assert called == []
