"""The N > 1 path on the CPU: two gloo ranks, the replica synchronisation that
bench.py uses (barrier + max of step times) and the whole-job value; plus the
property replicas rely on - the same seeded inputs give every rank identical
oracle results."""

import os
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    import oracle
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    barrier, allmax = bench.replica_sync(world, device="cpu")
    barrier()
    ms = allmax(1.0 + rank)                        # rank 1 is the slower one
    value = bench.whole_job_value(world, ms)
    cfg = synth.preset("tiny")
    W = synth.make_weights(cfg, seed=5)
    h = synth.make_hiddens(cfg, 12, seed=5)
    k, v, _ = oracle.inject_context(cfg, W, h, np.arange(12), "none")
    L = cfg["n_layers"]
    d = oracle.draft_block(cfg, W, [[k[l] for l in range(L)]], [[v[l] for l in range(L)]],
                           synth.make_anchors(cfg, 1, seed=5), [12], 8, "none")
    q.put((rank, ms, value, d["ids"].tolist(), float(d["logits"].sum())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert out[0][1] == out[1][1] == 2.0           # both ranks see the slowest time
    assert out[0][2] == pytest.approx(2 * 1e3 / 2.0)
    assert out[0][3] == out[1][3] and out[0][4] == out[1][4]
