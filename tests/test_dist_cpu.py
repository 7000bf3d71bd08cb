"""Replica (weak-scaling) glue on two gloo ranks on the CPU: every rank owns
its own sequences; timing is reduced as the max over ranks, token counts as
the sum."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    from sparse_attention_prolog_gb300 import dist as D
    from sparse_attention_prolog_gb300 import workloads as W
    r, w, _ = D.init("gloo")
    seed = D.replica_seed(1002, r)
    inp = W.make_decode_inputs(B=2, n_q=2, seq_lens=[256, 256], H_I=4, d_I=64, topk=8, H=2, seed=seed,
                               with_attention=False)
    mx = D.max_over_ranks(1.5 + r)
    tot = D.sum_over_ranks(inp.T)
    D.barrier()
    q.put((r, w, seed, mx, tot, int(inp.k_cache[0, :4].astype(int).sum())))
    D.shutdown()


def test_two_rank_replicas_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert res[0][2] != res[1][2]                 # distinct replica seeds
    assert all(r[3] == 2.5 for r in res)          # max over ranks
    assert all(r[4] == 8 for r in res)            # tokens summed over ranks
