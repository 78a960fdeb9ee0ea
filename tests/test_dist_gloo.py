"""The multi-process benchmark path on CPU: two gloo ranks, each an
independent replica with its own seeded batch (the decode step has no data
exchange between replicas).  Only the timing and byte totals cross ranks:
the slowest rank's time and the sum of bytes."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from paged_kv_cache_279_gb300 import workloads as wl
    r, w, local = bench.dist_env()
    bench.init_dist(w, "gloo")
    # every rank draws its own batch: the seed moves with the rank
    lens = wl.draw_lengths(wl.GQA_BF16, 1000 * r).tolist()
    slowest = bench.max_over_ranks(1.0 + r, w)
    total = bench.sum_over_ranks(bench.kv_bytes(lens, wl.GQA_BF16), w)
    bench.barrier(w)
    q.put((r, slowest, total, sum(lens)))
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_time_is_max_and_bytes_are_summed():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert res[0][1] == res[1][1] == 2.0
    per_rank_tokens = [r[3] for r in res]
    assert per_rank_tokens[0] != per_rank_tokens[1]  # independent replicas
    want = sum(t * 8 * 128 * 2 * 2 for t in per_rank_tokens)
    assert res[0][2] == res[1][2] == want
