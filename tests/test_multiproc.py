"""Replica scaling on N ranks: each rank compresses its own prompt and the
benchmark reduces two host scalars (max step time, total tokens).  Checked
here with the gloo backend, world size 2, on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, tokens = bench.aggregate(10.0 * (rank + 1), 32768.0, dist)
    # a rank's shape-only work (budget bytes) must not depend on other ranks
    from eviction_kvc_score_gb300 import workloads as wk
    wl = wk.ZIGZAG_32K
    alg = bench.algorithmic_bytes(wl, [2048] * wl.n_layers)
    q.put((rank, ms, tokens, alg))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tokens, alg in got:
        assert ms == 20.0            # max over ranks
        assert tokens == 65536.0     # sum over ranks
        assert alg == 2_787_115_008  # the 32K workload's algorithmic bytes per prompt


def test_algorithmic_bytes_closed_form():
    import bench
    from eviction_kvc_score_gb300 import workloads as wk
    wl = wk.ZIGZAG_32K
    # K 2^31 + Q 2^25 + scores 2^25 + idx 4*8*65536 + 4 * 8 * 69632 * 256
    assert bench.algorithmic_bytes(wl, [2048] * 32) == (2**31 + 2**25 + 2**25 + 4 * 8 * 65536
                                                        + 4 * 8 * 69632 * 256)
    assert bench.score_flops(wl) == 4 * 32 * 128 * 128 * 32768 * 32
