"""The multi-GPU path (independent replicas, one batch per rank) on CPU with gloo,
world size 2: per-rank batches differ, and the job's time is the slowest rank's while its
tokens are the sum over ranks."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist
    from rank_delta_paged_gb300 import workloads as W
    from rank_delta_paged_gb300.replicas import job_totals, replica_seed, tokens_per_s_per_layer
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = W.decode_7b(seed=replica_seed(0, rank), T=64, n_adapters=20)
        elapsed = [3.0, 5.0][rank]                      # rank 1 is the slower one
        ms, tokens = job_totals(elapsed, float(w.T), "cpu", world)
        out[rank] = (ms, tokens, tokens_per_s_per_layer(tokens, w.n_layers, ms),
                     w.token_adapter_idx.tolist())
    finally:
        dist.destroy_process_group()


def test_two_replicas_gloo():
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(2):
        ms, tokens, value, _ = res[r]
        assert ms == 5.0                      # max over ranks
        assert tokens == 128.0                # 64 tokens on each rank
        assert value == pytest.approx(128.0 / 5e-3)
    assert res[0][3] != res[1][3]            # each rank drew its own batch
