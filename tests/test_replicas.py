"""Replica aggregation across ranks with the gloo backend on CPU (world size 2)."""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, port, out):
    import torch.distributed as dist
    from sparse_entmax_attention_gb300 import replicas
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        assert replicas.world() == (rank, 2)
        replicas.barrier()
        out[rank] = replicas.max_over_ranks(100.0 + 7.5 * rank)
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs)
        assert dict(out) == {0: 107.5, 1: 107.5}


def test_single_process_is_identity():
    from sparse_entmax_attention_gb300 import replicas
    assert replicas.world() == (0, 1)
    assert replicas.max_over_ranks(3.25) == 3.25
