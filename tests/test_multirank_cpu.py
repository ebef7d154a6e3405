"""The multi-rank path of bench.py on CPU (gloo, world size 2): each rank
draws its own batch (weak scaling over samples, no collective on the data
path) and the job's step time is the maximum over ranks."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, local = bench.dist_env()
    xq, _, params = bench.make_rank_inputs(r, 1)
    step_ms = 1.0 + r  # rank 1 is slower
    out[r] = (w, r, float(xq[0, :4, :4].sum()), bench.max_over_ranks(step_ms, w))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_own_batches_and_max_time():
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork of this (threaded) process
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    (w0, r0, s0, m0), (w1, r1, s1, m1) = out[0], out[1]
    assert (w0, r0, w1, r1) == (2, 0, 2, 1)
    assert s0 != s1            # different tokens per rank
    assert m0 == m1 == 2.0     # both ranks report the slowest


def test_rank0_tokens_are_the_workload_tokens():
    import bench
    import synth
    xq, kv, _ = bench.make_rank_inputs(0, 2)
    ref, _, _ = synth.make_inputs(bench.WORKLOAD_ID, 2)
    assert np.array_equal(xq, ref)
    assert kv is xq  # attention within one graph: key/value are the query tokens


def test_bipartite_workload_has_its_own_key_tokens():
    import bench
    import synth
    saved = bench.WORKLOAD_ID
    try:
        bench.WORKLOAD_ID = 4
        xq, kv, _ = bench.make_rank_inputs(1, 1)
        w = synth.workload(4)
        assert xq.shape == (1, w.query_features, w.embed_dim)
        assert kv.shape == (1, w.key_features, w.embed_dim)
    finally:
        bench.WORKLOAD_ID = saved
