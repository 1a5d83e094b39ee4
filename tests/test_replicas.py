"""The replica (N > 1) host path of bench.py, run as two gloo ranks on CPU:
disjoint batch indices per rank, the slowest rank's time, counters summed
over ranks, and each rank's edges equal to the oracle's for its batches."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
import synth


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, n_batches, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.workload("tiny")
        g = synth.chung_lu(w.n_nodes, w.mean_deg, w.gamma, w.wmax, w.rng_seed)
        bs = synth.BatchStream(w)
        batches = bench.replica_batches(rank, world, n_batches)
        edges = 0
        for b in batches:
            ref = oracle.sampler_run(g.indptr, g.indices, bs.seeds(b), w.fanouts, w.sampler_seed(b))
            edges += sum(len(i) for i in ref.idx)
        elapsed, (tot_edges, tot_batches) = bench.combine_ranks(torch, 10.0 + rank, [edges, len(batches)], "cpu")
        out.put((rank, batches, edges, elapsed, tot_edges, tot_batches))
    finally:
        dist.destroy_process_group()


def test_replica_host_path_two_gloo_ranks():
    world, n_batches = 2, 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, n_batches, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    all_batches = [b for r in res for b in r[1]]
    assert sorted(all_batches) == list(range(world * n_batches))  # disjoint, complete
    # the oracle over every batch in one process gives the same total
    w = synth.workload("tiny")
    g = synth.chung_lu(w.n_nodes, w.mean_deg, w.gamma, w.wmax, w.rng_seed)
    bs = synth.BatchStream(w)
    want = 0
    for b in range(world * n_batches):
        ref = oracle.sampler_run(g.indptr, g.indices, bs.seeds(b), w.fanouts, w.sampler_seed(b))
        want += sum(len(i) for i in ref.idx)
    for r in res:
        _, _, edges, elapsed, tot_edges, tot_batches = r
        assert elapsed == 10.0 + (world - 1)  # the slowest rank
        assert tot_edges == want and tot_batches == world * n_batches
    assert sum(r[2] for r in res) == want


def test_combine_ranks_single_process_is_identity():
    assert bench.combine_ranks(torch, 3.5, [7, 8], "cpu") == (3.5, [7, 8])
