"""Multi-rank host logic on CPU (gloo, world size 2).

The path shards by request with no data exchange: each rank runs its own
requests, and the only cross-rank operations are the barrier and the max of
the step times.  These tests run two gloo ranks as child processes and
check (1) the max-over-ranks reduction and the whole-job rate the bench
reports, (2) that ranks draw disjoint inputs, and (3) that verification of
a request batch split across the ranks, gathered afterwards, equals the
oracle on the whole batch (requests are independent)."""
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


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import bench
    import oracle
    import workloads as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.reduce_max(1.5 + rank, dist, "cpu")
        rate = bench.whole_job_rate(384, world, ms)
        # disjoint per-rank inputs
        a = W.attn_inputs(**W.CONFIGS["tiny"], seed=bench.rank_seed(rank, 0))
        q = torch.from_numpy(a["q"].astype(np.int64))
        gathered = [torch.zeros_like(q) for _ in range(world)]
        dist.all_gather(gathered, q)
        distinct = not torch.equal(gathered[0], gathered[1])
        # request-sharded verification
        full = W.verify_inputs(R=8, B=5, V=300, seed=7)
        lo, hi = rank * 4, rank * 4 + 4
        shard = dict(full, R=4, target=full["target"][lo:hi], draft=full["draft"][lo:hi], y=full["y"][lo:hi],
                     u_accept=full["u_accept"][lo:hi], u_sample=full["u_sample"][lo:hi])
        mine = torch.from_numpy(oracle.spec_verify(shard)["out_tokens"].astype(np.int64))
        parts = [torch.zeros_like(mine) for _ in range(world)]
        dist.all_gather(parts, mine)
        np.save(os.path.join(out_dir, "rank%d.npy" % rank),
                np.array([ms, rate, float(distinct)], np.float64))
        if rank == 0:
            np.save(os.path.join(out_dir, "tokens.npy"), torch.cat(parts).numpy())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    assert r0[0] == r1[0] == pytest.approx(2.5)          # slowest rank sets the time
    assert r0[1] == pytest.approx(2 * 384 / 2.5e-3)       # all ranks' units / that time
    assert r0[2] == 1.0 and r1[2] == 1.0                  # ranks never share a request
    sys.path.insert(0, ROOT)
    import oracle
    import workloads as W

    whole = oracle.spec_verify(W.verify_inputs(R=8, B=5, V=300, seed=7))["out_tokens"]
    np.testing.assert_array_equal(np.load(tmp_path / "tokens.npy"), whole)
