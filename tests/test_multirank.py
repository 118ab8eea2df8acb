"""bench.py's multi-rank logic on CPU: world size 2 over gloo (no GPU).

The decode path shards by request with no collective, so the only
cross-rank steps are the barrier around the timed region and the max over
ranks of the elapsed time; each rank also draws its own requests.
"""
import os
import socket

import torch.multiprocessing as tmp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    dist = bench.dist_init(w, "gloo")
    bench.barrier(dist)
    t = bench.max_over_ranks(0.5 + rank, dist)           # rank 1 is the slow one
    from adaptive_sparse_paged_gb300 import synth
    wl = synth.Workload("t", 2, 1, 8, 2, 64, 16, seq_len=16 * 9)
    sh = synth.make_shared(wl, 1 + 1000 * rank, "cpu")
    lay = synth.make_layer(wl, sh, 1 + 1000 * rank, 0, "cpu")
    out[rank] = (t, float(lay.q.sum()))
    bench.barrier(dist)
    dist.destroy_process_group()


def test_two_ranks_gloo():
    world, port = 2, _free_port()
    mgr = tmp.get_context("spawn").Manager()
    out = mgr.dict()
    tmp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 1.5          # max over ranks on every rank
    assert out[0][1] != out[1][1]                 # each rank decodes its own requests


def test_reference_arm_other_ranks_exit(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "start_oracle_pool", lambda: called.append(1))
    bench.run_reference(bench.parse_args(["--impl", "reference"]))
    assert not called  # rank 1 does no work and returns
