"""The multi-GPU path (independent replicas) on CPU with gloo, world size 2."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from nano_intra_device_gb300 import replicas, workload as wl


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _init(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return replicas.setup("gloo")


def _timing_worker(rank, world, port, out):
    r, w, _ = _init(rank, world, port)
    replicas.barrier(w)
    out[rank] = (r, w, replicas.max_over_ranks(1.5 + r, w), replicas.sum_over_ranks(2048, w))
    replicas.teardown(w)


def test_replica_reductions_gloo_world2():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_timing_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == (0, 2, 2.5, 4096.0) and res[1] == (1, 2, 2.5, 4096.0)


def test_shard_covers_requests_once():
    for n in (1, 7, 1792):
        for world in (1, 2, 3, 8):
            parts = [replicas.shard(n, r, world) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))


def _oracle_worker(rank, world, port, out):
    from oracle import layer as orc
    r, w, _ = _init(rank, world, port)
    shape = wl.tiny_shape()
    ctx = [17, 33, 48, 64, 5, 90]
    full = wl.make_batch(shape, ctx, [], seed_bt=3)
    wts = wl.make_weights(shape, seed=2, gain_std=0.1)
    x = wl.make_x(shape, len(ctx), seed=2)
    kp, vp = wl.make_pools(shape, full, "cpu")
    b0, b1 = replicas.shard(len(ctx), r, w)
    # this replica's own requests: its rows of x, its rows of the block table
    res = orc.layer_step(shape, orc.weights_f64(wts), x[b0:b1], kp, vp, full.block_table[b0:b1],
                         full.seq_lens[b0:b1], full.q_lens[b0:b1])
    out[rank] = (b0, b1, res["y"])
    replicas.teardown(w)


def test_request_shards_on_replicas_equal_one_batch():
    """Each replica runs the layer on its own requests only; together they give
    exactly the single-process result: the step needs no data exchange."""
    from oracle import layer as orc
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_oracle_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    shape = wl.tiny_shape()
    ctx = [17, 33, 48, 64, 5, 90]
    full = wl.make_batch(shape, ctx, [], seed_bt=3)
    wts = wl.make_weights(shape, seed=2, gain_std=0.1)
    x = wl.make_x(shape, len(ctx), seed=2)
    kp, vp = wl.make_pools(shape, full, "cpu")
    ref = orc.layer_step(shape, orc.weights_f64(wts), x, kp, vp, full.block_table, full.seq_lens,
                         full.q_lens)["y"]
    y = np.zeros_like(ref)
    for b0, b1, part in res.values():
        y[b0:b1] = part
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
