"""The refit over a batch sharded across ranks, on CPU with gloo (world size
2): each rank accumulates the labels of its own block of sequences (the
oracle's sums, packed in the library's accumulator layout), the ranks sum
the blocks with one all-reduce, and every rank's solve equals the oracle's
refit of the whole batch ("Adaptive Verification without a confidence head",
"Fitting the coefficients": one theta from every label of the round)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from speculative_decoding_verification_03_gb300 import shard


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _labelled(seed, B, K):
    """Features from a spread of draft sharpness, accept lengths drawn from a
    known logistic (omega 0.5, beta decreasing from 0.55), ragged kept
    lengths."""
    rng = np.random.default_rng(seed)
    x = rng.normal(1.0, 2.0, (B, K))
    beta = 0.55 - 0.1 * np.arange(K)
    p = 1.0 / (1.0 + np.exp(-(0.5 * x + beta)))
    kept = rng.integers(0, K + 1, B).astype(np.int32)
    acc = np.zeros(B, np.int32)
    for b in range(B):
        a = 0
        while a < kept[b] and rng.random() < p[b, a]:
            a += 1
        acc[b] = a
    return x, acc, kept


def _round_sharded(rank, world, steps, theta0, B, K, damping_c):
    th = np.array(theta0, np.float64)
    for r, blocks in enumerate(steps):
        block = np.zeros(4 * K + 2)
        for (x, acc, kept) in blocks:
            b0, b1 = shard.shard_range(B, world, rank)
            d = oracle.av_accumulate(th, x[b0:b1], acc[b0:b1], kept[b0:b1])
            block += shard.block_from_dense(d["g"], d["H"], d["n"])
        t = torch.from_numpy(block)
        shard.sum_over_ranks_(t)
        th, _, _ = oracle.av_solve_update(th, shard.dense_from_block(t.numpy()), damping_c)
    return th


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, K = 301, 5
        rounds = [[_labelled(100 * r + s, B, K) for s in range(3)] for r in range(4)]  # 4 rounds of 3 steps
        out[rank] = _round_sharded(rank, world, rounds, [1.0] + [0.0] * K, B, K, 10.0).tolist()
    finally:
        dist.destroy_process_group()


def test_shard_range_partitions_the_batch():
    for B in (0, 1, 7, 64, 301, 1024):
        for world in (1, 2, 3, 8):
            parts = [shard.shard_range(B, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == B
            for (a0, a1), (b0, b1) in zip(parts, parts[1:]):
                assert a1 == b0
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
    with pytest.raises(ValueError):
        shard.shard_range(4, 2, 2)


def test_block_layout_round_trip():
    K = 4
    rng = np.random.default_rng(0)
    x, acc, kept = _labelled(1, 50, K)
    d = oracle.av_accumulate(rng.normal(size=K + 1), x, acc, kept)
    blk = shard.block_from_dense(d["g"], d["H"], d["n"])
    assert blk.size == 4 * K + 2
    back = shard.dense_from_block(blk)
    # the refit's Hessian is arrow-shaped: the block holds all of it
    np.testing.assert_array_equal(back["H"], d["H"])
    np.testing.assert_array_equal(back["g"], d["g"])
    np.testing.assert_array_equal(back["n"], d["n"])


def test_two_rank_refit_equals_whole_batch_gloo():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(180)
            assert p.exitcode == 0
        got0, got1 = np.array(out[0]), np.array(out[1])
    # every rank applies the identical update
    np.testing.assert_array_equal(got0, got1)
    # the whole batch on one process, rounds of 3 steps (oracle.AVFit)
    B, K = 301, 5
    fit = oracle.AVFit([1.0] + [0.0] * K, round_len=3, damping_c=10.0)
    for r in range(4):
        for s in range(3):
            x, acc, kept = _labelled(100 * r + s, B, K)
            fit.step(x, acc, kept)
    np.testing.assert_allclose(got0, fit.theta, rtol=1e-12, atol=1e-12)
    assert not np.allclose(fit.theta, [1.0] + [0.0] * K)  # the rounds moved theta
