"""Sharded use of the casts across ranks (world size 2, gloo, CPU).

Every GPU machine in this pool has one GPU, so the benchmark runs independent
replicas; these tests cover the host-side logic of the paths that do shard:

* NVFP4 over row shards: the one exchange is an all-reduce(MAX) of the
  per-tensor amax; each rank quantizes its rows with the global amax and the
  global element offset of its first row, which keeps the stochastic-rounding
  stream identical to the unsharded call.
* The transposed ragged conversion over expert shards: each rank owns whole
  groups; its columns of the transposed output and its scale slots equal the
  unsharded result's.
* bench.py's max-over-ranks timing reduction.

The arithmetic runs in the CPU oracle (test infrastructure); the GPU library
uses the same offset and group conventions (checked by the GPU parity tests).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _nvfp4_shards(rank, world, port, result):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    from fp8_quantization_gb300 import workloads
    _init(rank, world, port)
    try:
        M, K = 96, 160
        bits = workloads.nvfp4_act(M, K, seed=11)
        rows = np.array_split(np.arange(M), world)[rank]
        r0, r1 = int(rows[0]), int(rows[-1]) + 1
        local = torch.tensor([float(oracle.nvfp4_amax(bits[r0:r1]))], dtype=torch.float32)
        dist.all_reduce(local, op=dist.ReduceOp.MAX)
        A = np.float32(local.item())
        q, sb, g = oracle.nvfp4_quantize(bits[r0:r1], A, use_sr=True, seed=77, offset=r0 * K)
        obj = [None] * world
        dist.all_gather_object(obj, (r0, q, sb, float(g)))
        if rank == 0:
            obj.sort(key=lambda t: t[0])
            Aw = oracle.nvfp4_amax(bits)
            qw, sbw, gw = oracle.nvfp4_quantize(bits, Aw, use_sr=True, seed=77)
            ok = (A == Aw and np.array_equal(np.concatenate([o[1] for o in obj]), qw)
                  and np.array_equal(np.concatenate([o[2] for o in obj]), sbw)
                  and all(o[3] == float(gw) for o in obj))
            result["nvfp4"] = bool(ok)
    finally:
        dist.destroy_process_group()


def _expert_shards(rank, world, port, result):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    from fp8_quantization_gb300 import workloads
    _init(rank, world, port)
    try:
        M, K, G = 700, 256, 8
        rng = np.random.default_rng(3)
        q = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
        s = rng.integers(100, 130, (M, K // 32), dtype=np.uint8)
        offs = workloads.random_group_offsets(M, G, seed=9)
        mine = np.array_split(np.arange(G), world)[rank]
        g0, g1 = int(mine[0]), int(mine[-1]) + 1
        t0, t1 = int(offs[g0]), int(offs[g1])
        loc = offs[g0:g1 + 1] - t0
        yT, yTs = oracle.fp4_to_fp8_cols(q[t0:t1], s[t0:t1], loc, 2)
        nb = int(((np.diff(loc) + 127) // 128).sum())
        obj = [None] * world
        dist.all_gather_object(obj, (g0, t0, t1, yT, yTs[:nb]))
        if rank == 0:
            fyT, fyTs = oracle.fp4_to_fp8_cols(q, s, offs, 2)
            ok = True
            for (gg0, a, b, y, ys) in obj:
                base = int(((np.diff(offs[:gg0 + 1]) + 127) // 128).sum())
                ok &= np.array_equal(fyT[:, a:b], y)
                ok &= np.array_equal(fyTs[base:base + ys.shape[0]], ys)
            result["experts"] = bool(ok)
    finally:
        dist.destroy_process_group()


def _bench_max(rank, world, port, result):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    _init(rank, world, port)
    try:
        v = bench.max_over_ranks(1.5 + rank, None)
        if rank == 0:
            result["max"] = v
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("fn,key,want", [(_nvfp4_shards, "nvfp4", True),
                                         (_expert_shards, "experts", True),
                                         (_bench_max, "max", 2.5)])
def test_two_ranks(fn, key, want):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        result = mgr.dict()
        port = free_port()
        mp.start_processes(fn, args=(2, port, result), nprocs=2, join=True, start_method="spawn")
        assert result.get(key) == want
