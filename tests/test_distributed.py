"""Multi-process paths on the CPU (gloo, world size 2): the amax all-reduce
that sharded quantization needs, checked with the oracle (a shard encoded
with the global amax equals the rows of the whole tensor's encoding), and
the bench's max-over-ranks of the timing."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _sharded_worker(rank, world, port, block2d, q):
    try:
        _init(rank, world, port)
        from nvfp4_bit_block_02_b300.distributed import global_amax
        rng = np.random.default_rng(5)
        full = (rng.standard_normal((256, 192)) * np.where(rng.random((256, 192)) < 0.01, 40.0, 1.0)).astype(np.float32)
        rows = full.shape[0] // world
        shard = full[rank * rows:(rank + 1) * rows]
        # the shard's amax (on a GPU rank this is nvfp4_amax), then the 4-byte all-reduce
        a = torch.tensor([float(np.max(np.abs(shard)))], dtype=torch.float32)
        global_amax(a)
        mine = oracle.quantize(shard, block2d=block2d, amax=float(a[0]))
        whole = oracle.quantize(full, block2d=block2d)
        sl = slice(rank * rows, (rank + 1) * rows)
        ok = (float(a[0]) == whole.amax and mine.g == whole.g and (mine.codes == whole.codes[sl]).all()
              and (mine.scales == whole.scales[sl]).all())
        q.put((rank, ok, float(a[0]), whole.amax))
    except Exception as e:  # reported to the parent
        q.put((rank, False, repr(e), None))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


@pytest.mark.parametrize("block2d", [False, True])
def test_sharded_quantization_equals_whole_tensor(block2d):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_sharded_worker, args=(r, world, port, block2d, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
    for rank, ok, a, whole in sorted(results):
        assert ok, f"rank {rank}: amax {a} vs whole {whole}"


def _timing_worker(rank, world, port, q):
    try:
        _init(rank, world, port)
        from bench import max_over_ranks
        got = max_over_ranks([1.0 + rank, 10.0 - rank], world)
        q.put((rank, got))
    except Exception as e:
        q.put((rank, repr(e)))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_bench_takes_the_max_over_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_timing_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
    for rank, got in results:
        assert got == [2.0, 10.0], f"rank {rank}: {got}"
