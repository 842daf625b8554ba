"""Multi-rank host logic on CPU (gloo, world size 2): the bench's max-over-ranks
timing and weak-scaling arithmetic, and chunk-range sharding of the oracle
(ranks encode disjoint chunk ranges of one input; concatenating their blocks in
rank order reproduces the single-process stream)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    import oracle
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # timing: every rank sees the slowest rank's time
    t = bench.max_over_ranks(10.0 + rank, dist, "cpu")
    # sharding: rank r encodes chunks [r*C/world, (r+1)*C/world) of the same input
    x = synth.generate(1)
    cs = 2048
    chunks = -(-x.size // cs)
    c0, c1 = chunks * rank // world, chunks * (rank + 1) // world
    blocks = np.zeros(chunks * cs, np.uint8)
    sizes = np.zeros(chunks, np.uint32)
    entries = np.zeros(2 * chunks, np.uint32)
    lib = oracle._load()
    lib.orc_encode_chunk_range(oracle._u8(x), x.size, 4, cs, 1, c0, c1, oracle._u8(blocks),
                               oracle._u32(sizes), oracle._u32(entries))
    body = b"".join(bytes(blocks[c * cs: c * cs + int(sizes[c])]) for c in range(c0, c1))
    parts = [None] * world
    dist.all_gather_object(parts, (c0, c1, body, entries[2 * c0: 2 * c1].tobytes()))
    results[rank] = (t, parts)
    dist.destroy_process_group()


def test_two_rank_gloo_aggregation_and_sharding(orc):
    world = 2
    port = _free_port()
    manager = mp.Manager()
    results = manager.dict()
    mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
    import synth
    x = synth.generate(1)
    ref = orc.compress(x, 4, 2048, 1)
    chunks = -(-x.size // 2048)
    for rank in range(world):
        t, parts = results[rank]
        assert t == 11.0
        table = b"".join(p[3] for p in parts)
        body = b"".join(p[2] for p in parts)
        assert [p[0] for p in parts] == [0, chunks // 2]
        assert table == bytes(ref[32: 32 + 8 * chunks])
        assert body == bytes(ref[32 + 8 * chunks:])
