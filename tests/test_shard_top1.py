"""Vocabulary-sharded lm_head top-1 on CPU ranks (gloo, world size 2 and 3).

The lm_head rows shard by tile rows over the devices; each device reduces its
shard to one 64-bit key (q4nx_gemv_top1_key's format) and one MAX all-reduce
of int64 keys gives the global winner: the largest logit, the lowest row among
equal maxima, and a NaN logit winning (the first one), as the oracle's argmax
decides on the whole vector.  Here each rank's shard of logits comes from the
oracle (a q4_1 lm_head-shaped weight) or is planted (ties across shards, NaN,
-0/+0), its local key is built with the binding's host encoder, and the keys
are exchanged through torch.distributed on gloo.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _local_key(q, logits, row_base):
    # the shard's key: max over its rows' keys (the kernel folds rows the same way)
    return max(q.top1_key(float(v), row_base + i) for i, v in enumerate(logits))


def _rank(rank, world, port, cases, out):
    import torch.distributed as dist

    import dequant_gemv_gb300 as q

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = []
        for logits in cases:
            tr0, tr1 = q.shard_tile_rows(len(logits) // 32, rank, world)
            key = torch.tensor([_local_key(q, logits[tr0 * 32:tr1 * 32], tr0 * 32)], dtype=torch.int64)
            dist.all_reduce(key, op=dist.ReduceOp.MAX)
            res.append(q.top1_key_row(key.item()))
        out[rank] = res
    finally:
        dist.destroy_process_group()


def _cases():
    # an lm_head-shaped q4_1 GEMV (vocabulary 8192 rows x 512) from the oracle
    N, K = 8192, 512
    f, w = synth.make(synth.Q4_1, N, K, synth.rng(41, 0, 1))
    x = synth.activations(synth.rng(41, 1, 1), 1, K)[0]
    y64, _ = oracle.matmul(w, synth.Q4_1, N, K, x)
    real = y64.astype(np.float32)
    n = 96 * 32
    base = np.random.default_rng(5).standard_normal(n).astype(np.float32)
    tie = base.copy()
    tie[[100, 2000, 3000]] = 9.0                     # equal maxima in different shards: the lowest row wins
    nan = base.copy()
    nan[[2500, 2900]] = np.nan                       # NaN in a later shard wins; the first NaN
    zero = np.full(n, -1.0, np.float32)
    zero[1500] = -0.0
    zero[40] = 0.0                                   # -0 and +0 are equal: the lower row
    neg = np.full(n, -np.inf, np.float32)
    neg[3071] = -3.0e38
    return [real, tie, nan, zero, neg]


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_top1_keys_combine_to_the_global_argmax(world):
    cases = _cases()
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, cases, out), nprocs=world, join=True)
        res = dict(out)
    expect = [int(oracle.argmax(c.reshape(1, -1))[0]) for c in cases]
    for r in range(world):
        assert res[r] == expect, (r, res[r], expect)


def test_shard_tile_rows_partition():
    import dequant_gemv_gb300 as q

    for tr in (1, 7, 96, 4748):
        for world in (1, 2, 3, 8):
            parts = [q.shard_tile_rows(tr, r, world) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == tr
            assert all(parts[i][1] == parts[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        q.shard_tile_rows(10, 2, 2)
