"""Row-sharded execution on one GPU, shard after shard, as each device of a
row-sharded deployment would run its part: a tile-row range of a weight is a
weight of its own (no copy), and the lm_head's shards reduce to 64-bit top-1
keys (q4nx_gemv_top1_key) whose maximum is the global top-1.

Checks: the shards' GEMV outputs, concatenated, within the bar of the other
GPU tests against the binary64 oracle; each shard's key equals the host
encoding of the largest of that shard's own q4nx_gemv fp32 outputs (same
kernel partition, so the same bits); the combined key's row equals the
unsharded q4nx_gemv_top1 and the oracle's argmax when the oracle's top-2 gap
clears twice the tolerance.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from test_gpu_parity import DEV, assert_within, out_values, to_dev_bf16, to_dev_bytes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import dequant_gemv_gb300

    return dequant_gemv_gb300


@pytest.mark.parametrize("world", [2, 3, 8])
@pytest.mark.parametrize("kind,N,K", [(synth.Q8_KR, 8192, 2560), (synth.Q8_BLK, 4096, 2560), (synth.Q4_1, 12288, 1024)])
def test_row_shards(q, kind, N, K, world):
    f, w = synth.make(kind, N, K, synth.rng(51, world, N + K))
    x = synth.activations(synth.rng(51, 100 + world, N + K), 1, K)[0]
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    xd = to_dev_bf16(x)
    ys, keys = [], []
    for r in range(world):
        S, row_base = W.row_shard(r, world)
        assert S.chunks.data_ptr() == W.chunks.data_ptr() + (row_base // 32) * (K // 256) * q.q4nx_chunk_bytes(kind)
        y = q.q4nx_gemv(S, xd, out_dtype="f32")
        k = q.q4nx_gemv_top1_key(S, xd, row_base=row_base)
        yv = y.cpu().numpy()
        i = int(oracle.argmax(yv.reshape(1, -1))[0])
        assert int(k.item()) == q.top1_key(float(yv[i]), row_base + i), f"shard {r}: key does not match its outputs"
        ys.append(yv)
        keys.append(int(k.item()))
    y_all = np.concatenate(ys).astype(np.float64)
    Y64, A = oracle.matmul(w, kind, N, K, x)
    assert_within(y_all, Y64, A, False, f"shards of {N}x{K}")
    row = q.top1_key_row(max(keys))
    full = int(q.q4nx_gemv_top1(W, xd).item())
    order = np.argsort(-Y64)
    gap = Y64[order[0]] - Y64[order[1]]
    if gap > 2 * 1e-3 * (A[order[0]] + A[order[1]]):
        assert row == full == int(order[0])


def test_top1_key_row_base_limits(q):
    W = q.Weight(torch.zeros(5120, dtype=torch.uint8, device=DEV), synth.Q4_1, 32, 256)
    xd = torch.zeros(256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(q.Q4NXError):
        q.q4nx_gemv_top1_key(W, xd, row_base=-1)
    with pytest.raises(q.Q4NXError):
        q.q4nx_gemv_top1_key(W, xd, row_base=2**31 - 32)
    k = q.q4nx_gemv_top1_key(W, xd, row_base=2**31 - 33)    # all outputs 0: the shard's first row
    assert q.top1_key_row(k.item()) == 2**31 - 33
