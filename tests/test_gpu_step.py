"""The launch configuration bench.py times, at full size: the 28-layer
Qwen3-0.6B-shaped decode step (196 q4_1 GEMVs, 275.25 MB of chunks) in one
q4nx_gemv_batch launch, on the bench's own seeded inputs; and a batch of the
maximum item count.  Outputs are checked on sampled rows of every matrix
against the binary64 oracle, within the bar of the other GPU tests."""
import numpy as np
import pytest
import torch

import oracle
import synth
from test_gpu_parity import DEV, assert_within, out_values, to_dev_bf16, to_dev_bytes

pytestmark = pytest.mark.gpu

WORKLOAD_ID = 2          # the decode-step workload's seed stream (bench.py)


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import dequant_gemv_gb300

    return dequant_gemv_gb300


def test_decode_step_one_launch(q):
    mats = [(l, mi, n, k) for l in range(synth.QWEN3_06B_LAYERS) for mi, (_, n, k) in enumerate(synth.QWEN3_06B_LAYER)]
    assert len(mats) == 196
    items, host = [], []
    for (l, mi, n, k) in mats:
        f, w = synth.workload_weight(WORKLOAD_ID, mi, layer=l, shape=(n, k))
        x = synth.workload_activations(WORKLOAD_ID, mi, 1, k, layer=l)[0]
        items.append((q.Weight(to_dev_bytes(w), synth.Q4_1, n, k), to_dev_bf16(x),
                      torch.empty(n, dtype=torch.bfloat16, device=DEV)))
        host.append((w, x, n, k))
    assert sum(int(W.chunks.numel()) for W, _, _ in items) == 275_251_200
    batch = q.GemvBatch(items, out_dtype="bf16")
    for _ in range(2):                                   # the second launch runs on the workspace the first left
        batch()
    torch.cuda.synchronize()
    q.q4nx_check(batch.ws)
    rng = np.random.default_rng(196)
    for (W, xd, y), (w, x, n, k), (l, mi, _, _) in zip(items, host, mats):
        rows = np.unique(np.concatenate([[0, 31, 32, n - 1], rng.integers(0, n, 24)]))
        Y64, A = oracle.matmul(w, synth.Q4_1, n, k, x, rows=rows)
        assert_within(out_values(y)[rows], Y64, A, True, f"layer {l} matrix {mi} {n}x{k}")


def test_max_batch_items(q):
    n_items = q.Q4NX_MAX_BATCH
    rng = np.random.default_rng(7)
    shapes = [(32 * int(rng.integers(1, 5)), 256 * int(rng.integers(1, 4))) for _ in range(n_items)]
    items, host = [], []
    for i, (n, k) in enumerate(shapes):
        f, w = synth.make(synth.Q4_1, n, k, synth.rng(61, i, n + k))
        x = synth.activations(synth.rng(61, 1000 + i, n + k), 1, k)[0]
        items.append((q.Weight(to_dev_bytes(w), synth.Q4_1, n, k), to_dev_bf16(x),
                      torch.empty(n, dtype=torch.float32, device=DEV)))
        host.append((w, x, n, k))
    q.q4nx_gemv_batch(items, out_dtype="f32")
    torch.cuda.synchronize()
    for i, ((W, xd, y), (w, x, n, k)) in enumerate(zip(items, host)):
        Y64, A = oracle.matmul(w, synth.Q4_1, n, k, x)
        assert_within(out_values(y), Y64, A, False, f"item {i} {n}x{k}")
    with pytest.raises(ValueError):                     # one item past the maximum: refused before any launch
        q.q4nx_gemv_batch(items + items[:1], out_dtype="f32")


def test_layer_phases_on_merged_weights(q):
    """A decode layer's projections that read the same activations as one
    weight each: q|k|v (2048 + 1024 + 1024 rows of 1024 columns, parts of
    different heights) and gate|up (2 x 3072 rows), their chunk arrays
    concatenated; o and down as they are.  The four phases run as one
    q4nx_gemv_batch each, in order, every phase on one x; each part's rows are
    checked against the oracle of its own weight, around every seam."""
    layer = 3
    parts = {mi: synth.workload_weight(WORKLOAD_ID, mi, layer=layer, shape=(n, k))[1]
             for mi, (_, n, k) in enumerate(synth.QWEN3_06B_LAYER)}
    shapes = [(n, k) for (_, n, k) in synth.QWEN3_06B_LAYER]
    phases = [(0, 1, 2), (3,), (4, 5), (6,)]
    rng = np.random.default_rng(17)
    for p, grp in enumerate(phases):
        K = shapes[grp[0]][1]
        assert all(shapes[mi][1] == K for mi in grp)
        N = sum(shapes[mi][0] for mi in grp)
        x = synth.activations(synth.rng(62, layer, p), 1, K)[0]
        W = q.Weight(to_dev_bytes(np.concatenate([parts[mi] for mi in grp])), synth.Q4_1, N, K)
        y = torch.empty(N, dtype=torch.bfloat16, device=DEV)
        q.q4nx_gemv_batch([(W, to_dev_bf16(x), y)], out_dtype="bf16")
        got = out_values(y)
        base = 0
        for mi in grp:
            n = shapes[mi][0]
            rows = np.unique(np.concatenate([np.arange(0, 40), np.arange(n - 40, n), rng.integers(0, n, 64)]))
            Y64, A = oracle.matmul(parts[mi], synth.Q4_1, n, K, x, rows=rows)
            assert_within(got[base + rows], Y64, A, True, f"phase {p} part {mi} ({n}x{K} at row {base})")
            base += n
    q.q4nx_check(device=DEV)
