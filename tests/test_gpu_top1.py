"""q4nx_gemv_top1: the lm_head GEMV fused with top-1 (the logits never reach memory).

The index must equal, bit for bit, the argmax (lowest row on ties, first NaN)
of the fp32 logits q4nx_gemv computes for the same call; and where the binary64
oracle's top two logits are further apart than twice the GEMV tolerance, it
must equal the oracle's argmax.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from test_gpu_parity import DEV, to_dev_bf16, to_dev_bytes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import dequant_gemv_gb300

    return dequant_gemv_gb300


def _weight(q, kind, N, K, seed, wid=5):
    f, w = synth.make(kind, N, K, synth.rng(wid, 0, seed))
    return f, w, q.Weight(to_dev_bytes(w), kind, N, K)


def _fused_vs_separate(q, W, x):
    logits = q.q4nx_gemv(W, x, out_dtype="f32")
    sep = int(q.q4nx_argmax(logits.view(1, -1)).item())
    fused = int(q.q4nx_gemv_top1(W, x).item())
    return fused, sep, logits


@pytest.mark.parametrize("kind", [synth.Q8_KR, synth.Q8_BLK])
def test_top1_lm_head_matches_argmax_of_the_logits_and_the_oracle(q, kind):
    N, K = 151936, 2560
    f, w, W = _weight(q, kind, N, K, 11)
    xb = synth.activations(synth.rng(5, 1, 11), 1, K)[0]
    fused, sep, _ = _fused_vs_separate(q, W, to_dev_bf16(xb))
    assert fused == sep
    Y64, A = oracle.matmul(w, kind, N, K, xb[None, :])
    y64, a64 = Y64[0], A[0]
    order = np.argsort(-y64, kind="stable")
    gap = y64[order[0]] - y64[order[1]]
    if gap > 2e-3 * max(a64[order[0]], a64[order[1]]):
        assert fused == int(order[0])


@pytest.mark.parametrize("kind,N,K", [(synth.Q4_1, 12288, 4096), (synth.Q4_K, 9728, 2560), (synth.Q4_1, 1024, 1024),
                                      (synth.Q8_KR, 4096, 2560), (synth.Q4_1, 64, 65536), (synth.Q8_BLK, 64, 65536),
                                      # 4-bit weights large enough for two CTAs per SM
                                      (synth.Q4_1, 151936, 2560), (synth.Q4_K, 4864, 38912)])
def test_top1_other_kinds_and_sizes(q, kind, N, K):
    f, w, W = _weight(q, kind, N, K, 12, wid=4)
    x = to_dev_bf16(synth.activations(synth.rng(4, 1, 12), 1, K)[0])
    fused, sep, _ = _fused_vs_separate(q, W, x)
    assert fused == sep


def test_top1_ties_pick_the_lowest_row(q):
    N, K = 8192, 1024
    f, w, W = _weight(q, synth.Q8_BLK, N, K, 13)
    x = torch.zeros(K, dtype=torch.bfloat16, device=DEV)       # every logit is 0
    assert int(q.q4nx_gemv_top1(W, x).item()) == 0


def test_top1_first_nan_wins(q):
    N, K = 8192, 1024
    f, w = synth.make(synth.Q8_KR, N, K, synth.rng(5, 0, 14))
    T = (N // 32) * (K // 256)
    chunks = w.reshape(T, 8704).copy()
    d = chunks[:, 8192:].view(np.uint16)                     # d bf16 [T][32 r][8 g]
    TC = K // 256
    for row in (5000, 3000):                                # tile row 93 / 78, in-tile row 8 / 24
        tr, r = divmod(row, 32)
        d[tr * TC + 1, r * 8 + 3] = 0x7FC0                  # a NaN scale: the whole row's logit is NaN
    W = q.Weight(to_dev_bytes(chunks.reshape(-1)), synth.Q8_KR, N, K)
    x = to_dev_bf16(synth.activations(synth.rng(5, 1, 14), 1, K)[0])
    fused, sep, logits = _fused_vs_separate(q, W, x)
    assert torch.isnan(logits[3000]) and torch.isnan(logits[5000])
    assert fused == sep == 3000


def test_top1_repeat_calls_leave_the_workspace_clean(q):
    N, K = 151936, 2560
    f, w, W = _weight(q, synth.Q8_KR, N, K, 15)
    x = to_dev_bf16(synth.activations(synth.rng(5, 1, 15), 1, K)[0])
    ws = torch.zeros(int(q.lib.q4nx_gemv_workspace(__import__("ctypes").byref(W.c()))), dtype=torch.uint8, device=DEV)
    got = [int(q.q4nx_gemv_top1(W, x, ws=ws).item()) for _ in range(3)]
    assert got[0] == got[1] == got[2]
    torch.cuda.synchronize()
    assert int(ws[4:16].count_nonzero().item()) == 0
    q.q4nx_check(device=DEV)


def test_argmax_waits_for_the_gemv_that_writes_its_logits(q):
    """The argmax starts while the GEMV that writes its logits drains: before
    every GEMV the buffer holds a planted maximum far above any logit, so an
    argmax that read it early would return the planted row.  Back to back on
    one stream, no synchronisation in between."""
    N, K = 151936, 2560
    Ws, xs = [], []
    for s in range(3):
        _, _, W = _weight(q, synth.Q8_KR, N, K, 30 + s)
        Ws.append(W)
        xs.append(to_dev_bf16(synth.activations(synth.rng(5, 1, 30 + s), 1, K)[0]))
    logits = torch.empty((1, N), dtype=torch.float32, device=DEV)
    idx = torch.empty(1, dtype=torch.int32, device=DEV)
    got = []
    for it in range(12):
        W, x = Ws[it % 3], xs[it % 3]
        logits.fill_(0.0)
        logits[0, (7919 * (it + 1)) % N] = 1e30
        q.q4nx_gemv(W, x, out=logits[0], out_dtype="f32")
        q.q4nx_argmax(logits, out=idx)
        got.append(idx.clone())
    torch.cuda.synchronize()
    ref = [int(q.q4nx_gemv_top1(Ws[i], xs[i]).item()) for i in range(3)]
    for it in range(12):
        assert int(got[it].item()) == ref[it % 3]
