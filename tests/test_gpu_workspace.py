"""Workspace contract of the GEMV family (q4nx.h): a zero-filled workspace is
left zero-filled by every q4nx_gemv, q4nx_gemv_top1 and q4nx_gemv_batch call,
so one workspace serves any sequence of such calls; and the GEMM, whose
workspace keeps partial tiles, does not disturb the GEMV's results when the
binding runs both on one stream.  The shapes split tile rows between warps
and between CTAs (the cases that post partial sums)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import dequant_gemv_gb300

    return dequant_gemv_gb300


def _weight(q, kind, N, K, seed):
    f, w = synth.make(kind, N, K, synth.rng(21, seed, N + K))
    x = synth.activations(synth.rng(21, seed + 1, N + K), 1, K)[0]
    W = q.Weight(torch.from_numpy(w).to(DEV), kind, N, K)
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(DEV).view(torch.bfloat16)
    return w, x, W, xd


SHAPES = [(synth.Q4_1, 96, 768), (synth.Q4_1, 32, 2816), (synth.Q4_K, 160, 1280), (synth.Q8_KR, 4096, 12288),
          (synth.Q8_BLK, 12288, 4096), (synth.Q4_1, 151936 // 4, 2560), (synth.Q4_1, 12288, 4096),
          (synth.Q8_KR, 151936, 2560)]


@pytest.mark.parametrize("kind,N,K", SHAPES)
def test_gemv_leaves_workspace_zero(q, kind, N, K):
    w, x, W, xd = _weight(q, kind, N, K, 0)
    need = int(q.lib.q4nx_gemv_workspace(ctypes.byref(W.c())))
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for out in ("bf16", "f32"):
        q.q4nx_gemv(W, xd, out_dtype=out, ws=ws)
        torch.cuda.synchronize()
        nz = torch.nonzero(ws).flatten()
        assert nz.numel() == 0, f"{out}: {nz.numel()} workspace bytes left non-zero, first at {nz[:8].tolist()}"
    q.q4nx_gemv_top1(W, xd, ws=ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(ws).item() == 0, "top-1 left the workspace non-zero"


def test_gemv_batch_leaves_workspace_zero(q):
    mats = [(synth.Q4_1, n, k) for n, k in [(2048, 1024), (1024, 1024), (1024, 2048), (3072, 1024), (1024, 3072)]]
    made = [_weight(q, kind, N, K, 10 + i) for i, (kind, N, K) in enumerate(mats)]
    ys = [torch.empty(N, dtype=torch.bfloat16, device=DEV) for (_, N, _) in mats]
    batch = q.GemvBatch([(W, xd, y) for (_, _, W, xd), y in zip(made, ys)], out_dtype="bf16")
    ws = batch.ws
    ws.zero_()
    for _ in range(3):
        batch()
    torch.cuda.synchronize()
    assert torch.count_nonzero(ws).item() == 0


def test_gemv_after_gemm_on_one_stream(q):
    # the binding's default workspaces: a GEMM call between two GEMV calls
    kind, N, K = synth.Q4_1, 4096, 12288
    w, x, W, xd = _weight(q, kind, N, K, 30)
    y0 = q.q4nx_gemv(W, xd, out_dtype="f32").clone()
    X = torch.from_numpy(synth.activations(synth.rng(21, 31, 7), 64, K).view(np.int16)).to(DEV).view(torch.bfloat16)
    q.q4nx_gemm_m64(W, X)
    y1 = q.q4nx_gemv(W, xd, out_dtype="f32")
    torch.cuda.synchronize()
    assert torch.equal(y0, y1), "GEMV result changed after a GEMM on the same stream"
    rows = np.arange(0, N, 97)
    Y64, A = oracle.matmul(w, kind, N, K, x, rows=rows)
    got = y1.cpu().numpy().astype(np.float64)[rows]
    assert np.all(np.abs(got - Y64) <= 1e-3 * A)
    q.q4nx_check()
