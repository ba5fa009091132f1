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


def _planted_gemm(q):
    """A GEMM whose first tile is split between CTAs (1024x4096, M = 64: 32
    CTAs of 4 k-steps each, tile 0 finished by CTA 0 once its 3 contributors
    have counted themselves in)."""
    kind, N, K = synth.Q4_1, 1024, 4096
    f, w = synth.make(kind, N, K, synth.rng(21, 40, 0))
    X = synth.activations(synth.rng(21, 41, 0), 64, K)
    W = q.Weight(torch.from_numpy(w).to(DEV), kind, N, K)
    Xd = torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).to(DEV).view(torch.bfloat16)
    need = int(q.lib.q4nx_gemm_workspace(ctypes.byref(W.c()), 64))
    return w, X, W, Xd, need


def test_gemm_weights_of_different_sizes_share_one_workspace(q):
    """One GEMM workspace, sized for the largest, serves weights with
    different tile counts one after another, tensor-core blocks and
    few-token calls alike: the regions whose place depends on the weight (the
    posting counters, the few-token part) are left zero-filled, so the
    partial tiles that one weight's calls leave behind never reach another
    weight's counters."""
    shapes = [(synth.Q4_1, 1024, 4096, 64), (synth.Q4_1, 12288, 4096, 64), (synth.Q4_1, 4096, 1536, 2),
              (synth.Q4_1, 640, 12288, 33), (synth.Q4_1, 12288, 4096, 64), (synth.Q4_1, 2048, 2560, 2)]
    made = []
    for i, (kind, N, K, M) in enumerate(shapes):
        f, w = synth.make(kind, N, K, synth.rng(23, 50 + i, 0))
        X = synth.activations(synth.rng(23, 60 + i, 0), M, K)
        W = q.Weight(torch.from_numpy(w).to(DEV), kind, N, K)
        Xd = torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).to(DEV).view(torch.bfloat16)
        made.append((kind, N, K, M, w, X, W, Xd))
    need = max(int(q.lib.q4nx_gemm_workspace(ctypes.byref(W.c()), M)) for (_, _, _, M, _, _, W, _) in made)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for kind, N, K, M, w, X, W, Xd in made:
        Y = q.q4nx_gemm_m64(W, Xd, out_dtype="f32", ws=ws).cpu().numpy().astype(np.float64)
        q.q4nx_check(ws)
        rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(N - 64, N),
                                         np.random.default_rng(N + K).integers(0, N, 128)]))
        Y64, A = oracle.matmul(w, kind, N, K, X, rows=rows)
        bar = 1e-3 if M <= 2 else 1e-3 + 2.0 ** -9                 # CUDA-core / tensor-core path
        assert np.all(np.abs(Y[:, rows] - Y64) <= bar * A), (N, K, M)


# GEMM workspace: a 16-byte error block, the partial tiles (one per CTA, at
# most 1024 CTAs, each 64 tokens x 128 rows of fp32), then the posting
# counters (one per tile).
GEMM_COUNTERS = 16 + 1024 * 64 * 128 * 4


def _plant(ws):
    """Tile 0's posting counter far above any count its contributors can
    reach: the finisher's wait cannot succeed."""
    ws.zero_()
    ws[GEMM_COUNTERS:GEMM_COUNTERS + 4] = torch.tensor([0, 0, 0, 0x40], dtype=torch.uint8, device=ws.device)


def test_gemm_bounded_wait_reports_timeout_and_recovers(q):
    """A wait that cannot succeed gives up after its bounded time: the launch
    completes, q4nx_check reports Q4NX_E_DEVICE_TIMEOUT, and the context and
    the library stay usable; with the workspace zero-filled again the same
    call is correct."""
    kind, N, K = synth.Q4_1, 1024, 4096
    w, X, W, Xd, need = _planted_gemm(q)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    _plant(ws)
    q.q4nx_gemm_m64(W, Xd, out_dtype="f32", ws=ws)
    with pytest.raises(q.Q4NXError) as e:
        q.q4nx_check(ws)
    assert e.value.status == q.Q4NX_E_DEVICE_TIMEOUT
    ws.zero_()
    Y = q.q4nx_gemm_m64(W, Xd, out_dtype="f32", ws=ws).cpu().numpy().astype(np.float64)
    q.q4nx_check(ws)
    Y64, A = oracle.matmul(w, kind, N, K, X)
    assert np.all(np.abs(Y - Y64) <= (1e-3 + 2.0 ** -9) * A)


def test_default_workspace_is_zeroed_after_a_reported_timeout(q):
    """The binding's own GEMM workspace: q4nx_check raises and zero-fills it,
    so the next call through the default workspace is correct."""
    kind, N, K = synth.Q4_1, 1024, 4096
    w, X, W, Xd, need = _planted_gemm(q)
    _plant(q.workspace(torch.device(DEV), need, "gemm"))
    q.q4nx_gemm_m64(W, Xd, out_dtype="f32")
    with pytest.raises(q.Q4NXError):
        q.q4nx_check()
    Y = q.q4nx_gemm_m64(W, Xd, out_dtype="f32").cpu().numpy().astype(np.float64)
    q.q4nx_check()
    Y64, A = oracle.matmul(w, kind, N, K, X)
    assert np.all(np.abs(Y - Y64) <= (1e-3 + 2.0 ** -9) * A)


def test_gemv_on_two_streams_at_once(q):
    """Two streams, each with its own workspace (the binding keys them by
    stream), running GEMVs of different weights concurrently: every result
    equals the same call made alone."""
    kind = synth.Q4_1
    a = _weight(q, kind, 12288, 4096, 50)
    b = _weight(q, kind, 4096, 12288, 51)
    ref_a = q.q4nx_gemv(a[2], a[3], out_dtype="f32").clone()
    ref_b = q.q4nx_gemv(b[2], b[3], out_dtype="f32").clone()
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    outs_a, outs_b = [], []
    for _ in range(8):
        with torch.cuda.stream(s1):
            outs_a.append(q.q4nx_gemv(a[2], a[3], out_dtype="f32"))
        with torch.cuda.stream(s2):
            outs_b.append(q.q4nx_gemv(b[2], b[3], out_dtype="f32"))
    torch.cuda.synchronize()
    for ya, yb in zip(outs_a, outs_b):
        assert torch.equal(ya, ref_a) and torch.equal(yb, ref_b)
    for s in (s1, s2):
        with torch.cuda.stream(s):
            q.q4nx_check()
