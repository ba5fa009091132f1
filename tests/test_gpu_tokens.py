"""q4nx_gemm_m64 for a few tokens: q4_1 at M <= 2 and Q4_K at M <= 4 run on
the CUDA cores, each chunk read once and entering the dot products of every
token with the per-token arithmetic of q4nx_gemv (M = 1: q4nx_gemv's kernel
for every kind); the other cases take the tensor-core path, checked here to
the same bar.

Checks: every output within the bar of the other GPU tests against the binary64
oracle; a repeated call bit-identical (partials are added in a fixed order);
Q4_K accepted up to four tokens; the workspace's few-token part left
zero-filled.
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


def _case(q, kind, N, K, M, seed):
    f, w = synth.make(kind, N, K, synth.rng(31, seed, N + K))
    X = synth.activations(synth.rng(31, seed + 1, N + K), M, K)
    return w, X, q.Weight(to_dev_bytes(w), kind, N, K), to_dev_bf16(X)


SHAPES = [(32, 256), (2080, 256), (96, 768), (160, 2816), (1024, 1024), (4096, 4096)]


def tensor_path(kind, M):
    """True when q4nx_gemm_m64 runs M tokens of this kind on the tensor cores."""
    return M > {synth.Q4_1: 2, synth.Q4_K: 4}.get(kind, 1)


@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K, synth.Q8_KR, synth.Q8_BLK])
def test_tokens_match_oracle(q, kind, N, K, M, out):
    w, X, W, Xd = _case(q, kind, N, K, M, 3 * M + (kind << 4))
    Y = q.q4nx_gemm_m64(W, Xd, out_dtype=out)
    got = out_values(Y)
    assert got.shape == (M, N)
    rows = None if N * K <= 4_000_000 else np.unique(np.concatenate([
        np.arange(0, 96), np.arange(N - 96, N), np.random.default_rng(M).integers(0, N, 200)]))
    Y64, A = oracle.matmul(w, kind, N, K, X, rows=rows)
    # (q4_1 and Q8 at larger M take the tensor-core path: bf16 weights, reading o21)
    assert_within(got if rows is None else got[:, rows], Y64, A, out == "bf16", f"tokens kind {kind} {N}x{K} M={M}",
                  bf16_weights=tensor_path(kind, M) and K < 2560)
    again = q.q4nx_gemm_m64(W, Xd, out_dtype=out)
    bits = torch.int16 if out == "bf16" else torch.int32
    assert torch.equal(Y.view(bits), again.view(bits)), "a repeated call gave different bits"


@pytest.mark.parametrize("M", [2, 4])
@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K])
def test_tokens_row_split_over_many_ctas(q, kind, M):
    """64 x 65536: each tile row's 256 chunks spread over 64 CTAs, whose
    per-token row sums the owner of the row's first chunk adds up."""
    N, K = 64, 65536
    w, X, W, Xd = _case(q, kind, N, K, M, 70 + M)
    got = out_values(q.q4nx_gemm_m64(W, Xd, out_dtype="f32"))
    Y64, A = oracle.matmul(w, kind, N, K, X)
    assert_within(got, Y64, A, False, f"tokens kind {kind} {N}x{K} M={M}",
                  bf16_weights=tensor_path(kind, M) and K < 2560)


def test_q4k_tokens_then_unsupported_beyond(q):
    w, X, W, Xd = _case(q, synth.Q4_K, 2560, 9728, 5, 90)
    rows = np.arange(0, 2560, 5)
    Y64, A = oracle.matmul(w, synth.Q4_K, 2560, 9728, X[:4], rows=rows)
    got = out_values(q.q4nx_gemm_m64(W, Xd[:4].contiguous(), out_dtype="bf16"))
    assert_within(got[:, rows], Y64, A, True, "Q4_K 2560x9728 M=4")
    with pytest.raises(q.Q4NXError):
        q.q4nx_gemm_m64(W, Xd, out_dtype="bf16")        # five tokens: tensor-core path, no Q4_K


def test_tokens_workspace_part_left_zero(q):
    kind, N, K, M = synth.Q4_1, 4096, 12288, 2
    w, X, W, Xd = _case(q, kind, N, K, M, 70)
    need = int(q.lib.q4nx_gemm_workspace(ctypes.byref(W.c()), M))
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for _ in range(3):
        q.q4nx_gemm_m64(W, Xd, out_dtype="f32", ws=ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(ws).item() == 0          # the tensor-core part is untouched by few-token calls
    q.q4nx_check(ws)
