"""Parity of the tensor-core decode + GEMM (q4nx_gemm_m64) with the oracle, for
q4_1 chunks and Q8 chunks in both code layouts.

Bar: every output within 1e-3 * sum_k |w_k x_k| of the binary64 oracle (plus
2^-8 |y| for bf16 outputs), per-row cosine >= 0.99999.  Shapes narrower than
the configurations (K < 2560) add 2^-9 * sum_k |w_k x_k| for the bf16 rounding
of the weights the tensor cores multiply (reading o21), which short sums do
not average out.  The kernel multiplies
bf16-decoded weights with fp32 accumulation on tcgen05 tensor cores.
"""
import dataclasses

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


def run(q, kind, N, K, M, out="f32", rows=None, seed=0, wid=4):
    f, w = synth.make(kind, N, K, synth.rng(wid, 0, 50 + seed))
    X = synth.activations(synth.rng(wid, 0, 60 + seed), M, K)
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    Y = out_values(q.q4nx_gemm_m64(W, to_dev_bf16(X), out_dtype=out))
    assert Y.shape == (M, N)
    Y64, A = oracle.matmul(w, kind, N, K, X, rows=rows)
    # the configurations' widths (K >= 2560) meet the plain 1e-3 bar: over long
    # sums the weights' bf16 rounding averages out; short ones take reading o21
    assert_within(Y if rows is None else Y[:, rows], Y64, A, out == "bf16", f"gemm {N}x{K} M={M}",
                  bf16_weights=K < 2560)
    return Y


@pytest.mark.parametrize("N,K", [(128, 512), (96, 768), (256, 1024), (1024, 1024), (160, 2816), (4224, 512)])
@pytest.mark.parametrize("M", [64, 1, 5, 17])
def test_gemm_q4_1_small(q, N, K, M):
    run(q, synth.Q4_1, N, K, M)


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q8_KR, synth.Q8_BLK])
@pytest.mark.parametrize("N", [32, 256, 4096])
@pytest.mark.parametrize("M", [64, 9])
def test_gemm_single_k_step(q, kind, N, M):
    """K = 256: every tile is a single k-step (no tile is split between CTAs)."""
    run(q, kind, N, 256, M, wid=5 if kind != synth.Q4_1 else 4)


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q8_KR, synth.Q8_BLK])
@pytest.mark.parametrize("N,K", [(128, 12288), (96, 16384), (256, 12288)])
@pytest.mark.parametrize("M", [64, 17])
def test_gemm_tile_split_many_ways(q, kind, N, K, M):
    """Narrow, deep weights: a 128-row tile's k-steps spread over 8-16 CTAs,
    so its finisher takes the later partials through all 5 shared-memory
    gather slots and reads the rest directly."""
    run(q, kind, N, K, M, wid=5 if kind != synth.Q4_1 else 4)


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_gemm_q4_1_output_dtypes(q, out):
    run(q, synth.Q4_1, 512, 1536, 64, out=out)


@pytest.mark.parametrize("N,K", [(12288, 4096), (4096, 12288)])
def test_gemm_prefill_block_8b_width(q, N, K):
    """The 64-token prefill block at 8B width (gate/up 12288x4096, down 4096x12288)."""
    rows = np.unique(np.concatenate([np.arange(0, 160), np.arange(N - 160, N),
                                     np.random.default_rng(2).integers(0, N, 600)]))
    run(q, synth.Q4_1, N, K, 64, out="bf16", rows=rows)


@pytest.mark.parametrize("M", [1, 64])
def test_merged_gate_up_weight(q, M):
    """gate and up of the 8B-width block (12288x4096 each) as one 24576x4096
    weight, their chunk arrays concatenated: rows below 12288 are gate's
    outputs, the rest up's, each checked against the oracle of its own weight
    (sampled rows around both ends and the seam)."""
    Nh, K = 12288, 4096
    _, wg = synth.make(synth.Q4_1, Nh, K, synth.rng(4, 10, 0))
    _, wu = synth.make(synth.Q4_1, Nh, K, synth.rng(4, 11, 0))
    X = synth.activations(synth.rng(4, 12, 0), M, K)
    W = q.Weight(to_dev_bytes(np.concatenate([wg, wu])), synth.Q4_1, 2 * Nh, K)
    Xd = to_dev_bf16(X)
    if M == 1:
        Y = out_values(q.q4nx_gemv(W, Xd[0].contiguous(), out_dtype="bf16"))[None]
    else:
        Y = out_values(q.q4nx_gemm_m64(W, Xd, out_dtype="bf16"))
    assert Y.shape == (M, 2 * Nh)
    g = np.random.default_rng(3)
    for w, base in ((wg, 0), (wu, Nh)):
        r = np.unique(np.concatenate([np.arange(0, 96), np.arange(Nh - 96, Nh), g.integers(0, Nh, 300)]))
        Y64, A = oracle.matmul(w, synth.Q4_1, Nh, K, X, rows=r)
        assert_within(Y[:, base + r], Y64, A, True, f"merged gate|up M={M} half {base // Nh}")


def test_gemm_repeat_runs_are_byte_identical(q):
    f, w = synth.make(synth.Q4_1, 4096, 12288, synth.rng(4, 0, 70))
    X = to_dev_bf16(synth.activations(synth.rng(4, 0, 71), 64, 12288))
    W = q.Weight(to_dev_bytes(w), synth.Q4_1, 4096, 12288)
    a = q.q4nx_gemm_m64(W, X, out_dtype="f32").clone()
    b = q.q4nx_gemm_m64(W, X, out_dtype="f32").clone()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    q.q4nx_check(device=DEV)


def test_gemm_tokens_beyond_m_untouched(q):
    """Rows m >= M of the output are neither read nor written."""
    N, K, M = 256, 512, 5
    f, w = synth.make(synth.Q4_1, N, K, synth.rng(4, 0, 80))
    X = synth.activations(synth.rng(4, 0, 81), M, K)
    W = q.Weight(to_dev_bytes(w), synth.Q4_1, N, K)
    big = torch.full((8, N), 7.0, dtype=torch.float32, device=DEV)
    q.q4nx_gemm_m64(W, to_dev_bf16(X), out=big[:M], out_dtype="f32")
    assert (big[M:] == 7.0).all()
    Y64, A = oracle.matmul(w, synth.Q4_1, N, K, X)
    assert_within(out_values(big[:M]), Y64, A, False, "M=5", bf16_weights=True)


def test_gemm_matches_gemv_per_token(q):
    """Each token row of the GEMM agrees with a GEMV of that token (both within
    tolerance of the oracle; checked against each other at twice the bar)."""
    N, K, M = 1024, 2048, 8
    f, w = synth.make(synth.Q4_1, N, K, synth.rng(4, 0, 90))
    X = synth.activations(synth.rng(4, 0, 91), M, K)
    W = q.Weight(to_dev_bytes(w), synth.Q4_1, N, K)
    Xd = to_dev_bf16(X)
    Y = out_values(q.q4nx_gemm_m64(W, Xd, out_dtype="f32"))
    _, A = oracle.matmul(w, synth.Q4_1, N, K, X)
    for m in range(M):
        y = out_values(q.q4nx_gemv(W, Xd[m].contiguous(), out_dtype="f32"))
        assert np.all(np.abs(Y[m] - y) <= 2e-3 * A[m])


# ---- Q8 chunks (both code layouts): w = d * code, the lm_head kind ----

@pytest.mark.parametrize("kind", [synth.Q8_KR, synth.Q8_BLK])
@pytest.mark.parametrize("N,K", [(128, 512), (256, 1024), (4224, 512), (160, 2816)])
@pytest.mark.parametrize("M", [64, 1, 5, 17])
def test_gemm_q8_small(q, kind, N, K, M):
    run(q, kind, N, K, M, wid=5)


@pytest.mark.parametrize("kind", [synth.Q8_KR, synth.Q8_BLK])
def test_gemm_q8_bf16_output(q, kind):
    run(q, kind, 512, 1536, 64, out="bf16", wid=5)


@pytest.mark.parametrize("kind", [synth.Q8_KR, synth.Q8_BLK])
def test_gemm_q8_lm_head_64_tokens(q, kind):
    """The Q8 lm_head 151936x2560 at 64 tokens, fp32 logits (rows sampled for the oracle)."""
    N, K = 151936, 2560
    rows = np.unique(np.concatenate([np.arange(0, 160), np.arange(N - 160, N),
                                     np.random.default_rng(5).integers(0, N, 600)]))
    run(q, kind, N, K, 64, out="f32", rows=rows, wid=5)


def test_gemm_q4_1_lm_head_64_tokens(q):
    """An lm_head-sized q4_1 matrix (151936x2560, 243 MB) at 64 tokens, bf16 out (rows sampled)."""
    N, K = 151936, 2560
    rows = np.unique(np.concatenate([np.arange(0, 160), np.arange(N - 160, N),
                                     np.random.default_rng(6).integers(0, N, 600)]))
    run(q, synth.Q4_1, N, K, 64, out="bf16", rows=rows, wid=6)


def test_gemm_q8_layouts_agree_on_the_same_weights(q):
    """The same logical codes packed in layout KR and in layout BLK give the same products, bit for bit."""
    N, K, M = 512, 2048, 64
    f, wkr = synth.make(synth.Q8_KR, N, K, synth.rng(5, 0, 95))
    wblk = synth.pack(dataclasses.replace(f, kind=synth.Q8_BLK))
    X = to_dev_bf16(synth.activations(synth.rng(5, 0, 96), M, K))
    a = q.q4nx_gemm_m64(q.Weight(to_dev_bytes(wkr), synth.Q8_KR, N, K), X, out_dtype="f32")
    b = q.q4nx_gemm_m64(q.Weight(to_dev_bytes(wblk), synth.Q8_BLK, N, K), X, out_dtype="f32")
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


# ---- small token blocks (verify windows, multi-token prediction blocks): M in {2, 4, 8, 16} ----

@pytest.mark.parametrize("M", [2, 4, 8, 16])
@pytest.mark.parametrize("kind,N,K,wid", [(synth.Q4_1, 4096, 4096, 4), (synth.Q8_BLK, 2048, 2560, 5)])
def test_gemm_small_token_blocks(q, M, kind, N, K, wid):
    rows = np.unique(np.concatenate([np.arange(0, 128), np.arange(N - 128, N),
                                     np.random.default_rng(M).integers(0, N, 300)]))
    run(q, kind, N, K, M, out="bf16" if kind == synth.Q4_1 else "f32", rows=rows, wid=wid)
