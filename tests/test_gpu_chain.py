"""Dependent launches back to back: each call reads the previous call's
output, on one stream, with no synchronisation in between.  The kernels
start while the previous grid drains and wait for it before reading their
input; the intermediate buffers are pre-filled with ones, so a kernel that
read its input early would be checked against the wrong input and fail.
Every stage is compared with the oracle applied to the input the stage
actually received (read back after the chain)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from test_gpu_parity import DEV, assert_within, bf16_np, out_values, to_dev_bf16, to_dev_bytes

pytestmark = pytest.mark.gpu

DIMS = [1024, 2048, 1024, 3072, 1024]          # K of stage 0, then each stage's N (= the next stage's K)


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import dequant_gemv_gb300

    return dequant_gemv_gb300


def _stages(q):
    st = []
    for i in range(len(DIMS) - 1):
        N, K = DIMS[i + 1], DIMS[i]
        _, w = synth.make(synth.Q4_1, N, K, synth.rng(4, 20 + i, 0))
        st.append((w, q.Weight(to_dev_bytes(w), synth.Q4_1, N, K), N, K))
    return st


def _check(stages, inputs, outputs, tensor_cores, what):
    g = np.random.default_rng(7)
    for i, (w, _, N, K) in enumerate(stages):
        rows = np.unique(np.concatenate([np.arange(0, 48), np.arange(N - 48, N), g.integers(0, N, 200)]))
        Y64, A = oracle.matmul(w, synth.Q4_1, N, K, bf16_np(inputs[i]), rows=rows)
        assert_within(out_values(outputs[i])[:, rows], Y64, A, True, f"{what} stage {i}", bf16_weights=tensor_cores)


@pytest.mark.parametrize("M", [1, 2, 64])
def test_chain_of_dependent_products(q, M):
    """GEMV (M = 1), few-token GEMV (M = 2) or tensor-core GEMM (M = 64),
    four stages of alternating width."""
    stages = _stages(q)
    X0 = to_dev_bf16(synth.activations(synth.rng(4, 30, 0), M, DIMS[0]))
    outs = [torch.ones((M, N), dtype=torch.bfloat16, device=DEV) for (_, _, N, _) in stages]
    torch.cuda.synchronize()
    cur = X0
    for i, (_, W, _, _) in enumerate(stages):
        if M == 1:
            q.q4nx_gemv(W, cur[0], out=outs[i][0], out_dtype="bf16")
        else:
            q.q4nx_gemm_m64(W, cur, out=outs[i], out_dtype="bf16")
        cur = outs[i]
    torch.cuda.synchronize()
    q.q4nx_check(device=DEV)
    _check(stages, [X0] + outs[:-1], outs, M > 2, f"M={M} chain")


def test_chain_across_kernels(q):
    """Tensor-core GEMM -> GEMV of one of its output rows -> GEMV -> few-token
    GEMV of two rows of the first output, all without synchronisation."""
    stages = _stages(q)
    X0 = to_dev_bf16(synth.activations(synth.rng(4, 31, 0), 64, DIMS[0]))
    Y0 = torch.ones((64, DIMS[1]), dtype=torch.bfloat16, device=DEV)
    y1 = torch.ones((1, DIMS[2]), dtype=torch.bfloat16, device=DEV)
    y2 = torch.ones((1, DIMS[3]), dtype=torch.bfloat16, device=DEV)
    y3 = torch.ones((2, DIMS[2]), dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    q.q4nx_gemm_m64(stages[0][1], X0, out=Y0, out_dtype="bf16")
    q.q4nx_gemv(stages[1][1], Y0[5], out=y1[0], out_dtype="bf16")
    q.q4nx_gemv(stages[2][1], y1[0], out=y2[0], out_dtype="bf16")
    X3 = Y0[10:12]
    q.q4nx_gemm_m64(stages[1][1], X3, out=y3, out_dtype="bf16")
    torch.cuda.synchronize()
    q.q4nx_check(device=DEV)
    _check(stages[:1], [X0], [Y0], True, "GEMM")
    _check(stages[1:3], [Y0[5:6], y1], [y1, y2], False, "GEMV after GEMM")
    _check(stages[1:2], [X3], [y3], False, "two tokens after GEMV")
