"""q4nx_pack_q4_1 (GGUF-type tensor -> q4_1 chunks) against the oracle, byte for byte.

Q4_0 and Q4_1 map exactly (codes unchanged, bf16 rounding of scale and zero);
Q8_0 and the dense types go through a min/max q4_1 whose every step is one IEEE
binary32 operation, so the GPU's chunks must equal the oracle's exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from test_gpu_parity import DEV

pytestmark = pytest.mark.gpu

TYPES = [synth.SRC_Q4_0, synth.SRC_Q4_1, synth.SRC_Q8_0, synth.SRC_F32, synth.SRC_F16, synth.SRC_BF16]


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import dequant_gemv_gb300

    return dequant_gemv_gb300


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("N,K", [(32, 256), (96, 768), (1024, 1024), (4096, 12288)])
def test_pack_matches_the_oracle_byte_for_byte(q, t, N, K):
    src, _ = synth.gguf_tensor(t, N, K, synth.rng(30, t, N + K))
    got = q.q4nx_pack_q4_1(torch.from_numpy(src).to(DEV), t, N, K).cpu().numpy()
    want = oracle.pack_q4_1(src, t, N, K)
    assert np.array_equal(got, want)


def test_pack_special_groups(q):
    """Constant groups (scale 0), groups on their own grid (exact), +-0 minima, huge and tiny magnitudes."""
    N, K = 32, 512
    g = np.random.default_rng(31)
    x = g.normal(0, 0.02, size=(N, K)).astype(np.float32)
    x[0, :32] = 0.0371                                   # constant
    x[1, :32] = -0.09375 + 2.0 ** -7 * g.integers(0, 16, 32)
    x[1, 0], x[1, 1] = -0.09375, -0.09375 + 15 * 2.0 ** -7
    x[2, :32] = np.abs(x[2, :32])
    x[2, 3], x[2, 7] = 0.0, -0.0                          # equal minima of both signs
    x[3, :32] *= 1e30
    x[4, :32] *= 1e-30
    got = q.q4nx_pack_q4_1(torch.from_numpy(x).to(DEV), synth.SRC_F32, N, K).cpu().numpy()
    assert np.array_equal(got, oracle.pack_q4_1(x, synth.SRC_F32, N, K))


def test_packed_q4_0_feeds_the_gemv(q):
    """A Q4_0 tensor packed on the GPU and multiplied by the GEMV matches the oracle's product of the same chunks."""
    N, K = 2048, 2048
    src, _ = synth.gguf_tensor(synth.SRC_Q4_0, N, K, synth.rng(32))
    chunks = q.q4nx_pack_q4_1(torch.from_numpy(src).to(DEV), synth.SRC_Q4_0, N, K)
    x = synth.activations(synth.rng(33), 1, K)[0]
    y = q.q4nx_gemv(q.Weight(chunks, q.Q4NX_Q4_1, N, K),
                    torch.from_numpy(x.view(np.int16)).to(DEV).view(torch.bfloat16), out_dtype="f32")
    Y64, A = oracle.matmul(chunks.cpu().numpy(), oracle.Q4_1, N, K, x[None, :])
    assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - Y64[0]) <= 1e-3 * A[0])
