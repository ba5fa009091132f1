"""q4nx_gemv_noalloc: the GEMV for callers that may not allocate device memory.

Some callers cannot hand the library a scratch buffer: a decode loop held to a
no-allocation policy once it is set up, or a plug-in whose host framework owns
every device allocation and passes in only inputs and outputs.  This entry
point uses scratch compiled into the library instead.  The test calls it
through the C ABI twice in a row (the second call runs on whatever the first
left in the shared scratch) and checks that both outputs are bit for bit those
of q4nx_gemv (the entry point that takes a caller-owned workspace; both run
the same deterministic kernel), that they lie within the other GPU tests' bar
of the binary64 oracle, and that q4nx_check_noalloc then reports no failed
wait.  The shapes include a 151936 x 2560 q4_1 weight, whose launch runs two
CTAs per SM and splits tile rows between CTAs.

This file is named so that pytest collects it last.
"""
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


def _dev_bytes(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


@pytest.mark.parametrize("kind,N,K,out", [
    (synth.Q4_1, 4096, 12288, "bf16"),      # tile rows shared between CTAs
    (synth.Q4_1, 1024, 1024, "f32"),
    (synth.Q4_K, 2560, 9728, "bf16"),
    (synth.Q8_BLK, 8192, 2560, "f32"),
    (synth.Q4_1, 151936, 2560, "f32"),      # two CTAs per SM, 304 CTAs
])
def test_noalloc_matches_workspace_entry_point(q, kind, N, K, out):
    f, w = synth.make(kind, N, K, synth.rng(11, 0, N + K))
    x = synth.activations(synth.rng(11, 1, N + K), 1, K)[0]
    W = q.Weight(_dev_bytes(w), kind, N, K)
    xd = _dev_bf16(x)
    ref = q.q4nx_gemv(W, xd, out_dtype=out).clone()
    bits = torch.int32 if out == "f32" else torch.int16
    code = q.Q4NX_OUT_F32 if out == "f32" else q.Q4NX_OUT_BF16
    dt = torch.float32 if out == "f32" else torch.bfloat16
    cw = W.c()
    stream = torch.cuda.current_stream().cuda_stream
    rows = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N), np.arange(0, N, max(1, N // 1024))]))
    Y64, A = oracle.matmul(w, kind, N, K, x, rows=rows)
    tol = 1e-3 * A + (2.0 ** -8 * (np.abs(Y64) + 1e-3 * A) + 2.0 ** -134 if out == "bf16" else 0.0)
    for call in range(2):
        y = torch.full((N,), float("nan"), dtype=dt, device=DEV)
        st = q.lib.q4nx_gemv_noalloc(ctypes.byref(cw), xd.data_ptr(), y.data_ptr(), code, stream)
        assert st == 0, q.q4nx_status_str(st)
        assert torch.equal(y.view(bits), ref.view(bits)), f"call {call}: not bit-identical to q4nx_gemv"
        got = y.float().cpu().numpy().astype(np.float64)[rows]
        assert np.all(np.abs(got - Y64) <= tol), f"call {call}: outside the bar of the oracle"
    assert q.lib.q4nx_check_noalloc(stream) == 0


def test_noalloc_scratch_covers_any_weight(q):
    # host-side sizes only: the scratch a GEMV needs does not grow with the
    # weight, so the built-in array serves every shape q4nx_gemv accepts
    cap = int(q.lib.q4nx_noalloc_scratch_bytes())
    assert cap == 1 << 20
    for rows, cols in [(32, 256), (151936, 2560), (32 * 300000, 256), (32 * 4096, 256 * 4096)]:
        cw = q.q4nx_weight(0x1000, 1 << 62, synth.Q4_1, 0, rows, cols)
        need = int(q.lib.q4nx_gemv_workspace(ctypes.byref(cw)))
        assert 0 < need <= cap, (rows, cols, need)
