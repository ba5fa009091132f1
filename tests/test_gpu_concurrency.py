"""Cross-CTA waits with most SMs taken by another kernel.

The GEMV's split tile rows and the GEMM's split tiles are finished by the CTA
holding their first chunk (k-step), which waits, bounded, for the later CTAs'
posted partials.  A later CTA posts after its own first tile row (tile), not
at its end, and CTAs are dispatched in index order, so a launch completes
without all its CTAs being resident at once.  This test holds all SMs but 8
with a kernel on another stream (one CTA per SM through its shared-memory
request; it spins on %globaltimer for 30 ms and exits, a bounded wait) and
runs the GEMV, the fused top-1, a batched decode layer and the M=64 GEMM
meanwhile: every output must equal, bit for bit, the same call's output on
an idle GPU, q4nx_check must report no failed wait, and the spinner must
still be running when the calls are done (so they ran beside it).

The spinner is a test-only helper compiled here with nvcc; it is not part of
the library.
"""
import ctypes
import os
import subprocess
import tempfile
import time

import numpy as np
import pytest
import torch

import synth
from test_gpu_parity import DEV, to_dev_bf16, to_dev_bytes

pytestmark = pytest.mark.gpu

SPIN_SRC = r"""
#include <cuda_runtime.h>
extern "C" __global__ void hold_sm(unsigned long long ns, unsigned int* done) {
  extern __shared__ unsigned char pad[];
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  do {
    __nanosleep(2000);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < ns);
  if (threadIdx.x == 0) { pad[0] = 1; atomicAdd(done, 1u); }
}
extern "C" int launch_hold(void* stream, int blocks, int smem, unsigned long long ns, unsigned int* done) {
  cudaError_t e = cudaFuncSetAttribute(hold_sm, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return (int)e;
  hold_sm<<<blocks, 32, smem, (cudaStream_t)stream>>>(ns, done);
  return (int)cudaGetLastError();
}
"""


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import dequant_gemv_gb300

    return dequant_gemv_gb300


@pytest.fixture(scope="module")
def spinner():
    d = tempfile.mkdtemp(prefix="q4nx_hold_")
    src, lib = os.path.join(d, "hold.cu"), os.path.join(d, "libhold.so")
    with open(src, "w") as f:
        f.write(SPIN_SRC)
    nvcc = os.environ.get("NVCC", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    "-o", lib, src], check=True)
    L = ctypes.CDLL(lib)
    L.launch_hold.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_ulonglong, ctypes.c_void_p]
    L.launch_hold.restype = ctypes.c_int
    return L


def test_calls_complete_beside_a_kernel_holding_most_sms(q, spinner):
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    free_sms = 8
    # calls and their idle-GPU outputs
    f1, w1 = synth.make(synth.Q4_1, 12288, 4096, synth.rng(60, 1))
    W1 = q.Weight(to_dev_bytes(w1), synth.Q4_1, 12288, 4096)
    x1 = to_dev_bf16(synth.activations(synth.rng(60, 2), 1, 4096)[0])
    f2, w2 = synth.make(synth.Q8_KR, 32768, 2560, synth.rng(60, 3))
    W2 = q.Weight(to_dev_bytes(w2), synth.Q8_KR, 32768, 2560)
    x2 = to_dev_bf16(synth.activations(synth.rng(60, 4), 1, 2560)[0])
    X3 = to_dev_bf16(synth.activations(synth.rng(60, 5), 64, 4096))
    layer = []
    for mi, (_, N, K) in enumerate(synth.QWEN3_06B_LAYER):
        f, w = synth.workload_weight(2, mi, layer=7)
        layer.append((q.Weight(to_dev_bytes(w), synth.Q4_1, N, K),
                      to_dev_bf16(synth.workload_activations(2, mi, 1, K, layer=7)[0]),
                      torch.empty(N, dtype=torch.bfloat16, device=DEV)))

    def run():
        a = q.q4nx_gemv(W1, x1, out_dtype="f32").clone()
        b = q.q4nx_gemv_top1(W2, x2).clone()
        c = q.q4nx_gemm_m64(W1, X3, out_dtype="bf16").clone()
        ys = [y.clone() for y in q.q4nx_gemv_batch(layer)]
        return [a, b, c] + ys

    ref = run()
    torch.cuda.synchronize()
    q.q4nx_check(device=DEV)

    done = torch.zeros(1, dtype=torch.int32, device=DEV)
    hold_stream = torch.cuda.Stream(DEV)
    smem = int(props.shared_memory_per_block_optin) - 1024
    st = spinner.launch_hold(ctypes.c_void_p(hold_stream.cuda_stream), sms - free_sms, smem, 30_000_000,
                             ctypes.c_void_p(done.data_ptr()))
    assert st == 0, f"spinner launch failed: {st}"
    time.sleep(0.002)                                      # let it take its SMs
    got = run()
    torch.cuda.current_stream().synchronize()
    still_running = not hold_stream.query()
    hold_stream.synchronize()
    assert int(done.item()) == sms - free_sms
    assert still_running, "the calls did not run beside the spinner (it had finished first)"
    for i, (r, g) in enumerate(zip(ref, got)):
        bits = {torch.float32: torch.int32, torch.bfloat16: torch.int16, torch.int32: torch.int32}[r.dtype]
        assert torch.equal(r.view(bits), g.view(bits)), f"output {i} differs beside the spinner"
    q.q4nx_check(device=DEV)
