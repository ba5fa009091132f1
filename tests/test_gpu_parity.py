"""Parity of the CUDA path (through the C ABI) with the oracle, on a GB300.

Bars (the pass criteria of the path):
  * decode, repack, argmax: bit-exact (NaN compares equal to NaN);
  * GEMV / GEMM: |y - y64| <= 1e-3 * sum_k |w_k x_k| of the binary64 oracle
    (+ 2^-8 |y64| for bf16-typed outputs, the output's own rounding), and
    per-row cosine >= 0.99999;
  * lm_head: GPU top-1 of GPU logits equals the oracle's top-1 of the same
    logits, and equals the top-1 of the fp64 logits wherever the fp64 top-2
    gap exceeds twice the tolerance.
Inputs are the seeded synthetic workloads (synth/): small grids that span
several tiles and a ragged tail, and the full workload sizes with sampled
rows.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

REL = 1e-3
COS = 0.99999
BF16_OUT = 2.0 ** -8


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import dequant_gemv_gb300

    return dequant_gemv_gb300


DEV = "cuda:0"


def to_dev_bytes(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def out_values(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_bits_equal(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.uint16)
    ref = np.asarray(ref, np.uint16)
    nan_g = (got & 0x7F80) == 0x7F80
    nan_g &= (got & 0x7F) != 0
    nan_r = ((ref & 0x7F80) == 0x7F80) & ((ref & 0x7F) != 0)
    assert np.array_equal(nan_g, nan_r)
    diff = (got != ref) & ~nan_g
    assert not diff.any(), f"{int(diff.sum())} of {diff.size} values differ, first at {np.argwhere(diff)[0]}"


# Tensor-core products multiply bf16 weights (the decode to bf16 that feeds the
# MMA): rounding a weight to bf16 moves it by at most 2^-9 of itself, so those
# outputs may be off by up to 2^-9 * sum|w x| more (reading o21).
BF16_WEIGHTS = 2.0 ** -9


# Below 2^-126 binary32 and bf16 keep an absolute spacing (2^-149, 2^-133):
# a bf16 output adds half of the latter to the half-ulp of its rounding, and
# inputs whose products fall there add `f32_floor` = K * 2^-147, a few binary32
# subnormal roundings per column (reading o22).
BF16_OUT_SUBNORMAL = 2.0 ** -134


def f32_floor(K: int) -> float:
    return K * 2.0 ** -147


def assert_within(y: np.ndarray, Y64: np.ndarray, A: np.ndarray, bf16_out: bool, what="", bf16_weights=False,
                  floor: float = 0.0, cosine: bool = True):
    y = np.atleast_2d(y)
    Y64 = np.atleast_2d(Y64)
    A = np.atleast_2d(A)
    rel = REL + (BF16_WEIGHTS if bf16_weights else 0.0)
    tol = rel * A + floor
    if bf16_out:
        tol = tol + BF16_OUT * (np.abs(Y64) + tol) + BF16_OUT_SUBNORMAL
    err = np.abs(y - Y64)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs outside tolerance; worst err/tol "
                           f"{float(np.nanmax(err / np.maximum(tol, 1e-300))):.3g}")
    if not cosine:
        return
    for m in range(y.shape[0]):
        n1, n2 = np.linalg.norm(y[m]), np.linalg.norm(Y64[m])
        if n1 == 0 and n2 == 0:
            continue
        cos = float(np.dot(y[m], Y64[m]) / (n1 * n2))
        assert cos >= COS, f"{what}: row {m} cosine {cos}"


def weight(q, kind, N, K, seed=0, wid=9, **kw):
    f, w = synth.make(kind, N, K, synth.rng(wid, 0, seed + 10 * kind), **kw)
    return f, w, q.Weight(to_dev_bytes(w), kind, N, K)


SMALL = [(32, 256), (64, 512), (96, 768), (160, 1280), (1024, 1024), (32, 2816), (2080, 256)]
KINDS = [synth.Q4_1, synth.Q4_K, synth.Q8_KR, synth.Q8_BLK]


# ------------------------------------------------------------------ decode --

@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("N,K", SMALL[:5])
def test_decode_bit_exact_small(q, kind, N, K):
    f, w, W = weight(q, kind, N, K)
    assert_bits_equal(bf16_np(q.q4nx_decode(W)), oracle.decode(w, kind, N, K))


@pytest.mark.parametrize("kind,N,K,wid", [(synth.Q4_1, 1024, 1024, 1), (synth.Q4_K, 9728, 2560, 3),
                                          (synth.Q8_KR, 151936, 2560, 5), (synth.Q8_BLK, 151936, 2560, 5)])
def test_decode_bit_exact_full_size_sampled(q, kind, N, K, wid):
    f, w = synth.make(kind, N, K, synth.rng(wid, 0, 0))
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    dec = q.q4nx_decode(W)
    TR, TC = N // 32, K // 256
    cb = synth.CHUNK_BYTES[kind]
    g = np.random.default_rng(0)
    trs = sorted(set([0, TR - 1] + list(g.integers(0, TR, size=min(TR, 24)))))
    for tr in trs:
        sub = w[tr * TC * cb:(tr + 1) * TC * cb]
        ref = oracle.decode(sub, kind, 32, K)
        assert_bits_equal(bf16_np(dec[tr * 32:(tr + 1) * 32]), ref)


def test_decode_edge_values(q):
    """Tiny and large scales (subnormal products, big magnitudes), zero and
    negative zeros: still bit-exact."""
    N, K = 64, 512
    f = synth.q4_1_fields(synth.rng(77), N, K)
    g = np.random.default_rng(5)
    vals = np.array([1e-38, 3e-39, 1e-30, 2.0 ** -126, 1e30, 3e38, 0.0, -0.0, 1.0, -1.5], np.float32)
    f.scale[:] = synth.bf16_bits(g.choice(vals, size=f.scale.shape))
    f.zero[:] = synth.bf16_bits(g.choice(vals, size=f.zero.shape) * np.float32(-1))
    w = synth.pack(f)
    W = q.Weight(to_dev_bytes(w), synth.Q4_1, N, K)
    assert_bits_equal(bf16_np(q.q4nx_decode(W)), oracle.decode(w, synth.Q4_1, N, K))


# -------------------------------------------------------------------- GEMV --

@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("N,K", SMALL)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_gemv_small(q, kind, N, K, out):
    f, w, W = weight(q, kind, N, K)
    x = synth.activations(synth.rng(9, 1, kind), 1, K)[0]
    y = out_values(q.q4nx_gemv(W, to_dev_bf16(x), out_dtype=out))
    Y64, A = oracle.matmul(w, kind, N, K, x)
    assert_within(y, Y64, A, out == "bf16", f"kind {kind} {N}x{K}")


@pytest.mark.parametrize("kind,N,K,wid,out", [
    (synth.Q4_1, 1024, 1024, 1, "bf16"),
    (synth.Q4_1, 2048, 1024, 2, "bf16"), (synth.Q4_1, 1024, 2048, 2, "bf16"),
    (synth.Q4_1, 3072, 1024, 2, "bf16"), (synth.Q4_1, 1024, 3072, 2, "bf16"),
    (synth.Q4_K, 9728, 2560, 3, "bf16"), (synth.Q4_K, 2560, 9728, 3, "bf16"),
    (synth.Q4_1, 12288, 4096, 4, "bf16"), (synth.Q4_1, 4096, 12288, 4, "bf16"),
    (synth.Q8_KR, 151936, 2560, 5, "f32"), (synth.Q8_BLK, 151936, 2560, 5, "f32"),
    (synth.Q4_1, 151936, 2560, 6, "f32"),
])
def test_gemv_workload_sizes(q, kind, N, K, wid, out):
    f, w = synth.make(kind, N, K, synth.rng(wid, 0, 0))
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    x = synth.workload_activations(wid, 0, 1, K)[0]
    y = out_values(q.q4nx_gemv(W, to_dev_bf16(x), out_dtype=out))
    rows = None if N * K <= 40_000_000 else np.unique(np.concatenate([
        np.arange(64), np.arange(N - 64, N), np.random.default_rng(1).integers(0, N, 2048)]))
    Y64, A = oracle.matmul(w, kind, N, K, x, rows=rows)
    assert_within(y if rows is None else y[rows], Y64, A, out == "bf16", f"kind {kind} {N}x{K}")


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K])
def test_gemv_two_ctas_per_sm_threshold(q, kind):
    """A 4-bit weight of at least 128 chunks per SM runs two CTAs per SM, a smaller
    one a single CTA per SM: shapes on both sides of that point, one of them with
    tile rows of 152 chunks spread over several CTAs, match the oracle on sampled
    rows, and a repeated call gives the same bytes."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shapes = [(4 * sms, 32), (4 * sms - 1, 32), (-(-128 * sms // 152), 152)]   # (tile rows, tile columns)
    for i, (TR, TC) in enumerate(shapes):
        N, K = 32 * TR, 256 * TC
        f, w = synth.make(kind, N, K, synth.rng(12, kind, i))
        W = q.Weight(to_dev_bytes(w), kind, N, K)
        x = synth.activations(synth.rng(12, 1, i), 1, K)[0]
        xd = to_dev_bf16(x)
        yd = q.q4nx_gemv(W, xd, out_dtype="f32").clone()
        again = q.q4nx_gemv(W, xd, out_dtype="f32")
        assert torch.equal(yd.view(torch.int32), again.view(torch.int32)), f"{N}x{K} not repeatable"
        rows = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N), np.arange(0, N, 7)]))
        Y64, A = oracle.matmul(w, kind, N, K, x, rows=rows)
        assert_within(out_values(yd)[rows], Y64, A, False, f"kind {kind} {N}x{K}")
    q.q4nx_check(device=DEV)


def test_gemv_wide_k(q):
    """Any number of columns (x is streamed with each chunk, not staged whole)."""
    for kind in (synth.Q4_1, synth.Q8_BLK):
        N, K = 64, 65536
        f, w, W = weight(q, kind, N, K)
        x = synth.activations(synth.rng(9, 2, kind), 1, K)[0]
        y = out_values(q.q4nx_gemv(W, to_dev_bf16(x), out_dtype="f32"))
        Y64, A = oracle.matmul(w, kind, N, K, x)
        assert_within(y, Y64, A, False, f"kind {kind} wide")


@pytest.mark.parametrize("kind", KINDS)
def test_gemv_batch_mixed_shapes(q, kind):
    """One launch over many weights of one kind: each output matches the oracle."""
    shapes = [(2048, 1024), (1024, 1024), (1024, 1024), (1024, 2048), (3072, 1024), (3072, 1024), (1024, 3072),
              (32, 256), (96, 768)]
    items, refs = [], []
    for i, (N, K) in enumerate(shapes):
        f, w = synth.make(kind, N, K, synth.rng(2, 0, i))
        x = synth.workload_activations(2, i, 1, K)[0]
        W = q.Weight(to_dev_bytes(w), kind, N, K)
        y = torch.empty(N, dtype=torch.float32, device=DEV)
        items.append((W, to_dev_bf16(x), y))
        refs.append((w, x, N, K))
    q.q4nx_gemv_batch(items, out_dtype="f32")
    for (W, xt, y), (w, x, N, K) in zip(items, refs):
        rows = np.arange(0, N, 3)
        Y64, A = oracle.matmul(w, kind, N, K, x, rows=rows)
        assert_within(out_values(y)[rows], Y64, A, False, f"batch kind {kind} {N}x{K}")
    q.q4nx_check(device=DEV)


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_gemv_batch_small_launches(q, kind, out):
    """Batches small enough (at most 8 chunks per SM) that the launch takes
    quarters of chunks as units: the {q, k, v} and {gate, up} phases of a
    Qwen3-0.6B-shaped layer, and a mix of tiny weights whose quarters fall
    across item boundaries at every offset; every row matches the oracle."""
    batches = [[(2048, 1024), (1024, 1024), (1024, 1024)],
               [(3072, 1024), (3072, 1024)],
               [(32, 256), (96, 768), (64, 512), (160, 1280), (32, 2304), (256, 256)]]
    for bi, shapes in enumerate(batches):
        items, refs = [], []
        for i, (N, K) in enumerate(shapes):
            f, w = synth.make(kind, N, K, synth.rng(33, bi, i))
            x = synth.activations(synth.rng(34, bi, i), 1, K)[0]
            y = torch.empty(N, dtype=torch.float32 if out == "f32" else torch.bfloat16, device=DEV)
            items.append((q.Weight(to_dev_bytes(w), kind, N, K), to_dev_bf16(x), y))
            refs.append((w, x, N, K))
        q.q4nx_gemv_batch(items, out_dtype=out)
        for (W, xt, y), (w, x, N, K) in zip(items, refs):
            Y64, A = oracle.matmul(w, kind, N, K, x)
            assert_within(out_values(y), Y64, A, out == "bf16", f"small batch {bi} kind {kind} {N}x{K}")
    q.q4nx_check(device=DEV)


def test_gemv_batch_qwen3_layer_bf16(q):
    """A Qwen3-0.6B-shaped layer (7 projections) in one launch, bf16 outputs."""
    items, refs = [], []
    for mi, (_, N, K) in enumerate(synth.QWEN3_06B_LAYER):
        f, w = synth.workload_weight(2, mi, layer=3)
        x = synth.workload_activations(2, mi, 1, K, layer=3)[0]
        y = torch.empty(N, dtype=torch.bfloat16, device=DEV)
        items.append((q.Weight(to_dev_bytes(w), synth.Q4_1, N, K), to_dev_bf16(x), y))
        refs.append((w, x, N, K))
    q.q4nx_gemv_batch(items)
    for (W, xt, y), (w, x, N, K) in zip(items, refs):
        Y64, A = oracle.matmul(w, synth.Q4_1, N, K, x)
        assert_within(out_values(y), Y64, A, True, f"layer {N}x{K}")


def test_gemv_repeat_runs_are_byte_identical(q):
    f, w, W = weight(q, synth.Q4_1, 4096, 12288)
    x = to_dev_bf16(synth.activations(synth.rng(3), 1, 12288)[0])
    a = q.q4nx_gemv(W, x, out_dtype="f32").clone()
    b = q.q4nx_gemv(W, x, out_dtype="f32").clone()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_gemv_degenerate_inputs(q):
    N, K = 96, 768
    f, w, W = weight(q, synth.Q4_1, N, K)
    zero_x = torch.zeros(K, dtype=torch.bfloat16, device=DEV)
    assert (q.q4nx_gemv(W, zero_x, out_dtype="f32") == 0).all()
    # zero scale and zero: every weight is 0
    f.scale[:] = 0
    f.zero[:] = 0
    W0 = q.Weight(to_dev_bytes(synth.pack(f)), synth.Q4_1, N, K)
    x = to_dev_bf16(synth.activations(synth.rng(4), 1, K)[0])
    assert (q.q4nx_gemv(W0, x, out_dtype="f32") == 0).all()
    # basis vectors pick columns
    Wd = oracle.weights_f64(w, synth.Q4_1, N, K)
    for k in (0, 1, 255, 256, 767):
        e = np.zeros(K, np.uint16)
        e[k] = synth.bf16_bits(np.array([1.0], np.float32))[0]
        y = out_values(q.q4nx_gemv(W, to_dev_bf16(e), out_dtype="f32"))
        assert np.all(np.abs(y - Wd[:, k]) <= 1e-6 * np.abs(Wd[:, k]) + 1e-30)


def test_gemv_large_magnitudes(q):
    """Activations far beyond fp16 range accumulate in fp32 without overflow."""
    N, K = 64, 1024
    f, w, W = weight(q, synth.Q8_KR, N, K)
    x = synth.bf16_bits(np.random.default_rng(2).normal(0, 3e4, K).astype(np.float32))
    y = out_values(q.q4nx_gemv(W, to_dev_bf16(x), out_dtype="f32"))
    Y64, A = oracle.matmul(w, synth.Q8_KR, N, K, x)
    assert_within(y, Y64, A, False, "large x")


def test_gemv_tile_row_shards_match_whole(q):
    """Contiguous tile-row ranges are weights of their own: the shards'
    outputs, gathered, equal the whole weight's (bit for bit)."""
    N, K = 1024, 2048
    f, w, W = weight(q, synth.Q4_1, N, K)
    x = to_dev_bf16(synth.activations(synth.rng(6), 1, K)[0])
    whole = q.q4nx_gemv(W, x, out_dtype="f32")
    parts = [q.q4nx_gemv(W.tile_rows(tr0, cnt), x, out_dtype="f32") for tr0, cnt in ((0, 11), (11, 16), (27, 5))]
    assert torch.equal(torch.cat(parts), whole)


def test_gemv_status_errors_on_gpu(q):
    f, w, W = weight(q, synth.Q4_1, 64, 512)
    x = to_dev_bf16(synth.activations(synth.rng(7), 1, 512)[0])
    short = q.Weight(W.chunks[:5120 * 3], synth.Q4_1, 64, 512)
    with pytest.raises(q.Q4NXError) as e:
        q.q4nx_gemv(short, x)
    assert e.value.status == 4
    odd = q.Weight(W.chunks[8:8 + 5120 * 4], synth.Q4_1, 32, 512)
    with pytest.raises(q.Q4NXError) as e:
        q.q4nx_gemv(odd, x)
    assert e.value.status == 5
    q.q4nx_check(device=DEV)


# ------------------------------------------------------------------ repack --

@pytest.mark.parametrize("N,K", [(32, 256), (64, 512), (96, 768), (9728, 2560), (2560, 9728)])
def test_repack_bit_exact(q, N, K):
    f, w = synth.make(synth.Q4_K, N, K, synth.rng(3, 0, 1))
    rep = q.q4nx_repack_q4k(to_dev_bytes(w), N, K).cpu().numpy()
    ref = oracle.repack_q4k(w, N, K)
    assert np.array_equal(rep, ref)


def test_repacked_weights_run_on_q4_1_gemv(q):
    """Code that reads q4_1 runs Q4_K weights unchanged after the repack."""
    N, K = 9728, 2560
    f, w = synth.make(synth.Q4_K, N, K, synth.rng(3, 0, 0))
    rep = q.q4nx_repack_q4k(to_dev_bytes(w), N, K)
    x = synth.workload_activations(3, 0, 1, K)[0]
    y = out_values(q.q4nx_gemv(q.Weight(rep, synth.Q4_1, N, K), to_dev_bf16(x), out_dtype="f32"))
    rows = np.arange(0, N, 7)
    Y64, A = oracle.matmul(rep.cpu().numpy(), synth.Q4_1, N, K, x, rows=rows)
    assert_within(y[rows], Y64, A, False, "repacked")


# ------------------------------------------------------------------ argmax --

@pytest.mark.parametrize("M,V", [(1, 1), (1, 7), (3, 1000), (1, 151936), (64, 151936), (5, 151937), (2, 33),
                                 (19, 151936), (20, 151936), (1, 1 << 20), (2, 1000003)])
def test_argmax_bit_exact(q, M, V):
    g = np.random.default_rng(M * 7 + V)
    L = g.normal(size=(M, V)).astype(np.float32)
    if V > 10:
        L[0, [3, V // 2, V - 1]] = 9.0                  # ties -> lowest index
        if M > 1:
            L[1, [V - 2, 5]] = np.nan                   # first NaN wins
        if M > 2:
            L[2, :] = -np.inf
    got = q.q4nx_argmax(torch.from_numpy(L).to(DEV)).cpu().numpy()
    assert np.array_equal(got, oracle.argmax(L))
    assert np.array_equal(got, np.argmax(L, axis=1))


def test_argmax_signed_zeros_and_infs(q):
    L = np.full((4, 300), -0.0, np.float32)
    L[0, 10] = 0.0                                      # +0 == -0: index 0 wins
    L[1, 299] = np.inf
    L[1, 298] = np.inf
    L[2, :] = -np.inf
    L[3, 100] = np.nan
    L[3, 5] = np.inf
    got = q.q4nx_argmax(torch.from_numpy(L).to(DEV)).cpu().numpy()
    assert got.tolist() == [0, 298, 0, 100]
    assert np.array_equal(got, oracle.argmax(L))


def _ambiguous_and_check(idx_gpu, logits, w, kind, N, K, X, bar_rel, what):
    """Reading o24: per row, the top-1 of the GPU logits must equal the top-1 of
    the binary64 oracle logits wherever the oracle's top-2 gap exceeds twice the
    bar.  Rows below that gap are ambiguous (several answers are within the
    bar): there the GPU's choice must be a row whose oracle logit lies within
    twice the bar of the oracle's maximum, and it must still equal the oracle's
    top-1 wherever the gap exceeds twice the GPU's own largest observed error on
    the row's candidates (|y - y64| <= e everywhere and a gap > 2e fix the
    answer).  The candidates are the row's 64 largest GPU logits.  Returns the
    number of ambiguous rows."""
    ambiguous = 0
    for m in range(logits.shape[0]):
        cand = np.argsort(-logits[m])[:64]
        Y64, A = oracle.matmul(w, kind, N, K, X[m], rows=cand)
        order = np.argsort(-Y64)
        best, second = order[0], order[1]
        gap = Y64[best] - Y64[second]
        bar = bar_rel * max(A[best], A[second])
        if gap > 2 * bar:
            assert idx_gpu[m] == cand[best], f"{what}: row {m} top-1 {idx_gpu[m]} != oracle {cand[best]}"
            continue
        ambiguous += 1
        chosen = np.nonzero(cand == idx_gpu[m])[0]
        assert chosen.size == 1, f"{what}: row {m} top-1 {idx_gpu[m]} not among the 64 largest logits"
        assert Y64[best] - Y64[chosen[0]] <= 2 * bar, f"{what}: row {m} chose a row outside the bar"
        e_obs = float(np.max(np.abs(logits[m][cand].astype(np.float64) - Y64)))
        if gap > 2 * e_obs:
            assert idx_gpu[m] == cand[best], f"{what}: row {m}: gap {gap} > 2 x observed error {e_obs}"
    return ambiguous


@pytest.mark.parametrize("kind", [synth.Q8_KR, synth.Q8_BLK])
def test_lm_head_top1(q, kind):
    """lm_head logits then argmax, one token (GEMV) and 64 tokens (tensor-core
    GEMM): q4nx_argmax equals the oracle's scan of the same GPU logits bit for
    bit, and the end-to-end top-1 equals the binary64 oracle's on every
    unambiguous row (see _ambiguous_and_check).  At these seeds the rows'
    top-2 gaps are often inside twice the bar (the one-token row: 0.63 against
    1.13), so the ambiguous count is printed, not assumed to be 0."""
    N, K = 151936, 2560
    f, w = synth.make(kind, N, K, synth.rng(5, 0, 0))
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    x = synth.workload_activations(5, 0, 1, K)[0]
    logits = q.q4nx_gemv(W, to_dev_bf16(x), out_dtype="f32")
    idx = q.q4nx_argmax(logits.view(1, N)).cpu().numpy()
    lg = logits.cpu().numpy().reshape(1, N)
    assert np.array_equal(idx, oracle.argmax(lg))
    amb1 = _ambiguous_and_check(idx, lg, w, kind, N, K, x.reshape(1, K), REL, f"kind {kind} M=1")
    X = synth.workload_activations(5, 0, 64, K)
    L64 = q.q4nx_gemm_m64(W, to_dev_bf16(X), out_dtype="f32")
    idx64 = q.q4nx_argmax(L64).cpu().numpy()
    lg64 = L64.cpu().numpy()
    assert np.array_equal(idx64, oracle.argmax(lg64))
    # the tensor-core logits multiply bf16 weights: reading o21's bar
    amb64 = _ambiguous_and_check(idx64, lg64, w, kind, N, K, X, REL + BF16_WEIGHTS, f"kind {kind} M=64")
    print(f"lm_head top-1 kind {kind}: ambiguous rows {amb1} of 1 (GEMV), {amb64} of 64 (GEMM)")
