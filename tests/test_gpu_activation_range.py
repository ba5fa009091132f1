"""The 4-bit GEMV (and the few-token and tensor-core paths) against the oracle
on activations whose magnitudes spread far apart inside a 32-column group.

The weight formulas are those of the chunk-kind table ("NPU engine" page,
section "Q4NX chunks"); the Q4_0 mapping scale d, zero -8d comes from its
section "From a GGUF".  With that mapping, code 8 is an exact zero weight,
so an activation on such a weight adds nothing to sum_k |w_k x_k| while a
computation that multiplies scale and zero separately sees it at full size.

Cases:
  * the worked case: one activation of 1.0 per group on a zero weight, the
    other 31 at 2^-20 on weights of 7 scale units;
  * LLM-style outlier channels (a fixed few columns at 10^2 - 10^3 times
    N(0, 1)) at the decode-layer and 8B-width shapes;
  * log-uniform magnitudes over 2^+-30 with exact zeros of both signs;
  * bf16 subnormals mixed with +0 and -0 (outputs below 2^-126: the bar adds
    the binary32 / bf16 spacing there, and no cosine is taken);
  * groups whose magnitudes span exactly 2^14 and just beyond;
  * every weight an exact zero: the output is exactly zero;
  * scales near 2^+-100;
  * several tokens whose x slices, prepared once per CTA for all of them,
    need different numbers of digit planes (the few-token x-slice cache),
    also beside a token holding +Inf or NaN and an all-zero token;
  * one +Inf, -Inf or NaN activation (GEMV of every kind, the batched layer
    on the x-slice cache path, the tensor-core GEMM): each row meets the
    special value exactly as the binary64 sum does (0 * Inf = NaN).
Every finite output is checked against the binary64 oracle at
1e-3 * sum_k |w_k x_k|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from test_gpu_parity import DEV, assert_within, f32_floor, out_values, to_dev_bf16, to_dev_bytes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import dequant_gemv_gb300

    return dequant_gemv_gb300


BF16_ONE = 0x3F80


def bf16_of(v: float) -> int:
    return int(synth.bf16_bits(np.array([v], np.float32))[0])


def q4_0_mapped_weight(kind: int, N: int, K: int, seed: int = 0):
    """Weight whose every group has scale 2^-7 and zero -8 * 2^-7 (the Q4_0
    mapping), code 8 in the group's first column (w = 0) and 15 in the other
    31 (w = 7 * 2^-7).  Q4_K: S = 2^-7, sc = 1, M = -2^-7, mn = 8."""
    f, _ = synth.make(kind, N, K, synth.rng(40, kind, seed))
    codes = np.full_like(f.codes, 15)
    codes[:, :, 0::32] = 8
    f.codes[:] = codes
    if kind == synth.Q4_1:
        f.scale[:] = bf16_of(2.0 ** -7)
        f.zero[:] = bf16_of(-8 * 2.0 ** -7)
    else:
        f.S[:] = bf16_of(2.0 ** -7)
        f.M[:] = bf16_of(-(2.0 ** -7))
        f.sc[:] = 1
        f.mn[:] = 8
    return f, synth.pack(f)


def worked_x(K: int, big: float = 1.0, small_exp: int = -20) -> np.ndarray:
    x = np.full(K, 2.0 ** small_exp, np.float32)
    x[0::32] = big
    return synth.bf16_bits(x)


def check_gemv(q, kind, w, N, K, x, out, what, rows=None, floor=0.0, cosine=True):
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    y = out_values(q.q4nx_gemv(W, to_dev_bf16(x), out_dtype=out))
    Y64, A = oracle.matmul(w, kind, N, K, x, rows=rows)
    assert_within(y if rows is None else y[rows], Y64, A, out == "bf16", what, floor=floor, cosine=cosine)
    return y, Y64


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K])
@pytest.mark.parametrize("N,K", [(32, 256), (1024, 1024), (2560, 9728)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_worked_case_zero_weight_outlier(q, kind, N, K, out):
    f, w = q4_0_mapped_weight(kind, N, K)
    x = worked_x(K)
    y, Y64 = check_gemv(q, kind, w, N, K, x, out, f"worked case kind {kind} {N}x{K}")
    # the exact value: per group 31 * 7 * 2^-7 * 2^-20
    assert np.allclose(Y64, (K // 32) * 31 * 7 * 2.0 ** -27, rtol=0, atol=0)


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K])
@pytest.mark.parametrize("small_exp", [-8, -14, -15, -16, -40, -100])
def test_worked_case_spreads(q, kind, small_exp):
    """The outlier at 1 and the rest at 2^small_exp: at 2^-14 the group still
    fits the 24-bit fixed point, from 2^-15 on it does not."""
    N, K = 64, 2048
    f, w = q4_0_mapped_weight(kind, N, K, seed=1)
    check_gemv(q, kind, w, N, K, worked_x(K, small_exp=small_exp), "f32", f"spread 2^{small_exp}")


@pytest.mark.parametrize("kind,N,K", [(synth.Q4_1, 12288, 4096), (synth.Q4_1, 4096, 12288),
                                      (synth.Q4_K, 9728, 2560), (synth.Q4_K, 2560, 9728),
                                      (synth.Q4_1, 1024, 3072), (synth.Q4_1, 151936, 2560)])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_outlier_channels_workload_shapes(q, kind, N, K, out):
    f, w = synth.make(kind, N, K, synth.rng(41, kind, N + K))
    x = synth.activations_outliers(synth.rng(41, 1, K), 1, K)[0]
    rows = None if N * K <= 8_000_000 else np.unique(np.concatenate([
        np.arange(64), np.arange(N - 64, N), np.random.default_rng(2).integers(0, N, 1024)]))
    check_gemv(q, kind, w, N, K, x, out, f"outliers kind {kind} {N}x{K}", rows=rows)


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K])
def test_outlier_channels_on_q4_0_mapped_weights(q, kind):
    """Q4_0-mapped weights (zero exactly -8 scale, so code 8 is an exact zero)
    under 10^3 outlier channels."""
    N, K = 2048, 4096
    f, _ = synth.make(kind, N, K, synth.rng(42, kind))
    if kind == synth.Q4_1:
        f.zero[:] = synth.bf16_bits(np.float32(-8.0) * synth.bf16_values(f.scale))
    else:
        f.M[:] = synth.bf16_bits(-synth.bf16_values(f.S))
        f.mn[:] = 8
        f.sc[:] = 1
    w = synth.pack(f)
    x = synth.activations_outliers(synth.rng(42, 1), 1, K, frac=0.01, lo=500.0, hi=1000.0)[0]
    check_gemv(q, kind, w, N, K, x, "f32", f"Q4_0-mapped outliers kind {kind}")


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_log_uniform_magnitudes(q, kind, out):
    N, K = 2080, 2816
    f, w = synth.make(kind, N, K, synth.rng(43, kind))
    x = synth.activations_log_uniform(synth.rng(43, 1), 1, K)[0]
    check_gemv(q, kind, w, N, K, x, out, f"log-uniform kind {kind}")


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K, synth.Q8_KR])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_subnormals_mixed_with_signed_zeros(q, kind, out):
    N, K = 96, 768
    f, w = synth.make(kind, N, K, synth.rng(44, kind))
    x = synth.activations_subnormal(synth.rng(44, 1), 1, K)[0]
    check_gemv(q, kind, w, N, K, x, out, f"subnormal x kind {kind}", floor=f32_floor(K), cosine=False)
    # groups mixing subnormals, zeros and normal values (those fall outside the fixed point)
    x2 = x.copy()
    x2[5::64] = synth.bf16_bits(np.full(len(x2[5::64]), 3.0, np.float32))
    check_gemv(q, kind, w, N, K, x2, out, f"subnormal + normal x kind {kind}", floor=f32_floor(K))


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K])
def test_all_zero_weights_give_exact_zero(q, kind):
    """Code 8 everywhere under the Q4_0 mapping: every weight is exactly 0, so
    every output must be exactly 0 whatever x is (on both arithmetic paths)."""
    N, K = 256, 2048
    f, _ = q4_0_mapped_weight(kind, N, K)
    f.codes[:] = 8
    w = synth.pack(f)
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    for x in (synth.activations(synth.rng(45), 1, K)[0], synth.activations_outliers(synth.rng(45, 1), 1, K)[0],
              synth.activations_log_uniform(synth.rng(45, 2), 1, K)[0]):
        y = q.q4nx_gemv(W, to_dev_bf16(x), out_dtype="f32")
        assert torch.count_nonzero(y).item() == 0


def test_large_and_small_scales(q):
    """Scales and zeros near 2^+-100 with moderate x."""
    N, K = 128, 1024
    for e in (100, -100):
        f, _ = synth.make(synth.Q4_1, N, K, synth.rng(46, e + 200))
        s = synth.bf16_values(f.scale) * np.float32(2.0 ** e)
        f.scale[:] = synth.bf16_bits(s)
        f.zero[:] = synth.bf16_bits(np.float32(-7.5) * s)
        w = synth.pack(f)
        for x in (synth.activations(synth.rng(46, 1), 1, K)[0], synth.activations_outliers(synth.rng(46, 2), 1, K)[0]):
            check_gemv(q, synth.Q4_1, w, N, K, x, "f32", f"scales 2^{e}")


def test_decode_layer_batch_with_outliers(q):
    """The seven projections of a Qwen3-0.6B-shaped layer in one launch, each
    activation vector with outlier channels."""
    items, refs = [], []
    for mi, (_, N, K) in enumerate(synth.QWEN3_06B_LAYER):
        f, w = synth.workload_weight(2, mi, layer=5)
        x = synth.activations_outliers(synth.rng(47, mi), 1, K)[0]
        y = torch.empty(N, dtype=torch.bfloat16, device=DEV)
        items.append((q.Weight(to_dev_bytes(w), synth.Q4_1, N, K), to_dev_bf16(x), y))
        refs.append((w, x, N, K))
    q.q4nx_gemv_batch(items)
    for (W, xt, y), (w, x, N, K) in zip(items, refs):
        Y64, A = oracle.matmul(w, synth.Q4_1, N, K, x)
        assert_within(out_values(y), Y64, A, True, f"layer {N}x{K} with outliers")


# ------------------------------------------------------- several tokens --

def token_block(K: int, M: int) -> np.ndarray:
    """M rows: the worked case, outlier channels, log-uniform, N(0, 1)."""
    rows = [worked_x(K), synth.activations_outliers(synth.rng(48, 1), 1, K)[0],
            synth.activations_log_uniform(synth.rng(48, 2), 1, K)[0], synth.activations(synth.rng(48, 3), 1, K)[0]]
    return np.stack(rows[:M])


@pytest.mark.parametrize("kind,M", [(synth.Q4_1, 2), (synth.Q4_K, 2), (synth.Q4_K, 3), (synth.Q4_K, 4)])
@pytest.mark.parametrize("N,K", [(1024, 1024), (2560, 9728)])
def test_few_tokens_dynamic_range(q, kind, M, N, K):
    """q4nx_gemm_m64's CUDA-core path (each chunk read once for all tokens)."""
    f, w = q4_0_mapped_weight(kind, N, K)
    X = token_block(K, M)
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    got = out_values(q.q4nx_gemm_m64(W, to_dev_bf16(X), out_dtype="f32"))
    Y64, A = oracle.matmul(w, kind, N, K, X)
    assert_within(got, Y64, A, False, f"tokens kind {kind} M={M} {N}x{K}")
    f2, w2 = synth.make(kind, N, K, synth.rng(49, kind))
    W2 = q.Weight(to_dev_bytes(w2), kind, N, K)
    got = out_values(q.q4nx_gemm_m64(W2, to_dev_bf16(X), out_dtype="bf16"))
    Y64, A = oracle.matmul(w2, kind, N, K, X)
    assert_within(got, Y64, A, True, f"tokens kind {kind} M={M} {N}x{K} (random weights)")


@pytest.mark.parametrize("kind,M", [(synth.Q4_1, 2), (synth.Q4_K, 2), (synth.Q4_K, 3), (synth.Q4_K, 4)])
@pytest.mark.parametrize("N,K", [(16384, 1024), (12288, 4096), (10240, 1024)])
@pytest.mark.parametrize("order", ["as_built", "reversed"])
def test_few_tokens_cached_x_slices(q, kind, M, N, K, order):
    """Shapes whose CTAs read each touched x slice more than twice (16384 x
    1024: about 13 chunks per CTA over 4 slices; 12288 x 4096: about 40 over
    16), so that the few-token kernel prepares every slice once for all
    tokens, in the largest number of digit planes any token's group needs
    (Q4_K at 3-4 tokens on 12288 x 4096 excepted: 16 slices of 4 tokens do
    not fit beside its ring, and it prepares x per chunk).  10240 x 1024
    mixes both in one launch: CTAs of 9 chunks over 4 slices use the cache,
    those of 8 prepare x per chunk.  The tokens mix
    N(0, 1), outlier channels, the worked case and log-uniform magnitudes
    (which need the binary32 path), in either order."""
    f, w = q4_0_mapped_weight(kind, N, K, seed=M)
    X = token_block(K, 4)
    X = np.stack([X[3], X[1], X[0], X[2]])[:M]         # N(0, 1) first: its slices share a wider token's mode
    if order == "reversed":
        X = X[::-1].copy()
    rows = None if N * K <= 20_000_000 else np.unique(np.concatenate([
        np.arange(0, 128), np.arange(N - 128, N), np.random.default_rng(M).integers(0, N, 384)]))
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    for out in ("f32", "bf16"):
        got = out_values(q.q4nx_gemm_m64(W, to_dev_bf16(X), out_dtype=out))
        Y64, A = oracle.matmul(w, kind, N, K, X, rows=rows)
        assert_within(got if rows is None else got[:, rows], Y64, A, out == "bf16",
                      f"cached tokens kind {kind} M={M} {N}x{K} {order} {out}")
    f2, w2 = synth.make(kind, N, K, synth.rng(53, kind, M))
    W2 = q.Weight(to_dev_bytes(w2), kind, N, K)
    got = out_values(q.q4nx_gemm_m64(W2, to_dev_bf16(X), out_dtype="f32"))
    Y64, A = oracle.matmul(w2, kind, N, K, X, rows=rows)
    assert_within(got if rows is None else got[:, rows], Y64, A, False,
                  f"cached tokens kind {kind} M={M} {N}x{K} {order} (random weights)")


@pytest.mark.parametrize("N,K", [(12288, 4096), (4096, 12288)])
def test_gemm_64_tokens_with_outliers(q, N, K):
    """The tensor-core path at the prefill block's shapes with outlier channels
    in every token.  It multiplies bf16-rounded weights (each within 2^-9 of
    itself); under outliers a few columns carry much of sum_k |w_k x_k|, so
    their rounding no longer averages out over the long sum, and the bar is
    reading o21's (1e-3 + 2^-9) * sum_k |w_k x_k| at every width."""
    f, w = synth.make(synth.Q4_1, N, K, synth.rng(50, N))
    X = synth.activations_outliers(synth.rng(50, 1), 64, K)
    W = q.Weight(to_dev_bytes(w), synth.Q4_1, N, K)
    got = out_values(q.q4nx_gemm_m64(W, to_dev_bf16(X), out_dtype="bf16"))
    rows = np.unique(np.concatenate([np.arange(128), np.arange(N - 128, N),
                                     np.random.default_rng(3).integers(0, N, 256)]))
    Y64, A = oracle.matmul(w, synth.Q4_1, N, K, X, rows=rows)
    assert_within(got[:, rows], Y64, A, True, f"gemm 64 tokens outliers {N}x{K}", bf16_weights=True)


# ---------------------------------------------- x-slice cache coverage --

@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K])
@pytest.mark.parametrize("N,K", [(1024, 7168), (160, 1280), (4096, 7680), (96, 8192)])
def test_cached_x_slices_partial_rows(q, kind, N, K):
    """Shapes whose CTAs hold fewer chunks than a tile row (the touched tile
    columns start mid-row and wrap) or exactly the cache's capacity, with
    activations that make some x slices exact in 24-bit fixed point and
    others not (outliers next to N(0, 1) columns, and one log-uniform slice)."""
    f, w = synth.make(kind, N, K, synth.rng(51, kind, N))
    x = synth.activations_outliers(synth.rng(51, 1, K), 1, K, frac=0.002)[0]
    x[256:512] = synth.activations_log_uniform(synth.rng(51, 2), 1, 256)[0]
    for out in ("f32", "bf16"):
        check_gemv(q, kind, w, N, K, x, out, f"cache kind {kind} {N}x{K}")


def test_cached_x_slices_many_items_per_cta(q):
    """A batch of 40 small q4_1 matrices of mixed widths: some CTAs touch more
    items than the cache's item table holds and prepare x per chunk, others
    use the cache; every output matches the oracle."""
    items, refs = [], []
    g = np.random.default_rng(7)
    for i in range(40):
        N, K = 32 * int(g.integers(1, 4)), 256 * int(g.integers(1, 6))
        f, w = synth.make(synth.Q4_1, N, K, synth.rng(52, 0, i))
        x = (synth.activations_outliers if i % 3 == 0 else synth.activations)(synth.rng(52, 1, i), 1, K)[0]
        y = torch.empty(N, dtype=torch.float32, device=DEV)
        items.append((q.Weight(to_dev_bytes(w), synth.Q4_1, N, K), to_dev_bf16(x), y))
        refs.append((w, x, N, K))
    q.q4nx_gemv_batch(items, out_dtype="f32")
    for (W, xt, y), (w, x, N, K) in zip(items, refs):
        Y64, A = oracle.matmul(w, synth.Q4_1, N, K, x)
        assert_within(out_values(y), Y64, A, False, f"batch item {N}x{K}")


# ------------------------------------------------- Inf and NaN activations --

def special_x(K: int, which: str, col: int, seed: int) -> np.ndarray:
    """N(0, 1) activations with one +Inf, -Inf or NaN at column `col`."""
    x = synth.activations(synth.rng(49, seed), 1, K)[0].copy()
    x[col] = {"+inf": 0x7F80, "-inf": 0xFF80, "nan": 0x7FC0}[which]
    return x


def assert_same_specials(y, Y64, what):
    """IEEE outcome, row by row: NaN where the binary64 sum is NaN, an
    infinity of the same sign where it is infinite, nothing else."""
    y, Y64 = np.asarray(y, np.float64), np.asarray(Y64, np.float64)
    assert np.array_equal(np.isnan(y), np.isnan(Y64)), f"{what}: NaN pattern"
    inf = np.isinf(Y64)
    assert np.array_equal(np.isinf(y), inf), f"{what}: infinity pattern"
    assert np.array_equal(np.sign(y[inf]), np.sign(Y64[inf])), f"{what}: infinity signs"
    assert np.all(np.isnan(Y64) | inf), f"{what}: every row meets the special value"


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K, synth.Q8_KR])
@pytest.mark.parametrize("which", ["+inf", "-inf", "nan"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_inf_and_nan_activations(q, kind, which, out):
    """One infinite or NaN activation: a row's sum is +-Inf where its weight
    at that column is nonzero (sign of the product), NaN where that weight is
    exactly zero (0 * Inf) or the activation is NaN, as in binary64."""
    N, K = 2048, 2560
    f, w = synth.make(kind, N, K, synth.rng(49, kind, 1))
    x = special_x(K, which, 1337, kind)
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    y = out_values(q.q4nx_gemv(W, to_dev_bf16(x), out_dtype=out))
    Y64, _ = oracle.matmul(w, kind, N, K, x)
    assert_same_specials(y, Y64, f"kind {kind} {which} {out}")


@pytest.mark.parametrize("kind", [synth.Q4_1, synth.Q4_K])
def test_infinity_on_exact_zero_weights(q, kind):
    """Q4_0-mapped weights (code 8 = an exact zero weight in every group's
    first column) with +Inf there: every row is 0 * Inf = NaN."""
    N, K = 1024, 1024
    f, w = q4_0_mapped_weight(kind, N, K, seed=3)
    x = special_x(K, "+inf", 256, 7)
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    y = out_values(q.q4nx_gemv(W, to_dev_bf16(x), out_dtype="f32"))
    Y64, _ = oracle.matmul(w, kind, N, K, x)
    assert np.all(np.isnan(Y64))
    assert_same_specials(y, Y64, f"kind {kind} Inf on zero weights")


def test_decode_layer_batch_with_inf_and_nan(q):
    """The seven projections of a layer in one launch (the x-slice cache
    path): q's activations hold a +Inf, v's a NaN, the others are N(0, 1)
    and stay within the bar."""
    items, refs = [], []
    for mi, (_, N, K) in enumerate(synth.QWEN3_06B_LAYER):
        f, w = synth.workload_weight(2, mi, layer=6)
        if mi == 0:
            x = special_x(K, "+inf", 700, 30)
        elif mi == 2:
            x = special_x(K, "nan", 5, 31)
        else:
            x = synth.activations(synth.rng(49, 40 + mi), 1, K)[0]
        y = torch.empty(N, dtype=torch.float32, device=DEV)
        items.append((q.Weight(to_dev_bytes(w), synth.Q4_1, N, K), to_dev_bf16(x), y))
        refs.append((mi, w, x, N, K))
    q.q4nx_gemv_batch(items, out_dtype="f32")
    for (W, xt, y), (mi, w, x, N, K) in zip(items, refs):
        Y64, A = oracle.matmul(w, synth.Q4_1, N, K, x)
        if mi in (0, 2):
            assert_same_specials(out_values(y), Y64, f"layer matrix {mi}")
        else:
            assert_within(out_values(y), Y64, A, False, f"layer matrix {mi} beside special values")


@pytest.mark.parametrize("kind,M", [(synth.Q4_1, 2), (synth.Q4_K, 2), (synth.Q4_K, 3), (synth.Q4_K, 4)])
def test_few_tokens_cached_slices_with_special_values(q, kind, M):
    """The few-token kernel with its x-slice cache (16384 x 1024: each CTA
    reads its 4 slices about three times) when token 0 holds a +Inf, at four
    tokens token 1 a NaN, and from three tokens the last is all zeros: a slice
    holding a special value is prepared for every token on the binary32 path.
    The special tokens' rows meet it as in binary64, the zero token's rows are
    exactly 0 and the N(0, 1) token stays within the bar."""
    N, K = 16384, 1024
    f, w = synth.make(kind, N, K, synth.rng(54, kind, M))
    X = synth.activations(synth.rng(54, 1, M), M, K).copy()
    X[0, 700] = 0x7F80                                  # +Inf (slice 2)
    specials = [0]
    if M == 4:
        X[1, 5] = 0x7FC0                                # NaN (slice 0)
        specials.append(1)
    zero = M - 1 if M >= 3 else None
    if zero is not None:
        X[zero, :] = 0
    finite = [m for m in range(M) if m not in specials and m != zero]
    assert len(finite) == 1
    W = q.Weight(to_dev_bytes(w), kind, N, K)
    got = out_values(q.q4nx_gemm_m64(W, to_dev_bf16(X), out_dtype="f32"))
    Y64, A = oracle.matmul(w, kind, N, K, X)
    for m in specials:
        assert_same_specials(got[m], Y64[m], f"kind {kind} M={M} token {m}")
    if zero is not None:
        assert np.all(got[zero] == 0.0), "the all-zero token's rows"
    m = finite[0]
    assert_within(got[m], Y64[m], A[m], False, f"kind {kind} M={M} token {m} beside special values")


def test_gemm_64_tokens_with_inf_and_nan(q):
    """The tensor-core GEMM: one token with a +Inf activation, one with a
    NaN; those tokens' rows meet the special value as in binary64 (on the
    bf16 weights the tensor cores multiply), the other tokens stay within
    the tensor-core bar."""
    N, K, M = 4096, 4096, 64
    f, w = synth.make(synth.Q4_1, N, K, synth.rng(49, 50))
    X = synth.activations(synth.rng(49, 51), M, K).copy()
    X[5, 1000] = 0x7F80
    X[9, 3] = 0x7FC0
    W = q.Weight(to_dev_bytes(w), synth.Q4_1, N, K)
    Y = q.q4nx_gemm_m64(W, to_dev_bf16(X), out_dtype="f32").cpu().numpy().astype(np.float64)
    rows = np.unique(np.concatenate([np.arange(0, 256), np.random.default_rng(5).integers(0, N, 512)]))
    # (a weight's sign, and whether it is exactly zero, survive its bf16
    # rounding, so the binary64 pattern on the exact weights is the one the
    # tensor cores must give)
    Ys, _ = oracle.matmul(w, synth.Q4_1, N, K, X[[5, 9]], rows=rows)
    for i, m in enumerate((5, 9)):
        assert_same_specials(Y[m, rows], Ys[i], f"token {m}")
    others = [m for m in range(M) if m not in (5, 9)]
    Y64, A = oracle.matmul(w, synth.Q4_1, N, K, X[others], rows=rows)
    assert np.all(np.abs(Y[others][:, rows] - Y64) <= (1e-3 + 2.0 ** -9) * A)
