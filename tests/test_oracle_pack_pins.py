"""Pins of the oracle's GGUF-type -> q4_1 packer ("NPU engine" page, "From a GGUF").

The page's table fixes what each source type becomes: Q4_0 -> scale d, zero -8d;
Q4_1 -> scale d, zero m; codes unchanged; the only error is the bf16 rounding
of scale and zero.  Q8_0 and dense types are dequantized and then quantized to
a min/max q4_1 per 32 columns.  These checks tie the oracle to those facts
through the oracle's own, separately pinned decoders (codes, weights_f64).
"""
import numpy as np
import pytest

import oracle
import synth

U = 2.0 ** -8                       # bf16 unit round-off (nearest-even)


def _logical(codes_blocks: np.ndarray, N: int, K: int) -> np.ndarray:
    return codes_blocks.reshape(N, K)


def _f16(h):
    return oracle.f16_to_f32(h).astype(np.float64)


@pytest.mark.parametrize("t", [synth.SRC_Q4_0, synth.SRC_Q4_1])
def test_codes_are_carried_over_unchanged(t):
    N, K = 64, 512
    src, f = synth.gguf_tensor(t, N, K, synth.rng(20, t))
    out = oracle.pack_q4_1(src, t, N, K)
    assert np.array_equal(oracle.codes(out, oracle.Q4_1, N, K), _logical(f["codes"], N, K))


def test_q4_0_is_exact_when_d_is_a_short_binary_fraction():
    # d = 2^-e is exact in fp16 and bf16: every weight must equal d * (q - 8)
    N, K = 32, 256
    src, f = synth.gguf_tensor(synth.SRC_Q4_0, N, K, synth.rng(21))
    blk = src.reshape(N, K // 32, 18).copy()
    e = synth.rng(22).integers(6, 12, size=(N, K // 32))
    blk[:, :, 0:2] = np.asarray(2.0 ** -e, dtype=np.float16).view(np.uint8).reshape(N, K // 32, 2)
    out = oracle.pack_q4_1(blk.reshape(-1), synth.SRC_Q4_0, N, K)
    d = np.repeat(2.0 ** -e, 32, axis=1)
    want = d * (_logical(f["codes"], N, K) - 8.0)
    assert np.array_equal(oracle.weights_f64(out, oracle.Q4_1, N, K), want)


def test_q4_0_within_the_bf16_rounding_bound():
    N, K = 64, 768
    src, f = synth.gguf_tensor(synth.SRC_Q4_0, N, K, synth.rng(23))
    out = oracle.pack_q4_1(src, synth.SRC_Q4_0, N, K)
    d = np.repeat(_f16(f["d"]), 32, axis=1)
    q = _logical(f["codes"], N, K).astype(np.float64)
    w = oracle.weights_f64(out, oracle.Q4_1, N, K)
    err = np.abs(w - d * (q - 8.0))
    assert np.all(err <= q * U * d + U * 8.0 * d)
    assert err.max() > 0                              # fp16 d is not bf16: the rounding is really there


def test_q4_1_exact_cases_and_bound():
    N, K = 64, 512
    src, f = synth.gguf_tensor(synth.SRC_Q4_1, N, K, synth.rng(24))
    out = oracle.pack_q4_1(src, synth.SRC_Q4_1, N, K)
    d = np.repeat(_f16(f["d"]), 32, axis=1)
    m = np.repeat(_f16(f["m"]), 32, axis=1)
    q = _logical(f["codes"], N, K).astype(np.float64)
    w = oracle.weights_f64(out, oracle.Q4_1, N, K)
    assert np.all(np.abs(w - (d * q + m)) <= q * U * d + U * np.abs(m))
    # d and m exact in bf16 (8 significant bits): the pack is exact
    blk = src.reshape(N, K // 32, 20).copy()
    dd = np.asarray([[0.00390625, 0.0078125, 0.01171875, 0.0234375] * (K // 128)] * N, dtype=np.float16)
    mm = np.asarray(-8.5 * dd.astype(np.float64), dtype=np.float16)      # 8.5 * d keeps 8 significant bits
    blk[:, :, 0:2] = dd.view(np.uint8).reshape(N, K // 32, 2)
    blk[:, :, 2:4] = mm.view(np.uint8).reshape(N, K // 32, 2)
    out2 = oracle.pack_q4_1(blk.reshape(-1), synth.SRC_Q4_1, N, K)
    want = np.repeat(dd.astype(np.float64), 32, axis=1) * q + np.repeat(mm.astype(np.float64), 32, axis=1)
    assert np.array_equal(oracle.weights_f64(out2, oracle.Q4_1, N, K), want)


def _dense_fields(out, N, K):
    T = out.reshape(-1, 5120)
    TC = K // 256
    s = oracle.bf16_to_f32(T[:, 4096:4608].view(np.uint16)).astype(np.float64).reshape(N // 32, TC, 32, 8)
    z = oracle.bf16_to_f32(T[:, 4608:5120].view(np.uint16)).astype(np.float64).reshape(N // 32, TC, 32, 8)
    # [N, K/32] per (row, group)
    s = s.transpose(0, 2, 1, 3).reshape(N, K // 32)
    z = z.transpose(0, 2, 1, 3).reshape(N, K // 32)
    return s, z


def test_min_max_reproduces_values_on_its_own_grid():
    # x = lo + step * q with lo, step exact in bf16 and step = (hi - lo)/15 exactly
    N, K = 32, 256
    g = synth.rng(25)
    q = g.integers(0, 16, size=(N, K))
    q[:, ::32] = 0
    q[:, 1::32] = 15                                   # every group spans the full range
    lo, step = -0.09375, 2.0 ** -7
    x = (lo + step * q).astype(np.float32)
    out = oracle.pack_q4_1(x, synth.SRC_F32, N, K)
    assert np.array_equal(oracle.codes(out, oracle.Q4_1, N, K), q)
    assert np.array_equal(oracle.weights_f64(out, oracle.Q4_1, N, K), x.astype(np.float64))


def test_min_max_constant_group_has_zero_scale():
    N, K = 32, 256
    x = np.full((N, K), 0.0371, dtype=np.float32)
    out = oracle.pack_q4_1(x, synth.SRC_F32, N, K)
    s, z = _dense_fields(out, N, K)
    assert np.all(s == 0) and np.all(oracle.codes(out, oracle.Q4_1, N, K) == 0)
    assert np.all(z == oracle.bf16_to_f32(oracle.f32_to_bf16(np.float32(0.0371))))


@pytest.mark.parametrize("t", [synth.SRC_F32, synth.SRC_F16, synth.SRC_BF16, synth.SRC_Q8_0])
def test_min_max_codes_are_the_nearest_level_and_errors_are_bounded(t):
    N, K = 32, 512
    src, f = synth.gguf_tensor(t, N, K, synth.rng(26, t))
    if t == synth.SRC_Q8_0:
        x = (np.repeat(_f16(f["d"]), 32, axis=1) * f["codes"].reshape(N, K)).astype(np.float64)
    elif t == synth.SRC_BF16:
        x = oracle.bf16_to_f32(f["values"]).astype(np.float64)
    else:
        x = f["values"].astype(np.float64)
    out = oracle.pack_q4_1(src, t, N, K)
    s, z = _dense_fields(out, N, K)
    S, Z = np.repeat(s, 32, axis=1), np.repeat(z, 32, axis=1)
    code = oracle.codes(out, oracle.Q4_1, N, K)
    # brute force: the stored code is a nearest level (near-ties excepted)
    levels = np.arange(16)[None, None, :] * S[..., None] + Z[..., None]
    dist = np.abs(x[..., None] - levels)
    best = dist.min(axis=-1)
    mine = np.take_along_axis(dist, code[..., None], axis=-1)[..., 0]
    assert np.all(mine <= best + 1e-6 * S)
    # every value is reproduced within half a step plus the bf16 rounding of the result
    grp = x.reshape(N, K // 32, 32)
    lo, hi = np.repeat(grp.min(-1), 32, axis=1), np.repeat(grp.max(-1), 32, axis=1)
    w = oracle.weights_f64(out, oracle.Q4_1, N, K)
    assert np.all(np.abs(w - x) <= 0.5 * S + U * (np.abs(lo) + np.abs(hi) + 15 * S) + 1e-12)


def test_the_three_dense_types_agree_on_equal_values():
    N, K = 32, 256
    v = np.asarray(synth.rng(27).normal(0, 0.02, size=(N, K)), dtype=np.float16)   # exact in f32, f16; bf16 not
    a = oracle.pack_q4_1(v.astype(np.float32), synth.SRC_F32, N, K)
    b = oracle.pack_q4_1(v, synth.SRC_F16, N, K)
    assert np.array_equal(a, b)
    vb = synth.bf16_bits(v.astype(np.float64))
    c = oracle.pack_q4_1(oracle.bf16_to_f32(vb).astype(np.float32), synth.SRC_F32, N, K)
    d = oracle.pack_q4_1(vb, synth.SRC_BF16, N, K)
    assert np.array_equal(c, d)
