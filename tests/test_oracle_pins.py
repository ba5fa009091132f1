"""Pins of the oracle to facts outside itself (CPU only).

Each test ties the oracle to something the pages or mathematics fix:
the chunk-kind table and Q8 layout expressions of the "Q4NX chunks" section of
the 1bit engine "NPU engine" page, closed forms of the weight formulas,
library routines (numpy binary64 matmul, numpy binary32 arithmetic, torch's
bf16 conversion, numpy argmax), exact rational arithmetic, and the repack's
rounding bound stated on the same page.  The byte order inside a chunk is not
printed on any page: tests of it below pin the oracle to the documented
reading, not to the pages (parity unpinned for that reading).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
KINDS = (oracle.Q4_1, oracle.Q4_K, oracle.Q8_KR, oracle.Q8_BLK)


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _bf16(x):
    return synth.bf16_bits(np.asarray(x, dtype=np.float32))


def _q4_1_const(T, code, s, z):
    f = synth.Fields(synth.Q4_1, 32, 256 * T, np.full((T, 32, 256), code, np.uint8),
                     scale=np.full((T, 32, 8), _bf16(s), np.uint16),
                     zero=np.full((T, 32, 8), _bf16(z), np.uint16))
    return f


# ----------------------------------------------------------------- sizes ----

def test_chunk_bytes_match_page_table():
    table = {r[0]: int(r[1]) for r in _golden_rows("chunk_kinds.txt")}
    assert oracle.chunk_bytes(oracle.Q4_1) == table["q4_1"]
    assert oracle.chunk_bytes(oracle.Q4_K) == table["q4_k"]
    assert oracle.chunk_bytes(oracle.Q8_KR) == table["q8"]
    assert oracle.chunk_bytes(oracle.Q8_BLK) == table["q8"]
    assert oracle.chunk_bytes(0) == 0 and oracle.chunk_bytes(5) == 0
    # The sizes are exactly the fields the table lists for a 32x256 tile:
    codes4, codes8, groups = 32 * 256 // 2, 32 * 256, 32 * 8
    assert table["q4_1"] == codes4 + groups * 2 * 2            # bf16 scale + bf16 zero
    assert table["q4_k"] == codes4 + groups * 1 * 2 + 32 * 2 * 2  # u8 sc, mn + bf16 S, M
    assert table["q8"] == codes8 + groups * 2                   # bf16 d
    for k in KINDS:
        assert synth.CHUNK_BYTES[k] == oracle.chunk_bytes(k)


# ------------------------------------------------------------------ bf16 ----

def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(7)
    vals = np.concatenate([
        g.normal(0, 1, 4000).astype(np.float32),
        (g.normal(0, 1, 1000) * 1e-39).astype(np.float32),         # subnormal range
        (np.clip(g.normal(0, 1, 1000), -3, 3) * 1.1e38).astype(np.float32),  # near overflow
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38], np.float32),
    ])
    # exact ties: low 16 bits == 0x8000, with even and odd kept parts
    ties = (np.arange(0x3F80, 0x3FC0, dtype=np.uint32) << 16) | 0x8000
    vals = np.concatenate([vals, ties.view(np.float32), (ties | 0x80000000).view(np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f32_to_bf16(vals)
    assert np.array_equal(got, ref)
    nan = np.array([np.nan, -np.nan], np.float32)
    back = oracle.bf16_to_f32(oracle.f32_to_bf16(nan))
    assert np.isnan(back).all()
    h = np.arange(0, 65536, 97, dtype=np.uint16)
    h = h[(h & 0x7F80) != 0x7F80]            # NaN payloads do not survive a round trip through a C float
    assert np.array_equal(oracle.bf16_to_f32(h).view(np.uint32), h.astype(np.uint32) << 16)


# -------------------------------------------------------------- Q8 layouts ----

@pytest.mark.parametrize("kind,col", [(oracle.Q8_KR, 2), (oracle.Q8_BLK, 3)])
def test_q8_layout_points_from_page(kind, col):
    """A single nonzero code byte at the page's offset decodes at (r, k)."""
    for row in _golden_rows("q8_layout_points.txt"):
        r, k, off = int(row[0]), int(row[1]), int(row[col])
        ch = np.zeros(8704, np.uint8)
        ch[off] = 3
        ch[8192:].view(np.uint16)[:] = _bf16(1.0)
        c = oracle.codes(ch, kind, 32, 256)
        nz = np.argwhere(c != 0)
        assert nz.tolist() == [[r, k]], (row, nz.tolist())


@pytest.mark.parametrize("kind", [oracle.Q8_KR, oracle.Q8_BLK])
def test_q8_layout_is_bijection_and_matches_expression(kind):
    """Brute force over all 8192 (r, k): the code byte the oracle reads is the
    page's expression, and the map is one-to-one onto the 8192 code bytes."""
    off = np.arange(8192)
    lo = np.zeros(8704, np.uint8)
    hi = np.zeros(8704, np.uint8)
    lo[:8192] = off & 0xFF
    hi[:8192] = off >> 8
    got = (oracle.codes(lo, kind, 32, 256) & 0xFF) | ((oracle.codes(hi, kind, 32, 256) & 0xFF) << 8)
    assert np.array_equal(np.sort(got.reshape(-1)), off)
    r = np.arange(32)[:, None]
    k = np.arange(256)[None, :]
    if kind == oracle.Q8_KR:
        expect = k * 32 + r
    else:
        expect = (r // 16) * 4096 + (k // 32) * 512 + (k % 32) * 16 + r % 16
    assert np.array_equal(got, expect)


def test_q8_wrong_layout_decorrelates():
    """Analogue of the page's layout check: decoding with the right layout
    correlates perfectly with the true weights, the wrong one hardly at all."""
    g = synth.rng(99)
    f, w = synth.make(synth.Q8_BLK, 64, 512, g)
    truth = oracle.weights_f64(w, oracle.Q8_BLK, 64, 512).reshape(-1)
    wrong = oracle.weights_f64(w, oracle.Q8_KR, 64, 512).reshape(-1)
    assert np.corrcoef(truth, truth)[0, 1] > 0.9999
    assert abs(np.corrcoef(truth, wrong)[0, 1]) < 0.05


# --------------------------------------------------- 4-bit code positions ----

@pytest.mark.parametrize("kind", [oracle.Q4_1, oracle.Q4_K])
def test_nibble_positions_by_probe(kind):
    """Every single-nibble probe lands on exactly one (r, k): the documented
    reading, byte r*128 + k/2 with the low nibble for even k (unpinned reading)."""
    cb = oracle.chunk_bytes(kind)
    base = np.zeros(cb, np.uint8)
    for b in range(0, 4096, 37):
        for hi in (0, 1):
            ch = base.copy()
            ch[b] = 0x50 if hi else 0x05
            c = oracle.codes(ch, kind, 32, 256)
            nz = np.argwhere(c != 0).tolist()
            assert nz == [[b // 128, 2 * (b % 128) + hi]]
            assert c[b // 128, 2 * (b % 128) + hi] == 5


def test_tile_grid_is_row_major():
    """Chunk t of a 2x3 grid covers rows (t//3)*32.., columns (t%3)*256.."""
    T = 6
    codes = np.repeat(np.arange(T, dtype=np.uint8)[:, None, None], 32, 1).repeat(256, 2)
    f = synth.Fields(synth.Q4_1, 64, 768, codes,
                     scale=np.full((T, 32, 8), _bf16(1.0), np.uint16),
                     zero=np.zeros((T, 32, 8), np.uint16))
    W = oracle.weights_f64(synth.pack(f), oracle.Q4_1, 64, 768)
    for t in range(T):
        tr, tc = divmod(t, 3)
        assert (W[tr * 32:(tr + 1) * 32, tc * 256:(tc + 1) * 256] == t).all()


@pytest.mark.parametrize("kind", KINDS)
def test_concatenated_chunk_arrays_stack_rows(kind):
    """The grid is row-major over whole tile rows, so two weights of the same
    width whose chunk arrays are concatenated form one weight with the first's
    rows above the second's (how gate and up become one matrix)."""
    _, wa = synth.make(kind, 64, 512, synth.rng(5, matrix_id=20 + kind))
    _, wb = synth.make(kind, 96, 512, synth.rng(5, matrix_id=40 + kind))
    Wab = oracle.weights_f64(np.concatenate([wa, wb]), kind, 160, 512)
    assert np.array_equal(Wab[:64], oracle.weights_f64(wa, kind, 64, 512))
    assert np.array_equal(Wab[64:], oracle.weights_f64(wb, kind, 96, 512))


@pytest.mark.parametrize("kind", KINDS)
def test_generator_round_trip(kind):
    g = synth.rng(5, matrix_id=kind)
    f, w = synth.make(kind, 96, 512, g)
    assert w.size == f.tiles * oracle.chunk_bytes(kind)
    assert np.array_equal(oracle.codes(w, kind, 96, 512), synth.logical_codes(f).astype(np.int32))


# ----------------------------------------------------------- closed forms ----

def test_q4_1_closed_forms():
    # constant code, scale 1, zero 0: w = code
    for c0 in (0, 1, 7, 15):
        w = synth.pack(_q4_1_const(2, c0, 1.0, 0.0))
        assert (oracle.weights_f64(w, oracle.Q4_1, 32, 512) == c0).all()
        assert (oracle.decode(w, oracle.Q4_1, 32, 512) == _bf16(float(c0))).all()
    # constant (code, scale, zero): w = code*scale + zero, y = w * sum(x)
    w = synth.pack(_q4_1_const(2, 11, 0.25, -1.5))
    assert (oracle.weights_f64(w, oracle.Q4_1, 32, 512) == 11 * 0.25 - 1.5).all()
    x = synth.activations(synth.rng(3), 1, 512)[0]
    y, A = oracle.matmul(w, oracle.Q4_1, 32, 512, x)
    sx = math.fsum(synth.bf16_values(x).astype(np.float64))
    assert np.allclose(y, 1.25 * sx, rtol=1e-12, atol=0)
    assert np.allclose(A, 1.25 * np.abs(synth.bf16_values(x)).astype(np.float64).sum(), rtol=1e-12)
    # the Q4_0 mapping of the "From a GGUF" table (zero = -8 d): code 8 is exactly 0
    for d in (0.5, 0.01171875, 3.0):
        w = synth.pack(_q4_1_const(1, 8, d, -8 * d))
        assert (oracle.weights_f64(w, oracle.Q4_1, 32, 256) == 0).all()
        assert (oracle.decode(w, oracle.Q4_1, 32, 256) == 0).all()
        y, _ = oracle.matmul(w, oracle.Q4_1, 32, 256, x[:256])
        assert (y == 0).all()


def _q4k_const(code, sc, mn, S, M):
    T = 1
    return synth.Fields(synth.Q4_K, 32, 256, np.full((T, 32, 256), code, np.uint8),
                        sc=np.full((T, 32, 8), sc, np.uint8), mn=np.full((T, 32, 8), mn, np.uint8),
                        S=np.full((T, 32), _bf16(S), np.uint16), M=np.full((T, 32), _bf16(M), np.uint16))


def test_q4_k_closed_forms():
    w = synth.pack(_q4k_const(9, 1, 0, 1.0, 0.0))              # S=1, scale=1, M=0: w = code
    assert (oracle.weights_f64(w, oracle.Q4_K, 32, 256) == 9).all()
    w = synth.pack(_q4k_const(5, 3, 4, 2.0, 0.5))              # 2*3*5 + 0.5*4 = 32 (sign +M*min)
    assert (oracle.weights_f64(w, oracle.Q4_K, 32, 256) == 32).all()
    assert (oracle.decode(w, oracle.Q4_K, 32, 256) == _bf16(32.0)).all()
    w = synth.pack(_q4k_const(5, 3, 4, 2.0, -0.5))             # negative M: 30 - 2 = 28
    assert (oracle.weights_f64(w, oracle.Q4_K, 32, 256) == 28).all()
    w = synth.pack(_q4k_const(15, 63, 63, 1.0, 1.0))           # largest fields: 945 + 63
    assert (oracle.weights_f64(w, oracle.Q4_K, 32, 256) == 1008).all()


@pytest.mark.parametrize("kind", [oracle.Q8_KR, oracle.Q8_BLK])
def test_q8_closed_forms(kind):
    g = synth.rng(11)
    f = synth.q8_fields(g, 32, 256, kind)
    f.d[:] = _bf16(1.0)
    w = synth.pack(f)
    assert np.array_equal(oracle.weights_f64(w, kind, 32, 256), synth.logical_codes(f).astype(np.float64))
    f.codes[:] = -127
    f.d[:] = _bf16(0.5)
    w = synth.pack(f)
    assert (oracle.weights_f64(w, kind, 32, 256) == -63.5).all()
    assert (oracle.decode(w, kind, 32, 256) == _bf16(-63.5)).all()


# ----------------------------------------------- decode rounding (bit-exact) ----

def _exact_weight(kind, fld, r, k):
    """The weight as an exact rational from the logical fields."""
    g = k // 32
    v = lambda bits: Fraction(float(synth.bf16_values(bits)))
    c = int(fld.codes[0, r, k])
    if kind == oracle.Q4_1:
        return c * v(fld.scale[0, r, g]) + v(fld.zero[0, r, g])
    if kind == oracle.Q4_K:
        return v(fld.S[0, r]) * int(fld.sc[0, r, g]) * c + v(fld.M[0, r]) * int(fld.mn[0, r, g])
    return v(fld.d[0, r, g]) * c


@pytest.mark.parametrize("kind", KINDS)
def test_decode_f32_is_one_correct_rounding(kind):
    """Every product is exact in binary32, so the binary32 weight is the exact
    weight correctly rounded once (|err| <= half an ulp, exact rationals)."""
    f, w = synth.make(kind, 32, 256, synth.rng(13, matrix_id=kind))
    got = oracle.decode_f32(w, kind, 32, 256)
    for r in range(0, 32, 5):
        for k in range(0, 256, 7):
            ex = _exact_weight(kind, f, r, k)
            v = got[r, k]
            ulp = Fraction(float(np.spacing(np.float32(abs(v))))) if v != 0 else Fraction(2) ** -149
            assert abs(Fraction(float(v)) - ex) <= ulp / 2


@pytest.mark.parametrize("kind", KINDS)
def test_decode_matches_numpy_f32_and_torch_bf16(kind):
    """The bf16 decode equals binary32 evaluation in numpy (one operation at a
    time) followed by torch's nearest-even bf16 conversion."""
    f, w = synth.make(kind, 64, 512, synth.rng(17, matrix_id=kind))
    c = synth.logical_codes(f).astype(np.float32)
    grid = lambda a: a.reshape(2, 2, 32, -1).transpose(0, 2, 1, 3).reshape(64, -1)
    rep = lambda a: np.repeat(grid(a), 32, axis=1)          # per (row, group) -> per column
    if kind == oracle.Q4_1:
        v = c * rep(synth.bf16_values(f.scale)) + rep(synth.bf16_values(f.zero))
    elif kind == oracle.Q4_K:
        S = np.repeat(grid(synth.bf16_values(f.S)[:, :, None]), 256, axis=1)   # per (row, tile)
        M = np.repeat(grid(synth.bf16_values(f.M)[:, :, None]), 256, axis=1)
        v = (S * rep(f.sc.astype(np.float32))) * c + M * rep(f.mn.astype(np.float32))
    else:
        v = rep(synth.bf16_values(f.d)) * c
    assert np.array_equal(oracle.decode_f32(w, kind, 64, 512), v.astype(np.float32))
    assert np.array_equal(oracle.decode(w, kind, 64, 512), synth.bf16_bits(v))


# --------------------------------------------------------------- matvec ----

@pytest.mark.parametrize("kind", KINDS)
def test_matvec_basis_vectors_give_columns(kind):
    """x = e_k gives y = W[:, k] exactly (catches a transposed operand on a
    non-square weight)."""
    N, K = 64, 512
    f, w = synth.make(kind, N, K, synth.rng(19, matrix_id=kind))
    W = oracle.weights_f64(w, kind, N, K)
    one = int(_bf16([1.0])[0])
    for k in (0, 1, 31, 32, 255, 256, 511):
        x = np.zeros(K, np.uint16)
        x[k] = one
        y, A = oracle.matmul(w, kind, N, K, x)
        assert np.array_equal(y, W[:, k])
        assert np.array_equal(A, np.abs(W[:, k]))


def test_matvec_non_finite_activations_follow_ieee():
    """Closed forms for a non-finite activation (IEEE arithmetic, which the
    products of the weight formulas inherit): with x = +Inf at one column and
    zeros elsewhere, a row gives +Inf where its weight at that column is
    positive, -Inf where it is negative and NaN (0 * Inf) where it is exactly
    zero; a NaN activation gives NaN on every row."""
    K = 256
    inf, ninf, nan = 0x7F80, 0xFF80, 0x7FC0
    # rows of three kinds at column 40: w > 0 (code 11, zero -1.5 at scale
    # 0.25: 1.25), w < 0 (code 2: -1.0) and w = 0 (the Q4_0 mapping, code 8)
    f = _q4_1_const(1, 11, 0.25, -1.5)
    f.codes[0, 10:20, :] = 2
    f.codes[0, 20:32, :] = 8
    f.scale[0, 20:32, :] = _bf16(0.25)
    f.zero[0, 20:32, :] = _bf16(-8 * 0.25)
    w = synth.pack(f)
    W = oracle.weights_f64(w, oracle.Q4_1, 32, K)
    assert (W[:10, 40] == 1.25).all() and (W[10:20, 40] == -1.0).all() and (W[20:, 40] == 0).all()
    for bits, sign in ((inf, 1.0), (ninf, -1.0)):
        x = np.zeros(K, np.uint16)
        x[40] = bits
        y, _ = oracle.matmul(w, oracle.Q4_1, 32, K, x)
        assert (y[:10] == sign * np.inf).all()
        assert (y[10:20] == -sign * np.inf).all()
        assert np.isnan(y[20:]).all()
    x = synth.activations(synth.rng(31), 1, K)[0].copy()
    x[7] = nan
    y, _ = oracle.matmul(w, oracle.Q4_1, 32, K, x)
    assert np.isnan(y).all()


@pytest.mark.parametrize("kind", KINDS)
def test_matmul_matches_numpy_float64(kind):
    N, K, M = 96, 768, 3
    f, w = synth.make(kind, N, K, synth.rng(23, matrix_id=kind))
    X = synth.activations(synth.rng(24), M, K)
    W = oracle.weights_f64(w, kind, N, K)
    Xf = synth.bf16_values(X).astype(np.float64)
    Y, A = oracle.matmul(w, kind, N, K, X)
    Yref = Xf @ W.T
    Aref = np.abs(Xf) @ np.abs(W.T)
    assert np.all(np.abs(Y - Yref) <= 1e-12 * Aref)
    assert np.allclose(A, Aref, rtol=1e-12, atol=0)
    # linearity: scaling x by 2 (exact in bf16) scales y by 2 exactly
    X2 = synth.bf16_bits(synth.bf16_values(X) * np.float32(2))
    Y2, _ = oracle.matmul(w, kind, N, K, X2)
    assert np.array_equal(Y2, 2 * Y)
    # a subset of rows equals the same rows of the full product
    rows = np.array([95, 0, 33, 64])
    Ys, As = oracle.matmul(w, kind, N, K, X, rows=rows)
    assert np.array_equal(Ys, Y[:, rows]) and np.array_equal(As, A[:, rows])


def test_matvec_within_binary64_bound_of_exact_sum():
    """Against exact rational arithmetic: |y - exact| <= K * 2^-53 * A."""
    N, K = 32, 512
    f, w = synth.make(oracle.Q4_1, N, K, synth.rng(29))
    x = synth.activations(synth.rng(30), 1, K)[0]
    y, A = oracle.matmul(w, oracle.Q4_1, N, K, x)
    W = oracle.weights_f64(w, oracle.Q4_1, N, K)
    xv = [Fraction(float(v)) for v in synth.bf16_values(x)]
    for n in range(0, N, 7):
        ex = sum(Fraction(float(W[n, k])) * xv[k] for k in range(K))
        assert abs(Fraction(float(y[n])) - ex) <= Fraction(K) * Fraction(2) ** -53 * Fraction(float(A[n]))


# --------------------------------------------------------------- repack ----

def test_repack_within_page_rounding_bound():
    """The page: the repack is exact apart from rounding S*scale and M*min to
    bf16.  Per weight |w_q41 - w_q4k| <= code*u*|S sc| + u*|M mn|, u = 2^-8."""
    N, K = 64, 512
    f, w = synth.make(oracle.Q4_K, N, K, synth.rng(31))
    rep = oracle.repack_q4k(w, N, K)
    assert rep.size == (N // 32) * (K // 256) * 5120
    Wk = oracle.weights_f64(w, oracle.Q4_K, N, K)
    W1 = oracle.weights_f64(rep, oracle.Q4_1, N, K)
    u = 2.0 ** -8
    S = np.repeat(np.repeat(synth.bf16_values(f.S).astype(np.float64)[:, :, None], 256, 2), 1, 0)
    grid = lambda a: a.reshape(2, 2, 32, 256).transpose(0, 2, 1, 3).reshape(N, K)
    rep_g = lambda a: np.repeat(a.astype(np.float64), 32, axis=2)
    Sg = grid(np.repeat(synth.bf16_values(f.S).astype(np.float64)[:, :, None], 256, 2))
    Mg = grid(np.repeat(synth.bf16_values(f.M).astype(np.float64)[:, :, None], 256, 2))
    sc, mn = grid(rep_g(f.sc)), grid(rep_g(f.mn))
    code = synth.logical_codes(f).astype(np.float64)
    bound = code * u * np.abs(Sg * sc) + u * np.abs(Mg * mn)
    assert np.all(np.abs(W1 - Wk) <= bound)
    assert np.any(W1 != Wk)          # the rounding is real for generic S, M
    # codes unchanged, byte for byte
    assert np.array_equal(rep.reshape(-1, 5120)[:, :4096], w.reshape(-1, 4736)[:, :4096])
    del S


def test_repack_exact_for_power_of_two_S_M():
    """With S and M powers of two, S*sc and M*mn are exact in bf16: no error."""
    N, K = 32, 512
    f = synth.q4_k_fields(synth.rng(37), N, K)
    g = np.random.default_rng(1)
    f.S[:] = _bf16(2.0 ** g.integers(-12, 2, size=f.S.shape))
    f.M[:] = _bf16(-(2.0 ** g.integers(-12, 2, size=f.M.shape)))
    w = synth.pack(f)
    rep = oracle.repack_q4k(w, N, K)
    assert np.array_equal(oracle.weights_f64(rep, oracle.Q4_1, N, K), oracle.weights_f64(w, oracle.Q4_K, N, K))


# --------------------------------------------------------------- argmax ----

def test_argmax_matches_numpy_with_ties_nan_inf():
    g = np.random.default_rng(41)
    L = g.normal(size=(12, 1000)).astype(np.float32)
    L[1, [10, 500, 999]] = 50.0                        # tie -> lowest index
    L[2, :] = 3.0                                      # all equal -> 0
    L[3, [7, 700]] = np.nan                            # first NaN wins
    L[3, 5] = np.inf
    L[4, 900] = np.inf
    L[4, 901] = np.inf
    L[5, :] = -np.inf
    L[6, 0] = np.nan
    L[7, 999] = np.nan
    L[8, :] = -0.0
    L[8, 3] = 0.0                                      # +0 == -0: first one wins
    got = oracle.argmax(L)
    assert np.array_equal(got, np.argmax(L, axis=1))
    assert got[1] == 10 and got[2] == 0 and got[3] == 7 and got[4] == 900 and got[8] == 0
    assert oracle.argmax(L[9]) == np.argmax(L[9])
