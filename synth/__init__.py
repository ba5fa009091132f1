"""Seeded synthetic inputs for the Q4NX path: logical fields and chunk bytes.

This module only MAKES inputs.  It holds none of the method's arithmetic (no
decode, no product, no repack, no top-1); the oracle and the CUDA library each
read what it writes with their own code.  Both sides get the same bytes from
here, and nothing here calls either of them.

Every draw comes from numpy's PCG64 seeded by
``SeedSequence([workload_id, layer, matrix_id, seed])``.  bf16 values are
binary32 draws rounded to nearest-even by torch's CPU conversion.

Chunk byte order (the reading used across the build; the Q4NX section of the
1bit engine "NPU engine" page gives sizes and formulas but not the order):

  q4_1 (5120 B): codes 4096 | scale bf16 [32 r][8 g] | zero bf16 [32 r][8 g]
  Q4_K (4736 B): codes 4096 | sc u8 [32][8] | mn u8 [32][8] | S bf16 [32] | M bf16 [32]
  Q8   (8704 B): codes 8192 (layout KR: k*32+r, layout BLK:
                 (r/16)*4096+(k/32)*512+(k%32)*16+r%16) | d bf16 [32 r][8 g]
  4-bit code (r, k): byte r*128 + k/2, low nibble for even k.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

Q4_1, Q4_K, Q8_KR, Q8_BLK = 1, 2, 3, 4
CHUNK_BYTES = {Q4_1: 5120, Q4_K: 4736, Q8_KR: 8704, Q8_BLK: 8704}
KIND_NAMES = {Q4_1: "q4_1", Q4_K: "q4_k", Q8_KR: "q8_kr", Q8_BLK: "q8_blk"}


def rng(workload_id: int, layer: int = 0, matrix_id: int = 0, seed: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([workload_id, layer, matrix_id, seed])))


def bf16_bits(a) -> np.ndarray:
    """binary32 -> bf16 bit patterns (uint16), nearest-even, via torch on the CPU."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float32)))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits) -> np.ndarray:
    """bf16 bit patterns -> binary32 values (exact widening)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


# --------------------------------------------------------------------------
# logical fields of a weight: arrays indexed [tile, r, ...] with tile = tr*TC + tc
# --------------------------------------------------------------------------

@dataclass
class Fields:
    kind: int
    N: int
    K: int
    codes: np.ndarray                     # [T, 32, 256] uint8 (0..15) or int8
    scale: np.ndarray | None = None       # q4_1  [T, 32, 8] bf16 bits
    zero: np.ndarray | None = None        # q4_1  [T, 32, 8] bf16 bits
    sc: np.ndarray | None = None          # Q4_K  [T, 32, 8] uint8
    mn: np.ndarray | None = None          # Q4_K  [T, 32, 8] uint8
    S: np.ndarray | None = None           # Q4_K  [T, 32] bf16 bits
    M: np.ndarray | None = None           # Q4_K  [T, 32] bf16 bits
    d: np.ndarray | None = None           # Q8    [T, 32, 8] bf16 bits
    extra: dict = field(default_factory=dict)

    @property
    def tiles(self) -> int:
        return (self.N // 32) * (self.K // 256)


def _tiles(N: int, K: int) -> int:
    if N <= 0 or K <= 0 or N % 32 or K % 256:
        raise ValueError(f"{N}x{K} is not a whole grid of 32x256 tiles")
    return (N // 32) * (K // 256)


def q4_1_fields(g: np.random.Generator, N: int, K: int, scale_sigma: float = 0.02) -> Fields:
    """codes U{0..15}; scale = bf16(|N(0, sigma)| / 8); zero = bf16(-8 scale (1 + U(-0.1, 0.1)))."""
    T = _tiles(N, K)
    codes = g.integers(0, 16, size=(T, 32, 256), dtype=np.uint8)
    s_bits = bf16_bits(np.abs(g.normal(0.0, scale_sigma, size=(T, 32, 8))).astype(np.float32) / np.float32(8))
    s = bf16_values(s_bits)
    jitter = g.uniform(-0.1, 0.1, size=(T, 32, 8)).astype(np.float32)
    z_bits = bf16_bits(np.float32(-8.0) * s * (np.float32(1.0) + jitter))
    return Fields(Q4_1, N, K, codes, scale=s_bits, zero=z_bits)


def q4_k_fields(g: np.random.Generator, N: int, K: int, sigma: float = 0.01) -> Fields:
    """codes U{0..15}; sc, mn U{0..63}; per-row S = bf16(|N(0, sigma)|), M = bf16(|N(0, sigma)|)."""
    T = _tiles(N, K)
    codes = g.integers(0, 16, size=(T, 32, 256), dtype=np.uint8)
    sc = g.integers(0, 64, size=(T, 32, 8), dtype=np.uint8)
    mn = g.integers(0, 64, size=(T, 32, 8), dtype=np.uint8)
    S = bf16_bits(np.abs(g.normal(0.0, sigma, size=(T, 32))))
    M = bf16_bits(np.abs(g.normal(0.0, sigma, size=(T, 32))))
    return Fields(Q4_K, N, K, codes, sc=sc, mn=mn, S=S, M=M)


def q8_fields(g: np.random.Generator, N: int, K: int, kind: int = Q8_KR, sigma: float = 0.005) -> Fields:
    """int8 codes U{-127..127}; d = bf16(|N(0, sigma)|) per (row, 32-column group)."""
    if kind not in (Q8_KR, Q8_BLK):
        raise ValueError("Q8 kind must be Q8_KR or Q8_BLK")
    T = _tiles(N, K)
    codes = g.integers(-127, 128, size=(T, 32, 256), dtype=np.int8)
    d = bf16_bits(np.abs(g.normal(0.0, sigma, size=(T, 32, 8))))
    return Fields(kind, N, K, codes, d=d)


def activations(g: np.random.Generator, M: int, K: int, sigma: float = 1.0) -> np.ndarray:
    """bf16 bits [M, K] of N(0, sigma) draws."""
    return bf16_bits(g.normal(0.0, sigma, size=(M, K)))


def activations_outliers(g: np.random.Generator, M: int, K: int, frac: float = 0.005, lo: float = 100.0,
                         hi: float = 1000.0) -> np.ndarray:
    """bf16 bits [M, K]: N(0, 1) with a fixed set of outlier channels (a fraction
    `frac` of the columns, at least one) scaled by U(lo, hi), the way a few
    channels of LLM hidden states run 10^2 - 10^3 times the rest."""
    x = g.normal(0.0, 1.0, size=(M, K))
    n = max(1, int(round(frac * K)))
    cols = g.choice(K, size=n, replace=False)
    x[:, cols] *= g.uniform(lo, hi, size=n)
    return bf16_bits(x)


def activations_log_uniform(g: np.random.Generator, M: int, K: int, lo_exp: float = -30.0,
                            hi_exp: float = 30.0, zero_frac: float = 0.05) -> np.ndarray:
    """bf16 bits [M, K]: random signs, magnitudes 2^U(lo_exp, hi_exp), a fraction
    of exact zeros (both signs): groups whose magnitudes span far more than
    any fixed-point width."""
    mag = np.exp2(g.uniform(lo_exp, hi_exp, size=(M, K)))
    x = np.where(g.random((M, K)) < 0.5, -mag, mag)
    z = g.random((M, K)) < zero_frac
    x[z] = np.where(g.random(int(z.sum())) < 0.5, -0.0, 0.0)
    return bf16_bits(x)


def activations_subnormal(g: np.random.Generator, M: int, K: int, zero_frac: float = 0.3) -> np.ndarray:
    """bf16 bits [M, K]: bf16 subnormals (exponent field 0, random nonzero
    mantissa and sign) mixed with +0 and -0."""
    mant = g.integers(1, 128, size=(M, K), dtype=np.uint16)
    sign = (g.random((M, K)) < 0.5).astype(np.uint16) << 15
    bits = sign | mant
    z = g.random((M, K)) < zero_frac
    bits[z] = sign[z]
    return bits


# --------------------------------------------------------------------------
# writers: logical fields -> chunk bytes
# --------------------------------------------------------------------------

def _nibbles(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).reshape(c.shape[0], 4096)


def _q8_code_bytes(codes: np.ndarray, kind: int) -> np.ndarray:
    T = codes.shape[0]
    c = codes.view(np.uint8)
    if kind == Q8_KR:          # byte k*32 + r
        return np.ascontiguousarray(c.transpose(0, 2, 1)).reshape(T, 8192)
    # byte (r/16)*4096 + (k/32)*512 + (k%32)*16 + r%16
    c5 = c.reshape(T, 2, 16, 8, 32)            # [T, r/16, r%16, k/32, k%32]
    return np.ascontiguousarray(c5.transpose(0, 1, 3, 4, 2)).reshape(T, 8192)


def pack(f: Fields) -> np.ndarray:
    """Chunk bytes (uint8, T * chunk_bytes) of a weight, row-major over the tile grid."""
    T = f.codes.shape[0]
    if f.kind == Q4_1:
        parts = [_nibbles(f.codes), f.scale.reshape(T, 256).view(np.uint8),
                 f.zero.reshape(T, 256).view(np.uint8)]
    elif f.kind == Q4_K:
        parts = [_nibbles(f.codes), f.sc.reshape(T, 256), f.mn.reshape(T, 256),
                 f.S.reshape(T, 32).view(np.uint8), f.M.reshape(T, 32).view(np.uint8)]
    elif f.kind in (Q8_KR, Q8_BLK):
        parts = [_q8_code_bytes(f.codes, f.kind), f.d.reshape(T, 256).view(np.uint8)]
    else:
        raise ValueError(f"unknown kind {f.kind}")
    out = np.concatenate([np.ascontiguousarray(p).reshape(T, -1) for p in parts], axis=1)
    assert out.shape[1] == CHUNK_BYTES[f.kind]
    return out.reshape(-1)


def logical_codes(f: Fields) -> np.ndarray:
    """The codes as a [N, K] matrix (tile grid unfolded), for round-trip checks."""
    TR, TC = f.N // 32, f.K // 256
    return f.codes.reshape(TR, TC, 32, 256).transpose(0, 2, 1, 3).reshape(f.N, f.K)


def make(kind: int, N: int, K: int, g: np.random.Generator, **kw) -> tuple[Fields, np.ndarray]:
    if kind == Q4_1:
        f = q4_1_fields(g, N, K, **kw)
    elif kind == Q4_K:
        f = q4_k_fields(g, N, K, **kw)
    else:
        f = q8_fields(g, N, K, kind, **kw)
    return f, pack(f)


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

QWEN3_06B_LAYER = (            # (name, N, K) of one Qwen3-0.6B-shaped decode layer
    ("q", 2048, 1024), ("k", 1024, 1024), ("v", 1024, 1024), ("o", 1024, 2048),
    ("gate", 3072, 1024), ("up", 3072, 1024), ("down", 1024, 3072),
)
QWEN3_06B_LAYERS = 28

WORKLOADS = {
    1: dict(name="q4_1 1024x1024 decode+GEMV", kind=Q4_1, shapes=[(1024, 1024)], M=1),
    2: dict(name="Qwen3-0.6B-shaped decode layer x28, q4_1, batch 1", kind=Q4_1,
            shapes=[(n, k) for _, n, k in QWEN3_06B_LAYER], layers=QWEN3_06B_LAYERS, M=1),
    3: dict(name="Q4_K 9728x2560 and 2560x9728 GEMV + repack", kind=Q4_K,
            shapes=[(9728, 2560), (2560, 9728)], M=1),
    4: dict(name="64-token prefill block, q4_1 8B width (gate/up 12288x4096, down 4096x12288)",
            kind=Q4_1, shapes=[(12288, 4096), (12288, 4096), (4096, 12288)], M=64),
    5: dict(name="Q8 lm_head 151936x2560, layouts KR and BLK, batch 1 and 64", kind=Q8_KR,
            shapes=[(151936, 2560)], M=64),
}


def workload_weight(workload_id: int, matrix_id: int, layer: int = 0, seed: int = 0,
                    kind: int | None = None, shape: tuple[int, int] | None = None):
    """Fields and chunk bytes of one weight of a workload."""
    spec = WORKLOADS[workload_id]
    N, K = shape if shape is not None else spec["shapes"][matrix_id]
    k = spec["kind"] if kind is None else kind
    return make(k, N, K, rng(workload_id, layer, matrix_id, seed))


def workload_activations(workload_id: int, matrix_id: int, M: int, K: int, layer: int = 0,
                         seed: int = 0) -> np.ndarray:
    """bf16 bits [M, K]; drawn from a stream separate from the weight's."""
    return activations(rng(workload_id, layer, 1000 + matrix_id, seed), M, K)


# --------------------------------------------------------------------------
# GGUF-type tensors (input of the q4_1 packer): blocks of 32 columns along a
# row, row-major.  Q4_0: fp16 d + 16 code bytes (element i < 16 = low nibble
# of byte i, i >= 16 = high nibble of byte i - 16); Q4_1: fp16 d, fp16 m + 16
# code bytes; Q8_0: fp16 d + 32 int8 codes; dense: F32 / F16 / BF16 values.
# --------------------------------------------------------------------------

SRC_Q4_0, SRC_Q4_1, SRC_Q8_0, SRC_F32, SRC_F16, SRC_BF16 = 1, 2, 3, 4, 5, 6


def _f16_bits(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def _gguf_nibbles(codes: np.ndarray) -> np.ndarray:
    """[N, K/32, 32] codes 0..15 -> [N, K/32, 16] bytes (element i and i + 16 share byte i)."""
    c = codes.astype(np.uint8)
    return c[..., :16] | (c[..., 16:] << 4)


def gguf_tensor(src_type: int, N: int, K: int, g: np.random.Generator) -> tuple[np.ndarray, dict]:
    """Bytes of a synthetic N x K GGUF-type tensor and its logical fields.

    Q4_0 / Q4_1: d = |N(0, 0.02)| / 8 (fp16), Q4_1 m = -8 d (1 + U(-0.1, 0.1)) (fp16), codes U{0..15};
    Q8_0: d = |N(0, 0.005)| (fp16), codes U{-127..127}; dense: N(0, 0.02) values.
    """
    if N % 32 or K % 256:
        raise ValueError("shape must be a whole grid of 32 x 256 tiles")
    nb = K // 32
    if src_type in (SRC_Q4_0, SRC_Q4_1):
        d = np.abs(g.normal(0.0, 0.02, size=(N, nb))) / 8
        codes = g.integers(0, 16, size=(N, nb, 32), dtype=np.int64)
        dh = _f16_bits(d)
        parts = [dh.reshape(N, nb, 1).view(np.uint8).reshape(N, nb, 2)]
        f = {"d": dh, "codes": codes}
        if src_type == SRC_Q4_1:
            m = -8.0 * d * (1.0 + g.uniform(-0.1, 0.1, size=(N, nb)))
            mh = _f16_bits(m)
            parts.append(mh.reshape(N, nb, 1).view(np.uint8).reshape(N, nb, 2))
            f["m"] = mh
        parts.append(_gguf_nibbles(codes))
        return np.concatenate(parts, axis=2).reshape(-1), f
    if src_type == SRC_Q8_0:
        d = _f16_bits(np.abs(g.normal(0.0, 0.005, size=(N, nb))))
        codes = g.integers(-127, 128, size=(N, nb, 32), dtype=np.int8)
        blk = np.concatenate([d.reshape(N, nb, 1).view(np.uint8).reshape(N, nb, 2), codes.view(np.uint8)], axis=2)
        return blk.reshape(-1), {"d": d, "codes": codes}
    x = g.normal(0.0, 0.02, size=(N, K))
    if src_type == SRC_F32:
        v = x.astype(np.float32)
    elif src_type == SRC_F16:
        v = x.astype(np.float16)
    elif src_type == SRC_BF16:
        v = bf16_bits(x)
    else:
        raise ValueError(f"unknown GGUF type {src_type}")
    return np.ascontiguousarray(v).view(np.uint8).reshape(-1), {"values": v}
