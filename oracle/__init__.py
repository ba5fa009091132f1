"""The oracle: a plain, slow, single-threaded CPU statement of the Q4NX path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``dequant_gemv_gb300``) never imports, links or runs it, and this
package imports nothing from the product path.

The arithmetic lives in ``q4nx_oracle.c`` (plain C, ``-ffp-contract=off``);
this module only compiles it with gcc, loads it with ctypes and converts numpy
arrays.  Format source: the 1bit engine "NPU engine" page, section "Q4NX
chunks" (chunk-kind table, the two Q8 code layouts, the repack paragraph).

Functions
---------
chunk_bytes(kind)                -> bytes of one chunk of that kind
bf16_to_f32(h) / f32_to_bf16(f)  -> bf16 conversions (ties to even)
codes(w, kind, N, K)             -> stored codes [N, K] (int32)
decode(w, kind, N, K)            -> bf16 bits [N, K] (uint16), bit-exact target
decode_f32(w, kind, N, K)        -> binary32 weights before the bf16 rounding
weights_f64(w, kind, N, K)       -> exact weights [N, K] (float64)
matmul(w, kind, N, K, X, rows)   -> (Y, A): Y = X . W^T in binary64, A = sum |w x|
repack_q4k(w, N, K)              -> q4_1 chunk bytes
pack_q4_1(src, type, N, K)       -> q4_1 chunk bytes of a GGUF-type tensor ("From a GGUF")
f16_to_f32(h)                    -> IEEE binary16 decoding
argmax(logits)                   -> first maximum per row (NaN wins)

Parity of the byte order inside a chunk is unpinned: no page prints it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q4_1, Q4_K, Q8_KR, Q8_BLK = 1, 2, 3, 4
SRC_Q4_0, SRC_Q4_1, SRC_Q8_0, SRC_F32, SRC_F16, SRC_BF16 = 1, 2, 3, 4, 5, 6
SRC_BYTES_PER_32 = {SRC_Q4_0: 18, SRC_Q4_1: 20, SRC_Q8_0: 34, SRC_F32: 128, SRC_F16: 64, SRC_BF16: 64}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4nx_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (single thread of plain C, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC",
             "-shared", "-Wall", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.oracle_chunk_bytes.argtypes = [I]
            lib.oracle_chunk_bytes.restype = I64
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f32.restype = ctypes.c_float
            lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
            for name in ("oracle_codes", "oracle_decode", "oracle_decode_f32", "oracle_weights_f64"):
                getattr(lib, name).argtypes = [P, I, I64, I64, P]
                getattr(lib, name).restype = None
            lib.oracle_matmul_rows.argtypes = [P, I, I64, I64, P, I64, P, I64, P, P]
            lib.oracle_matmul_rows.restype = None
            lib.oracle_repack_q4k.argtypes = [P, I64, I64, P]
            lib.oracle_repack_q4k.restype = None
            lib.oracle_argmax.argtypes = [P, I64, I64, P]
            lib.oracle_argmax.restype = None
            lib.oracle_pack_q4_1.argtypes = [P, I, I64, I64, P]
            lib.oracle_pack_q4_1.restype = None
            lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f32.restype = ctypes.c_float
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _chunks(w, kind, N, K) -> np.ndarray:
    w = np.ascontiguousarray(np.asarray(w, dtype=np.uint8).reshape(-1))
    need = (N // 32) * (K // 256) * chunk_bytes(kind)
    if N % 32 or K % 256 or N <= 0 or K <= 0:
        raise ValueError(f"shape {N}x{K} is not a whole grid of 32x256 tiles")
    if w.size < need:
        raise ValueError(f"{w.size} bytes given, {need} needed")
    return w


def chunk_bytes(kind: int) -> int:
    return int(_load().oracle_chunk_bytes(kind))


def bf16_to_f32(h) -> np.ndarray:
    lib = _load()
    h = np.asarray(h, dtype=np.uint16)
    return np.array([lib.oracle_bf16_to_f32(int(v)) for v in h.reshape(-1)],
                    dtype=np.float32).reshape(h.shape)


def f32_to_bf16(f) -> np.ndarray:
    lib = _load()
    f = np.asarray(f, dtype=np.float32)
    return np.array([lib.oracle_f32_to_bf16(float(v)) for v in f.reshape(-1)],
                    dtype=np.uint16).reshape(f.shape)


def codes(w, kind: int, N: int, K: int) -> np.ndarray:
    w = _chunks(w, kind, N, K)
    out = np.empty((N, K), dtype=np.int32)
    _load().oracle_codes(_ptr(w), kind, N, K, _ptr(out))
    return out


def decode(w, kind: int, N: int, K: int) -> np.ndarray:
    w = _chunks(w, kind, N, K)
    out = np.empty((N, K), dtype=np.uint16)
    _load().oracle_decode(_ptr(w), kind, N, K, _ptr(out))
    return out


def decode_f32(w, kind: int, N: int, K: int) -> np.ndarray:
    w = _chunks(w, kind, N, K)
    out = np.empty((N, K), dtype=np.float32)
    _load().oracle_decode_f32(_ptr(w), kind, N, K, _ptr(out))
    return out


def weights_f64(w, kind: int, N: int, K: int) -> np.ndarray:
    w = _chunks(w, kind, N, K)
    out = np.empty((N, K), dtype=np.float64)
    _load().oracle_weights_f64(_ptr(w), kind, N, K, _ptr(out))
    return out


def matmul(w, kind: int, N: int, K: int, X_bf16, rows=None):
    """Y[m, j] = sum_k w[rows[j], k] * X[m, k] in binary64 (k ascending).

    X_bf16: uint16 bf16 bits, shape [K] or [M, K].  Returns (Y, A), each
    [M, len(rows)] (or [len(rows)] for a 1-D X); A = sum_k |w x| per output.
    """
    w = _chunks(w, kind, N, K)
    X = np.ascontiguousarray(np.asarray(X_bf16, dtype=np.uint16))
    one_d = X.ndim == 1
    X = X.reshape(-1, K)
    M = X.shape[0]
    rows = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= N):
        raise ValueError("row index out of range")
    Y = np.empty((M, rows.size), dtype=np.float64)
    A = np.empty((M, rows.size), dtype=np.float64)
    _load().oracle_matmul_rows(_ptr(w), kind, N, K, _ptr(X), M, _ptr(rows), rows.size, _ptr(Y), _ptr(A))
    if one_d:
        return Y[0], A[0]
    return Y, A


def repack_q4k(w, N: int, K: int) -> np.ndarray:
    w = _chunks(w, Q4_K, N, K)
    out = np.empty((N // 32) * (K // 256) * 5120, dtype=np.uint8)
    _load().oracle_repack_q4k(_ptr(w), N, K, _ptr(out))
    return out


def argmax(logits) -> np.ndarray:
    L = np.ascontiguousarray(np.asarray(logits, dtype=np.float32))
    one_d = L.ndim == 1
    L = L.reshape(-1, L.shape[-1])
    out = np.empty(L.shape[0], dtype=np.int32)
    _load().oracle_argmax(_ptr(L), L.shape[0], L.shape[1], _ptr(out))
    return out[0] if one_d else out


def f16_to_f32(h) -> np.ndarray:
    """IEEE binary16 bits -> binary32 values (exact)."""
    h = np.asarray(h, dtype=np.uint16)
    lib = _load()
    return np.array([lib.oracle_f16_to_f32(int(v)) for v in h.reshape(-1)], dtype=np.float32).reshape(h.shape)


def pack_q4_1(src, src_type: int, N: int, K: int) -> np.ndarray:
    """q4_1 chunk bytes of the N x K tensor `src` (bytes) of GGUF type `src_type`."""
    if N % 32 or K % 256 or N <= 0 or K <= 0:
        raise ValueError(f"shape {N}x{K} is not a whole grid of 32x256 tiles")
    src = np.ascontiguousarray(np.asarray(src).view(np.uint8).reshape(-1))
    need = N * (K // 32) * SRC_BYTES_PER_32[src_type]
    if src.size < need:
        raise ValueError(f"{src.size} bytes given, {need} needed")
    out = np.zeros((N // 32) * (K // 256) * 5120, dtype=np.uint8)
    _load().oracle_pack_q4_1(_ptr(src), src_type, N, K, _ptr(out))
    return out
