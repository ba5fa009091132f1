"""Python binding of libq4nx.so: Q4NX dequant-GEMV / GEMM on GB300 (sm_103a).

A thin ctypes layer over the C ABI in ``include/q4nx.h``.  It only marshals
arguments: device pointers of torch tensors, the current CUDA stream, output
buffers and cached zero-filled workspaces.  Every step of the computation runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and
importing this package fails loudly if ``libq4nx.so`` has not been built
(``python dequant_gemv_gb300/_build.py``).

Functions keep the C names:

    q4nx_decode(w, out=None)                     -> bf16 [N, K]
    q4nx_gemv(w, x, out=None, out_dtype="bf16")  -> [N]
    q4nx_gemm_m64(w, X, out=None, out_dtype=...) -> [M, N]
    q4nx_repack_q4k(chunks, rows, cols, out=None)-> uint8 q4_1 chunks
    q4nx_argmax(logits, out=None)                -> int32 [M]

``w`` is a :class:`Weight`: a uint8 CUDA tensor of chunk bytes plus kind, rows
and cols (the tile grid of the "Q4NX chunks" section of the 1bit engine
"NPU engine" page).
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

Q4NX_Q4_1, Q4NX_Q4_K, Q4NX_Q8_KR, Q4NX_Q8_BLK = 1, 2, 3, 4
Q4NX_OUT_BF16, Q4NX_OUT_F32 = 0, 1
# statuses of include/q4nx.h
(Q4NX_OK, Q4NX_E_NULL, Q4NX_E_KIND, Q4NX_E_SHAPE, Q4NX_E_SHORT, Q4NX_E_ALIGN, Q4NX_E_M, Q4NX_E_WORKSPACE,
 Q4NX_E_UNSUPPORTED, Q4NX_E_CUDA, Q4NX_E_DEVICE_TIMEOUT, Q4NX_E_DTYPE) = range(12)
KINDS = {"q4_1": Q4NX_Q4_1, "q4_k": Q4NX_Q4_K, "q8_kr": Q4NX_Q8_KR, "q8_blk": Q4NX_Q8_BLK}

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libq4nx.so")


class Q4NXError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {q4nx_status_str(status)} (status {status})")


class q4nx_weight(ctypes.Structure):
    _fields_ = [("chunks_dev", ctypes.c_void_p), ("bytes", ctypes.c_uint64), ("kind", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class q4nx_gemv_item(ctypes.Structure):
    _fields_ = [("w", q4nx_weight), ("x_dev", ctypes.c_void_p), ("y_dev", ctypes.c_void_p)]


Q4NX_MAX_BATCH = 256


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python dequant_gemv_gb300/_build.py` "
                          "(there is no fallback path)")
    lib = ctypes.CDLL(LIB_PATH)
    P, U64, I, I64 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int64
    W = ctypes.POINTER(q4nx_weight)
    sig = {
        "q4nx_chunk_bytes": ([I], U64),
        "q4nx_status_str": ([I], ctypes.c_char_p),
        "q4nx_abi_version": ([], I),
        "q4nx_decode": ([W, P, U64, P], I),
        "q4nx_gemv": ([W, P, P, I, P, U64, P], I),
        "q4nx_gemv_workspace": ([W], U64),
        "q4nx_gemv_top1": ([W, P, P, P, U64, P], I),
        "q4nx_gemv_top1_key": ([W, P, I64, P, P, U64, P], I),
        "q4nx_gemv_batch": ([ctypes.POINTER(q4nx_gemv_item), I, I, P, U64, P], I),
        "q4nx_gemv_batch_workspace": ([ctypes.POINTER(q4nx_gemv_item), I], U64),
        "q4nx_gemm_m64": ([W, P, I, P, I, P, U64, P], I),
        "q4nx_gemm_workspace": ([W, I], U64),
        "q4nx_repack_q4k": ([P, U64, I64, I64, P, U64, P], I),
        "q4nx_pack_q4_1": ([I, P, U64, I64, I64, P, U64, P], I),
        "q4nx_argmax": ([P, I, I64, P, P], I),
        "q4nx_check": ([P, P], I),
        "q4nx_gemv_noalloc": ([W, P, P, I, P], I),
        "q4nx_noalloc_scratch_bytes": ([], U64),
        "q4nx_check_noalloc": ([P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()
EXPORTS = ("q4nx_chunk_bytes", "q4nx_status_str", "q4nx_abi_version", "q4nx_decode", "q4nx_gemv",
           "q4nx_gemv_workspace", "q4nx_gemv_top1", "q4nx_gemv_top1_key", "q4nx_gemv_batch", "q4nx_gemv_batch_workspace", "q4nx_gemm_m64", "q4nx_gemm_workspace", "q4nx_repack_q4k", "q4nx_pack_q4_1", "q4nx_argmax",
           "q4nx_check", "q4nx_gemv_noalloc", "q4nx_noalloc_scratch_bytes", "q4nx_check_noalloc")


def q4nx_chunk_bytes(kind: int) -> int:
    return int(lib.q4nx_chunk_bytes(kind))


def q4nx_status_str(status: int) -> str:
    return lib.q4nx_status_str(status).decode()


@dataclass
class Weight:
    """Chunk bytes (uint8 CUDA tensor, row-major over the tile grid) of a rows x cols weight."""
    chunks: torch.Tensor
    kind: int
    rows: int
    cols: int

    def c(self) -> q4nx_weight:
        t = self.chunks
        return q4nx_weight(t.data_ptr(), t.numel() * t.element_size(), int(self.kind), 0, int(self.rows),
                           int(self.cols))

    @property
    def device(self) -> torch.device:
        return self.chunks.device

    def tile_rows(self, tr0: int, count: int) -> "Weight":
        """The contiguous tile-row range [tr0, tr0+count) as a weight of its own."""
        tc = self.cols // 256
        cb = q4nx_chunk_bytes(self.kind)
        return Weight(self.chunks[tr0 * tc * cb:(tr0 + count) * tc * cb], self.kind, count * 32, self.cols)

    def row_shard(self, rank: int, world: int) -> tuple["Weight", int]:
        """Rank `rank`'s share of the rows when `world` devices split the weight by
        tile rows (contiguous, sizes within one tile row of each other): the
        shard as a weight of its own and its first global row."""
        tr0, tr1 = shard_tile_rows(self.rows // 32, rank, world)
        return self.tile_rows(tr0, tr1 - tr0), tr0 * 32


def _stream(dev: torch.device) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _check(status: int, where: str):
    if status != 0:
        raise Q4NXError(status, where)


def _cuda(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# Workspaces: zero-filled once.  The GEMV family (q4nx_gemv, _gemv_top1,
# _gemv_batch) leaves its workspace zero-filled after every call and relies on
# that; the GEMM leaves partial tiles behind, so the two families never share
# one.  One per (family, device, stream); calls on one stream are ordered, so
# they never overlap.
_ws_lock = threading.Lock()
_ws: dict[tuple[str, int, int], torch.Tensor] = {}
WS_FAMILIES = ("gemv", "gemm")


def workspace(device: torch.device, nbytes: int, family: str = "gemv") -> torch.Tensor:
    if family not in WS_FAMILIES:
        raise ValueError(f"unknown workspace family {family!r}")
    key = (family, device.index if device.index is not None else torch.cuda.current_device(), _stream(device))
    with _ws_lock:
        t = _ws.get(key)
        if t is None or t.numel() < nbytes:
            t = torch.zeros(max(nbytes, 1 << 16), dtype=torch.uint8, device=device)
            _ws[key] = t
        return t


def q4nx_decode(w: Weight, out: torch.Tensor | None = None) -> torch.Tensor:
    _cuda(w.chunks, "chunks")
    with torch.cuda.device(w.device):
        if out is None:
            out = torch.empty((w.rows, w.cols), dtype=torch.bfloat16, device=w.device)
        _cuda(out, "out")
        cw = w.c()
        _check(lib.q4nx_decode(ctypes.byref(cw), out.data_ptr(), out.numel() * out.element_size(),
                               _stream(w.device)), "q4nx_decode")
    return out


def _out_code(out_dtype) -> int:
    if out_dtype in ("bf16", torch.bfloat16, Q4NX_OUT_BF16):
        return Q4NX_OUT_BF16
    if out_dtype in ("f32", "fp32", torch.float32, Q4NX_OUT_F32):
        return Q4NX_OUT_F32
    raise ValueError(f"unknown out_dtype {out_dtype!r}")


def q4nx_gemv(w: Weight, x: torch.Tensor, out: torch.Tensor | None = None, out_dtype="bf16",
              ws: torch.Tensor | None = None) -> torch.Tensor:
    _cuda(w.chunks, "chunks")
    _cuda(x, "x")
    if x.dtype != torch.bfloat16 or x.numel() != w.cols:
        raise ValueError("x must be bf16 with cols elements")
    code = _out_code(out_dtype)
    with torch.cuda.device(w.device):
        if out is None:
            out = torch.empty(w.rows, dtype=torch.bfloat16 if code == Q4NX_OUT_BF16 else torch.float32,
                              device=w.device)
        _cuda(out, "out")
        cw = w.c()
        need = int(lib.q4nx_gemv_workspace(ctypes.byref(cw)))
        if ws is None:
            ws = workspace(w.device, need)
        _check(lib.q4nx_gemv(ctypes.byref(cw), x.data_ptr(), out.data_ptr(), code, ws.data_ptr(),
                             ws.numel(), _stream(w.device)), "q4nx_gemv")
    return out


def q4nx_gemv_top1(w: Weight, x: torch.Tensor, out: torch.Tensor | None = None,
                   ws: torch.Tensor | None = None) -> torch.Tensor:
    """int32 [1]: the row of the largest fp32 output of w @ x (lowest row on ties; a NaN wins)."""
    _cuda(w.chunks, "chunks")
    _cuda(x, "x")
    if x.dtype != torch.bfloat16 or x.numel() != w.cols:
        raise ValueError("x must be bf16 with cols elements")
    with torch.cuda.device(w.device):
        if out is None:
            out = torch.empty(1, dtype=torch.int32, device=w.device)
        _cuda(out, "out")
        cw = w.c()
        need = int(lib.q4nx_gemv_workspace(ctypes.byref(cw)))
        if ws is None:
            ws = workspace(w.device, need)
        _check(lib.q4nx_gemv_top1(ctypes.byref(cw), x.data_ptr(), out.data_ptr(), ws.data_ptr(), ws.numel(),
                                  _stream(w.device)), "q4nx_gemv_top1")
    return out


def q4nx_gemv_top1_key(w: Weight, x: torch.Tensor, row_base: int = 0, out: torch.Tensor | None = None,
                       ws: torch.Tensor | None = None) -> torch.Tensor:
    """int64 [1]: this shard's top-1 key (q4nx.h), rows numbered from row_base;
    the keys of all shards combine by a MAX reduction (top1_key_row decodes)."""
    _cuda(w.chunks, "chunks")
    _cuda(x, "x")
    if x.dtype != torch.bfloat16 or x.numel() != w.cols:
        raise ValueError("x must be bf16 with cols elements")
    with torch.cuda.device(w.device):
        if out is None:
            out = torch.empty(1, dtype=torch.int64, device=w.device)
        _cuda(out, "out")
        cw = w.c()
        need = int(lib.q4nx_gemv_workspace(ctypes.byref(cw)))
        if ws is None:
            ws = workspace(w.device, need)
        _check(lib.q4nx_gemv_top1_key(ctypes.byref(cw), x.data_ptr(), int(row_base), out.data_ptr(), ws.data_ptr(),
                                      ws.numel(), _stream(w.device)), "q4nx_gemv_top1_key")
    return out


# ---- host side of the sharded lm_head (no GPU work) ----

def shard_tile_rows(tile_rows: int, rank: int, world: int) -> tuple[int, int]:
    """[first, end) tile rows of `rank` when `world` devices split `tile_rows` tile rows."""
    if not 0 <= rank < world:
        raise ValueError("rank outside 0..world-1")
    return tile_rows * rank // world, tile_rows * (rank + 1) // world


def top1_key(value: float, row: int) -> int:
    """The key format of q4nx_gemv_top1_key for an fp32 `value` at global `row`
    (for combining keys on the host and for tests of the exchange)."""
    import struct

    v = float(value)
    if v != v:
        ord_ = 0xFFFFFFFF
    else:
        b = struct.unpack("<I", struct.pack("<f", 0.0 if v == 0.0 else v))[0]   # rounds to fp32
        ord_ = (~b & 0xFFFFFFFF) if b & 0x80000000 else (b | 0x80000000)
    key = (ord_ << 32) | (0xFFFFFFFF - row)
    key ^= 1 << 63
    return key - (1 << 64) if key >= 1 << 63 else key


def top1_key_row(key) -> int:
    """Global row of a (combined) top-1 key."""
    return 0xFFFFFFFF - (int(key) & 0xFFFFFFFF)


class GemvBatch:
    """A prepared batch of independent GEMVs of one chunk kind (one launch).

    items: list of (Weight, x, y) with x bf16 [cols] and y [rows] of out_dtype,
    all CUDA tensors on one device.  The ctypes array is built once; call()
    launches on the current stream (capturable in a CUDA graph)."""

    def __init__(self, items, out_dtype="bf16", ws: torch.Tensor | None = None):
        if not 1 <= len(items) <= Q4NX_MAX_BATCH:
            raise ValueError(f"a batch holds 1..{Q4NX_MAX_BATCH} items")
        self.code = _out_code(out_dtype)
        self.items = list(items)
        arr = (q4nx_gemv_item * len(items))()
        for i, (w, x, y) in enumerate(items):
            _cuda(x, "x")
            _cuda(y, "y")
            arr[i].w = w.c()
            arr[i].x_dev = x.data_ptr()
            arr[i].y_dev = y.data_ptr()
        self.arr = arr
        self.device = items[0][0].device
        self.need = int(lib.q4nx_gemv_batch_workspace(arr, len(items)))
        self.ws = ws if ws is not None else workspace(self.device, self.need)

    def __call__(self):
        _check(lib.q4nx_gemv_batch(self.arr, len(self.items), self.code, self.ws.data_ptr(), self.ws.numel(),
                                   _stream(self.device)), "q4nx_gemv_batch")


def q4nx_gemv_batch(items, out_dtype="bf16", ws: torch.Tensor | None = None):
    """Run a list of (Weight, x, y) GEMVs of one kind in one launch; returns the y tensors."""
    with torch.cuda.device(items[0][0].device):
        GemvBatch(items, out_dtype, ws)()
    return [y for _, _, y in items]


def q4nx_gemv_noalloc(w: Weight, x: torch.Tensor, out: torch.Tensor | None = None, out_dtype="bf16") -> torch.Tensor:
    """q4nx_gemv with the library's built-in scratch: allocates nothing on the device
    (the output tensor, when not given, is the only allocation, made here by torch)."""
    _cuda(w.chunks, "chunks")
    _cuda(x, "x")
    code = _out_code(out_dtype)
    with torch.cuda.device(w.device):
        if out is None:
            out = torch.empty(w.rows, dtype=torch.bfloat16 if code == Q4NX_OUT_BF16 else torch.float32,
                              device=w.device)
        _cuda(out, "out")
        cw = w.c()
        _check(lib.q4nx_gemv_noalloc(ctypes.byref(cw), x.data_ptr(), out.data_ptr(), code, _stream(w.device)),
               "q4nx_gemv_noalloc")
    return out


def q4nx_check_noalloc(device=None) -> None:
    """Raise Q4NXError if a bounded in-kernel wait of an earlier q4nx_gemv_noalloc
    call on this device gave up (synchronises the current stream)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib.q4nx_check_noalloc(_stream(dev)), "q4nx_check_noalloc")


def q4nx_gemm_m64(w: Weight, X: torch.Tensor, out: torch.Tensor | None = None, out_dtype="bf16",
                  ws: torch.Tensor | None = None) -> torch.Tensor:
    _cuda(w.chunks, "chunks")
    _cuda(X, "X")
    if X.dtype != torch.bfloat16 or X.dim() != 2 or X.shape[1] != w.cols:
        raise ValueError("X must be bf16 [M, cols]")
    M = X.shape[0]
    code = _out_code(out_dtype)
    with torch.cuda.device(w.device):
        if out is None:
            out = torch.empty((M, w.rows), dtype=torch.bfloat16 if code == Q4NX_OUT_BF16 else torch.float32,
                              device=w.device)
        _cuda(out, "out")
        cw = w.c()
        need = int(lib.q4nx_gemm_workspace(ctypes.byref(cw), M))
        if ws is None:
            ws = workspace(w.device, need, "gemm")
        _check(lib.q4nx_gemm_m64(ctypes.byref(cw), X.data_ptr(), M, out.data_ptr(), code, ws.data_ptr(),
                                 ws.numel(), _stream(w.device)), "q4nx_gemm_m64")
    return out


Q4NX_SRC_Q4_0, Q4NX_SRC_Q4_1, Q4NX_SRC_Q8_0, Q4NX_SRC_F32, Q4NX_SRC_F16, Q4NX_SRC_BF16 = 1, 2, 3, 4, 5, 6


def q4nx_pack_q4_1(src: torch.Tensor, src_type: int, rows: int, cols: int,
                   out: torch.Tensor | None = None) -> torch.Tensor:
    """q4_1 chunk bytes of a GGUF-type rows x cols tensor (`src`: its bytes, or a dense tensor)."""
    _cuda(src, "src")
    with torch.cuda.device(src.device):
        if out is None:
            out = torch.empty((rows // 32) * (cols // 256) * 5120, dtype=torch.uint8, device=src.device)
        _cuda(out, "out")
        _check(lib.q4nx_pack_q4_1(src_type, src.data_ptr(), src.numel() * src.element_size(), rows, cols,
                                  out.data_ptr(), out.numel() * out.element_size(), _stream(src.device)),
               "q4nx_pack_q4_1")
    return out


def q4nx_repack_q4k(chunks: torch.Tensor, rows: int, cols: int, out: torch.Tensor | None = None) -> torch.Tensor:
    _cuda(chunks, "chunks")
    with torch.cuda.device(chunks.device):
        if out is None:
            out = torch.empty((rows // 32) * (cols // 256) * 5120, dtype=torch.uint8, device=chunks.device)
        _cuda(out, "out")
        _check(lib.q4nx_repack_q4k(chunks.data_ptr(), chunks.numel(), rows, cols, out.data_ptr(), out.numel(),
                                   _stream(chunks.device)), "q4nx_repack_q4k")
    return out


def q4nx_argmax(logits: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    _cuda(logits, "logits")
    if logits.dtype != torch.float32:
        raise ValueError("logits must be fp32")
    L = logits.reshape(-1, logits.shape[-1])
    with torch.cuda.device(logits.device):
        if out is None:
            out = torch.empty(L.shape[0], dtype=torch.int32, device=logits.device)
        _cuda(out, "out")
        _check(lib.q4nx_argmax(L.data_ptr(), L.shape[0], L.shape[1], out.data_ptr(), _stream(logits.device)),
               "q4nx_argmax")
    return out


def q4nx_check(ws: torch.Tensor | None = None, device=None) -> None:
    """Raise if a bounded in-kernel wait of an earlier call on this workspace (default:
    this stream's GEMV and GEMM workspaces) gave up.  A workspace that reports
    such an error must be zero-filled before its next use: the default ones
    are zero-filled here before raising; a caller's own `ws` is left to the
    caller."""
    if ws is not None:
        _check(lib.q4nx_check(ws.data_ptr(), _stream(ws.device)), "q4nx_check")
        return
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    for family in WS_FAMILIES:
        w = workspace(device, 16, family)
        st = lib.q4nx_check(w.data_ptr(), _stream(w.device))
        if st != Q4NX_OK:
            with torch.cuda.device(w.device):
                w.zero_()
        _check(st, "q4nx_check")
