"""Host-side checks of the C-ABI library (no GPU needed).

libq4nx.so loads, exports every function include/q4nx.h declares, and
rejects bad arguments with the documented status before touching the GPU
(the "Q4NX chunks" section of the 1bit engine "NPU engine" page: refuse an
unknown chunk size or a tensor shorter than its layout needs).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q():
    import __graft_entry__

    __graft_entry__._load_build_module().build()
    import dequant_gemv_gb300

    return dequant_gemv_gb300


def _declared():
    src = open(os.path.join(ROOT, "include", "q4nx.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(q4nx_[a-z0-9_]+)\s*\(", src)))


def test_binding_constants_match_the_header(q):
    """The binding's status, kind and output-type numbers are the header's."""
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "q4nx.h")).read(), flags=re.S)
    vals = {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(Q4NX_[A-Z0-9_]+)\s*=\s*(\d+)", src)}
    for name in ("Q4NX_OK", "Q4NX_E_NULL", "Q4NX_E_KIND", "Q4NX_E_SHAPE", "Q4NX_E_SHORT", "Q4NX_E_ALIGN",
                 "Q4NX_E_M", "Q4NX_E_WORKSPACE", "Q4NX_E_UNSUPPORTED", "Q4NX_E_CUDA", "Q4NX_E_DEVICE_TIMEOUT",
                 "Q4NX_E_DTYPE", "Q4NX_Q4_1", "Q4NX_Q4_K", "Q4NX_Q8_KR", "Q4NX_Q8_BLK", "Q4NX_OUT_BF16",
                 "Q4NX_OUT_F32"):
        assert getattr(q, name) == vals[name], name


def test_exports_every_declared_symbol(q):
    names = _declared()
    assert "q4nx_gemv" in names and "q4nx_gemm_m64" in names and len(names) >= 11
    lib = ctypes.CDLL(q.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(q.EXPORTS)


def test_chunk_bytes_and_strings(q):
    assert [q.q4nx_chunk_bytes(k) for k in (1, 2, 3, 4)] == [5120, 4736, 8704, 8704]
    assert q.q4nx_chunk_bytes(0) == 0 and q.q4nx_chunk_bytes(9) == 0
    assert q.lib.q4nx_abi_version() == 1
    for s in range(0, 12):
        assert q.q4nx_status_str(s) != "unknown status"
    assert q.q4nx_status_str(99) == "unknown status"


def _w(q, ptr=16, nbytes=5120, kind=1, rows=32, cols=256, reserved=0):
    return q.q4nx_weight(ptr, nbytes, kind, reserved, rows, cols)


def test_validation_statuses(q):
    L = q.lib
    by = ctypes.byref
    P = 0x10000                      # a fake, 16-byte aligned "device" address: never dereferenced
    # decode
    assert L.q4nx_decode(None, P, 1 << 20, None) == 1
    assert L.q4nx_decode(by(_w(q, ptr=None)), P, 1 << 20, None) == 1
    assert L.q4nx_decode(by(_w(q, ptr=P, kind=7)), P, 1 << 20, None) == 2
    assert L.q4nx_decode(by(_w(q, ptr=P, reserved=1)), P, 1 << 20, None) == 2
    assert L.q4nx_decode(by(_w(q, ptr=P, rows=31)), P, 1 << 20, None) == 3
    assert L.q4nx_decode(by(_w(q, ptr=P, cols=255)), P, 1 << 20, None) == 3
    assert L.q4nx_decode(by(_w(q, ptr=P, rows=0)), P, 1 << 20, None) == 3
    assert L.q4nx_decode(by(_w(q, ptr=P, rows=-32)), P, 1 << 20, None) == 3
    assert L.q4nx_decode(by(_w(q, ptr=P, nbytes=5119)), P, 1 << 20, None) == 4
    assert L.q4nx_decode(by(_w(q, ptr=P, kind=3, nbytes=5120)), P, 1 << 20, None) == 4
    assert L.q4nx_decode(by(_w(q, ptr=P + 8)), P, 1 << 20, None) == 5
    assert L.q4nx_decode(by(_w(q, ptr=P)), None, 1 << 20, None) == 1
    assert L.q4nx_decode(by(_w(q, ptr=P)), P, 32 * 256 * 2 - 1, None) == 4
    assert L.q4nx_decode(by(_w(q, ptr=P)), P + 4, 1 << 20, None) == 5
    # gemv
    w = _w(q, ptr=P)
    need = L.q4nx_gemv_workspace(by(w))
    assert need >= 16
    assert L.q4nx_gemv(by(w), None, P, 0, P, need, None) == 1
    assert L.q4nx_gemv(by(w), P, P, 2, P, need, None) == 11
    assert L.q4nx_gemv(by(w), P, P, 0, None, need, None) == 7
    assert L.q4nx_gemv(by(w), P, P, 0, P, need - 1, None) == 7
    assert L.q4nx_gemv(by(w), P + 2, P, 0, P, need, None) == 5
    # GGUF-type pack: unknown source type, shape, short buffers, alignment
    assert L.q4nx_pack_q4_1(9, P, 1 << 30, 32, 256, P, 5120, None) == 2
    assert L.q4nx_pack_q4_1(1, P, 1 << 30, 31, 256, P, 5120, None) == 3
    assert L.q4nx_pack_q4_1(1, P, 32 * 8 * 18 - 1, 32, 256, P, 5120, None) == 4
    assert L.q4nx_pack_q4_1(1, P, 32 * 8 * 18, 32, 256, P, 5119, None) == 4
    assert L.q4nx_pack_q4_1(1, P + 2, 1 << 20, 32, 256, P, 5120, None) == 5
    assert L.q4nx_pack_q4_1(1, None, 1 << 20, 32, 256, P, 5120, None) == 1
    # fused top-1: same weight checks; the index pointer needs 4-byte alignment
    assert L.q4nx_gemv_top1(by(w), P, None, P, need, None) == 1
    assert L.q4nx_gemv_top1(by(w), P, P + 2, P, need, None) == 5
    assert L.q4nx_gemv_top1(by(w), P, P, P, need - 1, None) == 7
    # sharded top-1 key: 8-byte aligned key, row base within int32 rows, workspace
    assert L.q4nx_gemv_top1_key(by(w), P, 0, None, P, need, None) == 1
    assert L.q4nx_gemv_top1_key(by(w), P, 0, P + 4, P, need, None) == 5
    assert L.q4nx_gemv_top1_key(by(w), P, -1, P, P, need, None) == 3
    assert L.q4nx_gemv_top1_key(by(w), P, 2**31 - 32, P, P, need, None) == 3
    assert L.q4nx_gemv_top1_key(by(w), P, 0, P, P, need - 1, None) == 7
    assert L.q4nx_gemv_workspace(by(_w(q, rows=33))) == 0
    # gemv batch
    items = (q.q4nx_gemv_item * 3)()
    for i in range(3):
        items[i].w = _w(q, ptr=P, rows=64, cols=512, nbytes=4 * 5120)
        items[i].x_dev = P
        items[i].y_dev = P
    bneed = L.q4nx_gemv_batch_workspace(items, 3)
    assert bneed >= L.q4nx_gemv_workspace(by(items[0].w))
    assert L.q4nx_gemv_batch_workspace(items, 0) == 0
    assert L.q4nx_gemv_batch(None, 3, 0, P, bneed, None) == 1
    assert L.q4nx_gemv_batch(items, 0, 0, P, bneed, None) == 3
    assert L.q4nx_gemv_batch(items, 257, 0, P, bneed, None) == 3
    assert L.q4nx_gemv_batch(items, 3, 0, P, bneed - 1, None) == 7
    items[2].w = _w(q, ptr=P, kind=2, rows=64, cols=512, nbytes=4 * 4736)
    assert L.q4nx_gemv_batch(items, 3, 0, P, bneed, None) == 2
    items[2].w = _w(q, ptr=P, rows=64, cols=512, nbytes=4 * 5120 - 1)
    assert L.q4nx_gemv_batch(items, 3, 0, P, bneed, None) == 4
    items[2].w = _w(q, ptr=P, rows=64, cols=512, nbytes=4 * 5120)
    items[1].y_dev = P + 2
    assert L.q4nx_gemv_batch(items, 3, 0, P, bneed, None) == 5
    # gemm
    gneed = L.q4nx_gemm_workspace(by(w), 64)
    assert L.q4nx_gemm_workspace(by(w), 0) == 0 and L.q4nx_gemm_workspace(by(w), 65) == 0
    assert L.q4nx_gemm_m64(by(w), P, 0, P, 0, P, gneed, None) == 6
    assert L.q4nx_gemm_m64(by(w), P, 65, P, 0, P, gneed, None) == 6
    assert L.q4nx_gemm_m64(by(_w(q, ptr=P, kind=2, nbytes=4736)), P, 64, P, 0, P, gneed, None) == 8
    assert L.q4nx_gemm_m64(by(w), P, 64, P, 0, None, gneed, None) == 7
    # repack
    assert L.q4nx_repack_q4k(None, 4736, 32, 256, P, 5120, None) == 1
    assert L.q4nx_repack_q4k(P, 4735, 32, 256, P, 5120, None) == 4
    assert L.q4nx_repack_q4k(P, 4736, 32, 256, P, 5119, None) == 4
    assert L.q4nx_repack_q4k(P, 4736, 32, 250, P, 5120, None) == 3
    assert L.q4nx_repack_q4k(P + 1, 4736, 32, 256, P, 5120, None) == 5
    # argmax
    assert L.q4nx_argmax(None, 1, 10, P, None) == 1
    assert L.q4nx_argmax(P, 0, 10, P, None) == 3
    assert L.q4nx_argmax(P, 1, 0, P, None) == 3
    assert L.q4nx_argmax(P, 65536, 10, P, None) == 3
    assert L.q4nx_argmax(P + 2, 1, 10, P, None) == 5
    assert L.q4nx_check(None, None) == 1


def test_noalloc_statuses_equal_gemv_statuses(q):
    """q4nx_gemv_noalloc checks its arguments as q4nx_gemv does (the same shared
    checks, in the same order): every bad argument set gives both entry points
    the same status, before any CUDA call."""
    L = q.lib
    by = ctypes.byref
    P = 0x10000
    need = L.q4nx_gemv_workspace(by(_w(q, ptr=P)))
    cases = [
        (None, P, P, 0),                                        # NULL weight
        (_w(q, ptr=None), P, P, 0),                             # NULL chunks
        (_w(q, ptr=P, kind=7), P, P, 0),                        # unknown kind
        (_w(q, ptr=P, kind=2, nbytes=4735), P, P, 0),           # short Q4_K
        (_w(q, ptr=P, reserved=3), P, P, 0),                    # reserved field
        (_w(q, ptr=P, rows=33), P, P, 0),                       # shape
        (_w(q, ptr=P, cols=512), P, P, 0),                      # buffer too short for 32x512
        (_w(q, ptr=P + 8), P, P, 0),                            # misaligned chunks
        (_w(q, ptr=P), None, P, 0),                             # NULL x
        (_w(q, ptr=P), P, None, 0),                             # NULL y
        (_w(q, ptr=P), P, P, 5),                                # unknown dtype
        (_w(q, ptr=P), P + 4, P, 0),                            # misaligned x
        (_w(q, ptr=P), P, P + 2, 1),                            # misaligned y
    ]
    for w, x, y, od in cases:
        wp = None if w is None else by(w)
        a = L.q4nx_gemv(wp, x, y, od, P, need, None)
        b = L.q4nx_gemv_noalloc(wp, x, y, od, None)
        assert a == b != 0, (w, x, y, od, a, b)


def test_weight_tile_rows_is_pointer_arithmetic(q):
    import torch

    t = torch.zeros(6 * 5120, dtype=torch.uint8)
    W = q.Weight(t, 1, 96, 512)
    sub = W.tile_rows(1, 2)
    assert sub.rows == 64 and sub.cols == 512
    assert sub.chunks.data_ptr() == t.data_ptr() + 2 * 5120 and sub.chunks.numel() == 4 * 5120
