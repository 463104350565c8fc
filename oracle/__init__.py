"""The oracle: plain, slow, single-threaded fp64 CPU implementation of the
HiSparse sparse-decode step (index normalisation, hot-buffer lookup with LRU
assignment, SwapIn/BackUp, sparse attention, split-KV merge).

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg may import this package.  It shares no code with the CUDA
path in sparse_top_kv_gb300/ and never imports it.

Each wrapper takes numpy arrays (C-contiguous, the dtypes named below), calls
the C++ definition in hs_oracle.cpp through ctypes, and returns numpy arrays.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        L.hso_normalize_indices.argtypes = [P, i32, i32, i32, i32, P, P, P, i64, i32, P, i32,
                                            i32, i32, i32, P, P, P, P]
        L.hso_hot_lookup_assign.argtypes = [P, P, i32, i32, i32, P, P, P, i32, i64, P, P, P, P,
                                            P, P, P]
        L.hso_swap_in.argtypes = [P, i64, P, i64, P, P, P, i32, i32, P, i32, i64]
        L.hso_backup.argtypes = [P, P, P, P, i32, i64, i64, P]
        L.hso_sparse_decode.argtypes = [P, P, P, i64, i64, P, P, i32, i32, i32, i32, i32, i32,
                                        f64, P, P]
        L.hso_merge.argtypes = [P, P, P, i32, i32, i32, P, P, P]
        L.hso_layer_transfer.argtypes = [P, P, i64, i64, i32, i32, i32, i32, i64, i64, P, P,
                                         i32, i64, i32, P]
        L.hso_e4m3_decode.argtypes = [P, i64, P]
        L.hso_fp8ds_dequant.argtypes = [P, i64, P, i64, P]
        L.hso_swap_in_fp8ds.argtypes = [P, i64, i64, P, P, P, P, i32, i32, P, i32, i64]
        for f in ("hso_normalize_indices", "hso_hot_lookup_assign", "hso_swap_in",
                  "hso_backup", "hso_sparse_decode", "hso_merge", "hso_layer_transfer",
                  "hso_e4m3_decode", "hso_fp8ds_dequant", "hso_swap_in_fp8ds"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


class OracleError(RuntimeError):
    pass


def _check(rc, name):
    if rc != 0:
        raise OracleError(f"{name} returned {rc}")


def normalize_indices(cand, row_req, seq_lens, block_table, page_size, window=0, num_sinks=0,
                      page_owner=None, num_pages=None, cap=None):
    """S1.  cand int32 [rows, n_cand]; row_req int32 [rows]; seq_lens int32 [reqs];
    block_table int32 [reqs, max_blocks].  Returns (tok, slot, count, err)."""
    cand = _c(cand, np.int32)
    rows, n_cand = cand.shape
    row_req = _c(row_req, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    block_table = _c(block_table, np.int32)
    num_reqs, max_blocks = block_table.shape
    if num_pages is None:
        num_pages = int(block_table.max()) + 1 if block_table.size else 0
    if page_owner is not None:
        page_owner = _c(page_owner, np.int32)
    if cap is None:
        cap = n_cand + window + num_sinks
    tok = np.empty((rows, cap), np.int32)
    slot = np.empty((rows, cap), np.int32)
    count = np.empty(rows, np.int32)
    err = np.empty((rows, 4), np.int32)
    rc = lib().hso_normalize_indices(_p(cand), rows, n_cand, window, num_sinks, _p(row_req),
                                     _p(seq_lens), _p(block_table), max_blocks, max_blocks,
                                     _p(page_owner), num_reqs, num_pages, page_size, cap,
                                     _p(tok), _p(slot), _p(count), _p(err))
    _check(rc, "hso_normalize_indices")
    return tok, slot, count, err


def hot_lookup_assign(slot, count, newest_slot, dgi, lru, hot_size, region_stride,
                      num_real_rows=None, stats=None):
    """S2.  Updates dgi (int32 [rows, hot_size]) and lru (int16 [rows, hot_size])
    in place.  Returns (hot_idx, miss_mask, miss_src, miss_dst, miss_count, stats, err)."""
    slot = _c(slot, np.int32)
    rows, cap = slot.shape
    if count is not None:
        count = _c(count, np.int32)
    if newest_slot is not None:
        newest_slot = _c(newest_slot, np.int32)
    assert dgi.dtype == np.int32 and dgi.flags.c_contiguous
    assert lru.dtype == np.int16 and lru.flags.c_contiguous
    if num_real_rows is None:
        num_real_rows = rows
    hot_idx = np.empty((rows, cap), np.int32)
    miss_mask = np.empty((rows, cap), np.uint8)
    miss_src = np.empty((rows, cap), np.int32)
    miss_dst = np.empty((rows, cap), np.int64)
    miss_count = np.empty(rows, np.int32)
    if stats is None:
        stats = np.zeros(2, np.int64)
    err = np.empty(rows, np.int32)
    rc = lib().hso_hot_lookup_assign(_p(slot), _p(count), rows, cap, num_real_rows,
                                     _p(newest_slot), _p(dgi), _p(lru), hot_size, region_stride,
                                     _p(hot_idx), _p(miss_mask), _p(miss_src), _p(miss_dst),
                                     _p(miss_count), _p(stats), _p(err))
    _check(rc, "hso_hot_lookup_assign")
    return hot_idx, miss_mask, miss_src, miss_dst, miss_count, stats, err


def swap_in(host_pool, hot, row_bytes, miss_src, miss_dst, miss_count, dgi=None, hot_size=0,
            region_stride=0):
    """S3 SwapIn.  host_pool / hot: uint8 arrays (hot updated in place)."""
    miss_src = _c(miss_src, np.int32)
    miss_dst = _c(miss_dst, np.int64)
    miss_count = _c(miss_count, np.int32)
    rows, cap = miss_src.shape
    host_rows = host_pool.size // row_bytes
    rc = lib().hso_swap_in(_p(host_pool), host_rows, _p(hot), row_bytes, _p(miss_src),
                           _p(miss_dst), _p(miss_count), rows, cap, _p(dgi), hot_size,
                           region_stride)
    _check(rc, "hso_swap_in")


def backup(src, src_rows, host_pool, dst_slots, row_bytes):
    """BackUp.  host_pool[dst_slots[i]] = src[src_rows[i]]; returns bad-destination count."""
    src_rows = _c(src_rows, np.int64)
    dst_slots = _c(dst_slots, np.int32)
    bad = np.zeros(1, np.int32)
    host_rows = host_pool.size // row_bytes
    rc = lib().hso_backup(_p(src), _p(src_rows), _p(host_pool), _p(dst_slots), len(dst_slots),
                          row_bytes, host_rows, _p(bad))
    _check(rc, "hso_backup")
    return int(bad[0])


def layer_transfer(dev, host, host_tokens, row_bytes, src_idx, dst_idx, *, page_size,
                   page_first, direction):
    """HiCache layer transfer.  dev: list over buffers of lists over layers of
    uint8 arrays [dev_tokens * row_bytes] (updated in place for H2D); host:
    uint8 array of nbuf pools of host_tokens * layers rows each (updated in
    place for D2H); src_idx/dst_idx int32 or int64 [n].  Returns the number
    of skipped (buffer, layer, row) copies."""
    nbuf, layers = len(dev), len(dev[0])
    dev_tokens = dev[0][0].size // row_bytes
    ptrs = (ctypes.c_void_p * (nbuf * layers))(*[a.ctypes.data for bl in dev for a in bl])
    src_idx = np.ascontiguousarray(src_idx)
    dst_idx = np.ascontiguousarray(dst_idx, dtype=src_idx.dtype)
    ib = src_idx.dtype.itemsize
    bad = np.zeros(1, np.int64)
    rc = lib().hso_layer_transfer(ctypes.cast(ptrs, ctypes.c_void_p), _p(host), host_tokens,
                                  host_tokens * layers * row_bytes, nbuf, layers, page_size,
                                  1 if page_first else 0, dev_tokens, row_bytes, _p(src_idx),
                                  _p(dst_idx), ib, len(src_idx), direction, _p(bad))
    _check(rc, "hso_layer_transfer")
    return int(bad[0])


def sparse_decode(q, k_base, v_base, row_stride, kv_head_stride, kv_rows, count, scale,
                  d_v=None):
    """S4.  q: uint16 (bf16 bits) [rows, heads, d_qk]; k_base/v_base: uint16 flat
    arrays; kv_rows int32 [rows, kv_heads, cap]; count int32 [rows, kv_heads] or None.
    Returns (out float64 [rows, heads, d_v], lse float64 [rows, heads])."""
    q = _c(q, np.uint16)
    rows, heads, d_qk = q.shape
    kv_rows = _c(kv_rows, np.int32)
    _, kv_heads, cap = kv_rows.shape
    if count is not None:
        count = _c(count, np.int32)
    if d_v is None:
        d_v = d_qk
    out = np.empty((rows, heads, d_v), np.float64)
    lse = np.empty((rows, heads), np.float64)
    rc = lib().hso_sparse_decode(_p(q), _p(k_base), _p(v_base), row_stride, kv_head_stride,
                                 _p(kv_rows), _p(count), rows, cap, heads, kv_heads, d_qk, d_v,
                                 float(scale), _p(out), _p(lse))
    _check(rc, "hso_sparse_decode")
    return out, lse


def merge(m, l, o):
    """Eq. (7) merge.  m, l: float64 [n, parts]; o: float64 [n, parts, d_v]."""
    m = _c(m, np.float64)
    l = _c(l, np.float64)
    o = _c(o, np.float64)
    n, parts, d_v = o.shape
    mo = np.empty(n, np.float64)
    lo = np.empty(n, np.float64)
    oo = np.empty((n, d_v), np.float64)
    rc = lib().hso_merge(_p(m), _p(l), _p(o), n, parts, d_v, _p(mo), _p(lo), _p(oo))
    _check(rc, "hso_merge")
    return mo, lo, oo


FP8DS_ROW_BYTES = 656


def e4m3_decode(codes):
    """OCP FP8 E4M3 codes (uint8 array) -> float64 values (NaN for 0x7F / 0xFF)."""
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    _check(lib().hso_e4m3_decode(_p(codes), codes.size, _p(out)), "hso_e4m3_decode")
    return out


def fp8ds_dequant(rows8, ids=None):
    """fp8_ds_mla rows (uint8 [n_rows, row_bytes >= 656]) -> bf16 bits uint16
    [len(ids), 576]: latent column d = bf16(fp32(code) * fp32(scale[d // 128])),
    RoPE columns copied.  ids: row numbers (default: every row)."""
    rows8 = _c(rows8, np.uint8)
    n_rows, row_bytes = rows8.shape
    ids = np.arange(n_rows, dtype=np.int64) if ids is None else _c(ids, np.int64)
    if ids.size and (ids.min() < 0 or ids.max() >= n_rows):
        raise OracleError("fp8ds_dequant: row id out of range")
    out = np.empty((ids.size, 576), np.uint16)
    rc = lib().hso_fp8ds_dequant(_p(rows8), row_bytes, _p(ids), ids.size, _p(out))
    _check(rc, "hso_fp8ds_dequant")
    return out


def sparse_decode_fp8ds(q, rows8, kv_rows, count, scale):
    """S4 over fp8_ds_mla rows: every referenced row is reconstructed with
    fp8ds_dequant, then sparse_decode runs on those bf16 rows (K = all 576
    columns, V = the first 512).  Entries that are negative or beyond the
    rows are masked (no row).  kv_rows int32 [rows, 1, cap]; count int32
    [rows, 1] or None.  Returns (out float64 [rows, heads, 512], lse)."""
    rows8 = _c(rows8, np.uint8)
    kv_rows = _c(kv_rows, np.int32)
    ok = (kv_rows >= 0) & (kv_rows < rows8.shape[0])
    ids = np.unique(kv_rows[ok]).astype(np.int64)
    deq = fp8ds_dequant(rows8, ids)
    local = np.full(kv_rows.shape, -1, np.int32)
    local[ok] = np.searchsorted(ids, kv_rows[ok]).astype(np.int32)
    if deq.shape[0] == 0:
        deq = np.zeros((1, 576), np.uint16)
    flat = deq.reshape(-1)
    return sparse_decode(q, flat, flat, 576, 0, local, count, scale, d_v=512)


def swap_in_fp8ds(host_pool8, hot, miss_src, miss_dst, miss_count, dgi=None, hot_size=0,
                  region_stride=0):
    """S3 SwapIn from fp8_ds_mla pool rows (uint8 [host_rows, row_bytes >= 656])
    into bf16 hot rows (uint16 bits [hot_rows, 576], updated in place), each
    copied row reconstructed as in fp8ds_dequant."""
    host_pool8 = _c(host_pool8, np.uint8)
    miss_src = _c(miss_src, np.int32)
    miss_dst = _c(miss_dst, np.int64)
    miss_count = _c(miss_count, np.int32)
    assert hot.dtype == np.uint16 and hot.flags.c_contiguous and hot.shape[-1] == 576
    rows, cap = miss_src.shape
    rc = lib().hso_swap_in_fp8ds(_p(host_pool8), host_pool8.shape[0], host_pool8.shape[1],
                                 _p(hot), _p(miss_src), _p(miss_dst), _p(miss_count), rows, cap,
                                 _p(dgi), hot_size, region_stride)
    _check(rc, "hso_swap_in_fp8ds")
