"""Thin Python binding of libhs (include/hs_api.h), same names as the C ABI.

Argument marshalling only: checks dtypes/devices, allocates output tensors
when the caller does not pass them, and forwards raw pointers plus the current
CUDA stream.  Every step of the path runs in the CUDA kernels of libhs.so;
there is no CPU fallback.  If the library cannot be loaded this module raises.
"""
import ctypes

import torch

from . import _build

_lib = None

HS_OK = 0
STATUS_NAMES = {0: "HS_OK", 1: "HS_ERR_INVALID_ARG", 2: "HS_ERR_MISALIGNED", 3: "HS_ERR_CAPACITY",
                4: "HS_ERR_CUDA", 5: "HS_ERR_TIMEOUT", 6: "HS_ERR_BAD_INDEX",
                7: "HS_ERR_UNSUPPORTED"}


class HSError(RuntimeError):
    def __init__(self, name, code):
        super().__init__(f"{name} failed: {STATUS_NAMES.get(code, code)}")
        self.code = code


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F32 = ctypes.c_float

_SIGS = {
    "hs_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "hs_wait_selftest": ([_I32, ctypes.c_uint64, _P, _P, _P], ctypes.c_int),
    "hs_host_device_pointer": ([_P, ctypes.POINTER(_P)], ctypes.c_int),
    "hs_normalize_indices": ([_P, _I32, _I32, _I32, _I32, _P, _P, _P, _I64, _I32, _P, _I32, _I32,
                              _I32, _I32, _P, _P, _P, _P, _P], ctypes.c_int),
    "hs_hot_state_reset": ([_P, _P, _I32, _I32, _P], ctypes.c_int),
    "hs_normalize_lookup_assign": ([_P, _I32, _I32, _I32, _I32, _P, _P, _P, _I64, _I32, _P, _I32,
                                    _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _I32, _I64,
                                    _P, _P, _P, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "hs_hot_lookup_assign": ([_P, _P, _I32, _I32, _I32, _P, _P, _P, _I32, _I64, _P, _P, _P, _P,
                              _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "hs_layer_transfer": ([_P, _P, _I64, _I64, _I32, _I32, _I32, _I32, _I64, _I64, _P, _P, _I32,
                           _I64, _I32, _I32, _P, _P], ctypes.c_int),
    "hs_swap_in": ([_P, _I64, _P, _I64, _P, _P, _P, _I32, _I32, _P, _I32, _I64, _I32, _P, _P, _P],
                   ctypes.c_int),
    "hs_hot_lookup_swap_in": ([_P, _P, _I32, _I32, _I32, _P, _P, _P, _I32, _I64, _P, _P, _P, _P,
                               _P, _P, _P, _P, _P, _P, _I64, _P, _I64, _P], ctypes.c_int),
    "hs_backup": ([_P, _P, _P, _P, _I32, _I64, _I64, _P, _P], ctypes.c_int),
    "hs_sparse_decode_workspace_bytes": ([_I32, _I32, _I32, _I32, _I32, _I32], _I64),
    "hs_sparse_decode": ([_P, _P, _P, _I64, _I64, _I64, _P, _P, _I32, _I32, _I32, _I32, _I32,
                          _I32, _F32, _P, _P, _P, _I64, _P, _P], ctypes.c_int),
    "hs_merge_states": ([_P, _P, _P, _I32, _I32, _I32, _P, _P, _P], ctypes.c_int),
    "hs_sparse_decode_partial_splits": ([_I32, _I32, _I32, _I32, _I32, _I32], _I32),
    "hs_sparse_decode_partial": ([_P, _P, _P, _I64, _I64, _I64, _P, _P, _I32, _I32, _I32, _I32,
                                  _I32, _I32, _F32, _P, _P, _P, _I32, _I32, _P, _P],
                                 ctypes.c_int),
    "hs_sparse_decode_finish": ([_P, _P, _P, _I64, _I64, _I64, _P, _P, _I32, _I32, _I32, _I32,
                                 _I32, _I32, _F32, _P, _P, _P, _I32, _I32, _P, _P, _P, _P, _P],
                                ctypes.c_int),
    "hs_sparse_decode_noalloc": ([_P, _P, _P, _I64, _I64, _I64, _P, _P, _I32, _I32, _I32, _I32,
                                  _I32, _I32, _F32, _P, _P, _P, _P], ctypes.c_int),
    "hs_fp8ds_gather": ([_P, _I64, _I64, _P, _P, _I32, _I32, _P, _P, _P, _P], ctypes.c_int),
    "hs_sparse_decode_fp8ds_workspace_bytes": ([_I32, _I32, _I32], _I64),
    "hs_swap_in_fp8ds": ([_P, _I64, _I64, _P, _I64, _P, _P, _P, _I32, _I32, _P, _I32, _I64, _I32,
                          _P, _P, _P], ctypes.c_int),
    "hs_sparse_decode_fp8ds": ([_P, _P, _I64, _I64, _P, _P, _I32, _I32, _I32, _F32, _P, _P, _P,
                                _I64, _P, _P], ctypes.c_int),
}

NOALLOC_WORKSPACE_BYTES = 8 * 1024 * 1024  # HS_NOALLOC_WORKSPACE_BYTES

EXPORTS = tuple(_SIGS)


def lib_path():
    return _build.LIB


def lib():
    """Load libhs.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _ptr(t):
    """Device-visible address of a tensor argument: a CUDA tensor's own, or
    the mapped address of a pinned host tensor (the kernels then read or
    write host memory over the link)."""
    if t is None:
        return None
    if not t.is_cuda:
        return ctypes.c_void_p(host_device_pointer(t))
    return ctypes.c_void_p(t.data_ptr())


def device_address(t):
    """Device-visible address (int) of a CUDA tensor or a pinned host tensor."""
    return _ptr(t).value


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != HS_OK:
        raise HSError(name, rc)


def _check(t, dtype, name, cuda=True):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if cuda and not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name}: must be a CUDA tensor or pinned host memory")


def wait_selftest(mode, timeout_ns, *, stream=None):
    """Bounded-wait self-test (hs_wait_selftest); returns (status, elapsed_ns)."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    _call("hs_wait_selftest", mode, timeout_ns, _ptr(status), _ptr(elapsed), _stream(stream))
    torch.cuda.synchronize()
    return int(status.item()), int(elapsed.item())


def status_string(code):
    return lib().hs_status_string(code).decode()


def host_device_pointer(t):
    """Device-visible address of a pinned host tensor."""
    if not t.is_pinned():
        raise ValueError("host memory must be pinned (pin_memory())")
    out = ctypes.c_void_p()
    _call("hs_host_device_pointer", ctypes.c_void_p(t.data_ptr()), ctypes.byref(out))
    return out.value


# ---------------------------------------------------------------------------
def normalize_indices(cand, row_req, seq_lens, block_table, page_size, *, window=0, num_sinks=0,
                      page_owner=None, num_pages, max_blocks=None, cap=None, out=None,
                      stream=None):
    """S1.  Returns (tok, slot, count, err) int32 tensors."""
    for t, n in ((cand, "cand"), (row_req, "row_req"), (seq_lens, "seq_lens"),
                 (block_table, "block_table"), (page_owner, "page_owner")):
        _check(t, torch.int32, n)
    rows, n_cand = cand.shape
    num_reqs, bt_stride = block_table.shape
    max_blocks = bt_stride if max_blocks is None else max_blocks
    cap = n_cand + window + num_sinks if cap is None else cap
    if out is None:
        dev = cand.device
        out = (torch.empty(rows, cap, dtype=torch.int32, device=dev),
               torch.empty(rows, cap, dtype=torch.int32, device=dev),
               torch.empty(rows, dtype=torch.int32, device=dev),
               torch.empty(rows, 4, dtype=torch.int32, device=dev))
    tok, slot, count, err = out
    _call("hs_normalize_indices", _ptr(cand), rows, n_cand, window, num_sinks, _ptr(row_req),
          _ptr(seq_lens), _ptr(block_table), bt_stride, max_blocks, _ptr(page_owner), num_reqs,
          num_pages, page_size, cap, _ptr(tok), _ptr(slot), _ptr(count), _ptr(err),
          _stream(stream))
    return tok, slot, count, err


def normalize_lookup_assign(cand, row_req, seq_lens, block_table, page_size, newest_slot, dgi,
                            lru, region_stride, stats, *, window=0, num_sinks=0, page_owner=None,
                            num_pages, max_blocks=None, cap=None, s1_out=None, s2_out=None,
                            stream=None):
    """S1 and S2 in one kernel (hs_normalize_lookup_assign).  Returns
    (s1_out, s2_out): (tok, slot, count, err) as normalize_indices and the
    8-tuple (hot_idx, miss_mask, miss_src, miss_dst, miss_count, err,
    hit_idx, miss_rows) as hot_lookup_assign with split lists."""
    for t, n in ((cand, "cand"), (row_req, "row_req"), (seq_lens, "seq_lens"),
                 (block_table, "block_table"), (page_owner, "page_owner"),
                 (newest_slot, "newest_slot"), (dgi, "dgi")):
        _check(t, torch.int32, n)
    _check(lru, torch.int16, "lru")
    _check(stats, torch.int64, "stats")
    rows, n_cand = cand.shape
    num_reqs, bt_stride = block_table.shape
    max_blocks = bt_stride if max_blocks is None else max_blocks
    cap = n_cand + window + num_sinks if cap is None else cap
    hot_size = dgi.shape[1]
    dev = cand.device
    i32 = dict(dtype=torch.int32, device=dev)
    if s1_out is None:
        s1_out = (torch.empty(rows, cap, **i32), torch.empty(rows, cap, **i32),
                  torch.empty(rows, **i32), torch.empty(rows, 4, **i32))
    if s2_out is None:
        s2_out = (torch.empty(rows, cap, **i32),
                  torch.empty(rows, cap, dtype=torch.uint8, device=dev),
                  torch.empty(rows, cap, **i32),
                  torch.empty(rows, cap, dtype=torch.int64, device=dev),
                  torch.empty(rows, **i32), torch.empty(rows, **i32),
                  torch.empty(rows, cap, **i32), torch.empty(rows, cap, **i32))
    tok, slot, count, err = s1_out
    hot_idx, miss_mask, miss_src, miss_dst, miss_count, lerr, hit_idx, miss_rows = s2_out
    _call("hs_normalize_lookup_assign", _ptr(cand), rows, n_cand, window, num_sinks,
          _ptr(row_req), _ptr(seq_lens), _ptr(block_table), bt_stride, max_blocks,
          _ptr(page_owner), num_reqs, num_pages, page_size, cap, _ptr(tok), _ptr(slot),
          _ptr(count), _ptr(err), _ptr(newest_slot), _ptr(dgi), _ptr(lru), hot_size,
          region_stride, _ptr(hot_idx), _ptr(miss_mask), _ptr(miss_src), _ptr(miss_dst),
          _ptr(miss_count), _ptr(stats), _ptr(lerr), _ptr(hit_idx), _ptr(miss_rows),
          _stream(stream))
    return s1_out, s2_out


def hot_state_reset(dgi, lru, stream=None):
    _check(dgi, torch.int32, "dgi")
    _check(lru, torch.int16, "lru")
    rows, hot_size = dgi.shape
    _call("hs_hot_state_reset", _ptr(dgi), _ptr(lru), rows, hot_size, _stream(stream))


def hot_lookup_assign(slot, count, newest_slot, dgi, lru, region_stride, stats, *,
                      num_real_rows=None, out=None, with_mask=True, with_split_lists=False,
                      swap=None, stream=None):
    """S2.  dgi/lru are updated in place; stats int64 [2] accumulates.
    Returns (hot_idx, miss_mask, miss_src, miss_dst, miss_count, err) and, with
    with_split_lists (or an 8-tuple `out`), also (hit_idx, miss_rows).
    swap=(host_pool_dev, host_rows, hot, row_bytes): the same kernel also
    copies the misses into the hot rows (hs_hot_lookup_swap_in)."""
    _check(slot, torch.int32, "slot")
    _check(count, torch.int32, "count")
    _check(newest_slot, torch.int32, "newest_slot")
    _check(dgi, torch.int32, "dgi")
    _check(lru, torch.int16, "lru")
    _check(stats, torch.int64, "stats")
    rows, cap = slot.shape
    hot_size = dgi.shape[1]
    if out is None:
        dev = slot.device
        out = (torch.empty(rows, cap, dtype=torch.int32, device=dev),
               torch.empty(rows, cap, dtype=torch.uint8, device=dev) if with_mask else None,
               torch.empty(rows, cap, dtype=torch.int32, device=dev),
               torch.empty(rows, cap, dtype=torch.int64, device=dev),
               torch.empty(rows, dtype=torch.int32, device=dev),
               torch.empty(rows, dtype=torch.int32, device=dev))
        if with_split_lists:
            out = out + (torch.empty(rows, cap, dtype=torch.int32, device=dev),
                         torch.empty(rows, cap, dtype=torch.int32, device=dev))
    hot_idx, miss_mask, miss_src, miss_dst, miss_count, err = out[:6]
    hit_idx, miss_rows = (out[6], out[7]) if len(out) == 8 else (None, None)
    nrr = rows if num_real_rows is None else num_real_rows
    if swap is None:
        _call("hs_hot_lookup_assign", _ptr(slot), _ptr(count), rows, cap, nrr,
              _ptr(newest_slot), _ptr(dgi), _ptr(lru), hot_size, region_stride, _ptr(hot_idx),
              _ptr(miss_mask), _ptr(miss_src), _ptr(miss_dst), _ptr(miss_count), _ptr(stats),
              _ptr(err), _ptr(hit_idx), _ptr(miss_rows), _stream(stream))
    else:
        host_pool_dev, host_rows, hot, row_bytes = swap
        _call("hs_hot_lookup_swap_in", _ptr(slot), _ptr(count), rows, cap, nrr,
              _ptr(newest_slot), _ptr(dgi), _ptr(lru), hot_size, region_stride, _ptr(hot_idx),
              _ptr(miss_mask), _ptr(miss_src), _ptr(miss_dst), _ptr(miss_count), _ptr(stats),
              _ptr(err), _ptr(hit_idx), _ptr(miss_rows), ctypes.c_void_p(host_pool_dev),
              host_rows, _ptr(hot), row_bytes, _stream(stream))
    return out


def swap_in(host_pool_dev, host_rows, hot, row_bytes, miss_src, miss_dst, miss_count, *,
            dgi=None, hot_size=0, region_stride=0, max_ctas=0, ticket=None, status=None,
            stream=None):
    """S3 SwapIn.  host_pool_dev: device-visible address (int) of the pinned pool.
    ticket: None, or int32 [2] device counters, zero on entry and left zero
    (groups claimed dynamically by the warps)."""
    _check(miss_src, torch.int32, "miss_src")
    _check(miss_dst, torch.int64, "miss_dst")
    _check(miss_count, torch.int32, "miss_count")
    _check(dgi, torch.int32, "dgi")
    _check(ticket, torch.int32, "ticket")
    _check(status, torch.int32, "status")
    if ticket is not None and ticket.numel() < 2:
        raise ValueError("ticket needs 2 int32 words")
    rows, cap = miss_src.shape
    _call("hs_swap_in", ctypes.c_void_p(host_pool_dev), host_rows, _ptr(hot), row_bytes,
          _ptr(miss_src), _ptr(miss_dst), _ptr(miss_count), rows, cap, _ptr(dgi), hot_size,
          region_stride, max_ctas, _ptr(ticket), _ptr(status), _stream(stream))


def layer_pointer_table(dev_pools):
    """Device pointer table for layer_transfer: dev_pools is a list over
    buffers (K, V; or one for MLA) of lists over layers of CUDA tensors
    [dev_tokens, ...] (row-major rows).  Build it once, outside graph capture."""
    ptrs = [t.data_ptr() for pools in dev_pools for t in pools]
    return torch.tensor(ptrs, dtype=torch.int64, device=dev_pools[0][0].device)


def layer_transfer(table, nbuf, layers, dev_tokens, row_bytes, host_pool, host_tokens,
                   src_idx, dst_idx, *, page_size, page_first, direction, max_ctas=0,
                   status=None, stream=None):
    """HiCache layer transfer (see hs_layer_transfer): table from
    layer_pointer_table; host_pool a pinned host tensor holding nbuf pools of
    host_tokens * layers rows; src_idx/dst_idx int32 or int64 CUDA tensors [n];
    direction 0 host -> device, 1 device -> host."""
    _check(table, torch.int64, "table")
    if src_idx.dtype not in (torch.int32, torch.int64) or dst_idx.dtype != src_idx.dtype:
        raise TypeError("src_idx/dst_idx: int32 or int64, the same dtype")
    _check(src_idx, src_idx.dtype, "src_idx")
    _check(dst_idx, dst_idx.dtype, "dst_idx")
    _check(status, torch.int32, "status")
    if table.numel() != nbuf * layers:
        raise ValueError("table holds nbuf * layers pointers")
    n = src_idx.numel()
    if dst_idx.numel() != n:
        raise ValueError("src_idx and dst_idx differ in length")
    hdev = host_device_pointer(host_pool)
    _call("hs_layer_transfer", _ptr(table), ctypes.c_void_p(hdev), host_tokens,
          host_tokens * layers * row_bytes, nbuf, layers, page_size, 1 if page_first else 0,
          dev_tokens, row_bytes, _ptr(src_idx), _ptr(dst_idx), src_idx.element_size(), n,
          direction, max_ctas, _ptr(status), _stream(stream))


def backup(src, src_rows, host_pool_dev, dst_slots, row_bytes, host_rows, *, status=None,
           stream=None):
    """BackUp: host_pool[dst_slots[i]] = src[src_rows[i]]."""
    _check(src_rows, torch.int64, "src_rows")
    _check(dst_slots, torch.int32, "dst_slots")
    _check(status, torch.int32, "status")
    _call("hs_backup", _ptr(src), _ptr(src_rows), ctypes.c_void_p(host_pool_dev),
          _ptr(dst_slots), dst_slots.numel(), row_bytes, host_rows, _ptr(status),
          _stream(stream))


def sparse_decode_workspace_bytes(rows, heads, kv_heads, cap, d_qk, d_v):
    return int(lib().hs_sparse_decode_workspace_bytes(rows, heads, kv_heads, cap, d_qk, d_v))


def sparse_decode(q, k_base, v_base, row_stride, kv_head_stride, num_kv_rows, kv_rows, count,
                  scale, d_v, *, out=None, lse=None, workspace=None, status=None, stream=None):
    """S4.  q bf16 [rows, heads, d_qk]; kv_rows int32 [rows, kv_heads, cap];
    count int32 [rows, kv_heads] or None.  Returns (out bf16, lse fp32)."""
    _check(q, torch.bfloat16, "q")
    _check(kv_rows, torch.int32, "kv_rows")
    _check(count, torch.int32, "count")
    _check(status, torch.int32, "status")
    rows, heads, d_qk = q.shape
    _, kv_heads, cap = kv_rows.shape
    if out is None:
        out = torch.empty(rows, heads, d_v, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(rows, heads, dtype=torch.float32, device=q.device)
    ws = sparse_decode_workspace_bytes(rows, heads, kv_heads, cap, d_qk, d_v)
    if ws > 0 and (workspace is None or workspace.numel() * workspace.element_size() < ws):
        workspace = torch.empty(ws, dtype=torch.uint8, device=q.device)
    _call("hs_sparse_decode", _ptr(q), _ptr(k_base), _ptr(v_base), row_stride, kv_head_stride,
          num_kv_rows, _ptr(kv_rows), _ptr(count), rows, cap, heads, kv_heads, d_qk, d_v,
          float(scale), _ptr(out), _ptr(lse), _ptr(workspace) if ws > 0 else None,
          workspace.numel() * workspace.element_size() if (ws > 0) else 0, _ptr(status),
          _stream(stream))
    return out, lse


FP8DS_ROW_BYTES = 656


def fp8ds_gather(kv8, kv_rows, count, *, out=None, out_ids=None, status=None, stream=None):
    """Reconstruct fp8_ds_mla rows.  kv8 uint8 [num_kv_rows, row_bytes >= 656];
    kv_rows int32 [rows, cap]; count int32 [rows] or None.  Returns (out bf16
    [rows * cap, 576], out_ids int32 [rows * cap])."""
    _check(kv8, torch.uint8, "kv8")
    _check(kv_rows, torch.int32, "kv_rows")
    _check(count, torch.int32, "count")
    _check(status, torch.int32, "status")
    rows, cap = kv_rows.shape[0], kv_rows.shape[-1]
    if out is None:
        out = torch.empty(rows * cap, 576, dtype=torch.bfloat16, device=kv_rows.device)
    if out_ids is None:
        out_ids = torch.empty(rows * cap, dtype=torch.int32, device=kv_rows.device)
    _call("hs_fp8ds_gather", _ptr(kv8), kv8.shape[1], kv8.shape[0], _ptr(kv_rows), _ptr(count),
          rows, cap, _ptr(out), _ptr(out_ids), _ptr(status), _stream(stream))
    return out, out_ids


def swap_in_fp8ds(host_pool_dev, host_rows, host_row_bytes, hot, miss_src, miss_dst,
                  miss_count, *, dgi=None, hot_size=0, region_stride=0, max_ctas=0,
                  ticket=None, status=None, stream=None):
    """S3 SwapIn from a pool of fp8_ds_mla rows (device-visible address
    host_pool_dev) into bf16 hot rows [hot_rows, 576], reconstructing as the
    copy stores each row; arguments as for swap_in."""
    _check(hot, torch.bfloat16, "hot")
    _check(miss_src, torch.int32, "miss_src")
    _check(miss_dst, torch.int64, "miss_dst")
    _check(miss_count, torch.int32, "miss_count")
    _check(dgi, torch.int32, "dgi")
    _check(ticket, torch.int32, "ticket")
    _check(status, torch.int32, "status")
    if ticket is not None and ticket.numel() < 2:
        raise ValueError("ticket needs 2 int32 words")
    rows, cap = miss_src.shape
    _call("hs_swap_in_fp8ds", ctypes.c_void_p(host_pool_dev), host_rows, host_row_bytes,
          _ptr(hot), hot.shape[0], _ptr(miss_src), _ptr(miss_dst), _ptr(miss_count), rows, cap,
          _ptr(dgi), hot_size, region_stride, max_ctas, _ptr(ticket), _ptr(status),
          _stream(stream))


def sparse_decode_fp8ds_workspace_bytes(rows, heads, cap):
    return int(lib().hs_sparse_decode_fp8ds_workspace_bytes(rows, heads, cap))


def sparse_decode_fp8ds(q, kv8, kv_rows, count, scale, *, out=None, lse=None, workspace=None,
                        status=None, stream=None):
    """S4 over fp8_ds_mla rows (MLA shape).  q bf16 [rows, heads, 576]; kv8
    uint8 [num_kv_rows, row_bytes >= 656]; kv_rows int32 [rows, 1, cap] or
    [rows, cap]; count int32 [rows] / [rows, 1] or None.  Returns (out bf16
    [rows, heads, 512], lse fp32 [rows, heads])."""
    _check(q, torch.bfloat16, "q")
    _check(kv8, torch.uint8, "kv8")
    _check(kv_rows, torch.int32, "kv_rows")
    _check(count, torch.int32, "count")
    _check(status, torch.int32, "status")
    rows, heads, _ = q.shape
    cap = kv_rows.shape[-1]
    if out is None:
        out = torch.empty(rows, heads, 512, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(rows, heads, dtype=torch.float32, device=q.device)
    ws = sparse_decode_fp8ds_workspace_bytes(rows, heads, cap)
    if workspace is None or workspace.numel() * workspace.element_size() < ws:
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=q.device)
    _call("hs_sparse_decode_fp8ds", _ptr(q), _ptr(kv8), kv8.shape[1], kv8.shape[0],
          _ptr(kv_rows), _ptr(count), rows, cap, heads, float(scale), _ptr(out), _ptr(lse),
          _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
          _stream(stream))
    return out, lse


def sparse_decode_partial_splits(rows, heads, kv_heads, cap, d_qk, d_v):
    return int(lib().hs_sparse_decode_partial_splits(rows, heads, kv_heads, cap, d_qk, d_v))


def sparse_decode_partial(q, k_base, v_base, row_stride, kv_head_stride, num_kv_rows, kv_rows,
                          count, scale, d_v, part_m, part_l, part_o, part_base, *, status=None,
                          stream=None):
    """S4 partial states into columns [part_base, part_base + P) of
    part_m/part_l fp32 [rows*heads, parts] and part_o fp32 [rows*heads, parts, d_v];
    returns P.  Combine with merge_states."""
    _check(q, torch.bfloat16, "q")
    _check(kv_rows, torch.int32, "kv_rows")
    _check(count, torch.int32, "count")
    for t, n in ((part_m, "part_m"), (part_l, "part_l"), (part_o, "part_o")):
        _check(t, torch.float32, n)
    _check(status, torch.int32, "status")
    rows, heads, d_qk = q.shape
    _, kv_heads, cap = kv_rows.shape
    parts = part_m.shape[-1]
    _call("hs_sparse_decode_partial", _ptr(q), _ptr(k_base), _ptr(v_base), row_stride,
          kv_head_stride, num_kv_rows, _ptr(kv_rows), _ptr(count), rows, cap, heads, kv_heads,
          d_qk, d_v, float(scale), _ptr(part_m), _ptr(part_l), _ptr(part_o), parts, part_base,
          _ptr(status), _stream(stream))
    return sparse_decode_partial_splits(rows, heads, kv_heads, cap, d_qk, d_v)


def sparse_decode_finish(q, k_base, v_base, row_stride, kv_head_stride, num_kv_rows, kv_rows,
                         count, scale, d_v, part_m, part_l, part_o, parts_used, *, sync=None,
                         out=None, lse=None, status=None, stream=None):
    """Attend over kv_rows, merge with partial columns [0, parts_used) and
    write the final (out bf16 [rows, heads, d_v], lse fp32 [rows, heads]).
    sync: optional int32 scratch of rows*heads words (lets the MLA kernel split
    the rows over several CTAs and merge in the last one)."""
    _check(q, torch.bfloat16, "q")
    _check(sync, torch.int32, "sync")
    _check(kv_rows, torch.int32, "kv_rows")
    _check(count, torch.int32, "count")
    for t, n in ((part_m, "part_m"), (part_l, "part_l"), (part_o, "part_o")):
        _check(t, torch.float32, n)
    _check(status, torch.int32, "status")
    rows, heads, d_qk = q.shape
    _, kv_heads, cap = kv_rows.shape
    if out is None:
        out = torch.empty(rows, heads, d_v, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(rows, heads, dtype=torch.float32, device=q.device)
    _call("hs_sparse_decode_finish", _ptr(q), _ptr(k_base), _ptr(v_base), row_stride,
          kv_head_stride, num_kv_rows, _ptr(kv_rows), _ptr(count), rows, cap, heads, kv_heads,
          d_qk, d_v, float(scale), _ptr(part_m), _ptr(part_l), _ptr(part_o), part_m.shape[-1],
          parts_used, _ptr(sync), _ptr(out), _ptr(lse), _ptr(status), _stream(stream))
    return out, lse


def merge_states(m, l, o, *, out=None, lse=None, stream=None):
    """Eq. (7) merge: m, l fp32 [n, parts] (m in log2 units); o fp32 [n, parts, d_v]."""
    for t, n in ((m, "m"), (l, "l"), (o, "o")):
        _check(t, torch.float32, n)
    n, parts, d_v = o.shape
    if out is None:
        out = torch.empty(n, d_v, dtype=torch.bfloat16, device=o.device)
    if lse is None:
        lse = torch.empty(n, dtype=torch.float32, device=o.device)
    _call("hs_merge_states", _ptr(m), _ptr(l), _ptr(o), n, parts, d_v, _ptr(out), _ptr(lse),
          _stream(stream))
    return out, lse


def sparse_decode_noalloc(q, k_base, v_base, row_stride, kv_head_stride, num_kv_rows, kv_rows,
                          count, scale, d_v, *, out, lse, status=None, stream=None):
    """S4 without a workspace argument: for callers that may not allocate
    device memory on the decode path (the library's built-in scratch array is
    used; see hs_sparse_decode_noalloc in hs_api.h).  `out` and `lse` must be
    passed in, so that this call allocates nothing."""
    _check(q, torch.bfloat16, "q")
    _check(kv_rows, torch.int32, "kv_rows")
    _check(count, torch.int32, "count")
    _check(out, torch.bfloat16, "out")
    _check(lse, torch.float32, "lse")
    _check(status, torch.int32, "status")
    rows, heads, d_qk = q.shape
    _, kv_heads, cap = kv_rows.shape
    _call("hs_sparse_decode_noalloc", _ptr(q), _ptr(k_base), _ptr(v_base), row_stride,
          kv_head_stride, num_kv_rows, _ptr(kv_rows), _ptr(count), rows, cap, heads, kv_heads,
          d_qk, d_v, float(scale), _ptr(out), _ptr(lse), _ptr(status), _stream(stream))
    return out, lse
