"""The oracle's HiSparse decode step: the same stage order as the GPU path,
each stage the plain CPU definition of hs_oracle.cpp.  TEST INFRASTRUCTURE ONLY.

State: a hot buffer (uint8 rows), dgi, lru and the {hits, misses} counters;
the host pool is the caller's array (BackUp writes into it).  With
row_format "fp8ds" the pool and the new rows are fp8_ds_mla rows, the hot
buffer holds their bf16 reconstruction (fp8ds_dequant, swap_in_fp8ds), and
BackUp writes the new rows' 656 bytes to the pool.
"""
import numpy as np

from . import (backup, fp8ds_dequant, hot_lookup_assign, normalize_indices, sparse_decode,
               swap_in, swap_in_fp8ds)


class OracleHiSparse:
    def __init__(self, *, host_pool_u8, block_table, num_pages, page_size, top_k, hot_size,
                 region_stride, row_bytes, scale, d_v=512, window=0, num_sinks=0,
                 row_format="bf16"):
        self.fp8 = row_format == "fp8ds"
        self.pool = host_pool_u8.reshape(-1)  # uint8 view; backups write into it
        self.block_table = np.ascontiguousarray(block_table, np.int32)
        self.R = self.block_table.shape[0]
        self.num_pages, self.page_size = num_pages, page_size
        self.top_k, self.hot_size, self.region_stride = top_k, hot_size, region_stride
        self.row_bytes, self.scale, self.d_v = row_bytes, scale, d_v
        self.window, self.num_sinks = window, num_sinks
        hot_bytes = 576 * 2 if self.fp8 else row_bytes
        self.hot = np.zeros((self.R * region_stride, hot_bytes), np.uint8)
        self.dgi = np.full((self.R, hot_size), -1, np.int32)
        self.lru = np.tile(np.arange(hot_size, dtype=np.int16), (self.R, 1))
        self.stats = np.zeros(2, np.int64)
        self.row_req = np.arange(self.R, dtype=np.int32)

    def newest_slots(self, newest_pos, seq_lens):
        _, slot, _, _ = normalize_indices(np.asarray(newest_pos, np.int32).reshape(-1, 1),
                                          self.row_req, seq_lens, self.block_table,
                                          self.page_size, num_pages=self.num_pages)
        return slot[:, 0].copy()

    def step(self, cand, seq_lens, newest_slot, new_row_u8, q_bits, attend_rows=None):
        """Returns a dict with every stage's outputs; attention is computed for
        the request rows in `attend_rows` (all when None)."""
        R, hs_, rs = self.R, self.hot_size, self.region_stride
        reserved = np.arange(R, dtype=np.int64) * rs + hs_
        if self.fp8:
            new_row_u8 = np.ascontiguousarray(new_row_u8, np.uint8).reshape(R, self.row_bytes)
            self.hot[reserved] = fp8ds_dequant(new_row_u8).view(np.uint8)
        else:
            self.hot[reserved] = new_row_u8
        tok, slot, count, err = normalize_indices(cand, self.row_req, seq_lens, self.block_table,
                                                  self.page_size, window=self.window,
                                                  num_sinks=self.num_sinks,
                                                  num_pages=self.num_pages)
        hot_idx, mm, msrc, mdst, mcount, self.stats, lerr = hot_lookup_assign(
            slot, count, newest_slot, self.dgi, self.lru, hs_, rs, stats=self.stats)
        if self.fp8:
            swap_in_fp8ds(self.pool.reshape(-1, self.row_bytes), self.hot.view(np.uint16),
                          msrc, mdst, mcount, dgi=self.dgi, hot_size=hs_, region_stride=rs)
            bad = backup(new_row_u8.reshape(-1), np.arange(R, dtype=np.int64), self.pool,
                         newest_slot, self.row_bytes)
        else:
            swap_in(self.pool, self.hot.reshape(-1), self.row_bytes, msrc, mdst, mcount,
                    dgi=self.dgi, hot_size=hs_, region_stride=rs)
            bad = backup(self.hot.reshape(-1), reserved, self.pool, newest_slot, self.row_bytes)
        rows = np.arange(R) if attend_rows is None else np.asarray(attend_rows, dtype=np.int64)
        hot_bf16 = self.hot.view(np.uint16).reshape(-1)
        width = self.hot.shape[1] // 2
        out, lse = sparse_decode(q_bits[rows], hot_bf16, hot_bf16, width, 0,
                                 hot_idx[rows][:, None, :], count[rows][:, None], self.scale,
                                 d_v=self.d_v)
        return dict(tok=tok, slot=slot, count=count, err=err, hot_idx=hot_idx, miss_mask=mm,
                    miss_src=msrc, miss_dst=mdst, miss_count=mcount, lookup_err=lerr,
                    backup_bad=bad, out=out, lse=lse, rows=rows)
