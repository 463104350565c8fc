/*
 * hs_api.h -- C ABI of libhs: the HiSparse top-k sparse decode hot path on
 * GB300 (sm_103a).  One decode step is four stages:
 *
 *   S1 hs_normalize_indices   candidate union/dedup/validation, token -> slot
 *   S2 hs_hot_lookup_assign   hot-buffer lookup keyed by global slot id, LRU
 *   S3 hs_swap_in / hs_backup pinned host pool <-> HBM hot region row copies
 *   S4 hs_sparse_decode       softmax(q K_S^T scale) V_S, split-KV merged
 *
 * Sources (web pages, cited by title and section):
 *   [HS] vLLM HiSparse walkthrough (devpress.csdn.net): "Hisparse hot cache
 *        初始化", "swap_in 方法流程详解", "triton_convert_req_index_to_global_index",
 *        hisparse_swap_in_kernel Phase 1 .. Phase 5.
 *   [HC] SGLang PR "[HiCache] TMA-staged host<->device KV transfer kernel
 *        (sm_90+) - #40278": Motivation, Modifications.
 *   [PT] PaperTrace 5.1.1 "从索引到 Kernel": sections 1.1-1.2 (eqs. 1-2),
 *        3.1-3.2 (eqs. 4-7), 7.3 (eqs. 16-17, empty and illegal sets).
 *   [PA] "PagedAttention 与 RadixAttention：上游机制与海光实现对照": 1.3, 1.4.
 *
 * Conventions, for every entry point:
 *  - All buffers are caller-owned.  Device pointers are CUDA device memory;
 *    "host pool" pointers are the DEVICE-VISIBLE address of pinned host
 *    memory (see hs_host_device_pointer).  The library allocates nothing.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  The return value reports only the synchronous
 *    host-side argument checks and the launch itself.
 *  - Conditions found on the device (invalid indices, timeouts) are written
 *    to caller-provided counters or a status word, readable after the stream
 *    is synchronised.  Invalid indices are dropped and counted, never read
 *    ([PT] 7.3: never silently read page 0; a wrong-request page is an error).
 *  - Layouts are row-major and densely packed unless a stride is passed.
 */
#ifndef HS_API_H
#define HS_API_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* hs_stream_t; /* identical to cudaStream_t */

/* Status codes (return values, and the device status word). */
#define HS_OK 0
#define HS_ERR_INVALID_ARG 1  /* null pointer, negative size, overflow        */
#define HS_ERR_MISALIGNED 2   /* row_bytes % 16 != 0 or unaligned pointer     */
#define HS_ERR_CAPACITY 3     /* cap / hot_size / shared-memory limits        */
#define HS_ERR_CUDA 4         /* a CUDA runtime call or launch failed         */
#define HS_ERR_TIMEOUT 5      /* device: a bounded wait gave up               */
#define HS_ERR_BAD_INDEX 6    /* device: an index outside its buffer, skipped */
#define HS_ERR_UNSUPPORTED 7  /* a shape no kernel here implements            */

/* Human-readable name of a status code (static storage, never NULL). */
const char* hs_status_string(int status);

/* Device-visible address of pinned host memory (cudaHostGetDevicePointer).
 * host_ptr must come from cudaHostAlloc / cudaHostRegister (torch
 * pin_memory()).  Returns HS_ERR_CUDA if the memory is not mapped. */
int hs_host_device_pointer(const void* host_ptr, void** dev_ptr);

/* ---------------------------------------------------------------------------
 * S1  hs_normalize_indices -- [PT] 1.1 eq. (1) S = unique(D u W u A), 1.2
 * eq. (2) b = floor(t / B), 7.3 eq. (16)/(17); [HS]
 * triton_convert_req_index_to_global_index (slot = table[b] * B + t mod B).
 *
 * cand        int32 [rows, n_cand] dynamic candidates (token positions);
 *             -1 is padding and is skipped silently.
 * window      W: positions [max(0, T - W), T) join every row (0 = none).
 * num_sinks   A: positions [0, min(A, T)) join every row (0 = none).
 * row_req     int32 [rows]: request of each index row (several index rows
 *             may share a request, e.g. one row per KV head).
 * seq_lens    int32 [num_reqs]: T, the request's context length including
 *             the newest token; a position is causal iff 0 <= t < T.
 * block_table int32 [num_reqs, bt_stride]: logical block -> physical page;
 *             only the first max_blocks entries of a row are read.
 * page_owner  int32 [num_pages] or NULL: request that owns each page; when
 *             given, a page owned by another request is rejected.
 * cap         row capacity of the outputs; must be >= n_cand + window +
 *             num_sinks (else HS_ERR_CAPACITY), so no valid set can overflow.
 * out_tok     int32 [rows, cap]: S in ascending token order, -1 padded.
 * out_slot    int32 [rows, cap]: global slot table[t / B] * B + t mod B, -1 padded.
 * out_count   int32 [rows]: |S|.
 * err_counts  int32 [rows, 4]: rejected positions per row, by first failing
 *             check: [0] range (t < -1 or t < 0 from W/A, block >= max_blocks,
 *             page outside [0, num_pages), row_req outside [0, num_reqs)),
 *             [1] causal (t >= T), [2] owner, [3] duplicates (valid dynamic
 *             entries already in S from W, A or an earlier dynamic entry).
 * Output is bit-exact and independent of thread scheduling.
 * ------------------------------------------------------------------------- */
int hs_normalize_indices(const int32_t* cand, int32_t rows, int32_t n_cand, int32_t window,
                         int32_t num_sinks, const int32_t* row_req, const int32_t* seq_lens,
                         const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                         const int32_t* page_owner, int32_t num_reqs, int32_t num_pages,
                         int32_t page_size, int32_t cap, int32_t* out_tok, int32_t* out_slot,
                         int32_t* out_count, int32_t* err_counts, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * Hot-buffer state reset ([HS] "Hisparse hot cache初始化": the hot cache is
 * zero-initialised; the coordinator invalidates recycled slots before reuse).
 * dgi int32 [rows, hot_size] := -1 (empty); lru int16 [rows, hot_size] :=
 * 0, 1, .., hot_size-1 (identity order).  hot_size <= 32767.
 * ------------------------------------------------------------------------- */
int hs_hot_state_reset(int32_t* dgi, int16_t* lru, int32_t rows, int32_t hot_size,
                       hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * S2  hs_hot_lookup_assign -- [HS] hisparse_swap_in_kernel Phase 1 .. 4.
 *
 * Row r (one request) owns hot rows [r*region_stride, r*region_stride +
 * hot_size]; the last one (hot_base + hot_size) is reserved for the newest
 * token.  region_stride >= hot_size + 1 (the page uses hot_size + 1 rounded
 * up to 128; any larger stride is accepted).
 *
 * slot        int32 [rows, cap]: global slot ids (S1 out_slot), -1 = none.
 * count       int32 [rows] or NULL: entries i >= count[r] are treated as -1.
 * num_real_rows rows r >= num_real_rows (CUDA-graph padding) output -1 and
 *             keep their state.
 * newest_slot int32 [rows] or NULL: the newest token's slot (the engine's
 *             slot_mapping); it resolves to the reserved row and never
 *             enters dgi / lru.
 * dgi, lru    state, updated in place; lru must be a permutation of
 *             0..hot_size-1 and the valid (>= 0) dgi values of a row unique,
 *             which hs_hot_state_reset and this function maintain.
 * hot_idx     int32 [rows, cap]: hot row of each entry, or -1.
 * miss_mask   uint8 [rows, cap] or NULL: 1 where the entry was a miss.
 * miss_src    int32 [rows, cap]: global slot of miss m, in row order.
 * miss_dst    int64 [rows, cap]: hot row of miss m.
 * miss_count  int32 [rows]: M, the number of misses of row r.
 * stats       int64 [2]: {hits, misses} accumulated (atomically added).
 * err         int32 [rows]: entries dropped as repeats of an earlier entry
 *             of the row (only the first occurrence resolves).
 * hit_idx     int32 [rows, cap] or NULL: hot_idx with the misses set to -1
 *             (the rows that are already resident before the SwapIn).
 * miss_rows   int32 [rows, cap] or NULL: int32 copy of miss_dst (first
 *             miss_count[r] entries valid, the rest -1).
 * Semantics (bit-exact): walk lru from least to most recently used; a slot
 * whose dgi is among the row's pending ids is a hit; the rest, in LRU order,
 * are the evictable list E.  Misses, in row order m = 0, 1, .., take E[m].
 * New lru = E[M:] ++ E[:M] ++ hits.  Requires cap <= hot_size (capacity).
 * ------------------------------------------------------------------------- */
int hs_hot_lookup_assign(const int32_t* slot, const int32_t* count, int32_t rows, int32_t cap,
                         int32_t num_real_rows, const int32_t* newest_slot, int32_t* dgi,
                         int16_t* lru, int32_t hot_size, int64_t region_stride,
                         int32_t* hot_idx, uint8_t* miss_mask, int32_t* miss_src,
                         int64_t* miss_dst, int32_t* miss_count, int64_t* stats, int32_t* err,
                         int32_t* hit_idx, int32_t* miss_rows, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * S2 + S3  hs_hot_lookup_swap_in -- [HS] hisparse_swap_in_kernel as one
 * kernel: Phase 1 .. 4 exactly as hs_hot_lookup_assign (same arguments and
 * outputs), then Phase 5 in the same CTA: each miss row host_pool[miss_src]
 * is copied to hot[miss_dst] (a source outside [0, host_rows) zeroes the hot
 * row and revokes its slot, dgi = -1, as in hs_swap_in).  One CTA per
 * request copies that request's misses, so this suits steps with few misses
 * per request; with many, hs_hot_lookup_assign followed by hs_swap_in
 * spreads the copy over many SMs.
 * host_pool   device-visible pointer to the pinned pool, host_rows rows of
 *             row_bytes (16-byte aligned).
 * hot         device hot buffer, rows of row_bytes (16-byte aligned), at
 *             least rows * region_stride rows (the misses' destinations are
 *             the hot regions S2 assigns; no other row is written).
 * row_bytes   multiple of 16, at most 2048 (HS_ERR_CAPACITY above).
 * ------------------------------------------------------------------------- */
int hs_hot_lookup_swap_in(const int32_t* slot, const int32_t* count, int32_t rows, int32_t cap,
                          int32_t num_real_rows, const int32_t* newest_slot, int32_t* dgi,
                          int16_t* lru, int32_t hot_size, int64_t region_stride,
                          int32_t* hot_idx, uint8_t* miss_mask, int32_t* miss_src,
                          int64_t* miss_dst, int32_t* miss_count, int64_t* stats, int32_t* err,
                          int32_t* hit_idx, int32_t* miss_rows, const void* host_pool,
                          int64_t host_rows, void* hot, int64_t row_bytes, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * S1 + S2  hs_normalize_lookup_assign -- [PT] 1.1 eq. (1), 1.2 eq. (2), 7.3
 * eq. (16) and [HS] hisparse_swap_in_kernel Phase 1 .. 4 in one kernel: each
 * index row is normalised exactly as hs_normalize_indices does (same
 * arguments and outputs: out_tok, out_slot, out_count, err_counts) and its
 * slots are then looked up and assigned exactly as hs_hot_lookup_assign does
 * with slot = out_slot and count = out_count (same state and outputs; row r
 * of the index rows uses state row r, num_real_rows = rows).  One CTA per
 * row: the row's dgi / lru are copied into shared memory while S1 runs, and
 * S1's ascending set stays in shared memory for the lookup, so the two
 * stages cost one launch and no round trip through global memory.  Every
 * argument is checked as by the two calls; cap <= hot_size.
 * ------------------------------------------------------------------------- */
int hs_normalize_lookup_assign(const int32_t* cand, int32_t rows, int32_t n_cand, int32_t window,
                               int32_t num_sinks, const int32_t* row_req, const int32_t* seq_lens,
                               const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                               const int32_t* page_owner, int32_t num_reqs, int32_t num_pages,
                               int32_t page_size, int32_t cap, int32_t* out_tok,
                               int32_t* out_slot, int32_t* out_count, int32_t* err_counts,
                               const int32_t* newest_slot, int32_t* dgi, int16_t* lru,
                               int32_t hot_size, int64_t region_stride, int32_t* hot_idx,
                               uint8_t* miss_mask, int32_t* miss_src, int64_t* miss_dst,
                               int32_t* miss_count, int64_t* stats, int32_t* err,
                               int32_t* hit_idx, int32_t* miss_rows, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * S3  hs_swap_in -- [HS] Phase 5 (copy each miss row host -> hot; a source
 * outside [0, host_rows) zeroes the hot row and revokes its slot, dgi = -1),
 * [HC] Modifications (copies staged through a shared-memory ring; one TMA
 * bulk op per contiguous run).  Scattered rows are staged with 16-byte
 * cp.async by whole warps instead of per-row bulk ops.
 *
 * host_pool   device-visible pointer to the pinned host pool, host_rows rows
 *             of row_bytes each (16-byte aligned base).
 * hot         device hot buffer, rows of row_bytes.
 * row_bytes   multiple of 16 ([HS] HiSparseCoordinator rejects others).
 * miss_src/miss_dst/miss_count  as produced by hs_hot_lookup_assign.
 * dgi         int32 [rows, hot_size] or NULL: revocation target.
 * max_ctas    SMs the copy may occupy, one CTA each (0 = every SM).  A smaller budget
 *             leaves SMs to a kernel running concurrently on another stream
 *             ([HC] Motivation: the copy's SM footprint is the cost to the
 *             concurrent forward pass); a few dozen CTAs already keep enough
 *             bytes in flight to fill the host link.
 * ticket      NULL (groups of rows dealt round-robin to the warps), or int32
 *             [2] device counters, zero on entry (zero them once), that the
 *             call leaves zero: warps then claim groups one at a time, so a
 *             warp that runs ahead takes more and the copy ends together.
 *             Calls that may run at the same time need their own counters.
 * status      int32 device word or NULL: HS_ERR_TIMEOUT / HS_ERR_BAD_INDEX
 *             is stored there (first error wins) if the device hits one.
 * Destinations must be distinct within one call.
 * ------------------------------------------------------------------------- */
int hs_swap_in(const void* host_pool, int64_t host_rows, void* hot, int64_t row_bytes,
               const int32_t* miss_src, const int64_t* miss_dst, const int32_t* miss_count,
               int32_t rows, int32_t cap, int32_t* dgi, int32_t hot_size, int64_t region_stride,
               int32_t max_ctas, int32_t* ticket, int32_t* status, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * hs_backup -- [HS] overview "BackUp": after each step copy the newly
 * generated KV row to host memory.  host_pool[dst_slots[i]] := src[src_rows[i]]
 * for i < n.  src is a device buffer of rows of row_bytes; src_rows int64 [n]
 * and dst_slots int32 [n] are device arrays.  A destination of -1 is padding
 * (an inactive request of a fixed-size batch) and is skipped; any other
 * destination outside [0, host_rows) is skipped and reported as
 * HS_ERR_BAD_INDEX in *status.
 * ------------------------------------------------------------------------- */
int hs_backup(const void* src, const int64_t* src_rows, void* host_pool,
              const int32_t* dst_slots, int32_t n, int64_t row_bytes, int64_t host_rows,
              int32_t* status, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * hs_layer_transfer -- [HC] Motivation and Modifications: HiCache moves the
 * rows of cached tokens between the pinned host pool and the device's
 * per-layer pools, for every layer in one call (a pointer table), in either
 * direction.  For every buffer b < nbuf (K and V, or one buffer for MLA),
 * layer l < layers and i < n, the row of token src_idx[i] is copied to the
 * row of token dst_idx[i].  Rows are row_bytes long (a multiple of 16, at
 * most 8192).
 *
 * dev_layers  device array [nbuf * layers] (at most 4096) of device pointers: the pool of
 *             buffer b and layer l is dev_layers[b * layers + l], rows of
 *             token t at + t * row_bytes (16-byte aligned pools).
 * host_pool   device-visible address of the pinned host pool; buffer b
 *             starts host_buf_bytes * b into it (>= host_tokens * layers *
 *             row_bytes when nbuf > 1).  page_first = 0: token t of layer l
 *             at row l * host_tokens + t; page_first = 1: at row
 *             ((t / page_size) * layers + l) * page_size + t % page_size (a
 *             page's rows of one layer are contiguous; host_tokens is then a
 *             multiple of page_size).
 * src_idx, dst_idx  device arrays of n int32 (index_bytes 4) or int64 (8)
 *             token ids; the same ids serve every buffer and layer.
 * direction   0: host -> device (src ids on the host), 1: device -> host.
 * max_ctas    SMs the copy may occupy, one CTA each (0 = every SM).
 * status      int32 device word or NULL: an id outside its pool ([0,
 *             host_tokens) on the host side, [0, dev_tokens) on the device
 *             side) skips that row and stores HS_ERR_BAD_INDEX.
 * Staged through shared-memory rings: consecutive ids whose rows are one
 * contiguous run on both sides (whole pages) are one bulk copy; scattered
 * rows are 16-byte copies by whole warps.
 * ------------------------------------------------------------------------- */
int hs_layer_transfer(void* const* dev_layers, void* host_pool, int64_t host_tokens,
                      int64_t host_buf_bytes, int32_t nbuf, int32_t layers, int32_t page_size,
                      int32_t page_first, int64_t dev_tokens, int64_t row_bytes,
                      const void* src_idx, const void* dst_idx, int32_t index_bytes, int64_t n,
                      int32_t direction, int32_t max_ctas, int32_t* status, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * S4  hs_sparse_decode -- [PT] 3.1 eqs. (4)-(6) (online softmax over tiles of
 * the candidate set), 3.2 (mask before the exponent; an empty set gives a
 * zero output and LSE = -inf) and eq. (7) (split-KV merge); [PA] 1.4 (GQA:
 * one work unit per KV head serves its query-head group).
 *
 * q          bf16 [rows, heads, d_qk].
 * k_base     bf16: K element (row j, kv head g, dim d) at
 *            k_base[j * row_stride + g * kv_head_stride + d];  v_base likewise.
 *            MLA passes k_base == v_base (V = the first d_v columns of the row).
 *            Both bases 16-byte aligned; row_stride and kv_head_stride
 *            multiples of 8 elements.
 * num_kv_rows rows addressable from k_base / v_base; a kv_rows entry outside
 *            [0, num_kv_rows) is skipped and reported as HS_ERR_BAD_INDEX.
 * kv_rows    int32 [rows, kv_heads, cap]: candidate rows per (row, kv head);
 *            -1 entries are skipped.  Taken as given: pass a set (S1 output),
 *            a repeated row would be weighted twice.
 * count      int32 [rows, kv_heads] or NULL: entries j >= count are not read.
 * heads      query heads; heads % kv_heads == 0, head h reads kv head
 *            h / (heads / kv_heads).
 * scale      softmax scale (e.g. 1/sqrt(d_qk)).
 * out        bf16 [rows, heads, d_v] = sum_j softmax_j V_j (fp32 accumulate,
 *            round to nearest even).
 * lse        fp32 [rows, heads] natural-log LSE, or NULL.
 * workspace  device scratch of at least hs_sparse_decode_workspace_bytes(..)
 *            bytes (split-KV partial states, and one arrival counter per
 *            (row, kv head, head group), zeroed by the call, so that the
 *            split that finishes last merges the others in its epilogue
 *            instead of a second launch); may be NULL when that is 0.  With
 *            128 MLA heads and two splits per row, when every row's cluster
 *            of four CTAs fits on the GPU at once, the two splits merge
 *            through distributed shared memory and the size is 0.
 * status     int32 device word or NULL (HS_ERR_TIMEOUT from bounded waits,
 *            HS_ERR_BAD_INDEX from skipped rows).
 * Supported shapes: (d_qk, d_v) = (576, 512) with kv_heads == 1 and k_base
 * == v_base (MLA), or d_qk == d_v == 128 with heads / kv_heads <= 8 (GQA);
 * others return HS_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------- */
int64_t hs_sparse_decode_workspace_bytes(int32_t rows, int32_t heads, int32_t kv_heads,
                                         int32_t cap, int32_t d_qk, int32_t d_v);

int hs_sparse_decode(const void* q, const void* k_base, const void* v_base, int64_t row_stride,
                     int64_t kv_head_stride, int64_t num_kv_rows, const int32_t* kv_rows,
                     const int32_t* count,
                     int32_t rows, int32_t cap, int32_t heads, int32_t kv_heads, int32_t d_qk,
                     int32_t d_v, float scale, void* out, float* lse, void* workspace,
                     int64_t workspace_bytes, int32_t* status, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * hs_sparse_decode_partial -- S4 over a subset of a row's candidates, left as
 * unnormalised partial states to be combined with others by eq. (7)
 * (hs_merge_states).  [PT] 3.2 eq. (7): o_s must stay unnormalised until the
 * merge.  Used to attend over the rows already resident while the SwapIn of
 * the missing rows is still in flight, then over the swapped rows, and merge.
 *
 * Same inputs as hs_sparse_decode (no out / lse / workspace).  Writes, for
 * every (row, head) qh, the columns [part_base, part_base + P) of
 *   part_m fp32 [rows*heads, parts_total]      max logit, log2 units (-inf: empty)
 *   part_l fp32 [rows*heads, parts_total]      sum of 2^(s - m)      (0: empty)
 *   part_o fp32 [rows*heads, parts_total, d_v] sum of 2^(s - m) V
 * where P = hs_sparse_decode_partial_splits(rows, heads, kv_heads, cap,
 * d_qk, d_v) (every one of the P columns is written, empty ones with l = 0).
 * part_base + P > parts_total is HS_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------- */
int32_t hs_sparse_decode_partial_splits(int32_t rows, int32_t heads, int32_t kv_heads,
                                        int32_t cap, int32_t d_qk, int32_t d_v);

int hs_sparse_decode_partial(const void* q, const void* k_base, const void* v_base,
                             int64_t row_stride, int64_t kv_head_stride, int64_t num_kv_rows,
                             const int32_t* kv_rows, const int32_t* count, int32_t rows,
                             int32_t cap, int32_t heads, int32_t kv_heads, int32_t d_qk,
                             int32_t d_v, float scale, float* part_m, float* part_l,
                             float* part_o, int32_t parts_total, int32_t part_base,
                             int32_t* status, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * hs_sparse_decode_finish -- the last pass of a split computation: attend over
 * kv_rows, merge (eq. 7) with the partial states already in columns
 * [0, parts_used) of part_m / part_l / part_o (written by
 * hs_sparse_decode_partial), and write the final out (bf16 [rows, heads, d_v])
 * and lse (fp32 [rows, heads], natural log, or NULL).  Columns
 * [parts_used, parts_total) may be used as scratch: parts_total must be at
 * least parts_used + hs_sparse_decode_partial_splits(...).
 * sync: NULL, or int32 counters of rows * heads words that are zero on entry
 * (zero them once); every call that completes leaves them zero again (the
 * last split of each (row, head group) resets its counter), so consecutive
 * calls need no memset.  For the MLA shape on tensor cores, with sync
 * the new rows are split over several CTAs per (row, group of query heads);
 * each writes its partial column and the last to finish merges every column
 * in its epilogue (one launch).  Without sync (or when the split count plus
 * parts_used exceeds 8 or parts_total) one CTA per (row, head group) attends
 * and merges in its epilogue.  Other shapes merge with a second launch.
 * ------------------------------------------------------------------------- */
int hs_sparse_decode_finish(const void* q, const void* k_base, const void* v_base,
                            int64_t row_stride, int64_t kv_head_stride, int64_t num_kv_rows,
                            const int32_t* kv_rows, const int32_t* count, int32_t rows,
                            int32_t cap, int32_t heads, int32_t kv_heads, int32_t d_qk,
                            int32_t d_v, float scale, float* part_m, float* part_l,
                            float* part_o, int32_t parts_total, int32_t parts_used,
                            int32_t* sync, void* out, float* lse, int32_t* status,
                            hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * hs_sparse_decode_noalloc -- the paper has no counterpart; this is a
 * convenience of this library.
 *
 * Same arguments and results as hs_sparse_decode, minus the workspace: the
 * split-KV partial states go to a scratch array compiled into libhs
 * (HS_NOALLOC_WORKSPACE_BYTES per GPU, held by every GPU that loads the
 * library until the process exits).  It is meant for callers that must not
 * allocate device memory on the decode path -- plugin code running inside a
 * host engine that owns every device allocation, or latency-critical loops
 * where a cudaMalloc (which may synchronise the device) is not allowed.
 * No allocation happens in this call.
 *
 * - Shapes whose workspace (hs_sparse_decode_workspace_bytes) exceeds
 *   HS_NOALLOC_WORKSPACE_BYTES are rejected with HS_ERR_CAPACITY.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is kept for the life of the
 *   process: after cudaDeviceReset (or any reset of the primary context)
 *   the library's module is unloaded and the kept address is stale, so do
 *   not call this entry point again in that process.
 * - Every call on a device shares the one array, which keeps the previous
 *   call's contents (nothing in it needs to start at zero).  Calls whose
 *   executions overlap on the GPU (e.g. on two streams) race on it: order
 *   them on one stream or use hs_sparse_decode with separate workspaces.
 * ------------------------------------------------------------------------- */
#define HS_NOALLOC_WORKSPACE_BYTES (8 * 1024 * 1024)

int hs_sparse_decode_noalloc(const void* q, const void* k_base, const void* v_base,
                             int64_t row_stride, int64_t kv_head_stride, int64_t num_kv_rows,
                             const int32_t* kv_rows, const int32_t* count, int32_t rows,
                             int32_t cap, int32_t heads, int32_t kv_heads, int32_t d_qk,
                             int32_t d_v, float scale, void* out, float* lse, int32_t* status,
                             hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * hs_merge_states -- [PT] 3.2 eq. (7) / [PA] 1.4 combine, the split-KV merge
 * used inside hs_sparse_decode, exposed for testing.
 * m, l       fp32 [n, parts]: per-part maximum logit in log2 units (logit *
 *            log2 e) and the sum of 2^(s - m); l == 0 marks an empty part.
 * o          fp32 [n, parts, d_v]: unnormalised sum of 2^(s - m) V.
 * out        bf16 [n, d_v] = merged o / merged l (0 if every part is empty).
 * lse        fp32 [n] natural-log LSE (-inf if empty), or NULL.
 * ------------------------------------------------------------------------- */
int hs_merge_states(const float* m, const float* l, const float* o, int32_t n, int32_t parts,
                    int32_t d_v, void* out, float* lse, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * fp8_ds_mla rows -- [HS] the FlashMLASparseBackend cache shape and
 * FP8_DS_MLA_ROW_BYTES = 656 (512 B quantised latent + 16 B scales + 128 B
 * RoPE), the 656-byte row of the Phase 5 copy walk-through; [PT] 7.2
 * (quantised KV: the scale is applied to the stored codes before the
 * products).  One row, 656 bytes (rows may sit row_bytes >= 656 apart):
 *   bytes [0, 512)    latent columns 0..511 as OCP FP8 E4M3 codes;
 *   bytes [512, 528)  four fp32 scales; scale g covers latent columns
 *                     [128 g, 128 g + 128);
 *   bytes [528, 656)  RoPE columns 512..575 as bf16.
 * Value of latent column d: code_d * scale_{d/128} in fp32, rounded to bf16
 * (nearest, ties to even) -- the operand type of QK^T and PV.  The hot
 * buffer, SwapIn and BackUp move these rows as opaque 656-byte rows
 * (row_bytes = 656 is a multiple of 16).
 *
 * hs_fp8ds_gather -- reconstruct the selected rows into a bf16 scratch.
 * kv8        device (or mapped pinned) rows, 16-byte aligned, row_bytes apart
 *            (multiple of 16, >= 656), num_kv_rows rows.
 * kv_rows    int32 [rows, cap] row ids; entries j >= count[r] are ignored;
 *            a negative id is no row (-1 is padding); an id >= num_kv_rows
 *            is no row and sets HS_ERR_BAD_INDEX in *status.
 * count      int32 [rows] or NULL (= cap).
 * out        bf16 [rows * cap, 576], 16-byte aligned: row r * cap + j holds
 *            the reconstructed row of kv_rows[r][j] (rows with no row id and
 *            rows j >= count[r] are not written).
 * out_ids    int32 [rows * cap]: r * cap + j where a row was written, -1
 *            where kv_rows[r][j] is no row (j >= count[r] not written): the
 *            kv_rows of a hs_sparse_decode over `out`.
 * Returns HS_ERR_INVALID_ARG (negative sizes, null pointers, row_bytes <
 * 656), HS_ERR_MISALIGNED, HS_ERR_CAPACITY (rows * cap >= 2^31).
 *
 * hs_sparse_decode_fp8ds -- S4 (MLA shape: K = all 576 columns, V = the
 * first 512, kv_heads = 1) over fp8_ds_mla rows: hs_fp8ds_gather into the
 * workspace, then hs_sparse_decode over the reconstructed rows.  q, out, lse,
 * count, scale, status as for hs_sparse_decode; kv_rows int32 [rows, cap].
 * workspace  device, 256-byte aligned, at least
 *            hs_sparse_decode_fp8ds_workspace_bytes(rows, heads, cap) bytes
 *            (the bf16 scratch rows * cap * 1152 B, the ids, and
 *            hs_sparse_decode's own workspace); caller-owned, no contents
 *            need to survive between calls.
 * Returns the first failing status of the two launches (HS_ERR_CAPACITY
 * when the workspace is missing or too small).
 * ------------------------------------------------------------------------- */
int hs_fp8ds_gather(const void* kv8, int64_t row_bytes, int64_t num_kv_rows,
                    const int32_t* kv_rows, const int32_t* count, int32_t rows, int32_t cap,
                    void* out, int32_t* out_ids, int32_t* status, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * hs_swap_in_fp8ds -- S3 SwapIn ([HS] Phase 5) for a host pool of
 * fp8_ds_mla rows and a hot buffer of reconstructed bf16 rows: every miss row
 * crosses the host link in its 656-byte form (hs_swap_in's staged copy), and
 * the copy's store step writes its reconstruction (as in hs_fp8ds_gather) to
 * the hot row, so the attention reads the hot buffer as bf16 MLA rows (576
 * columns).
 * host_pool8  device-visible pointer to the pinned pool (or a device
 *             buffer), host_rows rows host_row_bytes apart (>= 656, multiple
 *             of 16, 16-byte aligned).
 * hot         device bf16 rows of 576 (1152 B), hot_rows rows.
 * miss_src/miss_dst/miss_count/rows/cap/dgi/hot_size/region_stride/max_ctas/
 * ticket      as for hs_swap_in: a source outside [0, host_rows) zeroes the
 *             hot row and revokes its slot (dgi = -1; HS_ERR_BAD_INDEX
 *             without dgi); a destination outside [0, hot_rows) is skipped
 *             with HS_ERR_BAD_INDEX.  Destinations must be distinct.
 * ------------------------------------------------------------------------- */
int hs_swap_in_fp8ds(const void* host_pool8, int64_t host_rows, int64_t host_row_bytes,
                     void* hot, int64_t hot_rows, const int32_t* miss_src,
                     const int64_t* miss_dst, const int32_t* miss_count, int32_t rows,
                     int32_t cap, int32_t* dgi, int32_t hot_size, int64_t region_stride,
                     int32_t max_ctas, int32_t* ticket, int32_t* status, hs_stream_t stream);

int64_t hs_sparse_decode_fp8ds_workspace_bytes(int32_t rows, int32_t heads, int32_t cap);

int hs_sparse_decode_fp8ds(const void* q, const void* kv8, int64_t row_bytes,
                           int64_t num_kv_rows, const int32_t* kv_rows, const int32_t* count,
                           int32_t rows, int32_t cap, int32_t heads, float scale, void* out,
                           float* lse, void* workspace, int64_t workspace_bytes_given,
                           int32_t* status, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * hs_wait_selftest -- no counterpart on the pages: a test of the bounded
 * wait that every mbarrier wait of this library goes through (a wait that
 * cannot complete reports an error instead of hanging).  One CTA waits on an
 * mbarrier:  mode 0: nothing arrives, the wait gives up after timeout_ns;
 * mode 1: the barrier completes, the wait returns at once;  mode 2: nothing
 * arrives and another warp raises the CTA's abort flag after about 20 us,
 * so the wait gives up early.  A wait that gives up stores HS_ERR_TIMEOUT in
 * *status (device int32); *elapsed_ns (device int64) receives the wait's
 * wall time.  The context stays usable afterwards.
 * ------------------------------------------------------------------------- */
int hs_wait_selftest(int32_t mode, uint64_t timeout_ns, int32_t* status, int64_t* elapsed_ns,
                     hs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HS_API_H */
