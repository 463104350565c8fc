// hs_lookup.cu -- S2, hot-buffer lookup keyed by global slot id, with the
// deterministic LRU slot assignment of the vLLM HiSparse walkthrough
// (hisparse_swap_in_kernel, Phase 1 .. Phase 4), and the state reset
// ("Hisparse hot cache初始化": zero-initialised buffer, recycled slots
// invalidated before reuse).
//
// GB300 design: one 1024-thread CTA per request row.  Phase 1 builds an
// open-addressing hash (4-slot buckets, load <= 1/4 where shared memory
// allows, else <= 1/2) of the row's pending slot ids in shared memory; the
// first occurrence of a repeated id is kept with atomicMin on its position,
// so repeats resolve deterministically (the walkthrough's hash overwrites on
// a repeated key, which is racy).  Phase 2 walks the LRU list with each
// thread owning a contiguous run of positions (dgi and lru staged in shared
// memory); hits and evictables are compacted in LRU order by one block-wide
// shuffle scan.  Phase 3 ranks the misses in row order with the same scan and
// hands them E[0], E[1], ...  Phase 4 writes
// E[M:] ++ E[:M] ++ hits.  Every global read is issued in one batch at the
// start, and the per-entry outputs are kept in shared memory until one
// coalesced pass at the end (hits land at random entries: storing them from
// the walk would cost one L1 wavefront per hit).  The output is bit-
// identical to the sequential definition for every thread schedule.
//
// hs_hot_lookup_swap_in is the walkthrough's single kernel (lookup, LRU,
// eviction and the row loads of Phase 5 in one CTA per request): after the
// lookup the same CTA copies its request's misses from the pinned pool into
// their hot rows, each warp two rows at a time with 16-byte loads.  It saves
// the SwapIn launch and its hand-off for steps with few misses; with many
// misses the separate SwapIn, which spreads one request's rows over many SMs
// and stages them through shared memory, is the faster copy.
#include "hs_norm_core.cuh"

namespace {

constexpr int kThreads = 1024;
constexpr int32_t kEmpty = -1;
constexpr int32_t kPend = -2;  // outv of an entry still looked for (hot rows are >= 0)
constexpr uint8_t kNone = 0, kHit = 1, kMiss = 2;
constexpr int kMaxSmem = 227 * 1024;

struct LookupArgs {
    const int32_t* slot;
    const int32_t* count;
    int32_t rows, cap, num_real_rows;
    const int32_t* newest_slot;
    int32_t* dgi;
    int16_t* lru;
    int32_t hot_size;
    int64_t region_stride;
    int32_t* hot_idx;
    uint8_t* miss_mask;
    int32_t* miss_src;
    int64_t* miss_dst;
    int32_t* miss_count;
    int64_t* stats;
    int32_t* err;
    int32_t hash_log2;
    int32_t* hit_idx;    // optional: hot_idx with the misses set to -1
    int32_t* miss_rows;  // optional: int32 copy of miss_dst
    // Fused SwapIn (hot != nullptr): rows of row_bytes from host_pool.
    const uint8_t* host_pool;
    int64_t host_rows;
    uint8_t* hot;
    int64_t row_bytes;
    // Fused S1 (kNorm): the row's candidates are normalised in the same CTA
    // (norm.cand ...; S1's outputs to norm.out_tok/out_slot/out_count/
    // err_counts) and `slot`/`count` above are not read.
    hs_norm::NormArgs norm;
    int32_t state_async;  // 1: dgi / lru rows 16-byte aligned, copied with cp.async
};

constexpr int kCopyVecs = 4;   // 16-byte vectors per lane and row: rows up to 2048 B
constexpr int kCopyRows = 2;   // rows a warp moves per round

__device__ __forceinline__ uint32_t hash_of(int32_t g, int log2n) {
    return (uint32_t(g) * 2654435761u) >> (32 - log2n);
}

// The hash is linear probing over aligned buckets of 4 slots: a key's probe
// sequence starts at the first slot of its bucket, so a lookup reads one
// bucket per 16-byte load, and at a load factor <= 1/4 almost every lookup
// ends in its first bucket (a warp then runs no divergent probe loop).
// Position of key g in the table, or -1 when absent.
__device__ __forceinline__ int find_key(const int32_t* keys, int32_t g, int log2n) {
    const uint32_t mask = (1u << log2n) - 1u;
    uint32_t b = hash_of(g, log2n) & ~3u;
    for (uint32_t probe = 0; probe <= mask; probe += 4) {
        const int4 k = *reinterpret_cast<const int4*>(keys + b);
        if (k.x == g) return int(b);
        if (k.x == kEmpty) return -1;
        if (k.y == g) return int(b + 1);
        if (k.y == kEmpty) return -1;
        if (k.z == g) return int(b + 2);
        if (k.z == kEmpty) return -1;
        if (k.w == g) return int(b + 3);
        if (k.w == kEmpty) return -1;
        b = (b + 4u) & mask;
    }
    return -1;
}

// Slot of key g, inserting it at the first empty slot of its probe sequence.
__device__ __forceinline__ int insert_key(int32_t* keys, int32_t g, int log2n) {
    const uint32_t mask = (1u << log2n) - 1u;
    uint32_t h = hash_of(g, log2n) & ~3u;
    for (uint32_t probe = 0; probe <= mask; ++probe) {
        const int32_t old = atomicCAS(&keys[h], kEmpty, g);
        if (old == kEmpty || old == g) return int(h);
        h = (h + 1u) & mask;
    }
    return -1;  // unreachable: the table holds at least 4x the keys
}

template <bool kSwap, bool kNorm>
__global__ void __launch_bounds__(kThreads) lookup_kernel(const LookupArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int scan_scratch[33];
    __shared__ int s_dup;

    const int HS = 1 << a.hash_log2;
    const int cap = a.cap;
    const int hot_size = a.hot_size;
    int32_t* keys = reinterpret_cast<int32_t*>(smem);
    int32_t* vals = keys + HS;
    int32_t* state = vals + HS;       // pending id of each entry whose outv is kPend
    int32_t* outv = state + cap;      // hot_idx value of each entry, or kPend
    int32_t* s_dgi = outv + cap;
    int16_t* s_lru = reinterpret_cast<int16_t*>(s_dgi + hot_size);
    int16_t* E = s_lru + hot_size;
    int16_t* H = E + hot_size;
    // kMiss for misses and kHit for the newest row; other hits are told by
    // outv >= 0 alone (one store per hit in the LRU walk).
    uint8_t* kind = reinterpret_cast<uint8_t*>(H + hot_size);
    // Fused S1 (kNorm): bitmap, word offsets, error counts, S1's tokens and
    // slots (swizzled, cap rounded up to 32), staged block-table row; 16-byte
    // aligned after `kind`.
    const int cap32 = kNorm ? (cap + 31) & ~31 : 0;
    uint32_t* n_bm = reinterpret_cast<uint32_t*>(
        (reinterpret_cast<uintptr_t>(kind + cap) + 15) & ~uintptr_t(15));
    int* n_wpos = reinterpret_cast<int*>(n_bm + hs_norm::kWindowWords);
    int* n_err = n_wpos + hs_norm::kWindowWords;
    int32_t* n_tok = n_err + 4;
    int32_t* n_slot = n_tok + cap32;
    int32_t* n_table = n_slot + cap32;

    hs::pdl_trigger();
    const int row = blockIdx.x;
    const int tid = threadIdx.x;
    // Before the predecessor has completed: the hash (and S1's bitmap) are
    // cleared.
    for (int h = tid * 4; h < HS; h += kThreads * 4) {
        *reinterpret_cast<int4*>(keys + h) = make_int4(kEmpty, kEmpty, kEmpty, kEmpty);
        *reinterpret_cast<int4*>(vals + h) = make_int4(INT32_MAX, INT32_MAX, INT32_MAX, INT32_MAX);
    }
    if constexpr (kNorm)
        for (int w = tid; w < hs_norm::kWindowWords; w += kThreads) n_bm[w] = 0u;
    hs::pdl_wait();
    const int32_t* g_row = a.slot + int64_t(row) * cap;
    int32_t* out = a.hot_idx + int64_t(row) * cap;
    uint8_t* mm = a.miss_mask ? a.miss_mask + int64_t(row) * cap : nullptr;
    int32_t* msrc = a.miss_src + int64_t(row) * cap;
    int64_t* mdst = a.miss_dst + int64_t(row) * cap;
    int32_t* hidx = a.hit_idx ? a.hit_idx + int64_t(row) * cap : nullptr;
    int32_t* mrow = a.miss_rows ? a.miss_rows + int64_t(row) * cap : nullptr;

    if (row >= a.num_real_rows) {  // CUDA-graph padding row
        for (int i = tid; i < cap; i += kThreads) {
            out[i] = -1;
            if (mm) mm[i] = 0;
            msrc[i] = -1;
            mdst[i] = -1;
            if (hidx) hidx[i] = -1;
            if (mrow) mrow[i] = -1;
        }
        if (tid == 0) {
            a.miss_count[row] = 0;
            a.err[row] = 0;
        }
        return;
    }
    int32_t* dgi = a.dgi + int64_t(row) * hot_size;
    int16_t* lru = a.lru + int64_t(row) * hot_size;
    const int64_t hot_base = int64_t(row) * a.region_stride;

    int n;
    const int32_t newest = a.newest_slot ? a.newest_slot[row] : -1;
    if constexpr (kNorm) {
        // The row's state lands in shared memory (16-byte cp.async) while the
        // same CTA runs S1; S1's ascending slots go straight to `state`.
        // 16-byte copies need 16-byte aligned rows on both sides (s_dgi sits
        // at 8 * HS + 8 * cap bytes: cap even; the host checks the rest).
        const bool async_ok = a.state_async &&
                              ((hs::smem_u32(s_dgi) | hs::smem_u32(s_lru)) & 15u) == 0 &&
                              ((reinterpret_cast<uintptr_t>(dgi) |
                                reinterpret_cast<uintptr_t>(lru)) & 15u) == 0;
        if (async_ok) {
            for (int j = tid * 4; j < hot_size; j += kThreads * 4)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                 hs::smem_u32(s_dgi + j)),
                             "l"(dgi + j)
                             : "memory");
            for (int j = tid * 8; j < hot_size; j += kThreads * 8)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                 hs::smem_u32(s_lru + j)),
                             "l"(lru + j)
                             : "memory");
            asm volatile("cp.async.commit_group;" ::: "memory");
        } else {
            for (int j = tid; j < hot_size; j += kThreads) {
                s_dgi[j] = dgi[j];
                s_lru[j] = lru[j];
            }
        }
        n = hs_norm::normalize_row<kThreads>(a.norm, row, a.norm.stage_table ? n_table : nullptr,
                                             n_tok, n_slot, 31, n_bm, true, n_wpos, scan_scratch,
                                             n_err);
        // S1's outputs, coalesced (the last emission is behind a barrier).
        int32_t* g_tok = a.norm.out_tok + int64_t(row) * cap;
        int32_t* g_slot = a.norm.out_slot + int64_t(row) * cap;
        for (int j = tid; j < cap; j += kThreads) {
            const int e = hs_norm::out_index(j, 31);
            g_tok[j] = j < n ? n_tok[e] : -1;
            g_slot[j] = j < n ? n_slot[e] : -1;
        }
        if (tid == 0) a.norm.out_count[row] = n;
        if (tid < 4) a.norm.err_counts[int64_t(row) * 4 + tid] = n_err[tid];
        if (async_ok) asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        // Every global read of the kernel is issued here, in one batch: the
        // row's state, its pending ids and its count.
        n = a.count ? min(max(a.count[row], 0), cap) : cap;
        for (int j = tid; j < hot_size; j += kThreads) {
            s_dgi[j] = dgi[j];
            s_lru[j] = lru[j];
        }
        for (int i = tid; i < cap; i += kThreads) state[i] = g_row[i];
    }
    if (tid == 0) s_dup = 0;
    __syncthreads();

    // Phase 1: classify entries, hash the pending ids (first occurrence wins).
    for (int i = tid; i < cap; i += kThreads) {
        int32_t g;
        if constexpr (kNorm) g = i < n ? n_slot[hs_norm::out_index(i, 31)] : -1;
        else g = i < n ? state[i] : -1;
        int32_t v = -1;
        uint8_t kd = kNone;
        if (g >= 0 && newest >= 0 && g == newest) {
            v = int32_t(hot_base + hot_size);
            kd = kHit;
        } else if (g >= 0) {
            const int h = insert_key(keys, g, a.hash_log2);
            if (h >= 0) atomicMin(&vals[h], i);
            v = kPend;
            if constexpr (kNorm) state[i] = g;
        }
        outv[i] = v;
        kind[i] = kd;
    }
    __syncthreads();
    // Repeats of an earlier pending id resolve to -1.  This runs in the
    // same phase as the LRU walk below: the walk writes only first
    // occurrences (vals[h]) and this only later ones, and a first occurrence
    // reads as pending or found here, never as a repeat.  S1's output (kNorm)
    // is a set: no repeats to look for.
    if constexpr (!kNorm) {
        int dups = 0;
        for (int i = tid; i < cap; i += kThreads) {
            if (outv[i] != kPend) continue;
            const int h = find_key(keys, state[i], a.hash_log2);
            if (h >= 0 && vals[h] != i) {
                outv[i] = -1;
                ++dups;
            }
        }
        if (dups) atomicAdd(&s_dup, dups);
    }

    // Phase 2: LRU walk, least -> most recently used.  Thread t owns the
    // contiguous positions [t*K2, t*K2 + K2); one block scan orders hits and
    // evictables exactly as a sequential walk would.  Results stay in shared
    // memory; the global outputs are written once, coalesced, at the end.
    const int K2 = (hot_size + kThreads - 1) / kThreads;  // <= 32
    uint32_t hitmask = 0;
    int nh = 0;
    const int p0 = tid * K2;
    for (int k = 0; k < K2; ++k) {
        const int pos = p0 + k;
        if (pos >= hot_size) break;
        const int16_t sl = s_lru[pos];
        if (sl < 0 || sl >= hot_size) continue;
        const int32_t cg = s_dgi[sl];
        if (cg < 0) continue;
        const int h = find_key(keys, cg, a.hash_log2);
        if (h < 0) continue;
        const int i = vals[h];
        outv[i] = int32_t(hot_base + sl);
        hitmask |= 1u << k;
        ++nh;
    }
    __syncthreads();  // every hit and repeat is marked

    // Phase 3 ranks the misses in row order: thread t owns the contiguous
    // entries [t*K3, t*K3 + K3).  One block scan serves both orders: the hit
    // count of the thread's LRU positions in the low 16 bits, its miss count
    // in the high 16 (each total is at most hot_size <= 32767).
    const int K3 = (cap + kThreads - 1) / kThreads;
    const int i0 = tid * K3;
    int nm = 0;
    for (int k = 0; k < K3; ++k) {
        const int i = i0 + k;
        if (i >= cap) break;
        nm += outv[i] == kPend;
    }
    int packed_total;
    const int packed = hs::block_excl_scan(nh | (nm << 16), scan_scratch, &packed_total);
    const int hexcl = packed & 0xffff;
    const int hits_total = packed_total & 0xffff;
    const int miss_total = packed_total >> 16;
    int m = packed >> 16;
    {
        int hp = hexcl, ep = min(p0, hot_size) - hexcl;
        for (int k = 0; k < K2; ++k) {
            const int pos = p0 + k;
            if (pos >= hot_size) break;
            const int16_t sl = s_lru[pos];
            if ((hitmask >> k) & 1u) H[hp++] = sl; else E[ep++] = sl;
        }
    }
    __syncthreads();  // E and H are complete
    const int nE = hot_size - hits_total;

    // Misses in row order take E[0], E[1], ...
    for (int k = 0; k < K3; ++k) {
        const int i = i0 + k;
        if (i >= cap) break;
        if (outv[i] != kPend) continue;
        const int32_t g = state[i];
        const int16_t sl = m < nE ? E[m] : int16_t(-1);
        if (sl >= 0 && sl < hot_size) {
            outv[i] = int32_t(hot_base + sl);
            kind[i] = kMiss;
            dgi[sl] = g;
            msrc[m] = g;
            mdst[m] = hot_base + sl;
            if (mrow) mrow[m] = int32_t(hot_base + sl);
        } else {
            outv[i] = -1;  // only reachable with a corrupted LRU list
            kind[i] = kNone;
            if (m < nE) {
                msrc[m] = -1;
                mdst[m] = -1;
                if (mrow) mrow[m] = -1;
            }
        }
        ++m;
    }
    const int M = min(miss_total, nE);
    __syncthreads();

    // Outputs, coalesced: hot_idx, hit_idx, miss_mask of every entry, and the
    // unused tails of the miss lists.
    for (int i = tid; i < cap; i += kThreads) {
        const int32_t v = outv[i];
        const uint8_t kd = v < 0 ? kNone : (kind[i] == kMiss ? kMiss : kHit);
        out[i] = v;
        if (hidx) hidx[i] = kd == kHit ? v : -1;
        if (mm) mm[i] = kd == kMiss ? 1 : 0;
        if (i >= M) {
            msrc[i] = -1;
            mdst[i] = -1;
            if (mrow) mrow[i] = -1;
        }
    }

    // Phase 4: new LRU order = E[M:] ++ E[:M] ++ hits.
    for (int j = tid; j < hot_size; j += kThreads) {
        int16_t sl;
        if (j < nE - M) sl = E[M + j];
        else if (j < nE) sl = E[j - (nE - M)];
        else sl = H[j - nE];
        lru[j] = sl;
    }
    if (tid == 0) {
        a.miss_count[row] = M;
        atomicAdd(reinterpret_cast<unsigned long long*>(a.stats),
                  static_cast<unsigned long long>(hits_total));
        atomicAdd(reinterpret_cast<unsigned long long*>(a.stats + 1),
                  static_cast<unsigned long long>(M));
        a.err[row] = s_dup;
    }
    if (!kSwap) return;

    // Phase 5 (fused): the M misses host -> hot.  The miss lists and dgi
    // were written to global memory by this CTA above.
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    const int nv = int(a.row_bytes >> 4);
    for (int m0 = warp * kCopyRows; m0 < M; m0 += kCopyRows * (kThreads / 32)) {
        uint4 buf[kCopyRows][kCopyVecs];
        int64_t dst[kCopyRows];
        bool has_src[kCopyRows];
#pragma unroll
        for (int u = 0; u < kCopyRows; ++u) {
            const int mi = m0 + u;
            dst[u] = mi < M ? mdst[mi] : -1;
            const int32_t g = mi < M ? msrc[mi] : -1;
            has_src[u] = dst[u] >= 0 && g >= 0 && int64_t(g) < a.host_rows;
            if (has_src[u]) {
                const uint4* src = reinterpret_cast<const uint4*>(a.host_pool + int64_t(g) * a.row_bytes);
#pragma unroll
                for (int k = 0; k < kCopyVecs; ++k) {
                    const int v = lane + 32 * k;
                    if (v < nv) buf[u][k] = __ldg(src + v);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyRows; ++u) {
            if (dst[u] < 0) continue;
            uint4* d = reinterpret_cast<uint4*>(a.hot + dst[u] * a.row_bytes);
#pragma unroll
            for (int k = 0; k < kCopyVecs; ++k) {
                const int v = lane + 32 * k;
                if (v < nv) d[v] = has_src[u] ? buf[u][k] : make_uint4(0, 0, 0, 0);
            }
            // No source row: the hot row is zeroed above and its slot revoked.
            if (!has_src[u] && lane == 0) {
                const int64_t sl = dst[u] - hot_base;
                if (sl >= 0 && sl < hot_size) dgi[sl] = -1;
            }
        }
    }
}

__global__ void reset_kernel(int32_t* dgi, int16_t* lru, int32_t hot_size) {
    hs::pdl_trigger();
    const int64_t base = int64_t(blockIdx.x) * hot_size;
    for (int j = threadIdx.x; j < hot_size; j += blockDim.x) {
        dgi[base + j] = -1;
        lru[base + j] = int16_t(j);
    }
}

}  // namespace

extern "C" int hs_hot_state_reset(int32_t* dgi, int16_t* lru, int32_t rows, int32_t hot_size,
                                  hs_stream_t stream) {
    if (rows < 0 || hot_size <= 0 || hot_size > 32767) return HS_ERR_INVALID_ARG;
    if (rows == 0) return HS_OK;
    if (dgi == nullptr || lru == nullptr) return HS_ERR_INVALID_ARG;
    reset_kernel<<<rows, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dgi, lru, hot_size);
    return hs_host::launch_status();
}

namespace {
template <bool kSwap, bool kNorm = false>
int lookup_launch(LookupArgs a, int32_t rows, int32_t cap, int32_t hot_size, hs_stream_t stream) {
    // Hash of load factor <= 1/4, or <= 1/2 when the larger table does not fit.
    // Fused S1: bitmap, word offsets and tokens (+ the staged block-table row).
    const size_t norm_bytes =
        kNorm ? 16 + size_t(8) * hs_norm::kWindowWords + 16 +
                    size_t(8) * ((size_t(cap) + 31) & ~size_t(31)) +
                    (a.norm.stage_table ? size_t(4) * a.norm.max_blocks : 0)
              : 0;
    const auto smem_for = [&](int l2) {
        return size_t(8) * (size_t(1) << l2) + size_t(9) * cap + size_t(10) * hot_size +
               norm_bytes;
    };
    int log2n = 6;
    while ((1 << log2n) < 4 * cap) ++log2n;
    if (smem_for(log2n) > size_t(kMaxSmem) && log2n > 6) --log2n;
    const size_t smem = smem_for(log2n);
    if (smem > size_t(kMaxSmem)) return HS_ERR_CAPACITY;
    static int smem_set[64] = {};
    const int rc = hs_host::ensure_dynamic_smem(
        reinterpret_cast<const void*>(lookup_kernel<kSwap, kNorm>), smem, smem_set);
    if (rc != HS_OK) return rc;
    a.hash_log2 = log2n;
    return hs_host::launch_pdl(lookup_kernel<kSwap, kNorm>, dim3(rows), dim3(kThreads), smem,
                               stream, a);
}
}  // namespace

extern "C" int hs_hot_lookup_assign(const int32_t* slot, const int32_t* count, int32_t rows,
                                    int32_t cap, int32_t num_real_rows,
                                    const int32_t* newest_slot, int32_t* dgi, int16_t* lru,
                                    int32_t hot_size, int64_t region_stride, int32_t* hot_idx,
                                    uint8_t* miss_mask, int32_t* miss_src, int64_t* miss_dst,
                                    int32_t* miss_count, int64_t* stats, int32_t* err,
                                    int32_t* hit_idx, int32_t* miss_rows, hs_stream_t stream) {
    if (rows < 0 || cap < 0 || hot_size <= 0 || hot_size > 32767 || num_real_rows < 0)
        return HS_ERR_INVALID_ARG;
    if (region_stride < int64_t(hot_size) + 1) return HS_ERR_INVALID_ARG;
    if (int64_t(rows) * region_stride > INT32_MAX) return HS_ERR_INVALID_ARG;
    if (cap > hot_size) return HS_ERR_CAPACITY;
    if (rows == 0) return HS_OK;
    if ((cap > 0 && slot == nullptr) || dgi == nullptr || lru == nullptr ||
        (cap > 0 && (hot_idx == nullptr || miss_src == nullptr || miss_dst == nullptr)) ||
        miss_count == nullptr || stats == nullptr || err == nullptr)
        return HS_ERR_INVALID_ARG;
    LookupArgs a{slot,     count,    rows,     cap,        num_real_rows, newest_slot,
                 dgi,      lru,      hot_size, region_stride, hot_idx,    miss_mask,
                 miss_src, miss_dst, miss_count, stats,    err,           0,
                 hit_idx,  miss_rows, nullptr, 0, nullptr, 0, {}, 0};
    return lookup_launch<false>(a, rows, cap, hot_size, stream);
}

extern "C" int hs_hot_lookup_swap_in(const int32_t* slot, const int32_t* count, int32_t rows,
                                     int32_t cap, int32_t num_real_rows,
                                     const int32_t* newest_slot, int32_t* dgi, int16_t* lru,
                                     int32_t hot_size, int64_t region_stride, int32_t* hot_idx,
                                     uint8_t* miss_mask, int32_t* miss_src, int64_t* miss_dst,
                                     int32_t* miss_count, int64_t* stats, int32_t* err,
                                     int32_t* hit_idx, int32_t* miss_rows, const void* host_pool,
                                     int64_t host_rows, void* hot, int64_t row_bytes,
                                     hs_stream_t stream) {
    if (rows < 0 || cap < 0 || hot_size <= 0 || hot_size > 32767 || num_real_rows < 0 ||
        host_rows < 0 || row_bytes <= 0)
        return HS_ERR_INVALID_ARG;
    if (row_bytes % 16 != 0) return HS_ERR_MISALIGNED;
    if (row_bytes > 16 * 32 * kCopyVecs) return HS_ERR_CAPACITY;
    if (region_stride < int64_t(hot_size) + 1) return HS_ERR_INVALID_ARG;
    if (int64_t(rows) * region_stride > INT32_MAX) return HS_ERR_INVALID_ARG;
    if (cap > hot_size) return HS_ERR_CAPACITY;
    if (rows == 0) return HS_OK;
    if ((cap > 0 && slot == nullptr) || dgi == nullptr || lru == nullptr ||
        (cap > 0 && (hot_idx == nullptr || miss_src == nullptr || miss_dst == nullptr)) ||
        miss_count == nullptr || stats == nullptr || err == nullptr || host_pool == nullptr ||
        hot == nullptr)
        return HS_ERR_INVALID_ARG;
    if (((reinterpret_cast<uintptr_t>(host_pool) | reinterpret_cast<uintptr_t>(hot)) & 15u) != 0)
        return HS_ERR_MISALIGNED;
    LookupArgs a{slot,     count,    rows,     cap,        num_real_rows, newest_slot,
                 dgi,      lru,      hot_size, region_stride, hot_idx,    miss_mask,
                 miss_src, miss_dst, miss_count, stats,    err,           0,
                 hit_idx,  miss_rows, static_cast<const uint8_t*>(host_pool), host_rows,
                 static_cast<uint8_t*>(hot), row_bytes, {}, 0};
    return lookup_launch<true>(a, rows, cap, hot_size, stream);
}

extern "C" int hs_normalize_lookup_assign(
    const int32_t* cand, int32_t rows, int32_t n_cand, int32_t window, int32_t num_sinks,
    const int32_t* row_req, const int32_t* seq_lens, const int32_t* block_table,
    int64_t bt_stride, int32_t max_blocks, const int32_t* page_owner, int32_t num_reqs,
    int32_t num_pages, int32_t page_size, int32_t cap, int32_t* out_tok, int32_t* out_slot,
    int32_t* out_count, int32_t* err_counts, const int32_t* newest_slot, int32_t* dgi,
    int16_t* lru, int32_t hot_size, int64_t region_stride, int32_t* hot_idx, uint8_t* miss_mask,
    int32_t* miss_src, int64_t* miss_dst, int32_t* miss_count, int64_t* stats, int32_t* err,
    int32_t* hit_idx, int32_t* miss_rows, hs_stream_t stream) {
    // S1's checks (as hs_normalize_indices) ...
    if (rows < 0 || n_cand < 0 || window < 0 || num_sinks < 0 || max_blocks < 0 ||
        num_reqs < 0 || num_pages < 0 || page_size <= 0 || cap < 0 || bt_stride < max_blocks)
        return HS_ERR_INVALID_ARG;
    if (int64_t(cap) < int64_t(n_cand) + window + num_sinks) return HS_ERR_CAPACITY;
    if (int64_t(num_pages) * page_size > INT32_MAX) return HS_ERR_INVALID_ARG;
    // ... and S2's (as hs_hot_lookup_assign).
    if (hot_size <= 0 || hot_size > 32767) return HS_ERR_INVALID_ARG;
    if (region_stride < int64_t(hot_size) + 1) return HS_ERR_INVALID_ARG;
    if (int64_t(rows) * region_stride > INT32_MAX) return HS_ERR_INVALID_ARG;
    if (cap > hot_size) return HS_ERR_CAPACITY;
    if (rows == 0) return HS_OK;
    if ((n_cand > 0 && cand == nullptr) || row_req == nullptr || out_tok == nullptr ||
        out_slot == nullptr || out_count == nullptr || err_counts == nullptr)
        return HS_ERR_INVALID_ARG;
    if (num_reqs > 0 && (seq_lens == nullptr || (max_blocks > 0 && block_table == nullptr)))
        return HS_ERR_INVALID_ARG;
    if (dgi == nullptr || lru == nullptr ||
        (cap > 0 && (hot_idx == nullptr || miss_src == nullptr || miss_dst == nullptr)) ||
        miss_count == nullptr || stats == nullptr || err == nullptr)
        return HS_ERR_INVALID_ARG;
    hs_norm::NormArgs na{};
    na.cand = cand;
    na.rows = rows;
    na.n_cand = n_cand;
    na.window = window;
    na.num_sinks = num_sinks;
    na.row_req = row_req;
    na.seq_lens = seq_lens;
    na.block_table = block_table;
    na.bt_stride = bt_stride;
    na.max_blocks = max_blocks;
    na.page_owner = page_owner;
    na.num_reqs = num_reqs;
    na.num_pages = num_pages;
    na.page_size = page_size;
    na.cap = cap;
    na.out_tok = out_tok;
    na.out_slot = out_slot;
    na.out_count = out_count;
    na.err_counts = err_counts;
    na.stage_table = max_blocks <= hs_norm::kMaxStagedBlocks ? 1 : 0;
    na.page_shift = -1;
    na.stage_out = 1;
    if ((page_size & (page_size - 1)) == 0) {
        int sh = 0;
        while ((1 << sh) < page_size) ++sh;
        na.page_shift = sh;
    }
    // State rows copied with 16-byte cp.async: rows of a multiple of 8 slots,
    // 16-byte aligned arrays, and an even cap (shared-memory offsets).
    const bool aligned = hot_size % 8 == 0 && cap % 2 == 0 &&
                         ((reinterpret_cast<uintptr_t>(dgi) | reinterpret_cast<uintptr_t>(lru)) &
                          15u) == 0;
    LookupArgs a{nullptr,  nullptr,  rows,     cap,        rows,       newest_slot,
                 dgi,      lru,      hot_size, region_stride, hot_idx,  miss_mask,
                 miss_src, miss_dst, miss_count, stats,    err,        0,
                 hit_idx,  miss_rows, nullptr, 0, nullptr, 0, na, aligned ? 1 : 0};
    int rc = lookup_launch<false, true>(a, rows, cap, hot_size, stream);
    if (rc == HS_ERR_CAPACITY && na.stage_table) {
        // Shared memory too small with the table staged: read it from global.
        a.norm.stage_table = 0;
        rc = lookup_launch<false, true>(a, rows, cap, hot_size, stream);
    }
    return rc;
}
