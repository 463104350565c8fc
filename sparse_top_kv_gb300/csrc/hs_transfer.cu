// hs_transfer.cu -- S3, SwapIn (pinned host pool -> HBM hot region) and
// BackUp (HBM -> pinned host pool) row copies.
//
// Semantics: vLLM HiSparse walkthrough, hisparse_swap_in_kernel Phase 5 (one
// row of row_bytes per miss; a source id outside the host pool zeroes the hot
// row and revokes the slot, dgi = -1) and the overview's BackUp interface.
// Design prior art: SGLang PR "[HiCache] TMA-staged host<->device KV transfer
// kernel (sm_90+)", Motivation and Modifications: a register-staging copy is
// bounded by bytes in flight, while cp.async.bulk keeps a deep shared-memory
// ring in flight with one issuing thread; contiguous runs become ONE bulk op,
// per-row ops remain only for scattered rows.
//
// GB300 design: a grid of 2-warp CTAs.  Work items are (list, segment of
// `seg` rows); each CTA derives the item -> list map from the device-side
// counts (no host round trip) and takes items blockIdx.x, +gridDim.x, ...
// Warp 0 prefetches the item's indices into shared memory, then its lane 0
// plans a stage (greedy run detection: consecutive rows whose source and
// destination both advance by one row are one piece), arms the stage's full
// mbarrier with the byte count and issues one cp.async.bulk global->shared
// per piece.  Warp 1 lane 0 waits on the full barrier, issues one
// cp.async.bulk shared->global per piece, waits until the ring slot has been
// read, and releases it on the empty barrier.  Every wait is bounded in wall
// time; a timeout stores HS_ERR_TIMEOUT in the status word, and each role
// drains its own copies in flight (again bounded) before leaving.
#include "hs_common.cuh"

namespace {

constexpr int kStages = 4;
constexpr uint32_t kStageBytes = 32768;
constexpr int kMaxPieces = 64;
constexpr int kMaxSeg = 64;
constexpr int kThreads = 64;

struct Piece {
    int64_t src_byte;
    int64_t dst_byte;
    uint32_t smem_off;
    uint32_t bytes;
};

struct StageMeta {
    int32_t npieces;  // -1: end of work
    int32_t pad[3];
    Piece p[kMaxPieces];
};

struct XferArgs {
    const uint8_t* src_base;
    uint8_t* dst_base;
    int64_t row_bytes;
    int64_t src_limit;  // rows of the source buffer (ids outside are invalid), or -1
    int64_t dst_limit;  // rows of the destination buffer, or -1
    const int32_t* src32;
    const int64_t* src64;
    const int32_t* dst32;
    const int64_t* dst64;
    const int32_t* counts;  // per list, or nullptr: every list has fixed_count rows
    int32_t fixed_count;
    int32_t nlists;
    int32_t list_stride;
    int32_t seg;
    int32_t* dgi;  // swap-in revocation target, or nullptr
    int32_t zero_bad_src;  // 1: a missing source zeroes the destination (SwapIn)
    int32_t hot_size;
    int64_t region_stride;
    int32_t* status;
    uint64_t timeout_ns;
};

struct Smem {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int32_t abort;
    int32_t pad;
    int64_t idx_src[kMaxSeg];
    int64_t idx_dst[kMaxSeg];
    StageMeta meta[kStages];
};

constexpr size_t kRingBytes = size_t(kStages) * kStageBytes;

__device__ __forceinline__ int64_t list_count(const XferArgs& a, int r) {
    const int64_t c = a.counts ? int64_t(a.counts[r]) : int64_t(a.fixed_count);
    return c < 0 ? 0 : (c > a.list_stride ? a.list_stride : c);
}

__global__ void __launch_bounds__(kThreads) xfer_kernel(const XferArgs a) {
    extern __shared__ __align__(128) unsigned char dsmem[];
    // Layout: [ring kStages * kStageBytes][Smem][prefix int32 nlists+1]
    unsigned char* ring = dsmem;
    Smem& S = *reinterpret_cast<Smem*>(dsmem + kRingBytes);
    int32_t* prefix = reinterpret_cast<int32_t*>(dsmem + kRingBytes + sizeof(Smem));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            hs::mbar_init(&S.full[s], 1);
            hs::mbar_init(&S.empty[s], 1);
        }
        S.abort = 0;
        hs::fence_mbar_init();
    }
    // Items per list -> prefix sums (warp 0).
    if (warp == 0) {
        int running = 0;
        if (lane == 0) prefix[0] = 0;
        for (int base = 0; base < a.nlists; base += 32) {
            const int r = base + lane;
            const int items = r < a.nlists ? int((list_count(a, r) + a.seg - 1) / a.seg) : 0;
            const int incl = hs::warp_incl_scan(items);
            if (r < a.nlists) prefix[r + 1] = running + incl;
            running += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    __syncthreads();
    const int total_items = prefix[a.nlists];
    const int64_t rb = a.row_bytes;
    volatile int* abort_flag = &S.abort;

    if (warp == 0) {
        // ------------------------------ loader ------------------------------
        int stage = 0;
        uint32_t ring_par = 0;  // flips each time the ring wraps
        bool pending[kStages];
        uint32_t pend_par[kStages];
#pragma unroll
        for (int s = 0; s < kStages; ++s) pending[s] = false, pend_par[s] = 0;
        int ok = 1;
        for (int item = blockIdx.x; item < total_items && ok; item += gridDim.x) {
            // List of this item: the last r with prefix[r] <= item.
            int lo = 0, hi = a.nlists;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (prefix[mid] <= item) lo = mid; else hi = mid;
            }
            const int r = lo;
            const int64_t m0 = int64_t(item - prefix[r]) * a.seg;
            const int nrows = int(hs::min64(list_count(a, r), m0 + a.seg) - m0);
            // Index prefetch into shared memory (whole warp, coalesced).
            const int64_t off = int64_t(r) * a.list_stride + m0;
            for (int k = lane; k < nrows; k += 32) {
                S.idx_src[k] = a.src32 ? int64_t(a.src32[off + k]) : a.src64[off + k];
                S.idx_dst[k] = a.dst32 ? int64_t(a.dst32[off + k]) : a.dst64[off + k];
            }
            __syncwarp();
            if (lane == 0) {
                int k = 0;
                while (k < nrows) {
                    if (!hs::mbar_wait_bounded(&S.empty[stage], ring_par ^ 1u, a.timeout_ns,
                                               abort_flag)) {
                        ok = 0;
                        break;
                    }
                    pending[stage] = false;
                    StageMeta& M = S.meta[stage];
                    int np = 0;
                    uint32_t used = 0;
                    while (k < nrows && np < kMaxPieces) {
                        const int64_t g = S.idx_src[k];
                        const int64_t d = S.idx_dst[k];
                        const bool src_ok = g >= 0 && (a.src_limit < 0 || g < a.src_limit);
                        const bool dst_ok = d >= 0 && (a.dst_limit < 0 || d < a.dst_limit);
                        if (!dst_ok) {  // nothing may be written there
                            hs::set_status(a.status, HS_ERR_BAD_INDEX);
                            ++k;
                            continue;
                        }
                        if (!src_ok && !a.zero_bad_src) {
                            hs::set_status(a.status, HS_ERR_BAD_INDEX);
                            ++k;
                            continue;
                        }
                        if (!src_ok) {
                            // No source row: zero the destination and revoke the slot.
                            uint4* z = reinterpret_cast<uint4*>(a.dst_base + d * rb);
                            for (int64_t v = 0; v < rb / 16; ++v) z[v] = make_uint4(0, 0, 0, 0);
                            if (a.dgi != nullptr) {
                                const int64_t s = d - int64_t(r) * a.region_stride;
                                if (s >= 0 && s < a.hot_size)
                                    a.dgi[int64_t(r) * a.hot_size + s] = -1;
                            } else {
                                hs::set_status(a.status, HS_ERR_BAD_INDEX);
                            }
                            ++k;
                            continue;
                        }
                        const int64_t room = (int64_t(kStageBytes) - used) / rb;
                        if (room <= 0) break;
                        int64_t run = 1;
                        while (k + run < nrows && run < room && S.idx_src[k + run] == g + run &&
                               S.idx_dst[k + run] == d + run &&
                               (a.src_limit < 0 || g + run < a.src_limit) &&
                               (a.dst_limit < 0 || d + run < a.dst_limit))
                            ++run;
                        M.p[np].src_byte = g * rb;
                        M.p[np].dst_byte = d * rb;
                        M.p[np].smem_off = used;
                        M.p[np].bytes = uint32_t(run * rb);
                        ++np;
                        used += uint32_t(run * rb);
                        k += int(run);
                    }
                    M.npieces = np;
                    unsigned char* buf = ring + size_t(stage) * kStageBytes;
                    // One arrival (count 1) carrying the byte count, then the copies.
                    hs::mbar_arrive_expect_tx(&S.full[stage], used);
                    for (int p = 0; p < np; ++p)
                        hs::bulk_g2s(buf + M.p[p].smem_off, a.src_base + M.p[p].src_byte,
                                     M.p[p].bytes, &S.full[stage]);
                    pending[stage] = true;
                    pend_par[stage] = ring_par;
                    if (++stage == kStages) {
                        stage = 0;
                        ring_par ^= 1u;
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        if (lane == 0) {
            if (ok) {
                // End-of-work marker for the storer.
                if (hs::mbar_wait_bounded(&S.empty[stage], ring_par ^ 1u, a.timeout_ns,
                                          abort_flag)) {
                    S.meta[stage].npieces = -1;
                    hs::mbar_arrive(&S.full[stage]);
                } else {
                    ok = 0;
                }
            }
            if (!ok) {
                hs::set_status(a.status, HS_ERR_TIMEOUT);
                S.abort = 1;
                // Drain the loads this thread issued (bounded).
                for (int s = 0; s < kStages; ++s)
                    if (pending[s])
                        hs::mbar_wait_bounded(&S.full[s], pend_par[s], a.timeout_ns, nullptr);
            }
        }
    } else if (lane == 0) {
        // ------------------------------ storer ------------------------------
        int stage = 0;
        uint32_t ring_par = 0;
        for (;;) {
            if (!hs::mbar_wait_bounded(&S.full[stage], ring_par, a.timeout_ns, abort_flag)) {
                if (!*abort_flag) hs::set_status(a.status, HS_ERR_TIMEOUT);
                S.abort = 1;
                break;
            }
            const StageMeta& M = S.meta[stage];
            const int np = M.npieces;
            if (np < 0) break;
            const unsigned char* buf = ring + size_t(stage) * kStageBytes;
            for (int p = 0; p < np; ++p)
                hs::bulk_s2g(a.dst_base + M.p[p].dst_byte, buf + M.p[p].smem_off, M.p[p].bytes);
            hs::bulk_commit();
            hs::bulk_wait_read_all();
            hs::mbar_arrive(&S.empty[stage]);
            if (++stage == kStages) {
                stage = 0;
                ring_par ^= 1u;
            }
        }
        hs::bulk_wait_all();
    }
}

size_t xfer_smem_bytes(int nlists) {
    return kRingBytes + sizeof(Smem) + sizeof(int32_t) * (size_t(nlists) + 1);
}

constexpr int kMaxSmem = 227 * 1024;

int launch_xfer(const XferArgs& a, int64_t max_items, hs_stream_t stream) {
    const size_t smem = xfer_smem_bytes(a.nlists);
    if (smem > size_t(kMaxSmem)) return HS_ERR_CAPACITY;
    static int smem_set[64] = {};
    const int rc = hs_host::ensure_dynamic_smem(reinterpret_cast<const void*>(xfer_kernel), smem,
                                                smem_set);
    if (rc != HS_OK) return rc;
    const int64_t grid = hs::max64(1, hs::min64(max_items, hs_host::num_sms()));
    xfer_kernel<<<int(grid), kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    return hs_host::launch_status();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int hs_swap_in(const void* host_pool, int64_t host_rows, void* hot, int64_t row_bytes,
                          const int32_t* miss_src, const int64_t* miss_dst,
                          const int32_t* miss_count, int32_t rows, int32_t cap, int32_t* dgi,
                          int32_t hot_size, int64_t region_stride, int32_t* status,
                          hs_stream_t stream) {
    if (rows < 0 || cap < 0 || host_rows < 0 || row_bytes <= 0) return HS_ERR_INVALID_ARG;
    if (row_bytes % 16 != 0) return HS_ERR_MISALIGNED;
    if (row_bytes > int64_t(kStageBytes)) return HS_ERR_CAPACITY;
    if (rows == 0 || cap == 0) return HS_OK;
    if (host_pool == nullptr || hot == nullptr || miss_src == nullptr || miss_dst == nullptr ||
        miss_count == nullptr)
        return HS_ERR_INVALID_ARG;
    if (!aligned16(host_pool) || !aligned16(hot)) return HS_ERR_MISALIGNED;
    if (dgi != nullptr && (hot_size <= 0 || region_stride < hot_size)) return HS_ERR_INVALID_ARG;
    XferArgs a{};
    a.src_base = static_cast<const uint8_t*>(host_pool);
    a.dst_base = static_cast<uint8_t*>(hot);
    a.row_bytes = row_bytes;
    a.src_limit = host_rows;
    a.dst_limit = region_stride > 0 ? int64_t(rows) * region_stride : -1;
    a.src32 = miss_src;
    a.dst64 = miss_dst;
    a.counts = miss_count;
    a.nlists = rows;
    a.list_stride = cap;
    a.seg = kMaxSeg;
    a.dgi = dgi;
    a.zero_bad_src = 1;
    a.hot_size = hot_size;
    a.region_stride = region_stride;
    a.status = status;
    a.timeout_ns = hs::kWaitTimeoutNs;
    const int64_t max_items = int64_t(rows) * ((cap + kMaxSeg - 1) / kMaxSeg);
    return launch_xfer(a, max_items, stream);
}

extern "C" int hs_backup(const void* src, const int64_t* src_rows, void* host_pool,
                         const int32_t* dst_slots, int32_t n, int64_t row_bytes,
                         int64_t host_rows, int32_t* status, hs_stream_t stream) {
    if (n < 0 || host_rows < 0 || row_bytes <= 0) return HS_ERR_INVALID_ARG;
    if (row_bytes % 16 != 0) return HS_ERR_MISALIGNED;
    if (row_bytes > int64_t(kStageBytes)) return HS_ERR_CAPACITY;
    if (n == 0) return HS_OK;
    if (src == nullptr || src_rows == nullptr || host_pool == nullptr || dst_slots == nullptr)
        return HS_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(host_pool)) return HS_ERR_MISALIGNED;
    constexpr int kBackupSeg = 8;
    XferArgs a{};
    a.src_base = static_cast<const uint8_t*>(src);
    a.dst_base = static_cast<uint8_t*>(host_pool);
    a.row_bytes = row_bytes;
    a.src_limit = -1;
    a.dst_limit = host_rows;
    a.src64 = src_rows;
    a.dst32 = dst_slots;
    a.counts = nullptr;
    a.fixed_count = n;
    a.nlists = 1;
    a.list_stride = n;
    a.seg = kBackupSeg;
    a.status = status;
    a.timeout_ns = hs::kWaitTimeoutNs;
    return launch_xfer(a, (int64_t(n) + kBackupSeg - 1) / kBackupSeg, stream);
}
