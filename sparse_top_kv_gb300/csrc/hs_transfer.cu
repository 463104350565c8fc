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
// GB300 design: every warp works on its own.  Work is cut into groups of up
// to 32 consecutive rows of one list (as many as fill an 8 KB stage); each
// CTA derives the group -> list map from the device-side counts (no host
// round trip) and its warps take groups round-robin over the grid.  A warp
// keeps a ring of 3 stages in shared memory: a group whose rows are one
// contiguous run in both source and destination is ONE cp.async.bulk
// global->shared op armed on the stage's mbarrier with its byte count;
// scattered rows are fetched with 16-byte cp.async by all 32 lanes (measured
// on GB300: a per-row bulk op from host memory costs ~0.5 us of the SM's
// TMA unit, so per-row bulk loads cap a CTA near 2 GB/s, while 16-byte
// cp.async from all lanes keeps dozens of rows in flight).  A landed stage is
// written out by the warp's lanes with 16-byte stores (the destinations are
// scattered slots, and plain stores need no completion tracking), two groups
// behind the loads so that three stages stay in flight per warp.  The
// mbarrier waits are bounded in wall time (HS_ERR_TIMEOUT on expiry).
//
// fp8_ds_mla rows (hs_swap_in_fp8ds): the 656-byte rows cross the link as
// they are and the store step writes each staged row's bf16 reconstruction
// (1152 bytes: E4M3 code x fp32 group scale, rounded to bf16; RoPE copied)
// to its hot row, so the hot buffer is read by the attention as bf16 rows.
#include "hs_common.cuh"
#include "hs_fp8.cuh"

namespace {

// Each warp owns a ring of kWS stages of kStageBytes in shared memory and
// copies groups of up to kMaxGroup consecutive rows of one list.  Eight
// warps' rings (192 KB) fill an SM's shared memory, so a CTA budget is an SM
// budget: the copy never takes a slice of many SMs that a concurrent kernel
// with large CTAs then cannot use.
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kWS = 3;
constexpr uint32_t kStageBytes = 8192;
constexpr int kMaxGroup = 32;

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
    int32_t group;          // rows per group (<= kMaxGroup, group * row_bytes <= kStageBytes)
    int32_t* dgi;           // swap-in revocation target, or nullptr
    int32_t zero_bad_src;   // 1: a missing source zeroes the destination (SwapIn)
    int32_t pad_dst;        // 1: a destination id of -1 is padding, skipped silently (BackUp)
    int32_t fp8_rows;       // 1: sources are fp8_ds_mla rows, destinations bf16 rows of 576
    int64_t dst_row_bytes;  // bytes per destination row (row_bytes unless fp8_rows)
    int32_t hot_size;
    int64_t region_stride;
    int32_t* status;
    uint64_t timeout_ns;
    int32_t* ticket;        // [2] claim and exit counters (zero on entry, left zero), or nullptr
    // Layer transfer: list r is (buffer r / layers, layer r % layers), every
    // list reads the same index arrays, and row addresses follow the pools'
    // layouts instead of base + id * row_bytes.
    int32_t layer_mode;
    int32_t layers, page_first, page_size, page_shift;  // page_shift = log2(page_size) or -1
    int32_t to_host;             // 1: device pools -> host pool, 0: host -> device
    uint8_t* const* dev_layers;  // device array [nbuf * layers] of per-layer pools
    uint8_t* host_base;          // device-visible host pool: nbuf pools of host_buf_bytes
    int64_t host_tokens, host_buf_bytes;
};

struct WarpRing {
    uint64_t full[kWS];
    int64_t dst[kWS][kMaxGroup];  // destination address of each staged row, -1 = none
};

constexpr size_t kRingBytes = size_t(kWarps) * kWS * kStageBytes;

__device__ __forceinline__ int64_t list_count(const XferArgs& a, int r) {
    const int64_t c = a.counts ? int64_t(a.counts[r]) : int64_t(a.fixed_count);
    return c < 0 ? 0 : (c > a.list_stride ? a.list_stride : c);
}

// Row t of the host pool for buffer b and layer l: page-first pools hold the
// layers' rows of one page next to each other ([page][layer][token in page]),
// layer-first pools one layer after the other ([layer][token]).
__device__ __forceinline__ uint8_t* host_row(const XferArgs& a, int b, int l, int64_t t) {
    int64_t r;
    if (a.page_first) {
        const int64_t pg = a.page_shift >= 0 ? (t >> a.page_shift) : t / a.page_size;
        r = (pg * a.layers + l) * a.page_size + (t - pg * a.page_size);
    } else {
        r = int64_t(l) * a.host_tokens + t;
    }
    return a.host_base + int64_t(b) * a.host_buf_bytes + r * a.row_bytes;
}

// Addresses of source row `id` and destination row `id` of list r.
__device__ __forceinline__ const uint8_t* src_row(const XferArgs& a, int r, int64_t id) {
    if (!a.layer_mode) return a.src_base + id * a.row_bytes;
    if (a.to_host) return a.dev_layers[r] + id * a.row_bytes;
    return host_row(a, r / a.layers, r % a.layers, id);
}
__device__ __forceinline__ uint8_t* dst_row(const XferArgs& a, int r, int64_t id) {
    if (!a.layer_mode) return a.dst_base + id * a.dst_row_bytes;
    if (a.to_host) return host_row(a, r / a.layers, r % a.layers, id);
    return a.dev_layers[r] + id * a.row_bytes;
}

// Writes one landed stage out: the warp's lanes copy 16-byte vectors from
// shared memory to each staged row's destination.
__device__ __forceinline__ void store_group(const XferArgs& a, const WarpRing& R, int st,
                                            const unsigned char* stage, int64_t rb, int nv,
                                            int lane) {
    for (int k = 0; k < a.group; ++k) {
        const int64_t d = R.dst[st][k];
        if (d < 0) continue;
        const uint4* src = reinterpret_cast<const uint4*>(stage + int64_t(k) * rb);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uintptr_t>(d));
        if (a.fp8_rows) {
            // Lane l: the 16 codes of latent columns 16 l .. 16 l + 15 (scale
            // group l / 8) -> 32 bf16 bytes; lanes 0-7: the RoPE bytes.
            const uint4 c = src[lane];
            const float sc = reinterpret_cast<const float*>(stage + int64_t(k) * rb + 512)[lane >> 3];
            dst[2 * lane] = hs::fp8_dequant8(make_uint2(c.x, c.y), sc);
            dst[2 * lane + 1] = hs::fp8_dequant8(make_uint2(c.z, c.w), sc);
            if (lane < 8) dst[64 + lane] = src[33 + lane];
        } else {
            for (int v = lane; v < nv; v += 32) dst[v] = src[v];
        }
    }
}

__global__ void __launch_bounds__(kThreads) xfer_kernel(const XferArgs a) {
    extern __shared__ __align__(128) unsigned char dsmem[];
    // Layout: [ring kWarps * kWS * kStageBytes][WarpRing x kWarps][prefix int32 nlists+1]
    WarpRing* rings = reinterpret_cast<WarpRing*>(dsmem + kRingBytes);
    int32_t* prefix = reinterpret_cast<int32_t*>(dsmem + kRingBytes + sizeof(WarpRing) * kWarps);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    WarpRing& R = rings[warp];
    unsigned char* ring = dsmem + size_t(warp) * kWS * kStageBytes;
    hs::pdl_trigger();
    if (lane == 0) {
        for (int s = 0; s < kWS; ++s) hs::mbar_init(&R.full[s], 32);
        hs::fence_mbar_init();
    }
    hs::pdl_wait();  // the lists and counts come from the predecessor
    // Groups per list -> prefix sums (warp 0).
    if (warp == 0) {
        int running = 0;
        if (lane == 0) prefix[0] = 0;
        for (int base = 0; base < a.nlists; base += 32) {
            const int r = base + lane;
            const int g = r < a.nlists ? int((list_count(a, r) + a.group - 1) / a.group) : 0;
            const int incl = hs::warp_incl_scan(g);
            if (r < a.nlists) prefix[r + 1] = running + incl;
            running += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    __syncthreads();
    const int total = prefix[a.nlists];
    const int64_t rb = a.row_bytes;
    const int nv = int(rb / 16);
    const int64_t drb = a.dst_row_bytes;  // destination row bytes
    const int dnv = int(drb / 16);
    const int gw = blockIdx.x * kWarps + warp;   // global warp id
    const int nw = gridDim.x * kWarps;
    // Groups of this warp: round-robin over the grid, or, with a ticket
    // counter, the first kWS round-robin and the rest claimed one at a time
    // past them (a warp that runs ahead takes more, so the copy ends
    // together); `mine` is then fixed at the first group past the last.  The
    // first rounds need no claim: every warp's first claim at once on one
    // counter serialised the warps' starts (measured on the headline step:
    // the median warp issued its first copy 11 us after the lists were
    // ready).
    const bool claim = a.ticket != nullptr;
    int mine = claim ? (1 << 30) : (gw < total ? (total - gw + nw - 1) / nw : 0);
    bool ok = true;
    bool bad = false;
    for (int j = 0; j < mine + kWS - 1 && ok; ++j) {
        // (a) Issue group j into stage j % kWS.
        int gidx = gw + j * nw;
        if (claim && j < mine) {
            if (j >= kWS) {
                int t = 0;
                if (lane == 0) t = atomicAdd(a.ticket, 1);
                gidx = kWS * nw + __shfl_sync(0xffffffffu, t, 0);
            }
            if (gidx >= total) mine = j;
        }
        if (j < mine) {
            const int st = j % kWS;
            unsigned char* stage = ring + size_t(st) * kStageBytes;
            int lo = 0, hi = a.nlists;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (prefix[mid] <= gidx) lo = mid; else hi = mid;
            }
            const int r = lo;
            const int64_t m0 = int64_t(gidx - prefix[r]) * a.group;
            const int nrows = int(hs::min64(list_count(a, r), m0 + a.group) - m0);
            const int64_t off = (a.layer_mode ? 0 : int64_t(r) * a.list_stride) + m0;
            int64_t g = -1, d = -1;
            if (lane < nrows) {
                g = a.src32 ? int64_t(a.src32[off + lane]) : a.src64[off + lane];
                d = a.dst32 ? int64_t(a.dst32[off + lane]) : a.dst64[off + lane];
            }
            const bool src_ok = g >= 0 && (a.src_limit < 0 || g < a.src_limit);
            const bool dst_ok = d >= 0 && (a.dst_limit < 0 || d < a.dst_limit);
            bool copy = lane < nrows && src_ok && dst_ok;
            // Row addresses (as integers, so that they shuffle and compare).
            int64_t sp = -1, dp = -1;
            if (copy) {
                sp = int64_t(reinterpret_cast<uintptr_t>(src_row(a, r, g)));
                dp = int64_t(reinterpret_cast<uintptr_t>(dst_row(a, r, d)));
            }
            if (lane < nrows && !dst_ok && !(a.pad_dst && d == -1)) bad = true;
            if (lane < nrows && dst_ok && !src_ok && (!a.zero_bad_src || a.dgi == nullptr))
                bad = true;
            // Rows without a source: zero the destination and revoke the slot.
            unsigned zmask = __ballot_sync(0xffffffffu, lane < nrows && dst_ok && !src_ok &&
                                                           a.zero_bad_src);
            while (zmask) {
                const int k = __ffs(zmask) - 1;
                zmask &= zmask - 1;
                const int64_t dk = __shfl_sync(0xffffffffu, d, k);
                uint4* z = reinterpret_cast<uint4*>(dst_row(a, r, dk));
                for (int v = lane; v < dnv; v += 32) z[v] = make_uint4(0, 0, 0, 0);
                if (lane == 0 && a.dgi != nullptr) {
                    const int64_t s = dk - int64_t(r) * a.region_stride;
                    if (s >= 0 && s < a.hot_size) a.dgi[int64_t(r) * a.hot_size + s] = -1;
                }
            }
            // The stage's previous group was written out (synchronously) at
            // an earlier iteration by every lane of this warp.
            __syncwarp();
            if (lane < kMaxGroup) R.dst[st][lane] = copy ? dp : int64_t(-1);
            const unsigned cmask = __ballot_sync(0xffffffffu, copy);
            // One contiguous run of valid rows (source and destination
            // addresses) -> one bulk op; otherwise 16-byte copies by the whole
            // warp.
            const int64_t sp0 = __shfl_sync(0xffffffffu, sp, 0);
            const int64_t dp0 = __shfl_sync(0xffffffffu, dp, 0);
            const bool in_run = !(lane < nrows) ||
                                (copy && sp == sp0 + lane * rb && dp == dp0 + lane * drb);
            const bool one_run = nrows > 1 && cmask == ((nrows == 32) ? 0xffffffffu : ((1u << nrows) - 1u)) &&
                                 __all_sync(0xffffffffu, in_run);
            __syncwarp();
            if (one_run) {
                if (lane == 0) {
                    const uint32_t bytes = uint32_t(nrows * rb);
                    hs::mbar_arrive_expect_tx(&R.full[st], bytes);
                    hs::bulk_g2s(stage, reinterpret_cast<const void*>(static_cast<uintptr_t>(sp0)),
                                 bytes, &R.full[st]);
                } else {
                    hs::mbar_arrive(&R.full[st]);
                }
            } else {
                unsigned m = cmask;
                while (m) {
                    const int k = __ffs(m) - 1;
                    m &= m - 1;
                    const int64_t spk = __shfl_sync(0xffffffffu, sp, k);
                    const unsigned char* src =
                        reinterpret_cast<const unsigned char*>(static_cast<uintptr_t>(spk));
                    const uint32_t dsm = hs::smem_u32(stage + int64_t(k) * rb);
                    for (int v = lane; v < nv; v += 32)
                        hs::tc_cp_async16(dsm + v * 16, src + v * 16);
                }
                hs::tc_cp_async_arrive_noinc(&R.full[st]);
            }
        }
        // (b) Store group j - (kWS - 1) once it has landed.
        const int js = j - (kWS - 1);
        if (js >= 0 && js < mine) {
            const int st = js % kWS;
            const bool landed = hs::mbar_wait_bounded(&R.full[st], (js / kWS) & 1, a.timeout_ns);
            if (!__all_sync(0xffffffffu, landed)) {
                ok = false;
                break;
            }
            __syncwarp();
            store_group(a, R, st, ring + size_t(st) * kStageBytes, rb, nv, lane);
            __syncwarp();
        }
    }
    if (!ok) hs::set_status(a.status, HS_ERR_TIMEOUT);
    if (bad) hs::set_status(a.status, HS_ERR_BAD_INDEX);
    if (claim && lane == 0) {
        // Every warp has made its last claim before it counts itself out; the
        // last one out resets both counters for the next launch.
        __threadfence();
        if (atomicAdd(a.ticket + 1, 1) == nw - 1) {
            a.ticket[0] = 0;
            a.ticket[1] = 0;
        }
    }
    // Leave no copy into shared memory in flight (bounded: the waits above
    // only give up after the wall-time limit).
    asm volatile("cp.async.wait_all;" ::: "memory");
}

size_t xfer_smem_bytes(int nlists) {
    return kRingBytes + sizeof(WarpRing) * kWarps + sizeof(int32_t) * (size_t(nlists) + 1);
}

constexpr int kMaxSmem = 227 * 1024;

int launch_xfer(XferArgs a, int64_t max_items_rows, int max_ctas, hs_stream_t stream) {
    const size_t smem = xfer_smem_bytes(a.nlists);
    if (smem > size_t(kMaxSmem)) return HS_ERR_CAPACITY;
    static int smem_set[64] = {};
    const int rc = hs_host::ensure_dynamic_smem(reinterpret_cast<const void*>(xfer_kernel), smem,
                                                smem_set);
    if (rc != HS_OK) return rc;
    if (a.dst_row_bytes == 0) a.dst_row_bytes = a.row_bytes;
    a.group = int32_t(hs::max64(1, hs::min64(kMaxGroup, int64_t(kStageBytes) / a.row_bytes)));
    // A group never spans two lists: at most ceil(list_stride / group) per list.
    const int64_t groups = hs::min64(int64_t(a.nlists) * ((a.list_stride + a.group - 1) / a.group),
                                     max_items_rows);
    // One CTA (192 KB of stages) per SM.
    const int64_t budget = max_ctas > 0 ? max_ctas : int64_t(hs_host::num_sms());
    const int64_t grid = hs::max64(1, hs::min64((groups + kWarps - 1) / kWarps, budget));
    return hs_host::launch_pdl(xfer_kernel, dim3(unsigned(grid)), dim3(kThreads), smem, stream, a);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int hs_swap_in_fp8ds(const void* host_pool8, int64_t host_rows, int64_t host_row_bytes,
                                void* hot, int64_t hot_rows, const int32_t* miss_src,
                                const int64_t* miss_dst, const int32_t* miss_count, int32_t rows,
                                int32_t cap, int32_t* dgi, int32_t hot_size,
                                int64_t region_stride, int32_t max_ctas, int32_t* ticket,
                                int32_t* status, hs_stream_t stream) {
    if (rows < 0 || cap < 0 || host_rows < 0 || hot_rows < 0 || max_ctas < 0 ||
        host_row_bytes < 656)
        return HS_ERR_INVALID_ARG;
    if (host_row_bytes % 16 != 0) return HS_ERR_MISALIGNED;
    if (host_row_bytes > int64_t(kStageBytes)) return HS_ERR_CAPACITY;
    if (rows == 0 || cap == 0) return HS_OK;
    if (host_pool8 == nullptr || hot == nullptr || miss_src == nullptr || miss_dst == nullptr ||
        miss_count == nullptr)
        return HS_ERR_INVALID_ARG;
    if (!aligned16(host_pool8) || !aligned16(hot)) return HS_ERR_MISALIGNED;
    if (dgi != nullptr && (hot_size <= 0 || region_stride < hot_size)) return HS_ERR_INVALID_ARG;
    XferArgs a{};
    a.src_base = static_cast<const uint8_t*>(host_pool8);
    a.dst_base = static_cast<uint8_t*>(hot);
    a.row_bytes = host_row_bytes;
    a.fp8_rows = 1;
    a.dst_row_bytes = 576 * 2;
    a.src_limit = host_rows;
    a.dst_limit = hot_rows;
    a.src32 = miss_src;
    a.dst64 = miss_dst;
    a.counts = miss_count;
    a.nlists = rows;
    a.list_stride = cap;
    a.dgi = dgi;
    a.zero_bad_src = 1;
    a.hot_size = hot_size;
    a.region_stride = region_stride;
    a.status = status;
    a.timeout_ns = hs::kWaitTimeoutNs;
    a.ticket = ticket;
    return launch_xfer(a, int64_t(rows) * cap, max_ctas, stream);
}

extern "C" int hs_swap_in(const void* host_pool, int64_t host_rows, void* hot, int64_t row_bytes,
                          const int32_t* miss_src, const int64_t* miss_dst,
                          const int32_t* miss_count, int32_t rows, int32_t cap, int32_t* dgi,
                          int32_t hot_size, int64_t region_stride, int32_t max_ctas,
                          int32_t* ticket, int32_t* status, hs_stream_t stream) {
    if (rows < 0 || cap < 0 || host_rows < 0 || row_bytes <= 0 || max_ctas < 0)
        return HS_ERR_INVALID_ARG;
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
    a.dgi = dgi;
    a.zero_bad_src = 1;
    a.hot_size = hot_size;
    a.region_stride = region_stride;
    a.status = status;
    a.timeout_ns = hs::kWaitTimeoutNs;
    a.ticket = ticket;
    return launch_xfer(a, int64_t(rows) * cap, max_ctas, stream);
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
    XferArgs a{};
    a.src_base = static_cast<const uint8_t*>(src);
    a.dst_base = static_cast<uint8_t*>(host_pool);
    a.row_bytes = row_bytes;
    a.src_limit = -1;
    a.dst_limit = host_rows;
    a.src64 = src_rows;
    a.dst32 = dst_slots;
    a.pad_dst = 1;
    a.counts = nullptr;
    a.fixed_count = n;
    a.nlists = 1;
    a.list_stride = n;
    a.status = status;
    a.timeout_ns = hs::kWaitTimeoutNs;
    return launch_xfer(a, n, 0, stream);
}

extern "C" int hs_layer_transfer(void* const* dev_layers, void* host_pool, int64_t host_tokens,
                                 int64_t host_buf_bytes, int32_t nbuf, int32_t layers,
                                 int32_t page_size, int32_t page_first, int64_t dev_tokens,
                                 int64_t row_bytes, const void* src_idx, const void* dst_idx,
                                 int32_t index_bytes, int64_t n, int32_t direction,
                                 int32_t max_ctas, int32_t* status, hs_stream_t stream) {
    if (nbuf <= 0 || layers <= 0 || page_size <= 0 || host_tokens < 0 || dev_tokens < 0 ||
        n < 0 || n > INT32_MAX || max_ctas < 0 || row_bytes <= 0 ||
        (direction != 0 && direction != 1) || (index_bytes != 4 && index_bytes != 8) ||
        int64_t(nbuf) * layers > 4096)
        return HS_ERR_INVALID_ARG;
    if (row_bytes % 16 != 0 || host_buf_bytes % 16 != 0) return HS_ERR_MISALIGNED;
    if (row_bytes > int64_t(kStageBytes)) return HS_ERR_CAPACITY;
    if (page_first && host_tokens % page_size != 0) return HS_ERR_INVALID_ARG;
    if (host_buf_bytes < host_tokens * int64_t(layers) * row_bytes && nbuf > 1)
        return HS_ERR_INVALID_ARG;
    if (n == 0) return HS_OK;
    if (dev_layers == nullptr || host_pool == nullptr || src_idx == nullptr ||
        dst_idx == nullptr)
        return HS_ERR_INVALID_ARG;
    if (!aligned16(host_pool)) return HS_ERR_MISALIGNED;
    XferArgs a{};
    a.row_bytes = row_bytes;
    a.to_host = direction;
    a.src_limit = direction == 0 ? host_tokens : dev_tokens;
    a.dst_limit = direction == 0 ? dev_tokens : host_tokens;
    if (index_bytes == 4) {
        a.src32 = static_cast<const int32_t*>(src_idx);
        a.dst32 = static_cast<const int32_t*>(dst_idx);
    } else {
        a.src64 = static_cast<const int64_t*>(src_idx);
        a.dst64 = static_cast<const int64_t*>(dst_idx);
    }
    a.counts = nullptr;
    a.fixed_count = int32_t(n);
    a.nlists = nbuf * layers;
    a.list_stride = int32_t(n);
    a.zero_bad_src = 0;
    a.status = status;
    a.timeout_ns = hs::kWaitTimeoutNs;
    a.layer_mode = 1;
    a.layers = layers;
    a.page_first = page_first ? 1 : 0;
    a.page_size = page_size;
    a.page_shift = -1;
    if ((page_size & (page_size - 1)) == 0) {
        int sh = 0;
        while ((1 << sh) < page_size) ++sh;
        a.page_shift = sh;
    }
    a.dev_layers = reinterpret_cast<uint8_t* const*>(dev_layers);
    a.host_base = static_cast<uint8_t*>(host_pool);
    a.host_tokens = host_tokens;
    a.host_buf_bytes = host_buf_bytes;
    return launch_xfer(a, int64_t(a.nlists) * n, max_ctas, stream);
}
