// hs_fp8ds.cu -- S4 over fp8_ds_mla KV rows.
//
// Row format (vLLM HiSparse walkthrough: the FlashMLASparseBackend cache shape
// and FP8_DS_MLA_ROW_BYTES = 656): bytes [0, 512) hold the 512 latent
// columns as OCP FP8 E4M3 codes, bytes [512, 528) four fp32 scales (scale g
// for latent columns [128 g, 128 g + 128)), bytes [528, 656) the 64 RoPE
// columns as bf16.  Column d < 512 has the value code_d * scale_{d/128},
// formed in fp32 and rounded to bf16, the operand type of the products
// (PaperTrace 5.1.1 section 7.2: the scale is applied to the stored codes
// before QK^T and PV).
//
// GB300 design.  The attention runs in two launches:
//  * fp8ds_gather_kernel: a warp reads 32 entries' ids at once and moves
//    their rows four at a time; lane i loads the 16 codes of columns
//    16 i .. 16 i + 15 (one 16-byte load) and their group scale, lanes 0-7
//    the RoPE bytes; the codes go through the hardware e4m3x2 -> f16x2
//    conversion, fp32 scaling and bf16 rounding, and the warp writes the
//    1152-byte bf16 row into a per-request scratch [rows, cap, 576].
//  * the MLA attention (hs_attention_mla.cu on tensor cores for head counts
//    that are multiples of 16) over the scratch rows of each request (row
//    ids r * cap + j).
// The reconstructed rows cross HBM/L2 once more than a reconstructing load
// path would (PaperTrace section 7.2 prefers the latter).  Reconstructing in
// the tensor-core kernel's loaders was built and measured slower on GB300:
// the code -> fp32 * scale -> bf16 conversion of a whole 128-row unit lies
// between its arrival and the MMA, and the few warps that can do it bound
// the per-tile time.
#include <cuda_bf16.h>

#include "hs_common.cuh"
#include "hs_fp8.cuh"

namespace {

constexpr int kFp8RowBytes = 656;
constexpr int kBatch = 4;  // rows a warp moves with one round of loads
constexpr int kThreads = 256;

struct GatherArgs {
    const unsigned char* kv8;
    int64_t row_bytes;
    int64_t num_kv_rows;
    const int32_t* kv_rows;  // [rows, cap] source row ids
    const int32_t* count;    // [rows] or null (= cap)
    int32_t rows;
    int32_t cap;
    __nv_bfloat16* out;      // bf16 rows of 576
    int32_t* out_ids;        // [rows * cap]: r * cap + j, or -1 (no row)
    int32_t* status;
};

// A warp takes 32 consecutive entries at a time: lane l reads entry l's
// count and id (one coalesced load each), then the warp moves the entries
// that have a row in batches of kBatch rows, all loads of a batch in flight
// together (one memory latency per batch instead of three dependent ones per
// entry).  Within a row, lane l holds the 16 codes of latent columns
// 16 l .. 16 l + 15 (one 16-byte load; scale group l / 8) and writes their
// 32 bf16 bytes; lanes 0-7 also move the 128 RoPE bytes.
__global__ void __launch_bounds__(kThreads, 3) fp8ds_gather_kernel(const GatherArgs a) {
    hs::pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
    const int64_t total = int64_t(a.rows) * a.cap;
    bool bad = false;
    for (int64_t base = warp0 * 32; base < total; base += nwarps * 32) {
        const int64_t f = base + lane;
        bool live = false;
        int32_t id = -1;
        if (f < total) {
            const int r = int(f / a.cap), j = int(f - int64_t(r) * a.cap);
            const int n = a.count ? min(max(__ldg(a.count + r), 0), a.cap) : a.cap;
            if (j < n) {
                live = true;
                id = __ldg(a.kv_rows + f);
            }
        }
        const bool has_src = live && id >= 0 && int64_t(id) < a.num_kv_rows;
        if (live && int64_t(id) >= a.num_kv_rows) bad = true;
        if (live) a.out_ids[f] = has_src ? int32_t(f) : -1;
        unsigned todo = __ballot_sync(0xffffffffu, has_src);
        while (todo) {
            uint4 code[kBatch], rope[kBatch];
            float sc[kBatch];
            int64_t dst[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int u = todo ? __ffs(todo) - 1 : -1;  // the same on every lane
                todo &= todo - 1u;
                const int32_t iu = __shfl_sync(0xffffffffu, id, u < 0 ? 0 : u);
                dst[b] = u < 0 ? -1 : base + u;
                if (u >= 0) {
                    const unsigned char* row = a.kv8 + int64_t(iu) * a.row_bytes;
                    code[b] = __ldg(reinterpret_cast<const uint4*>(row) + lane);
                    sc[b] = __ldg(reinterpret_cast<const float*>(row + 512) + (lane >> 3));
                    if (lane < 8) rope[b] = __ldg(reinterpret_cast<const uint4*>(row + 528) + lane);
                }
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                if (dst[b] < 0) continue;
                uint4* o = reinterpret_cast<uint4*>(a.out + dst[b] * 576);
                o[2 * lane] = hs::fp8_dequant8(make_uint2(code[b].x, code[b].y), sc[b]);
                o[2 * lane + 1] = hs::fp8_dequant8(make_uint2(code[b].z, code[b].w), sc[b]);
                if (lane < 8) o[64 + lane] = rope[b];
            }
        }
    }
    if (bad) hs::set_status(a.status, HS_ERR_BAD_INDEX);
    // The stream successor (the attention) may start its set-up once every
    // CTA got here: triggered at the start, its waiting CTAs would hold SMs
    // this grid still needs.
    hs::pdl_trigger();
}

int gather_ctas_per_sm() {
    static int per_sm = 0;
    if (per_sm == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fp8ds_gather_kernel, kThreads, 0) !=
                cudaSuccess ||
            n <= 0) {
            cudaGetLastError();
            n = 1;
        }
        per_sm = n;
    }
    return per_sm;
}

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// Grid: enough warps for every entry, at most the resident CTAs of all SMs
// (or max_ctas CTAs when given).
int launch_gather(const GatherArgs& a, int64_t total, int32_t max_ctas, hs_stream_t stream) {
    const int64_t warps = (total + 31) / 32;
    int64_t ctas = hs::min64((warps * 32 + kThreads - 1) / kThreads,
                             int64_t(hs_host::num_sms()) * gather_ctas_per_sm());
    if (max_ctas > 0) ctas = hs::min64(ctas, max_ctas);
    return hs_host::launch_pdl(fp8ds_gather_kernel, dim3(unsigned(ctas)), dim3(kThreads), 0,
                               stream, a);
}

}  // namespace

extern "C" int hs_fp8ds_gather(const void* kv8, int64_t row_bytes, int64_t num_kv_rows,
                               const int32_t* kv_rows, const int32_t* count, int32_t rows,
                               int32_t cap, void* out, int32_t* out_ids, int32_t* status,
                               hs_stream_t stream) {
    if (rows < 0 || cap < 0 || num_kv_rows < 0 || row_bytes < kFp8RowBytes)
        return HS_ERR_INVALID_ARG;
    if (row_bytes % 16) return HS_ERR_MISALIGNED;
    const int64_t total = int64_t(rows) * cap;
    if (total == 0) return HS_OK;
    if (total > INT32_MAX) return HS_ERR_CAPACITY;
    if (kv8 == nullptr || kv_rows == nullptr || out == nullptr || out_ids == nullptr)
        return HS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(kv8) | reinterpret_cast<uintptr_t>(out)) & 15u)
        return HS_ERR_MISALIGNED;
    const GatherArgs a{static_cast<const unsigned char*>(kv8), row_bytes, num_kv_rows, kv_rows,
                       count, rows, cap, static_cast<__nv_bfloat16*>(out), out_ids, status};
    return launch_gather(a, total, 0, stream);
}

extern "C" int64_t hs_sparse_decode_fp8ds_workspace_bytes(int32_t rows, int32_t heads,
                                                          int32_t cap) {
    if (rows < 0 || heads <= 0 || cap < 0) return -1;
    const int64_t total = int64_t(rows) * cap;
    const int64_t dec = hs_sparse_decode_workspace_bytes(rows, heads, 1, cap, 576, 512);
    if (dec < 0) return -1;
    return align256(total * 576 * 2) + align256(total * 4) + dec;
}

extern "C" int hs_sparse_decode_fp8ds(const void* q, const void* kv8, int64_t row_bytes,
                                      int64_t num_kv_rows, const int32_t* kv_rows,
                                      const int32_t* count, int32_t rows, int32_t cap,
                                      int32_t heads, float scale, void* out, float* lse,
                                      void* workspace, int64_t workspace_bytes_given,
                                      int32_t* status, hs_stream_t stream) {
    if (rows < 0 || cap < 0 || heads <= 0) return HS_ERR_INVALID_ARG;
    if (rows == 0) return HS_OK;
    const int64_t need = hs_sparse_decode_fp8ds_workspace_bytes(rows, heads, cap);
    if (need < 0) return HS_ERR_INVALID_ARG;
    if (workspace == nullptr || workspace_bytes_given < need) return HS_ERR_CAPACITY;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return HS_ERR_MISALIGNED;
    const int64_t total = int64_t(rows) * cap;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    void* scratch = ws;
    int32_t* ids = reinterpret_cast<int32_t*>(ws + align256(total * 576 * 2));
    unsigned char* dec_ws = ws + align256(total * 576 * 2) + align256(total * 4);
    const int64_t dec_bytes = need - (dec_ws - ws);
    int rc = hs_fp8ds_gather(kv8, row_bytes, num_kv_rows, kv_rows, count, rows, cap, scratch,
                             ids, status, stream);
    if (rc != HS_OK) return rc;
    return hs_sparse_decode(q, scratch, scratch, 576, 0, total, ids, count, rows, cap, heads, 1,
                            576, 512, scale, out, lse, dec_bytes > 0 ? dec_ws : nullptr,
                            dec_bytes, status, stream);
}
