// hs_normalize.cu -- S1, candidate normalisation.
//
// PaperTrace 5.1.1 "从索引到 Kernel": section 1.1 eq. (1) S = unique(D u W u A)
// with range, causality and batch-ownership checks; section 1.2 eq. (2)
// b = floor(t / B) and the block-table lookup; section 7.3 eq. (16) (set
// semantics: membership by logical t, output ordered by t).  vLLM HiSparse
// walkthrough, "_convert_req_index_to_global_index_kernel": slot = table[b] *
// B + t mod B, invalid tokens propagate as -1.
//
// GB300 design: one CTA per index row.  The request's block-table row is
// copied to shared memory once (rows up to 16384 blocks), so the per-token
// page lookups never wait on global memory.  Membership is a bitmap over the
// row's positions in shared memory (a counting sort): W u A and then D are
// set with atomicOr (the returned old word tells a duplicate), and the
// ascending, de-duplicated output comes from a block-wide scan of the
// bitmap words' popcounts (warp shuffles + ballot-free popc).  The result is
// exactly the set definition, whatever the thread schedule.  Contexts longer
// than one bitmap window are processed in successive windows of kWindowBits
// positions.
#include "hs_norm_core.cuh"

namespace {

using namespace hs_norm;
constexpr int kThreads = 512;
constexpr int kMaxOutStageBytes = 160 * 1024;  // dynamic shared memory for table + outputs

__global__ void __launch_bounds__(kThreads) normalize_kernel(const NormArgs a) {
    // Dynamic: [max_blocks] table when a.stage_table, then [cap32] tokens and
    // [cap32] slots (cap rounded up to 32) when a.stage_out.
    extern __shared__ int32_t s_dyn[];
    __shared__ uint32_t bm[kWindowWords];
    __shared__ int wpos[kWindowWords];  // output offset of each bitmap word
    __shared__ int scan_scratch[33];
    __shared__ int s_err[4];

    hs::pdl_trigger();
    const int tid = threadIdx.x;
    // The first window's bitmap is cleared while the predecessor may still run.
    for (int w = tid; w < kWindowWords; w += kThreads) bm[w] = 0u;
    hs::pdl_wait();
    const int row = blockIdx.x;
    const int64_t cap32 = (int64_t(a.cap) + 31) & ~int64_t(31);
    int32_t* const g_tok = a.out_tok + int64_t(row) * a.cap;
    int32_t* const g_slot = a.out_slot + int64_t(row) * a.cap;
    int32_t* const s_table = s_dyn;
    int32_t* const s_tok = s_dyn + (a.stage_table ? a.max_blocks : 0);
    int32_t* const s_slot = s_tok + cap32;
    // Emission targets: shared memory (swizzled, written out coalesced at the
    // end) or the global rows directly.
    int32_t* const otok = a.stage_out ? s_tok : g_tok;
    int32_t* const oslot = a.stage_out ? s_slot : g_slot;
    const int out_n = normalize_row<kThreads>(a, row, s_table, otok, oslot,
                                              a.stage_out ? 31 : 0, bm, true, wpos,
                                              scan_scratch, s_err);
    if (a.stage_out) {
        __syncthreads();
        for (int j = tid; j < a.cap; j += kThreads) {
            const int e = out_index(j, 31);
            g_tok[j] = j < out_n ? s_tok[e] : -1;
            g_slot[j] = j < out_n ? s_slot[e] : -1;
        }
    } else {
        for (int j = out_n + tid; j < a.cap; j += kThreads) {
            g_tok[j] = -1;
            g_slot[j] = -1;
        }
    }
    __syncthreads();
    if (tid == 0) a.out_count[row] = out_n;
    if (tid < 4) a.err_counts[int64_t(row) * 4 + tid] = s_err[tid];
}

}  // namespace

extern "C" int hs_normalize_indices(const int32_t* cand, int32_t rows, int32_t n_cand,
                                    int32_t window, int32_t num_sinks, const int32_t* row_req,
                                    const int32_t* seq_lens, const int32_t* block_table,
                                    int64_t bt_stride, int32_t max_blocks,
                                    const int32_t* page_owner, int32_t num_reqs,
                                    int32_t num_pages, int32_t page_size, int32_t cap,
                                    int32_t* out_tok, int32_t* out_slot, int32_t* out_count,
                                    int32_t* err_counts, hs_stream_t stream) {
    if (rows < 0 || n_cand < 0 || window < 0 || num_sinks < 0 || max_blocks < 0 ||
        num_reqs < 0 || num_pages < 0 || page_size <= 0 || cap < 0 || bt_stride < max_blocks)
        return HS_ERR_INVALID_ARG;
    if (int64_t(cap) < int64_t(n_cand) + window + num_sinks) return HS_ERR_CAPACITY;
    if (int64_t(num_pages) * page_size > INT32_MAX) return HS_ERR_INVALID_ARG;
    if (rows == 0) return HS_OK;
    if ((n_cand > 0 && cand == nullptr) || row_req == nullptr || out_tok == nullptr ||
        out_slot == nullptr || out_count == nullptr || err_counts == nullptr)
        return HS_ERR_INVALID_ARG;
    if (num_reqs > 0 && (seq_lens == nullptr || (max_blocks > 0 && block_table == nullptr)))
        return HS_ERR_INVALID_ARG;
    NormArgs a{cand,      rows,      n_cand,     window,    num_sinks, row_req,
               seq_lens,  block_table, bt_stride, max_blocks, page_owner, num_reqs,
               num_pages, page_size, cap,        out_tok,   out_slot,  out_count,
               err_counts, max_blocks <= kMaxStagedBlocks ? 1 : 0, -1, 0};
    if ((page_size & (page_size - 1)) == 0) {
        int sh = 0;
        while ((1 << sh) < page_size) ++sh;
        a.page_shift = sh;
    }
    size_t smem = a.stage_table ? size_t(max_blocks) * sizeof(int32_t) : 0;
    // Outputs assembled in shared memory when they fit beside the table.
    const size_t out_bytes = size_t((int64_t(cap) + 31) & ~int64_t(31)) * 2 * sizeof(int32_t);
    if (smem + out_bytes <= size_t(kMaxOutStageBytes)) {
        a.stage_out = 1;
        smem += out_bytes;
    }
    static int smem_set[64] = {};
    const int rc = hs_host::ensure_dynamic_smem(reinterpret_cast<const void*>(normalize_kernel),
                                                smem, smem_set);
    if (rc != HS_OK) return rc;
    return hs_host::launch_pdl(normalize_kernel, dim3(rows), dim3(kThreads), smem, stream, a);
}
