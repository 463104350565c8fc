// hs_attention_internal.cuh -- internal interface between the S4 dispatcher
// (hs_attention.cu) and the tensor-core MLA kernel (hs_attention_mla.cu).
#pragma once

#include <cuda_bf16.h>

#include "hs_common.cuh"

namespace hs_attn {

struct MlaArgs {
    const __nv_bfloat16* q;   // [rows, heads, 576]
    const __nv_bfloat16* kv;  // rows of row_stride elements; K = [0,576), V = [0,512)
    int64_t row_stride;
    int64_t num_kv_rows;
    const int32_t* kv_rows;   // [rows, cap]
    const int32_t* count;     // [rows] or nullptr
    int32_t rows, cap, heads;
    float scale_log2;
    __nv_bfloat16* out;       // [rows, heads, 512]
    float* lse;               // [rows, heads] or nullptr
    float* part_m;            // partial states, index (row*heads+h)*part_stride + part_base + split
    float* part_l;
    float* part_o;
    int32_t splits;
    int32_t part_stride;
    int32_t part_base;
    int32_t force_partial;    // 1: write partial states even when splits == 1
    int32_t combine_parts;    // >0 (splits == 1): merge with partial columns [0, combine_parts)
                              // in the epilogue and write the final out / lse
    int32_t* sync;            // per (row, head group) arrival counters, zero on entry, or
                              // nullptr; with it every split writes its partial column and
                              // the last one to finish merges columns [0, merge_total)
    int32_t merge_total;
    int32_t* status;
    uint64_t timeout_ns;
};

// Columns the last-CTA merge of the tcgen05 kernel can combine.
constexpr int kMlaMaxMerge = 8;

// Splits of one row the CTA-pair kernel (128 heads) can merge in its epilogue.
constexpr int kMlaPairMaxSplits = 8;

// CTA-pair kernel for 128 heads: grid = 2 * rows * splits CTAs (clusters of
// two).  Workspace when splits > 1: part_o = [rows * 128, splits, 512] fp32,
// part_m = [2, rows * 128, splits, 2] fp32 (m, l per CTA rank), sync =
// [rows, 2, 2] int32 counters, zero on entry and left zero.
int launch_mla_pair(const MlaArgs& a, int pairs, hs_stream_t stream);
// True when launch_mla_pair merges a row's two splits inside a cluster of
// four CTAs (no partial states or counters in global memory).
bool mla_pair_cluster_merge(int rows, int splits);

// Query heads handled by one CTA (64, 32 or 16), or 0 when heads % 16 != 0.
int mla_tc_head_group(int heads);
// grid = (rows * heads / hg, splits).
int launch_mla_tc(const MlaArgs& a, int hg, dim3 grid, hs_stream_t stream);

}  // namespace hs_attn
