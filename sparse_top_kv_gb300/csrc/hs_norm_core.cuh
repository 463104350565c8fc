// hs_norm_core.cuh -- S1's normalisation of one index row, shared by the
// S1 kernel (hs_normalize.cu) and the fused S1 + S2 kernel (hs_lookup.cu).
//
// PaperTrace 5.1.1 "从索引到 Kernel": section 1.1 eq. (1) S = unique(D u W u A)
// with range, causality and batch-ownership checks; section 1.2 eq. (2)
// b = floor(t / B) and the block-table lookup; section 7.3 eq. (16) (set
// semantics: membership by logical t, output ordered by t).  vLLM HiSparse
// walkthrough, "_convert_req_index_to_global_index_kernel": slot = table[b] *
// B + t mod B, invalid tokens propagate as -1.
//
// Membership is a bitmap over the row's positions in shared memory (a
// counting sort): W u A and then D are set with atomicOr (the returned old
// word tells a duplicate), and the ascending, de-duplicated output comes from
// a block-wide scan of the bitmap words' popcounts.  The result is exactly
// the set definition, whatever the thread schedule.  Contexts longer than one
// bitmap window are processed in successive windows of kWindowBits positions.
#pragma once

#include "hs_common.cuh"

namespace hs_norm {

constexpr int kWindowWords = 4096;                          // bitmap words: 16 KB
constexpr int64_t kWindowBits = int64_t(kWindowWords) * 32;  // 131072 positions
constexpr int kMaxStagedBlocks = 16384;  // block-table rows up to this are copied to smem
constexpr int kUnroll = 4;               // candidates loaded per thread before use

struct NormArgs {
    const int32_t* cand;
    int32_t rows, n_cand, window, num_sinks;
    const int32_t* row_req;
    const int32_t* seq_lens;
    const int32_t* block_table;
    int64_t bt_stride;
    int32_t max_blocks;
    const int32_t* page_owner;
    int32_t num_reqs, num_pages, page_size, cap;
    int32_t* out_tok;
    int32_t* out_slot;
    int32_t* out_count;
    int32_t* err_counts;
    int32_t stage_table;  // 1: the request's block-table row is staged in shared memory
    int32_t page_shift;   // log2(page_size) when it is a power of two, else -1
    int32_t stage_out;    // 1: the outputs are assembled in shared memory, then written once
};

// Logical block and in-page offset of position t (0 <= t < 2^31): a shift and
// a mask for power-of-two pages, 32-bit division otherwise (no 64-bit divide).
__device__ __forceinline__ void split_pos(int64_t t, const NormArgs& a, int32_t* b, int32_t* off) {
    const uint32_t ut = uint32_t(t);
    if (a.page_shift >= 0) {
        *b = int32_t(ut >> a.page_shift);
        *off = int32_t(ut & ((1u << a.page_shift) - 1u));
    } else {
        const uint32_t ub = ut / uint32_t(a.page_size);
        *b = int32_t(ub);
        *off = int32_t(ut - ub * uint32_t(a.page_size));
    }
}

// Checks of a position already known to satisfy 0 <= t < T.
// Returns -1 when valid, else the rejection category (0 range, 2 owner).
__device__ __forceinline__ int classify_in_range(int64_t t, const int32_t* table,
                                                 const NormArgs& a, int32_t req) {
    int32_t b, off;
    split_pos(t, a, &b, &off);
    if (b >= a.max_blocks) return 0;
    const int32_t p = table[b];
    if (p < 0 || p >= a.num_pages) return 0;
    if (a.page_owner != nullptr && __ldg(a.page_owner + p) != req) return 2;
    return -1;
}

// Index of output entry j in a shared-memory output array: with swz = 31
// the low five bits are XORed with bits 5-9 (a permutation within every
// aligned run of 1024 entries, so the array needs its length rounded up to
// a multiple of 32).  A dense bitmap word puts 32 consecutive outputs on one
// thread, so the threads of a warp write entries 32 apart: without the
// swizzle those all fall on one bank.
__device__ __forceinline__ int out_index(int j, int swz) { return j ^ ((j >> 5) & swz); }

// Normalises index row `row` with the NT threads of the block (every thread
// must call it): the ascending set of valid positions goes to otok and their
// slots to oslot, entry j at out_index(j, swz) (swz = 31 for shared-memory
// targets, 0 for global ones), s_err[4] receives the rejected-candidate
// counts; returns n.  s_table: [max_blocks] shared ints when a.stage_table;
// bm / wpos: [kWindowWords] shared words, bm already zero when bm_zeroed
// (the zeros written by the block before the call); scan_scratch: >= 33
// shared ints.
template <int NT>
__device__ int normalize_row(const NormArgs& a, const int row, int32_t* s_table, int32_t* otok,
                             int32_t* oslot, int swz, uint32_t* bm, bool bm_zeroed, int* wpos,
                             int* scan_scratch, int* s_err) {
    constexpr int kWpt = kWindowWords / NT;
    static_assert(kWpt * NT == kWindowWords, "bitmap words per thread");
    const int tid = threadIdx.x;
    const int32_t* cand = a.cand + int64_t(row) * a.n_cand;
    // The request, then the first kUnroll candidates of this thread, whose
    // latency overlaps the table's copy below; later chunks, if any, are
    // loaded where they are used.
    const int32_t req = a.row_req[row];
    int32_t tv0[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int i = tid + u * NT;
        tv0[u] = i < a.n_cand ? __ldg(cand + i) : -1;
    }
    // One index row per request is the common layout (row r serves request
    // r): the length and the table row of request `row` are loaded before
    // the request id arrives, and loaded again for a row of another request.
    const bool guess = row < a.num_reqs;
    const int32_t t_guess = guess ? a.seq_lens[row] : 0;
    if (guess && a.stage_table) {
        const int32_t* tg = a.block_table + int64_t(row) * a.bt_stride;
        for (int b = tid; b < a.max_blocks; b += NT) s_table[b] = __ldg(tg + b);
    }
    if (tid < 4) s_err[tid] = 0;
    const bool has_req = req >= 0 && req < a.num_reqs;
    const bool same = guess && req == row;
    const int32_t t_len = has_req ? (same ? t_guess : a.seq_lens[req]) : 0;
    const int32_t* table = has_req ? a.block_table + int64_t(req) * a.bt_stride : nullptr;
    if (has_req && a.stage_table) {
        // One coalesced copy of the row; every later lookup hits shared
        // memory (each thread rewrites only the entries it wrote above).
        if (!same)
            for (int b = tid; b < a.max_blocks; b += NT) s_table[b] = __ldg(table + b);
        table = s_table;
    }
    __syncthreads();  // s_err and the staged table

    int out_n = 0;
    if (!has_req) {
        // No request: each dynamic candidate is a range error.
        int bad = 0;
        for (int i = tid; i < a.n_cand; i += NT) bad += (cand[i] != -1);
        if (bad) atomicAdd(&s_err[0], bad);
    } else {
        const int64_t T = max(t_len, 0);
        const int64_t a_hi = hs::min64(a.num_sinks, T);        // sinks  [0, a_hi)
        const int64_t s2 = hs::max64(hs::max64(T - a.window, 0), a_hi);  // window [s2, T)

        // Dynamic candidates outside [0, T) are rejected once, before the windows.
        {
            int er = 0, ec = 0;
            for (int i0 = tid; i0 < a.n_cand; i0 += NT * kUnroll) {
                int32_t tv[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int i = i0 + u * NT;
                    tv[u] = i0 == tid ? tv0[u] : (i < a.n_cand ? __ldg(cand + i) : -1);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int32_t t = tv[u];
                    if (t == -1) continue;
                    if (t < 0) ++er;
                    else if (t >= T) ++ec;
                }
            }
            if (er) atomicAdd(&s_err[0], er);
            if (ec) atomicAdd(&s_err[1], ec);
        }

        for (int64_t lo = 0; lo < T; lo += kWindowBits) {
            const int64_t hi = hs::min64(T, lo + kWindowBits);
            const int nw = int((hi - lo + 31) >> 5);
            if (lo > 0 || !bm_zeroed) {
                for (int w = tid; w < nw; w += NT) bm[w] = 0u;
                __syncthreads();
            }

            int er = 0, eo = 0, ed = 0;
            // Structural candidates: sinks [0, a_hi) and window [s2, T) (disjoint).
            for (int pass = 0; pass < 2; ++pass) {
                const int64_t b0 = pass == 0 ? hs::max64(lo, 0) : hs::max64(lo, s2);
                const int64_t b1 = pass == 0 ? hs::min64(hi, a_hi) : hs::min64(hi, T);
                for (int64_t t = b0 + tid; t < b1; t += NT) {
                    const int c = classify_in_range(t, table, a, req);
                    if (c < 0) {
                        const int64_t o = t - lo;
                        atomicOr(&bm[o >> 5], 1u << (o & 31));
                    } else if (c == 0) {
                        ++er;
                    } else {
                        ++eo;
                    }
                }
            }
            __syncthreads();
            // Dynamic candidates inside this window (kUnroll independent loads first).
            for (int i0 = tid; i0 < a.n_cand; i0 += NT * kUnroll) {
                int32_t tv[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int i = i0 + u * NT;
                    tv[u] = i0 == tid ? tv0[u] : (i < a.n_cand ? __ldg(cand + i) : -1);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int64_t t = tv[u];
                    if (t < lo || t >= hi) continue;
                    const int c = classify_in_range(t, table, a, req);
                    if (c == 0) { ++er; continue; }
                    if (c == 2) { ++eo; continue; }
                    const int64_t o = t - lo;
                    const uint32_t bit = 1u << (o & 31);
                    const uint32_t old = atomicOr(&bm[o >> 5], bit);
                    if (old & bit) ++ed;
                }
            }
            if (er) atomicAdd(&s_err[0], er);
            if (eo) atomicAdd(&s_err[2], eo);
            if (ed) atomicAdd(&s_err[3], ed);
            __syncthreads();

            // Ascending compaction of the window: the output offset of every
            // word from one block scan (thread tid counts words 8 tid ..
            // 8 tid + 7), then the words are emitted round-robin (word w by
            // thread w mod 512), so a dense run of positions -- recent tokens
            // under a recency-skewed selection -- is spread over consecutive
            // threads instead of falling on one.
            int cnt = 0;
            uint32_t words[kWpt];
#pragma unroll
            for (int k = 0; k < kWpt; ++k) {
                const int w = tid * kWpt + k;
                words[k] = w < nw ? bm[w] : 0u;
                cnt += __popc(words[k]);
            }
            int total;
            int run = out_n + hs::block_excl_scan(cnt, scan_scratch, &total);
#pragma unroll
            for (int k = 0; k < kWpt; ++k) {
                wpos[tid * kWpt + k] = run;
                run += __popc(words[k]);
            }
            __syncthreads();
            for (int w = tid; w < nw; w += NT) {
                uint32_t x = bm[w];
                int pos = wpos[w];
                const int64_t base = lo + int64_t(w) * 32;
                while (x) {
                    const int b = __ffs(x) - 1;
                    x &= x - 1;
                    const int64_t t = base + b;
                    int32_t blk, off;
                    split_pos(t, a, &blk, &off);
                    const int e = out_index(pos, swz);
                    otok[e] = int32_t(t);
                    oslot[e] = table[blk] * a.page_size + off;
                    ++pos;
                }
            }
            out_n += total;
            __syncthreads();
        }
    }
    return out_n;
}

}  // namespace hs_norm
