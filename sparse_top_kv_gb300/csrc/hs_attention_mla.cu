// hs_attention_mla.cu -- S4 for MLA rows (576 bf16: K = all 576 columns,
// V = the first 512) on the 5th-generation tensor cores.
//
// Math: PaperTrace 5.1.1 "从索引到 Kernel" section 3.1 eqs. (4)-(6) (tile
// logits, running maximum and exponent sums, rescaled accumulator), section
// 3.2 (mask before the exponent; empty set -> zero output, LSE = -inf) and
// eq. (7) (split-KV merge, done by merge_kernel in hs_attention.cu);
// "PagedAttention 与 RadixAttention" section 1.4 (exp2 with scale * log2 e).
//
// GB300 design.  One CTA per (index row, group of HG query heads, split of
// the row's candidate list); 128 candidate rows form a tile.
//  * Loader warps (4) gather the tile's K/V rows straight from the paged or
//    hot cache (no scratch gather, PaperTrace section 2.1 eq. (3)) with
//    16-byte cp.async into 128-byte-swizzled K-major blocks of 128 rows x 64
//    columns; rows that are invalid are zero-filled, never read.  Blocks
//    0..7 (the 512 V columns) travel in pairs so that a 128-wide slice of V
//    is one MN-major operand; block 8 (the RoPE tail) has its own ring.
//  * One MMA thread issues tcgen05.mma: S^T[128 tokens x HG] = K Q^T (M = 128
//    tokens, N = HG heads, K = 576) into TMEM, and O^T[512 x HG] += V^T P^T
//    (four M = 128 slices of d, K = 128 tokens).  Commits release the ring.
//  * Four softmax warps (thread = TMEM lane = token for S, = d for O) keep
//    a per-head reference maximum; a tile only rescales O (in TMEM) when some
//    logit exceeds the reference by more than 2^8 (the vote is one warp
//    reduction), so the common tile has no cross-thread max reduction.  The
//    exponent sums stay in registers per token lane and are reduced once.
// Every wait is bounded (HS_ERR_TIMEOUT in the status word on expiry).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "hs_attention_internal.cuh"
#include "hs_tcgen05.cuh"

namespace hs_attn {
namespace {

constexpr int kTok = 128;           // tokens per tile = M of the QK product
constexpr int kNB = 9;              // 64-column blocks of a 576-wide row
constexpr int kBlk = kTok * 128;    // bytes of one block (128 rows x 128 B)
constexpr int kPair = 2 * kBlk;
constexpr int kThreads = 288;       // 4 softmax + 4 loader warps + 1 MMA warp
constexpr int kLoaderThreads = 128;
constexpr float kThresh = 8.0f;     // log2 headroom before O is rescaled
constexpr int kMaxCombine = 4;      // partial columns a finishing pass can merge

template <int HG>
struct Cfg {
    static constexpr int NP = HG == 16 ? 5 : 4;        // V pair slots
    static constexpr int NR = HG == 64 ? 1 : 2;        // RoPE slots
    static constexpr bool kPInRope = HG == 64;         // P reuses the RoPE slot
    static constexpr int kQBytes = kNB * HG * 128;
    static constexpr int kPBytes = 2 * HG * 128;       // one P^T buffer
    static constexpr int kPairOff = 0;
    static constexpr int kRopeOff = kPairOff + NP * kPair;
    static constexpr int kQOff = kRopeOff + NR * kBlk;
    static constexpr int kPOff = kQOff + kQBytes;
    static constexpr int kBarOff = kPOff + (kPInRope ? 0 : 2 * kPBytes);
    static constexpr int kTmemCols = 6 * HG <= 128 ? 128 : (6 * HG <= 256 ? 256 : 512);
    static constexpr int kD1 = 0;                      // S^T buffers: cols [0, 2HG)
    static constexpr int kO = 2 * HG;                  // O^T slices: cols [2HG, 6HG)
};

struct Bars {
    uint64_t full_pair[8][2];
    uint64_t empty_pair[8];
    uint64_t full_rope[2];
    uint64_t empty_rope[2];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t pv_done[2];
    uint64_t drain;
    uint64_t group;
    uint32_t tmem_base;
    int32_t abort;
    uint32_t vote[2][4][2];
    float red[4][64];
    float cw[64][6];  // finishing merge, per head: w_own, 1/L_total, w_part[4]
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <int HG>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, float (&v)[HG]) {
#pragma unroll
    for (int c = 0; c < HG; c += 16) {
        float t[16];
        hs::tc::tmem_ld16(taddr + c, t);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[c + i] = t[i];
    }
}

template <int HG>
__device__ __forceinline__ void tmem_st_row(uint32_t taddr, const float (&v)[HG]) {
#pragma unroll
    for (int c = 0; c < HG; c += 16) {
        float t[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] = v[c + i];
        hs::tc::tmem_st16(taddr + c, t);
    }
}

template <int HG>
__global__ void __launch_bounds__(kThreads, 1) mla_tc_kernel(const MlaArgs a) {
    using C = Cfg<HG>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment of the swizzle atoms.
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars& B = *reinterpret_cast<Bars*>(smem + C::kBarOff);
    const uint32_t s_base = hs::smem_u32(smem);
    const uint32_t pair_base = s_base + C::kPairOff;
    const uint32_t rope_base = s_base + C::kRopeOff;
    const uint32_t q_base = s_base + C::kQOff;
    const uint32_t p_base = s_base + C::kPOff;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int groups = a.heads / HG;
    const int row = blockIdx.x / groups;
    const int grp = blockIdx.x % groups;
    const int split = blockIdx.y;
    const int n = a.count ? min(max(a.count[row], 0), a.cap) : a.cap;
    const int ntiles = (n + kTok - 1) / kTok;
    const int per = (ntiles + a.splits - 1) / a.splits;
    const int t_begin = min(ntiles, split * per);
    const int T = min(ntiles, t_begin + per) - t_begin;  // tiles of this CTA
    const int32_t* kv_rows = a.kv_rows + int64_t(row) * a.cap;
    const int head0 = grp * HG;
    const uint64_t tmo = a.timeout_ns;
    volatile int* abort_flag = &B.abort;

    if (tid == 0) {
        for (int i = 0; i < C::NP; ++i) {
            hs::mbar_init(&B.full_pair[i][0], kLoaderThreads);
            hs::mbar_init(&B.full_pair[i][1], kLoaderThreads);
            hs::mbar_init(&B.empty_pair[i], 1);
        }
        for (int i = 0; i < C::NR; ++i) {
            hs::mbar_init(&B.full_rope[i], kLoaderThreads);
            hs::mbar_init(&B.empty_rope[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            hs::mbar_init(&B.s_full[i], 1);
            hs::mbar_init(&B.p_full[i], 128);
            hs::mbar_init(&B.pv_done[i], 1);
        }
        hs::mbar_init(&B.drain, 1);
        hs::mbar_init(&B.group, 128);
        B.abort = 0;
        hs::fence_mbar_init();
    }
    if (warp == 8) {
        hs::tc::tmem_alloc(&B.tmem_base, C::kTmemCols);
        hs::tc::tmem_relinquish();
    }
    // Q rows of this head group -> 9 swizzled K-major blocks of [HG x 64].
    {
        const __nv_bfloat16* qg = a.q + (int64_t(row) * a.heads + head0) * 576;
        for (int e = tid; e < HG * 72; e += kThreads) {
            const int h = e / 72, c = e % 72;
            const int b = c >> 3, cc = c & 7;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(qg + int64_t(h) * 576) + c);
            *reinterpret_cast<uint4*>(smem + C::kQOff + b * HG * 128 + h * 128 +
                                      ((cc ^ (h & 7)) << 4)) = v;
        }
        hs::fence_proxy_async_shared();
    }
    hs::tc::fence_before_sync();
    __syncthreads();
    hs::tc::fence_after_sync();
    const uint32_t tmem = B.tmem_base;

    if (warp >= 4 && warp < 8) {
        // ------------------------------ loaders ------------------------------
        const int lt = tid - 128;
        const int c = lt & 7;          // 16-byte chunk of a 128-byte block row
        const int r0 = lt >> 3;        // rows r0 + 16 i, i < 8
        const uint32_t swz = uint32_t((c ^ (r0 & 7)) << 4);
        bool bad = false;
        for (int it = 0; it < T && !*abort_flag; ++it) {
            const int jt = (t_begin + it) * kTok;
            const char* src[8];
            uint32_t sz[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = jt + r0 + 16 * i;
                int64_t idx = j < n ? int64_t(__ldg(kv_rows + j)) : -1;
                if (idx >= a.num_kv_rows) { bad = true; idx = -1; }
                sz[i] = idx >= 0 ? 16u : 0u;
                src[i] = reinterpret_cast<const char*>(a.kv) +
                         (idx >= 0 ? idx : 0) * a.row_stride * 2 + c * 16;
            }
            bool ok = true;
            for (int half = 0; half < 4 && ok; ++half) {
                const int u = it * 4 + half;
                const int p = u % C::NP;
                if (!hs::mbar_wait_bounded(&B.empty_pair[p], ((u / C::NP) & 1) ^ 1, tmo,
                                           abort_flag)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                    const int blk = 2 * half + bb;
                    const uint32_t dst = pair_base + p * kPair + bb * kBlk + r0 * 128 + swz;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        hs::tc::cp_async16(dst + i * 16 * 128, src[i] + blk * 128, sz[i]);
                    hs::tc::cp_async_arrive_noinc(&B.full_pair[p][bb]);
                }
            }
            if (ok) {
                const int rs = it % C::NR;
                if (!hs::mbar_wait_bounded(&B.empty_rope[rs], ((it / C::NR) & 1) ^ 1, tmo,
                                           abort_flag)) {
                    ok = false;
                } else {
                    const uint32_t dst = rope_base + rs * kBlk + r0 * 128 + swz;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        hs::tc::cp_async16(dst + i * 16 * 128, src[i] + 8 * 128, sz[i]);
                    hs::tc::cp_async_arrive_noinc(&B.full_rope[rs]);
                }
            }
            if (!ok) {
                hs::set_status(a.status, HS_ERR_TIMEOUT);
                B.abort = 1;
            }
        }
        if (bad) hs::set_status(a.status, HS_ERR_BAD_INDEX);
        hs::tc::cp_async_wait_all();
    } else if (warp == 8) {
        // ---------------------------- MMA issuer -----------------------------
        if (lane == 0) {
            constexpr uint32_t idesc_qk = hs::tc::idesc_bf16(128, HG, 0, 0);
            constexpr uint32_t idesc_pv = hs::tc::idesc_bf16(128, HG, 1, 0);
            bool ok = true;
            auto issue_pv = [&](int it) -> bool {
                const int sb = it & 1;
                if (!hs::mbar_wait_bounded(&B.p_full[sb], (it >> 1) & 1, tmo, abort_flag))
                    return false;
                hs::fence_proxy_async_shared();
                hs::tc::fence_after_sync();
                const uint32_t pbuf =
                    C::kPInRope ? rope_base + (it % C::NR) * kBlk : p_base + sb * C::kPBytes;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t vbase = pair_base + ((it * 4 + c) % C::NP) * kPair;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = hs::tc::sdesc_sw128(vbase + kk * 2048, kBlk, 1024);
                        const uint64_t bd = hs::tc::sdesc_sw128(
                            pbuf + (kk >> 2) * HG * 128 + (kk & 3) * 32, 16, 1024);
                        hs::tc::mma_bf16(tmem + C::kO + c * HG, ad, bd, idesc_pv,
                                         (it > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                hs::tc::mma_commit(&B.pv_done[sb]);
#pragma unroll
                for (int c = 0; c < 4; ++c) hs::tc::mma_commit(&B.empty_pair[(it * 4 + c) % C::NP]);
                if (C::kPInRope) hs::tc::mma_commit(&B.empty_rope[it % C::NR]);
                return true;
            };
            auto issue_qk = [&](int it) -> bool {
                const int sb = it & 1;
                for (int b = 0; b < kNB; ++b) {
                    uint32_t abase;
                    bool got;
                    if (b < 8) {
                        const int u = it * 4 + (b >> 1);
                        const int p = u % C::NP;
                        got = hs::mbar_wait_bounded(&B.full_pair[p][b & 1], (u / C::NP) & 1, tmo,
                                                    abort_flag);
                        abase = pair_base + p * kPair + (b & 1) * kBlk;
                    } else {
                        const int rs = it % C::NR;
                        got = hs::mbar_wait_bounded(&B.full_rope[rs], (it / C::NR) & 1, tmo,
                                                    abort_flag);
                        abase = rope_base + rs * kBlk;
                    }
                    if (!got) return false;
                    hs::fence_proxy_async_shared();
                    hs::tc::fence_after_sync();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t ad = hs::tc::sdesc_sw128(abase + k * 32, 16, 1024);
                        const uint64_t bd =
                            hs::tc::sdesc_sw128(q_base + b * HG * 128 + k * 32, 16, 1024);
                        hs::tc::mma_bf16(tmem + C::kD1 + sb * HG, ad, bd, idesc_qk,
                                         (b | k) ? 1u : 0u);
                    }
                }
                if (!C::kPInRope) hs::tc::mma_commit(&B.empty_rope[it % C::NR]);
                hs::tc::mma_commit(&B.s_full[sb]);
                return true;
            };
            // Tile it+1 needs the ring slots that PV(it) releases, so PV(it)
            // is issued before QK(it+1).
            if (T > 0) ok = issue_qk(0);
            for (int it = 0; it < T && ok; ++it) {
                ok = issue_pv(it);
                if (ok && it + 1 < T) ok = issue_qk(it + 1);
            }
            if (!ok) {
                hs::set_status(a.status, HS_ERR_TIMEOUT);
                B.abort = 1;
            }
            // Drain: every MMA issued above has completed before TMEM is freed.
            hs::tc::mma_commit(&B.drain);
            hs::mbar_wait_bounded(&B.drain, 0, tmo, nullptr);
        }
        __syncwarp();
    } else {
        // ----------------------- softmax / epilogue (warps 0-3) ---------------
        const uint32_t lane_base = uint32_t(warp * 32) << 16;
        float m_ref[HG], l_part[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) {
            m_ref[h] = -CUDART_INF_F;
            l_part[h] = 0.f;
        }
        uint32_t gphase = 0;
        bool ok = true;
        // Bounded barrier of the 128 softmax threads (one mbarrier, 128 arrivals).
        auto group_sync = [&]() -> bool {
            hs::mbar_arrive(&B.group);
            const bool r = hs::mbar_wait_bounded(&B.group, gphase & 1, tmo, abort_flag);
            ++gphase;
            return r;
        };
        for (int it = 0; it < T && ok; ++it) {
            const int sb = it & 1;
            if (!hs::mbar_wait_bounded(&B.s_full[sb], (it >> 1) & 1, tmo, abort_flag)) {
                ok = false;
                break;
            }
            hs::tc::fence_after_sync();
            float s[HG];
            tmem_ld_row<HG>(tmem + lane_base + C::kD1 + sb * HG, s);
            hs::tc::tmem_wait_ld();
            const int j = (t_begin + it) * kTok + tid;
            bool valid = false;
            if (j < n) {
                const int32_t idx = __ldg(kv_rows + j);
                valid = idx >= 0 && int64_t(idx) < a.num_kv_rows;
            }
            uint32_t m0 = 0, m1 = 0;
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                s[h] = valid ? s[h] * a.scale_log2 : -CUDART_INF_F;
                if (s[h] > m_ref[h] + kThresh) {
                    if (h < 32) m0 |= 1u << h; else m1 |= 1u << (h - 32);
                }
            }
            m0 = __reduce_or_sync(0xffffffffu, m0);
            m1 = __reduce_or_sync(0xffffffffu, m1);
            if (lane == 0) {
                B.vote[sb][warp][0] = m0;
                B.vote[sb][warp][1] = m1;
            }
            if (!group_sync()) { ok = false; break; }
            m0 = B.vote[sb][0][0] | B.vote[sb][1][0] | B.vote[sb][2][0] | B.vote[sb][3][0];
            m1 = B.vote[sb][0][1] | B.vote[sb][1][1] | B.vote[sb][2][1] | B.vote[sb][3][1];
            if (m0 | m1) {
                // Exact tile maximum of the flagged heads, then rescale O and l.
#pragma unroll
                for (int h = 0; h < HG; ++h) {
                    const bool f = h < 32 ? (m0 >> h) & 1 : (m1 >> (h - 32)) & 1;
                    if (f) {
                        const float v = warp_max(s[h]);
                        if (lane == 0) B.red[warp][h] = v;
                    }
                }
                if (!group_sync()) { ok = false; break; }
                float alpha[HG];
#pragma unroll
                for (int h = 0; h < HG; ++h) {
                    alpha[h] = 1.f;
                    const bool f = h < 32 ? (m0 >> h) & 1 : (m1 >> (h - 32)) & 1;
                    if (f) {
                        const float tmax = fmaxf(fmaxf(B.red[0][h], B.red[1][h]),
                                                 fmaxf(B.red[2][h], B.red[3][h]));
                        const float mn = fmaxf(m_ref[h], tmax);
                        alpha[h] = m_ref[h] == -CUDART_INF_F ? 0.f : exp2f(m_ref[h] - mn);
                        m_ref[h] = mn;
                        l_part[h] *= alpha[h];
                    }
                }
                if (it > 0) {
                    // O holds PV(0..it-1): wait for PV(it-1), then rescale in TMEM.
                    if (!hs::mbar_wait_bounded(&B.pv_done[(it - 1) & 1], ((it - 1) >> 1) & 1,
                                               tmo, abort_flag)) {
                        ok = false;
                        break;
                    }
                    hs::tc::fence_after_sync();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float o[HG];
                        const uint32_t ta = tmem + lane_base + C::kO + c * HG;
                        tmem_ld_row<HG>(ta, o);
                        hs::tc::tmem_wait_ld();
#pragma unroll
                        for (int h = 0; h < HG; ++h) o[h] *= alpha[h];
                        tmem_st_row<HG>(ta, o);
                    }
                    hs::tc::tmem_wait_st();
                }
                // The red[] values are re-written only after the next group_sync.
            }
            // P^T tile, bf16, K-major: row h, token column tid.
            if (!C::kPInRope && it >= 2) {
                if (!hs::mbar_wait_bounded(&B.pv_done[sb], ((it - 2) >> 1) & 1, tmo, abort_flag)) {
                    ok = false;
                    break;
                }
            }
            const uint32_t pbuf = C::kPInRope ? C::kRopeOff + (it % C::NR) * kBlk
                                              : C::kPOff + sb * C::kPBytes;
            unsigned char* prow = smem + pbuf + (tid >> 6) * HG * 128;
            const int tcol = (tid & 63) * 2;
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                // A masked logit contributes 0 (also while m_ref is still -inf).
                const float p = s[h] == -CUDART_INF_F ? 0.f : exp2f(s[h] - m_ref[h]);
                const __nv_bfloat16 pb = __float2bfloat16_rn(p);
                l_part[h] += __bfloat162float(pb);
                *reinterpret_cast<__nv_bfloat16*>(prow + h * 128 +
                                                  ((((tcol >> 4) ^ (h & 7)) << 4) | (tcol & 15))) =
                    pb;
            }
            hs::fence_proxy_async_shared();
            hs::tc::fence_before_sync();
            hs::mbar_arrive(&B.p_full[sb]);
        }
        // Epilogue.
        if (ok && T > 0) {
            ok = hs::mbar_wait_bounded(&B.pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, tmo,
                                       abort_flag);
        }
        if (!ok) {
            hs::set_status(a.status, HS_ERR_TIMEOUT);
            B.abort = 1;
        } else {
            hs::tc::fence_after_sync();
            // l: per-lane partial sums -> per-head totals.
            float L[HG];
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                const float v = warp_sum(l_part[h]);
                L[h] = v;
            }
            // Reuse red[] only after every thread passed its last use.
            if (group_sync()) {
                if (lane == 0) {
#pragma unroll
                    for (int h = 0; h < HG; ++h) B.red[warp][h] = L[h];
                }
                if (group_sync()) {
#pragma unroll
                    for (int h = 0; h < HG; ++h)
                        L[h] = B.red[0][h] + B.red[1][h] + B.red[2][h] + B.red[3][h];
                    const int64_t qh0 = int64_t(row) * a.heads + head0;
                    // Eq. (7) with earlier partial states of the same rows (the
                    // resident-row pass): weights of every part, per head.
                    const int cp = min(a.combine_parts, kMaxCombine);
                    if (cp > 0) {
                        // Per-head merge weights, computed once (thread h) into smem.
                        if (tid < HG) {
                            float Lh = 0.f, Mo = -CUDART_INF_F;
#pragma unroll
                            for (int h = 0; h < HG; ++h)
                                if (h == tid) { Lh = L[h]; Mo = m_ref[h]; }
                            const int64_t base = (qh0 + tid) * a.part_stride;
                            float mp[kMaxCombine], lp[kMaxCombine];
                            float M = Lh > 0.f ? Mo : -CUDART_INF_F;
#pragma unroll
                            for (int pp = 0; pp < kMaxCombine; ++pp) {
                                mp[pp] = pp < cp ? a.part_m[base + pp] : -CUDART_INF_F;
                                lp[pp] = pp < cp ? a.part_l[base + pp] : 0.f;
                                if (lp[pp] > 0.f) M = fmaxf(M, mp[pp]);
                            }
                            float Lt = 0.f, wo = 0.f;
                            float* w = B.cw[tid];
#pragma unroll
                            for (int pp = 0; pp < kMaxCombine; ++pp) w[2 + pp] = 0.f;
                            if (M != -CUDART_INF_F) {
                                wo = Lh > 0.f ? exp2f(Mo - M) : 0.f;
                                Lt = wo * Lh;
#pragma unroll
                                for (int pp = 0; pp < kMaxCombine; ++pp) {
                                    if (lp[pp] > 0.f) {
                                        w[2 + pp] = exp2f(mp[pp] - M);
                                        Lt = fmaf(w[2 + pp], lp[pp], Lt);
                                    }
                                }
                            }
                            w[0] = wo;
                            w[1] = Lt > 0.f ? 1.f / Lt : 0.f;
                            if (a.lse != nullptr)
                                a.lse[qh0 + tid] = Lt > 0.f ? (M + log2f(Lt)) * 0.6931471805599453f
                                                            : -CUDART_INF_F;
                        }
                        if (!group_sync()) {
                            hs::set_status(a.status, HS_ERR_TIMEOUT);
                            B.abort = 1;
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float o[HG];
                        if (T > 0) {
                            tmem_ld_row<HG>(tmem + lane_base + C::kO + c * HG, o);
                            hs::tc::tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int h = 0; h < HG; ++h) o[h] = 0.f;
                        }
                        const int d = c * 128 + tid;
                        if (cp > 0) {
#pragma unroll
                            for (int h = 0; h < HG; ++h) {
                                const int64_t base = (qh0 + h) * a.part_stride;
                                const float* w = B.cw[h];
                                float acc = w[0] * o[h];
#pragma unroll
                                for (int pp = 0; pp < kMaxCombine; ++pp)
                                    if (pp < cp && w[2 + pp] != 0.f)
                                        acc = fmaf(w[2 + pp], a.part_o[(base + pp) * 512 + d], acc);
                                a.out[(qh0 + h) * 512 + d] = __float2bfloat16_rn(acc * w[1]);
                            }
                            continue;
                        }
#pragma unroll
                        for (int h = 0; h < HG; ++h) {
                            const int64_t qh = qh0 + h;
                            if (a.splits == 1 && !a.force_partial) {
                                a.out[qh * 512 + d] =
                                    __float2bfloat16_rn(L[h] > 0.f ? o[h] / L[h] : 0.f);
                            } else {
                                a.part_o[(qh * a.part_stride + a.part_base + split) * 512 + d] =
                                    L[h] > 0.f ? o[h] : 0.f;
                            }
                        }
                    }
                    if (tid < HG && cp == 0) {
                        float Lh = 0.f, Mh = -CUDART_INF_F;
#pragma unroll
                        for (int h = 0; h < HG; ++h)
                            if (h == tid) { Lh = L[h]; Mh = m_ref[h]; }
                        const int64_t qh = qh0 + tid;
                        if (a.splits == 1 && !a.force_partial) {
                            if (a.lse)
                                a.lse[qh] = Lh > 0.f ? (Mh + log2f(Lh)) * 0.6931471805599453f
                                                     : -CUDART_INF_F;
                        } else {
                            const int64_t pi = qh * a.part_stride + a.part_base + split;
                            a.part_m[pi] = Lh > 0.f ? Mh : -CUDART_INF_F;
                            a.part_l[pi] = Lh;
                        }
                    }
                }
            }
        }
        hs::tc::fence_before_sync();
    }
    __syncthreads();
    if (warp == 8) {
        hs::tc::fence_after_sync();
        hs::tc::tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int HG>
int launch_hg(const MlaArgs& a, dim3 grid, hs_stream_t stream) {
    using C = Cfg<HG>;
    static_assert(C::kBarOff + int(sizeof(Bars)) + 1024 <= 227 * 1024, "shared memory budget");
    const size_t smem = size_t(C::kBarOff) + sizeof(Bars) + 1024;
    static int smem_set[64] = {};
    const int rc = hs_host::ensure_dynamic_smem(reinterpret_cast<const void*>(mla_tc_kernel<HG>),
                                                smem, smem_set);
    if (rc != HS_OK) return rc;
    mla_tc_kernel<HG><<<grid, kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    return hs_host::launch_status();
}

}  // namespace

int mla_tc_head_group(int heads) {
    if (heads % 64 == 0) return 64;
    if (heads % 32 == 0) return 32;
    if (heads % 16 == 0) return 16;
    return 0;
}

int launch_mla_tc(const MlaArgs& a, int hg, dim3 grid, hs_stream_t stream) {
    switch (hg) {
        case 16: return launch_hg<16>(a, grid, stream);
        case 32: return launch_hg<32>(a, grid, stream);
        case 64: return launch_hg<64>(a, grid, stream);
        default: return HS_ERR_UNSUPPORTED;
    }
}

}  // namespace hs_attn
