// hs_attention_mla.cu -- S4 for MLA rows (576 bf16: K = all 576 columns,
// V = the first 512) on the 5th-generation tensor cores.
//
// Math: PaperTrace 5.1.1 "从索引到 Kernel" section 3.1 eqs. (4)-(6) (tile
// logits, running maximum and exponent sums, rescaled accumulator), section
// 3.2 (mask before the exponent; empty set -> zero output, LSE = -inf) and
// eq. (7) (split-KV merge, done by merge_kernel in hs_attention.cu or in this
// kernel's epilogue); "PagedAttention 与 RadixAttention" section 1.4 (exp2
// with scale * log2 e).
//
// GB300 design.  One CTA per (index row, group of HG query heads, split of
// the row's candidate list); 128 candidate rows form a tile.
//  * Two loader warps gather the tile's rows straight from the paged or hot
//    cache (no scratch gather, PaperTrace section 2.1 eq. (3)) with 16-byte
//    cp.async into 128-byte-swizzled K-major blocks of 128 rows x 64 columns;
//    invalid rows are zero-filled, never read.  Blocks travel in pair units
//    (32 KB) through a ring of NU units in the order the MMA thread consumes
//    them: QK(0), then per tile QK(t+1) and PV(t).  A QK unit holds two K
//    blocks (the ninth, RoPE, block travels alone); a PV unit holds the two
//    V blocks of one 128-wide slice of d, gathered a second time (from L2:
//    the same rows were read one tile earlier).  Re-reading V instead of
//    keeping the 144 KB tile resident keeps several units in flight per SM,
//    so the gathers of the next tile overlap this tile's softmax and MMAs.
//    The first tile's units that own a ring slot are filled by the loader
//    and softmax warps together (the softmax warps wait for its logits in
//    any case); the list's length and ids are prefetched into L2 before the
//    launch-chain wait.
//  * Splits of a list merge with eq. (7) in the epilogue of the split that
//    finishes last (arrival counter, partial states read from L2, every
//    column group's loads in flight at once).
//  * One MMA thread issues tcgen05.mma: S^T[128 tokens x HG] = K Q^T (M = 128
//    tokens, N = HG heads, K = 576) into one of two TMEM buffers, and
//    O^T[512 x HG] += V^T P^T (four M = 128 slices of d, K = 128 tokens, V
//    as an MN-major view of the pair unit).  Commits release ring units.
//  * Eight softmax warps: warp w reads TMEM lane quarter w % 4 (32 tokens)
//    and head half w / 4 (HG / 2 heads).  Each keeps a per-head reference
//    maximum; a tile rescales O (in TMEM) only when some logit exceeds the
//    reference by more than 2^8 (a warp vote, combined per head half), so the
//    common tile needs no cross-thread max reduction.  The exponent sums stay
//    in registers per token lane and are reduced once in the epilogue.
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
constexpr int kUnit = 2 * kBlk;     // one ring unit: two blocks
constexpr int kSoftWarps = 8;
constexpr int kLoadWarps = 2;
constexpr int kMmaWarp = kSoftWarps + kLoadWarps;
constexpr int kThreads = (kMmaWarp + 1) * 32;  // 352 (168 registers per thread)
constexpr int kLoadRows = kTok * 8 / (kLoadWarps * 32);  // rows per loader thread and block
constexpr int kLoaderThreads = kLoadWarps * 32;
constexpr int kSoftThreads = kSoftWarps * 32;
// Threads that fill the first tile's QK units: the loaders and the softmax
// warps (which have nothing to do before the first logits).  Every ring
// barrier counts this many arrivals; a unit the loaders fill alone gets the
// softmax threads' share from one loader thread.
constexpr int kFillThreads = kLoaderThreads + kSoftThreads;
constexpr int kHalfThreads = kSoftWarps * 16;  // softmax threads of one head half
constexpr float kThresh = 8.0f;     // log2 headroom before O is rescaled
constexpr int kMaxCombine = 4;      // partial columns a finishing pass can merge
constexpr int kQkUnits = 5;         // 4 K pairs + the RoPE block
constexpr int kPvUnits = 4;         // 4 V pairs
constexpr int kSmemLimit = 227 * 1024;
constexpr int kBarBytes = 6144;     // shared-memory budget of Bars

template <int HG>
struct Cfg {
    static constexpr int HH = HG / 2;                  // heads per softmax thread
    static constexpr int kQBytes = kNB * HG * 128;
    static constexpr int kPBytes = 2 * HG * 128;       // P^T: [2 token halves][HG][128 B]
    static constexpr int kFixed = kQBytes + kPBytes + kBarBytes + 1024;  // + alignment
    static constexpr int NU = (kSmemLimit - kFixed) / kUnit > 6 ? 6 : (kSmemLimit - kFixed) / kUnit;
    static constexpr int kRingOff = 0;
    static constexpr int kQOff = kRingOff + NU * kUnit;
    static constexpr int kPOff = kQOff + kQBytes;
    static constexpr int kBarOff = kPOff + kPBytes;
    static constexpr int kTmemCols = 6 * HG <= 128 ? 128 : (6 * HG <= 256 ? 256 : 512);
    static constexpr int kS = 0;                       // S^T buffers: cols [0, 2HG)
    static constexpr int kO = 2 * HG;                  // O^T slices: cols [2HG, 6HG)
    static_assert(NU >= 2, "ring needs two units");
};

struct Bars {
    uint64_t full[6][2];     // per block of a ring unit (one arrival per loader thread)
    uint64_t empty[6];       // ring unit consumed (MMA commit)
    uint64_t s_full[2];      // S^T buffer written (MMA commit)
    uint64_t p_full;         // P^T written (256 softmax arrivals)
    uint64_t pv_done[2];     // PV(t) complete (MMA commit), by t & 1
    uint64_t drain;
    uint64_t group[2];       // barrier of one head half (128 arrivals)
    uint64_t group_all;      // barrier of the 256 softmax threads
    uint32_t tmem_base;
    int32_t abort;
    int32_t last;            // this CTA arrived last for its (row, head group)
    uint32_t vote[2][2][4];  // [t & 1][half][quarter]
    float red[2][4][32];     // [half][quarter][head of the half]
    float alpha[2][32];      // O rescale factors of a rescaling tile, [half][head]
    float mref[2][2][32];    // reference maxima (log2 units), [buffer][half][head]
    // Merge weights per head: the fused finish uses w_own, 1/L_total,
    // w_part[4]; the last-CTA merge uses w[0 .. kMlaMaxMerge) and 1/L_total
    // at kMlaMaxMerge.
    float cw[64][kMlaMaxMerge + 2];
};
static_assert(sizeof(Bars) <= kBarBytes, "barrier block");

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

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
    if constexpr (N == 8) {
        hs::tc::tmem_ld8(taddr, v);
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 16) {
            float t[16];
            hs::tc::tmem_ld16(taddr + c, t);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[c + i] = t[i];
        }
    }
}

// Position of unit `u` of tile `t`'s QK (is_pv = 0) or PV (is_pv = 1) in the
// consumption sequence QK(0), {QK(t+1), PV(t)} for t = 0.. T-1.
__device__ __forceinline__ int unit_seq(int t, int is_pv, int u, int T) {
    if (!is_pv) return t == 0 ? u : kQkUnits + (t - 1) * (kQkUnits + kPvUnits) + u;
    // PV(t) follows QK(t+1) when that exists.
    const int before = kQkUnits + t * (kQkUnits + kPvUnits) + (t + 1 < T ? kQkUnits : 0);
    return before + u;
}

template <int HG>
__global__ void __launch_bounds__(kThreads, 1) mla_tc_kernel(const MlaArgs a) {
    using C = Cfg<HG>;
    constexpr int HH = C::HH;
    constexpr int NU = C::NU;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment of the swizzle atoms.
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars& B = *reinterpret_cast<Bars*>(smem + C::kBarOff);
    const uint32_t s_base = hs::smem_u32(smem);
    const uint32_t ring_base = s_base + C::kRingOff;
    const uint32_t q_base = s_base + C::kQOff;
    const uint32_t p_base = s_base + C::kPOff;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int groups = a.heads / HG;
    const int row = blockIdx.x / groups;
    const int grp = blockIdx.x % groups;
    const int split = blockIdx.y;
    const int32_t* kv_rows = a.kv_rows + int64_t(row) * a.cap;
    const int head0 = grp * HG;
    const uint64_t tmo = a.timeout_ns;
    volatile int* abort_flag = &B.abort;

    // Set-up that needs nothing from the stream predecessor (barriers, TMEM,
    // the query) runs before pdl_wait.
    hs::pdl_trigger();
    if (tid == 0) {
        for (int i = 0; i < NU; ++i) {
            hs::mbar_init(&B.full[i][0], kFillThreads);
            hs::mbar_init(&B.full[i][1], kFillThreads);
            hs::mbar_init(&B.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            hs::mbar_init(&B.s_full[i], 1);
            hs::mbar_init(&B.pv_done[i], 1);
            hs::mbar_init(&B.group[i], kHalfThreads);
        }
        hs::mbar_init(&B.p_full, kSoftWarps * 32);
        hs::mbar_init(&B.group_all, kSoftWarps * 32);
        hs::mbar_init(&B.drain, 1);
        for (int i = 0; i < 64; ++i) B.mref[0][i >> 5][i & 31] = -CUDART_INF_F;
        B.abort = 0;
        hs::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        hs::tc::tmem_alloc(&B.tmem_base, C::kTmemCols);
        hs::tc::tmem_relinquish();
    }
    // Q rows of this head group -> 9 swizzled K-major blocks of [HG x 64],
    // copied asynchronously (all copies in flight at once).
    {
        const __nv_bfloat16* qg = a.q + (int64_t(row) * a.heads + head0) * 576;
        for (int e = tid; e < HG * 72; e += kThreads) {
            const int h = e / 72, c = e % 72;
            const int b = c >> 3, cc = c & 7;
            hs::tc::cp_async16(q_base + b * HG * 128 + h * 128 + ((cc ^ (h & 7)) << 4),
                               qg + int64_t(h) * 576 + c * 8, 16u);
        }
        hs::tc::cp_async_wait_all();
        hs::fence_proxy_async_shared();
    }
    // The count and this row's candidate ids may still be written by a stream
    // predecessor: an L2 prefetch (it returns no data) of their lines lets the
    // loads after the wait hit L2.
    {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(kv_rows) & ~uintptr_t(127);
        const uintptr_t hi = reinterpret_cast<uintptr_t>(kv_rows + a.cap);
        for (uintptr_t p = lo + uintptr_t(tid) * 128; p < hi; p += uintptr_t(kThreads) * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
        if (tid == 0 && a.count != nullptr)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a.count + row));
    }
    hs::pdl_wait();
    const int n = a.count ? min(max(a.count[row], 0), a.cap) : a.cap;
    const int ntiles = (n + kTok - 1) / kTok;
    const int per = (ntiles + a.splits - 1) / a.splits;
    const int t_begin = min(ntiles, split * per);
    const int T = min(ntiles, t_begin + per) - t_begin;  // tiles of this CTA
    // A CTA with one tile keeps the four K-pair units of QK(0) (blocks 0-7 =
    // the V columns) for PV(0) instead of gathering V again, when the ring
    // holds all five QK units at once (16 and 32 heads per CTA); with more
    // tiles the ring is needed for the next QK, so V is re-gathered.
    const bool reuse_v = T == 1 && NU >= kQkUnits;
    hs::tc::fence_before_sync();
    __syncthreads();
    hs::tc::fence_after_sync();
    const uint32_t tmem = B.tmem_base;
    // The first tile's QK units that own their ring slot (units k < NU, phase
    // 0: no wait for a release), filled by the loader and softmax threads
    // together; `gt` in [0, kFillThreads) takes the 16-byte chunks e = gt +
    // kFillThreads i of every block (row e / 8, chunk e % 8).
    constexpr int kFirstUnits = NU < kQkUnits ? NU : kQkUnits;
    auto fill_first = [&](int gt) {
        constexpr int kPer = (kTok * 8 + kFillThreads - 1) / kFillThreads;
        const int jt = t_begin * kTok;
        int32_t id[kPer];
        bool bad0 = false;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = gt + kFillThreads * i;
            const int j = jt + (e >> 3);
            id[i] = (e < kTok * 8 && j < n) ? __ldg(kv_rows + j) : -1;
            if (int64_t(id[i]) >= a.num_kv_rows) bad0 = true;
        }
#pragma unroll 1
        for (int u = 0; u < kFirstUnits; ++u) {
            const uint32_t ub = ring_base + u * kUnit;
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const int blk = 2 * u + bb;
                if (blk >= kNB) break;
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int e = gt + kFillThreads * i;
                    if (e >= kTok * 8) continue;
                    const int r = e >> 3, c = e & 7;
                    const bool v = id[i] >= 0 && int64_t(id[i]) < a.num_kv_rows;
                    const char* src = reinterpret_cast<const char*>(a.kv) +
                                      (v ? int64_t(id[i]) : 0) * a.row_stride * 2 + blk * 128 +
                                      c * 16;
                    hs::tc::cp_async16(ub + bb * kBlk + r * 128 + ((c ^ (r & 7)) << 4), src,
                                       v ? 16u : 0u);
                }
            }
            hs::tc::cp_async_arrive_noinc(&B.full[u][0]);
            hs::tc::cp_async_arrive_noinc(&B.full[u][1]);
        }
        if (bad0) hs::set_status(a.status, HS_ERR_BAD_INDEX);
    };

    if (warp >= kSoftWarps && warp < kMmaWarp) {
        // ------------------------------ loaders ------------------------------
        const int lt = tid - kSoftWarps * 32;
        constexpr int kRowStep = kLoaderThreads / 8;
        const int c = lt & 7;          // 16-byte chunk of a 128-byte block row
        const int r0 = lt >> 3;        // rows r0 + kRowStep * i, i < kLoadRows
        const uint32_t swz = uint32_t((c ^ (r0 & 7)) << 4);
        bool bad = false;
        // Row ids of four tiles: PV(t) uses tile t, QK(t+1) tile t+1, and the
        // ids of tiles t+2 and t+3 are in flight (fetched two steps ahead).
        int32_t id_prev[kLoadRows], id_cur[kLoadRows], id_next[kLoadRows], id_far[kLoadRows];
        auto fetch = [&](int t, int32_t (&id)[kLoadRows]) {
            const int jt = (t_begin + t) * kTok;
#pragma unroll
            for (int i = 0; i < kLoadRows; ++i) {
                const int j = jt + r0 + kRowStep * i;
                id[i] = (t < T && j < n) ? __ldg(kv_rows + j) : -1;
            }
        };
        // Fills unit `k` of the sequence with blocks b0 (and b1 >= 0) of the
        // rows `id`; invalid ids zero-fill.
        auto fill = [&](int k, const int32_t (&id)[kLoadRows], int b0, int b1) -> bool {
            const int slot = k % NU;
            if (!hs::mbar_wait_bounded(&B.empty[slot], ((k / NU) & 1) ^ 1, tmo, abort_flag))
                return false;
            const uint32_t dst = ring_base + slot * kUnit + r0 * 128 + swz;
#pragma unroll
            for (int i = 0; i < kLoadRows; ++i) {
                const bool v = id[i] >= 0 && int64_t(id[i]) < a.num_kv_rows;
                const char* src = reinterpret_cast<const char*>(a.kv) +
                                  (v ? int64_t(id[i]) : 0) * a.row_stride * 2 + c * 16;
                hs::tc::cp_async16(dst + i * kRowStep * 128, src + b0 * 128, v ? 16u : 0u);
                if (b1 >= 0)
                    hs::tc::cp_async16(dst + kBlk + i * kRowStep * 128, src + b1 * 128,
                                       v ? 16u : 0u);
            }
            hs::tc::cp_async_arrive_noinc(&B.full[slot][0]);
            // The second block's barrier completes its phase in every unit.
            hs::tc::cp_async_arrive_noinc(&B.full[slot][1]);
            if (lt == 0) {
                // The softmax threads' share of the arrivals (they fill only
                // the first tile's units).
                hs::mbar_arrive_count(&B.full[slot][0], kSoftThreads);
                hs::mbar_arrive_count(&B.full[slot][1], kSoftThreads);
            }
            return true;
        };
        auto load_qk = [&](int t, const int32_t (&id)[kLoadRows], int u0) -> bool {
#pragma unroll
            for (int i = 0; i < kLoadRows; ++i)
                if (int64_t(id[i]) >= a.num_kv_rows) bad = true;
            const int k0 = unit_seq(t, 0, 0, T);
            for (int u = u0; u < kQkUnits; ++u)
                if (!fill(k0 + u, id, u < 4 ? 2 * u : 8, u < 4 ? 2 * u + 1 : -1)) return false;
            return true;
        };
        auto load_pv = [&](int t, const int32_t (&id)[kLoadRows]) -> bool {
            const int k0 = unit_seq(t, 1, 0, T);
            for (int u = 0; u < kPvUnits; ++u)
                if (!fill(k0 + u, id, 2 * u, 2 * u + 1)) return false;
            return true;
        };
        fetch(0, id_cur);
        fetch(1, id_next);
        fetch(2, id_far);
        if (T > 0) fill_first(kSoftThreads + lt);
        bool ok = T == 0 || load_qk(0, id_cur, kFirstUnits);
        for (int t = 0; t < T && ok; ++t) {
            // id_prev = tile t, id_cur = t + 1, id_next = t + 2, id_far = t + 3.
#pragma unroll
            for (int i = 0; i < kLoadRows; ++i) {
                id_prev[i] = id_cur[i];
                id_cur[i] = id_next[i];
                id_next[i] = id_far[i];
            }
            fetch(t + 3, id_far);
            if (t + 1 < T) ok = load_qk(t + 1, id_cur, 0);
            if (ok && !reuse_v) ok = load_pv(t, id_prev);
        }
        if (!ok) {
            hs::set_status(a.status, HS_ERR_TIMEOUT);
            B.abort = 1;
        }
        if (bad) hs::set_status(a.status, HS_ERR_BAD_INDEX);
        hs::tc::cp_async_wait_all();
    } else if (warp == kMmaWarp) {
        // ---------------------------- MMA issuer -----------------------------
        if (lane == 0) {
            constexpr uint32_t idesc_qk = hs::tc::idesc_bf16(128, HG, 0, 0);
            constexpr uint32_t idesc_pv = hs::tc::idesc_bf16(128, HG, 1, 0);
            auto wait_full = [&](int k, int b) -> bool {
                return hs::mbar_wait_bounded(&B.full[k % NU][b], (k / NU) & 1, tmo, abort_flag);
            };
            auto issue_qk = [&](int t) -> bool {
                const int sb = t & 1;
                const int k0 = unit_seq(t, 0, 0, T);
                for (int b = 0; b < kNB; ++b) {
                    const int k = k0 + (b >> 1);
                    if (!wait_full(k, b & 1)) return false;
                    // The RoPE unit's second barrier completes without data;
                    // it is waited too, so that no arrival of the unit can
                    // outlive the slot's release.
                    if (b == kNB - 1 && !wait_full(k, 1)) return false;
                    hs::tc::fence_after_sync();
                    const uint32_t abase = ring_base + (k % NU) * kUnit + (b & 1) * kBlk;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = hs::tc::sdesc_sw128(abase + kk * 32, 16, 1024);
                        const uint64_t bd =
                            hs::tc::sdesc_sw128(q_base + b * HG * 128 + kk * 32, 16, 1024);
                        hs::tc::mma_bf16(tmem + C::kS + sb * HG, ad, bd, idesc_qk,
                                         (b | kk) ? 1u : 0u);
                    }
                    if (((b & 1) && !reuse_v) || b == kNB - 1)
                        hs::tc::mma_commit(&B.empty[k % NU]);
                }
                hs::tc::mma_commit(&B.s_full[sb]);
                return true;
            };
            auto issue_pv = [&](int t) -> bool {
                if (!hs::mbar_wait_bounded(&B.p_full, t & 1, tmo, abort_flag)) return false;
                hs::tc::fence_after_sync();
                // V from the QK units themselves (one tile: their full
                // barriers' phases have completed) or from the PV units.
                const int k0 = reuse_v ? unit_seq(t, 0, 0, T) : unit_seq(t, 1, 0, T);
#pragma unroll 1
                for (int cs = 0; cs < kPvUnits; ++cs) {
                    const int k = k0 + cs;
                    if (!wait_full(k, 0) || !wait_full(k, 1)) return false;
                    hs::tc::fence_after_sync();
                    const uint32_t vbase = ring_base + (k % NU) * kUnit;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = hs::tc::sdesc_sw128(vbase + kk * 2048, kBlk, 1024);
                        const uint64_t bd = hs::tc::sdesc_sw128(
                            p_base + (kk >> 2) * HG * 128 + (kk & 3) * 32, 16, 1024);
                        hs::tc::mma_bf16(tmem + C::kO + cs * HG, ad, bd, idesc_pv,
                                         (t > 0 || kk > 0) ? 1u : 0u);
                    }
                    hs::tc::mma_commit(&B.empty[k % NU]);
                }
                hs::tc::mma_commit(&B.pv_done[t & 1]);
                return true;
            };
            bool ok = T == 0 || issue_qk(0);
            for (int t = 0; t < T && ok; ++t) {
                if (t + 1 < T) ok = issue_qk(t + 1);
                if (ok) ok = issue_pv(t);
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
        // ----------------------- softmax / epilogue (warps 0-7) ---------------
        const int qd = warp & 3;            // TMEM lane quarter = tokens qd*32 ..
        const int hf = warp >> 2;           // head half
        const int ht = qd * 32 + lane;      // thread index within the half
        const int hoff = hf * HH;           // first head (within the group) of the half
        const uint32_t lane_base = uint32_t(qd * 32) << 16;
        if (T > 0) fill_first(tid);
        // The reference maxima are the same for every thread of the half:
        // they live in shared memory (buffer msel), written by thread 0 of
        // the half into the other buffer when a tile rescales.
        float l_part[HH];
#pragma unroll
        for (int h = 0; h < HH; ++h) l_part[h] = 0.f;
        int msel = 0;
        uint32_t gphase = 0, aphase = 0;
        bool ok = true;
        // Bounded barrier of the 128 threads of this head half.
        auto group_sync = [&]() -> bool {
            hs::mbar_arrive(&B.group[hf]);
            const bool r = hs::mbar_wait_bounded(&B.group[hf], gphase & 1, tmo, abort_flag);
            ++gphase;
            return r;
        };
        // Row id of this thread's token in the current and the next tile
        // (fetched one tile ahead, off the softmax's critical path).
        auto token_id = [&](int t) -> int32_t {
            const int j = (t_begin + t) * kTok + qd * 32 + lane;
            return (t < T && j < n) ? __ldg(kv_rows + j) : -1;
        };
        int32_t id_next = token_id(0);
        // Bounded barrier of all 256 softmax threads.
        auto all_sync = [&]() -> bool {
            hs::mbar_arrive(&B.group_all);
            const bool r = hs::mbar_wait_bounded(&B.group_all, aphase & 1, tmo, abort_flag);
            ++aphase;
            return r;
        };
        for (int t = 0; t < T && ok; ++t) {
            const int sb = t & 1;
            const int32_t id_t = id_next;
            id_next = token_id(t + 1);
            if (!hs::mbar_wait_bounded(&B.s_full[sb], (t >> 1) & 1, tmo, abort_flag)) {
                ok = false;
                break;
            }
            hs::tc::fence_after_sync();
            float s[HH];
            tmem_ld_cols<HH>(tmem + lane_base + C::kS + sb * HG + hoff, s);
            hs::tc::tmem_wait_ld();
            const bool valid = id_t >= 0 && int64_t(id_t) < a.num_kv_rows;
            const float* m_ref = B.mref[msel][hf];
            uint32_t m0 = 0;
#pragma unroll
            for (int h = 0; h < HH; ++h) {
                s[h] = valid ? s[h] * a.scale_log2 : -CUDART_INF_F;
                if (s[h] > m_ref[h] + kThresh) m0 |= 1u << h;
            }
            m0 = __reduce_or_sync(0xffffffffu, m0);
            if (lane == 0) B.vote[sb][hf][qd] = m0;
            if (!group_sync()) { ok = false; break; }
            m0 = B.vote[sb][hf][0] | B.vote[sb][hf][1] | B.vote[sb][hf][2] | B.vote[sb][hf][3];
            bool pv_prev_done = t == 0;
            if (m0) {
                // Exact tile maximum of the flagged heads, then rescale O and l.
#pragma unroll
                for (int h = 0; h < HH; ++h) {
                    if ((m0 >> h) & 1) {
                        const float v = warp_max(s[h]);
                        if (lane == 0) B.red[hf][qd][h] = v;
                    }
                }
                if (!group_sync()) { ok = false; break; }
                // Every thread of the half computes the same factors; thread 0
                // of the half publishes them for the O rescale below (shared
                // memory keeps them out of the registers).
#pragma unroll
                for (int h = 0; h < HH; ++h) {
                    float al = 1.f;
                    float mn = m_ref[h];
                    if ((m0 >> h) & 1) {
                        const float tmax = fmaxf(fmaxf(B.red[hf][0][h], B.red[hf][1][h]),
                                                 fmaxf(B.red[hf][2][h], B.red[hf][3][h]));
                        mn = fmaxf(m_ref[h], tmax);
                        al = m_ref[h] == -CUDART_INF_F ? 0.f : exp2f(m_ref[h] - mn);
                        l_part[h] *= al;
                    }
                    if (ht == 0) {
                        B.alpha[hf][h] = al;
                        B.mref[msel ^ 1][hf][h] = mn;
                    }
                }
                if (!group_sync()) { ok = false; break; }
                msel ^= 1;
                m_ref = B.mref[msel][hf];
                if (t > 0) {
                    // O holds PV(0..t-1): wait for PV(t-1), then rescale in TMEM.
                    if (!hs::mbar_wait_bounded(&B.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, tmo,
                                               abort_flag)) {
                        ok = false;
                        break;
                    }
                    pv_prev_done = true;
                    hs::tc::fence_after_sync();
#pragma unroll 1
                    for (int cs = 0; cs < 4; ++cs) {
#pragma unroll
                        for (int hc = 0; hc < HH; hc += 8) {
                            float o[8];
                            const uint32_t ta = tmem + lane_base + C::kO + cs * HG + hoff + hc;
                            hs::tc::tmem_ld8(ta, o);
                            hs::tc::tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 8; ++i) o[i] *= B.alpha[hf][hc + i];
                            hs::tc::tmem_st8(ta, o);
                        }
                    }
                    hs::tc::tmem_wait_st();
                }
                // red[] is re-written only after the next group_sync.
            }
            // The single P^T buffer: PV(t-1) must have read it.
            if (!pv_prev_done) {
                if (!hs::mbar_wait_bounded(&B.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, tmo,
                                           abort_flag)) {
                    ok = false;
                    break;
                }
            }
            // P^T tile, bf16, K-major: row h, token column qd*32 + lane.  The
            // reference maxima are copied to registers first: read through the
            // shared-memory pointer inside the loop, each load would have to
            // wait for the P stores before it (possible aliasing).
            float mr[HH];
#pragma unroll
            for (int h = 0; h < HH; ++h) mr[h] = m_ref[h];
            const int tok = qd * 32 + lane;
            unsigned char* prow = smem + C::kPOff + (tok >> 6) * HG * 128;
            const int tcol = (tok & 63) * 2;
#pragma unroll
            for (int h = 0; h < HH; ++h) {
                const int hg = hoff + h;
                // A masked logit contributes 0 (also while m_ref is still -inf).
                const float p = s[h] == -CUDART_INF_F ? 0.f : exp2f(s[h] - mr[h]);
                const __nv_bfloat16 pb = __float2bfloat16_rn(p);
                l_part[h] += __bfloat162float(pb);
                *reinterpret_cast<__nv_bfloat16*>(
                    prow + hg * 128 + ((((tcol >> 4) ^ (hg & 7)) << 4) | (tcol & 15))) = pb;
            }
            hs::fence_proxy_async_shared();
            hs::tc::fence_before_sync();
            hs::mbar_arrive(&B.p_full);
        }
        // Epilogue.  (This thread's copies of the first tile are complete
        // before the CTA can exit.)
        hs::tc::cp_async_wait_all();
        if (ok && T > 0) {
            ok = hs::mbar_wait_bounded(&B.pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, tmo,
                                       abort_flag);
        }
        if (ok) {
            hs::tc::fence_after_sync();
            // l: per-lane partial sums -> per-head totals of this half.  red[]
            // is reused only after every thread of the half passed its last
            // use of it.
            ok = group_sync();
            if (ok) {
#pragma unroll
                for (int h = 0; h < HH; ++h) {
                    const float v = warp_sum(l_part[h]);
                    if (lane == 0) B.red[hf][qd][h] = v;
                }
                ok = group_sync();
            }
        }
        if (!ok) {
            hs::set_status(a.status, HS_ERR_TIMEOUT);
            B.abort = 1;
        } else {
            const int64_t qh0 = int64_t(row) * a.heads + head0;
            const int cp = min(a.combine_parts, kMaxCombine);
            // Thread ht < HH owns head hoff + ht: its total, maximum, the
            // output scale (shared memory, per head) and the LSE / partial
            // state.
            if (ht < HH) {
                const int h = ht;
                const float Lh = B.red[hf][0][h] + B.red[hf][1][h] + B.red[hf][2][h] +
                                 B.red[hf][3][h];
                const float Mh = B.mref[msel][hf][h];
                const int64_t qh = qh0 + hoff + h;
                float* w = B.cw[hoff + h];
                if (cp > 0) {
                    // Eq. (7) with earlier partial states of the same rows
                    // (the resident-row pass): weights of every part.
                    const int64_t base = qh * a.part_stride;
                    float mp[kMaxCombine], lp[kMaxCombine];
                    float M = Lh > 0.f ? Mh : -CUDART_INF_F;
#pragma unroll
                    for (int pp = 0; pp < kMaxCombine; ++pp) {
                        mp[pp] = pp < cp ? a.part_m[base + pp] : -CUDART_INF_F;
                        lp[pp] = pp < cp ? a.part_l[base + pp] : 0.f;
                        if (lp[pp] > 0.f) M = fmaxf(M, mp[pp]);
                    }
                    float Lt = 0.f, wo = 0.f;
#pragma unroll
                    for (int pp = 0; pp < kMaxCombine; ++pp) w[2 + pp] = 0.f;
                    if (M != -CUDART_INF_F) {
                        wo = Lh > 0.f ? exp2f(Mh - M) : 0.f;
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
                        a.lse[qh] = Lt > 0.f ? (M + log2f(Lt)) * 0.6931471805599453f
                                             : -CUDART_INF_F;
                } else if (a.splits == 1 && !a.force_partial) {
                    w[0] = 1.f;
                    w[1] = Lh > 0.f ? 1.f / Lh : 0.f;
                    if (a.lse)
                        a.lse[qh] = Lh > 0.f ? (Mh + log2f(Lh)) * 0.6931471805599453f
                                             : -CUDART_INF_F;
                } else {
                    // Unnormalised partial state; an empty part stores o = 0.
                    w[0] = Lh > 0.f ? 1.f : 0.f;
                    w[1] = 1.f;
                    const int64_t pi = qh * a.part_stride + a.part_base + split;
                    a.part_m[pi] = Lh > 0.f ? Mh : -CUDART_INF_F;
                    a.part_l[pi] = Lh;
                }
            }
            if (!group_sync()) {
                hs::set_status(a.status, HS_ERR_TIMEOUT);
                B.abort = 1;
            } else {
                const bool to_out = cp > 0 || (a.splits == 1 && !a.force_partial);
#pragma unroll 1
                for (int cs = 0; cs < 4; ++cs) {
                    const int d = cs * 128 + qd * 32 + lane;
#pragma unroll 1
                    for (int hc = 0; hc < HH; hc += 8) {
                        float o[8];
                        if (T > 0) {
                            hs::tc::tmem_ld8(tmem + lane_base + C::kO + cs * HG + hoff + hc, o);
                            hs::tc::tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; ++i) o[i] = 0.f;
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int hl = hoff + hc + i;
                            const int64_t qh = qh0 + hl;
                            const float* w = B.cw[hl];
                            float acc = w[0] * o[i];
                            if (cp > 0) {
#pragma unroll
                                for (int pp = 0; pp < kMaxCombine; ++pp)
                                    if (pp < cp && w[2 + pp] != 0.f)
                                        acc = fmaf(w[2 + pp],
                                                   a.part_o[(qh * a.part_stride + pp) * 512 + d],
                                                   acc);
                            }
                            if (to_out) {
                                a.out[qh * 512 + d] = __float2bfloat16_rn(acc * w[1]);
                            } else {
                                a.part_o[(qh * a.part_stride + a.part_base + split) * 512 + d] =
                                    acc;
                            }
                        }
                    }
                }
                // Split merge inside the kernel: every split has written its
                // partial column; the split that arrives last for this (row,
                // head group) merges columns [0, merge_total) with eq. (7)
                // (writes made visible with a fence before the arrival,
                // partials read from L2 after it).
                if (a.sync != nullptr) {
                    __threadfence();
                    bool last = false;
                    bool synced = all_sync();
                    if (synced) {
                        if (tid == 0) {
                            const int old = atomicAdd(a.sync + blockIdx.x, 1);
                            B.last = old == a.splits - 1 ? 1 : 0;
                            // Every split has arrived: the counter is reset
                            // for the next call.
                            if (old == a.splits - 1) a.sync[blockIdx.x] = 0;
                        }
                        synced = all_sync();
                        last = synced && B.last != 0;
                    }
                    if (!synced) {
                        hs::set_status(a.status, HS_ERR_TIMEOUT);
                        B.abort = 1;
                    }
                    if (last) {
                        __threadfence();
                        const int nc = min(a.merge_total, kMlaMaxMerge);
                        if (ht < HH) {
                            // Every column's (m, l) in one round of loads.
                            const int64_t qh = qh0 + hoff + ht;
                            const int64_t base = qh * a.part_stride;
                            float* w = B.cw[hoff + ht];
                            float mc[kMlaMaxMerge], lc[kMlaMaxMerge];
#pragma unroll
                            for (int c = 0; c < kMlaMaxMerge; ++c) {
                                lc[c] = c < nc ? __ldcg(a.part_l + base + c) : 0.f;
                                mc[c] = c < nc ? __ldcg(a.part_m + base + c) : -CUDART_INF_F;
                            }
                            float M = -CUDART_INF_F;
#pragma unroll
                            for (int c = 0; c < kMlaMaxMerge; ++c)
                                if (lc[c] > 0.f) M = fmaxf(M, mc[c]);
                            float Lt = 0.f;
#pragma unroll
                            for (int c = 0; c < kMlaMaxMerge; ++c) {
                                float wc = 0.f;
                                if (lc[c] > 0.f && M != -CUDART_INF_F) {
                                    wc = exp2f(mc[c] - M);
                                    Lt = fmaf(wc, lc[c], Lt);
                                }
                                w[c] = wc;
                            }
                            w[kMlaMaxMerge] = Lt > 0.f ? 1.f / Lt : 0.f;
                            if (a.lse != nullptr)
                                a.lse[qh] = Lt > 0.f ? (M + log2f(Lt)) * 0.6931471805599453f
                                                     : -CUDART_INF_F;
                        }
                        if (!group_sync()) {
                            hs::set_status(a.status, HS_ERR_TIMEOUT);
                            B.abort = 1;
                        } else {
                            // 16-byte chunks of d (128 per head), distributed over the
                            // half's 128 threads, kPer chunks per thread and pass; the
                            // loads of up to four columns are in flight at once, and
                            // each chunk accumulates the columns in order.
                            constexpr int kChunks = HH * 128;
                            constexpr int kPer = 4;
#pragma unroll 1
                            for (int e0 = ht; e0 < kChunks; e0 += kPer * kHalfThreads) {
                                float4 acc[kPer];
#pragma unroll
                                for (int i = 0; i < kPer; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
                                for (int c0 = 0; c0 < nc; c0 += 4) {
                                    float4 v[4][kPer];
#pragma unroll
                                    for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
                                        for (int i = 0; i < kPer; ++i) {
                                            const int e = e0 + i * kHalfThreads;
                                            const int64_t qh = qh0 + hoff + e / 128;
                                            v[cc][i] = c0 + cc < nc && e < kChunks
                                                           ? __ldcg(reinterpret_cast<const float4*>(
                                                                        a.part_o + (qh * a.part_stride + c0 + cc) * 512) +
                                                                    (e & 127))
                                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                                        }
                                    }
#pragma unroll
                                    for (int cc = 0; cc < 4; ++cc) {
                                        if (c0 + cc >= nc) break;
#pragma unroll
                                        for (int i = 0; i < kPer; ++i) {
                                            const int e = e0 + i * kHalfThreads;
                                            const float wc = e < kChunks ? B.cw[hoff + e / 128][c0 + cc] : 0.f;
                                            acc[i].x = fmaf(wc, v[cc][i].x, acc[i].x);
                                            acc[i].y = fmaf(wc, v[cc][i].y, acc[i].y);
                                            acc[i].z = fmaf(wc, v[cc][i].z, acc[i].z);
                                            acc[i].w = fmaf(wc, v[cc][i].w, acc[i].w);
                                        }
                                    }
                                }
#pragma unroll
                                for (int i = 0; i < kPer; ++i) {
                                    const int e = e0 + i * kHalfThreads;
                                    if (e >= kChunks) continue;
                                    const int hl = hoff + e / 128;
                                    const float sc = B.cw[hl][kMlaMaxMerge];
                                    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x * sc, acc[i].y * sc);
                                    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z * sc, acc[i].w * sc);
                                    uint2 pk;
                                    pk.x = *reinterpret_cast<uint32_t*>(&lo);
                                    pk.y = *reinterpret_cast<uint32_t*>(&hi);
                                    *reinterpret_cast<uint2*>(a.out + (qh0 + hl) * 512 + (e & 127) * 4) = pk;
                                }
                            }
                        }
                    }
                }
            }
        }
        hs::tc::fence_before_sync();
    }
    __syncthreads();
    if (warp == kMmaWarp) {
        hs::tc::fence_after_sync();
        hs::tc::tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int HG>
int launch_hg(const MlaArgs& a, dim3 grid, hs_stream_t stream) {
    using C = Cfg<HG>;
    static_assert(C::kBarOff + int(sizeof(Bars)) + 1024 <= kSmemLimit, "shared memory budget");
    const size_t smem = size_t(C::kBarOff) + sizeof(Bars) + 1024;
    static int smem_set[64] = {};
    const int rc = hs_host::ensure_dynamic_smem(reinterpret_cast<const void*>(mla_tc_kernel<HG>),
                                                smem, smem_set);
    if (rc != HS_OK) return rc;
    return hs_host::launch_pdl(mla_tc_kernel<HG>, grid, dim3(kThreads), smem, stream, a);
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
