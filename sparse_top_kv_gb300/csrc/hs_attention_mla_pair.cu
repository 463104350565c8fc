// hs_attention_mla_pair.cu -- S4 for MLA rows with 128 query heads on a CTA
// pair (two SMs of a thread-block cluster) with the 2-SM tensor-core
// products.
//
// Math: PaperTrace 5.1.1 "从索引到 Kernel" section 3.1 eqs. (4)-(6) (tile
// logits, running maximum and exponent sums, rescaled accumulator), section
// 3.2 (mask before the exponent; empty set -> zero output, LSE = -inf) and
// eq. (7) (split-KV merge, inside the cluster or in the epilogue of the split
// that finishes last);
// "PagedAttention 与 RadixAttention" section 1.4 (exp2 with scale * log2 e).
// K = all 576 columns of a row, V = its first 512.
//
// GB300 design.  With 128 heads sharing every row, one SM cannot hold the
// fp32 output (128 heads x 512 columns = all of its tensor memory) next to
// the logits, and two independent 64-head CTAs would each gather every row.
// A CTA pair shares the work so that every row is read from HBM once:
//  * A pair tile is 256 candidate rows: CTA r gathers rows [128 r, 128 r +
//    128) with 16-byte cp.async into 128-byte-swizzled K-major blocks and
//    holds the query of heads [64 r, 64 r + 64).  One thread of the even CTA
//    issues S^T[256 tokens x 128 heads] = K Q^T with tcgen05.mma.cta_group::2
//    (M = 256: each CTA's 128 rows; N = 128: each CTA's 64 heads); each CTA's
//    tensor memory receives the logits of its own 128 tokens for all heads.
//  * Softmax in both CTAs against a per-head reference maximum shared by the
//    pair: every tile the CTAs exchange a 128-bit mask of the heads whose
//    logits exceed the reference by more than 2^8 (log2 units); only then do
//    they exchange tile maxima and rescale O in tensor memory.
//  * P^T is split by heads like the query: each CTA writes the P of its own
//    tokens for its own 64 heads in place and sends the other 64 heads' half
//    (16 KB) to the partner with one shared-to-shared bulk copy.
//  * O^T[512 x 128 heads] += V^T P^T as two 2-SM products of M = 256 columns
//    of d: CTA r holds d in [256 j + 128 r, 256 j + 128 r + 128) for j = 0, 1,
//    so it gathers those V columns of all 256 tokens of the tile (its own
//    rows' again from L2, the partner's rows' from L2 as well).  Every HBM
//    byte of a row enters an SM once; the V halves enter a second time.
//  * Ring units (two 16 KB blocks) are consumed in the order QK(0), then
//    {QK(t+1), PV(t)}, so the next tile's gather and product overlap this
//    tile's softmax.  The odd CTA's control thread relays its units' arrival
//    (and its P's) to the even CTA's issuing thread; commits are multicast to
//    both CTAs.
//  * A row split in two runs as one cluster of four CTAs, the two splits its
//    two pairs: each CTA parks its unnormalised O in its own shared memory,
//    and after one cluster barrier the CTAs merge with eq. (7) through
//    distributed shared memory, each its half of the heads for its d rows.
//    Other split counts run as separate pairs; the last pair of a row to
//    finish merges the others' partial states with eq. (7).
// Every wait is bounded (HS_ERR_TIMEOUT in the status word on expiry).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "hs_attention_internal.cuh"
#include "hs_pair.cuh"
#include "hs_tcgen05.cuh"

namespace hs_attn {
namespace {

namespace pr = hs::pair;

constexpr int kHeads = 128;
constexpr int kHalfHeads = 64;       // heads of one CTA in the B operands
constexpr int kTok = 128;            // rows per CTA per pair tile
constexpr int kPairTok = 2 * kTok;   // rows of a pair tile
constexpr int kNB = 9;               // 64-column blocks of a 576-wide row
constexpr int kBlk = kTok * 128;     // one block: 128 rows x 128 B
constexpr int kUnit = 2 * kBlk;
constexpr int kNU = 3;               // ring units
constexpr int kQkUnits = 5;          // 4 K pairs + the RoPE block
constexpr int kPvUnits = 4;          // (d pair j, token half h), j, h in {0, 1}
// Ring order per tile t: QK(t+1) units [0, kQkSplit), PV(t), QK(t+1) units
// [kQkSplit, 5).  All of QK(t+1) first measured fastest (70 us on the
// 32 x 128-head decode; PV(t) between QK(t+1)'s fourth and fifth unit: 74 us,
// the next tile's logits then wait for PV(t)).
constexpr int kQkSplit = 5;
constexpr int kSoftWarps = 8;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kLoadWarps = 2;
constexpr int kLoaderThreads = kLoadWarps * 32;
constexpr int kCtlWarp = kSoftWarps + kLoadWarps;
constexpr int kThreads = (kCtlWarp + 1) * 32;           // 352
constexpr int kLoadRows = kTok * 8 / kLoaderThreads;    // 16 rows per loader thread and block
constexpr float kThresh = 8.0f;
constexpr int kSoftBar = 1;                              // named barrier of the softmax warps

constexpr int kRingOff = 0;
constexpr int kQOff = kRingOff + kNU * kUnit;            // Q: 9 blocks of [64 heads x 128 B]
constexpr int kQBlk = kHalfHeads * 128;                  // 8 KB
constexpr int kPOff = kQOff + kNB * kQBlk;               // P^T: 4 token blocks of [64 heads x 128 B]
constexpr int kPBlk = kHalfHeads * 128;
constexpr int kStageOff = kPOff + 4 * kPBlk;             // outgoing P^T half: 2 token blocks
constexpr int kBarOff = kStageOff + 2 * kPBlk;
constexpr int kSmemLimit = 227 * 1024;
constexpr int kTmemCols = 512;
constexpr int kS = 0;                                    // S^T buffers: columns [0, 256)
constexpr int kO = 256;                                  // O^T slices j: [256 + 128 j, ...)

struct Bars {
    uint64_t full[kNU][2];   // per block of a unit: this CTA's loader arrivals
    uint64_t pfull[kNU];     // even CTA: the odd CTA's unit landed (relayed)
    uint64_t empty[kNU];     // unit consumed (pair commit, both CTAs)
    uint64_t s_full[2];      // S^T buffer written (pair commit)
    uint64_t pv_done[2];     // PV(t) complete (pair commit), by t & 1
    uint64_t p_full;         // this CTA's P^T complete: own half + the partner's copy
    uint64_t p_peer;         // even CTA: the odd CTA's P^T complete (relayed)
    uint64_t flag_full[2];   // partner's tile maxima arrived, by t & 1
    uint64_t l_full;         // partner's exponent sums arrived
    uint64_t drain;
    uint64_t q_full;         // this CTA's query copies landed
    uint32_t tmem_base;
    int32_t abort;
    int32_t last;
    int32_t pad;
    alignas(16) float tmax_out[2][kHeads];  // this CTA's flagged tile maxima, by t & 1
    alignas(16) float tmax_in[2][kHeads];   // the partner's
    alignas(16) float l_out[kHeads];
    alignas(16) float l_in[kHeads];
    alignas(16) float mref[2][kHeads];   // reference maxima (log2 units), double buffered
    alignas(16) float alpha[kHeads];
    alignas(16) float mlc[2][kHeads];    // cluster merge: this pair's (m, l) per head
    float cwc[kHalfHeads][3];            // cluster merge: w(split 0), w(split 1), 1 / L
    float red[4][kHeads];    // per TMEM lane quarter: warp maxima or sums
};
constexpr int kSmemBytes = kBarOff + int(sizeof(Bars)) + 1024;
static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
static_assert(kMlaPairMaxSplits * kHeads * 4 + kHeads * 4 <= kNU * kUnit, "merge weights fit the ring");

// Warp maxima of 16 values per lane by a butterfly that halves the values
// at each step (16 shuffles instead of 80): lanes 2 i and 2 i + 1 return the
// maximum over the warp of value index i.
__device__ __forceinline__ float warp_max16_scatter(const float (&v)[16], int lane) {
    float a[8], b[4], c[2];
    const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1, b1 = (lane >> 1) & 1;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a[i] = fmaxf(b4 ? v[8 + i] : v[i], __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[8 + i], 16));
#pragma unroll
    for (int i = 0; i < 4; ++i)
        b[i] = fmaxf(b3 ? a[4 + i] : a[i], __shfl_xor_sync(0xffffffffu, b3 ? a[i] : a[4 + i], 8));
#pragma unroll
    for (int i = 0; i < 2; ++i)
        c[i] = fmaxf(b2 ? b[2 + i] : b[i], __shfl_xor_sync(0xffffffffu, b2 ? b[i] : b[2 + i], 4));
    float d = fmaxf(b1 ? c[1] : c[0], __shfl_xor_sync(0xffffffffu, b1 ? c[0] : c[1], 2));
    return fmaxf(d, __shfl_xor_sync(0xffffffffu, d, 1));
}

// Warp sums of 64 values per lane (62 shuffles): lane L returns the sums of
// value indices 2 L and 2 L + 1.
__device__ __forceinline__ void warp_sum64_scatter(const float (&v)[64], int lane, float& s0,
                                                   float& s1) {
    float a[32], b[16], c[8], d[4];
    const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1,
               b1 = (lane >> 1) & 1, b0 = lane & 1;
#pragma unroll
    for (int i = 0; i < 32; ++i)
        a[i] = (b4 ? v[32 + i] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[32 + i], 16);
#pragma unroll
    for (int i = 0; i < 16; ++i)
        b[i] = (b3 ? a[16 + i] : a[i]) + __shfl_xor_sync(0xffffffffu, b3 ? a[i] : a[16 + i], 8);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        c[i] = (b2 ? b[8 + i] : b[i]) + __shfl_xor_sync(0xffffffffu, b2 ? b[i] : b[8 + i], 4);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        d[i] = (b1 ? c[4 + i] : c[i]) + __shfl_xor_sync(0xffffffffu, b1 ? c[i] : c[4 + i], 2);
    s0 = (b0 ? d[2] : d[0]) + __shfl_xor_sync(0xffffffffu, b0 ? d[0] : d[2], 1);
    s1 = (b0 ? d[3] : d[1]) + __shfl_xor_sync(0xffffffffu, b0 ? d[1] : d[3], 1);
}

// 2^x, PTX ex2.approx.ftz (relative error ~2^-22, far below the bf16
// rounding of P; 0 for x below -126).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Position of unit `u` of tile t's QK (is_pv = 0) or PV (1) in the
// consumption sequence QK(0), then for t = 0 .. T-1: QK(t+1) units below
// kQkSplit, PV(t), QK(t+1) units from kQkSplit on.
__device__ __forceinline__ int unit_seq(int t, int is_pv, int u, int T) {
    if (!is_pv) {
        if (t == 0) return u;
        const int base = kQkUnits + (t - 1) * (kQkUnits + kPvUnits);
        return u < kQkSplit ? base + u : base + kPvUnits + u;
    }
    return kQkUnits + t * (kQkUnits + kPvUnits) + (t + 1 < T ? kQkSplit : 0) + u;
}

// CL = 2: one pair per cluster.  CL = 4 (a row split in two): the row's two
// pairs form one cluster (ranks 2 s + r for split s) and merge through
// distributed shared memory; the pair forms of tcgen05 pair the CTAs whose
// cluster ranks differ in bit 0.
template <int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(kThreads, 1)
    mla_pair_kernel(const MlaArgs a) {
    constexpr bool kClusterMerge = CL == 4;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars& B = *reinterpret_cast<Bars*>(smem + kBarOff);
    const uint32_t s_base = hs::smem_u32(smem);
    const uint32_t ring_base = s_base + kRingOff;
    const uint32_t q_base = s_base + kQOff;
    const uint32_t p_base = s_base + kPOff;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = pr::cta_rank();        // rank in the cluster
    const uint32_t rank = crank & 1u;             // rank in the pair
    const uint32_t peer = crank ^ 1u;             // the other CTA of the pair
    const uint32_t pair_base = crank & ~1u;       // the pair's even CTA
    const uint16_t pmask = uint16_t(3u << pair_base);
    const int pair_id = blockIdx.x >> 1;
    const int row = pair_id / a.splits;
    const int split = pair_id % a.splits;
    const int32_t* kv_rows = a.kv_rows + int64_t(row) * a.cap;
    const uint64_t tmo = a.timeout_ns;
    volatile int* abort_flag = &B.abort;

    auto fail = [&]() {
        hs::set_status(a.status, HS_ERR_TIMEOUT);
        B.abort = 1;
        pr::st_remote_u32(pr::mapa(hs::smem_u32(&B.abort), peer), 1u);
    };

    hs::pdl_trigger();
    if (tid == 0) {
        for (int i = 0; i < kNU; ++i) {
            hs::mbar_init(&B.full[i][0], kLoaderThreads);
            hs::mbar_init(&B.full[i][1], kLoaderThreads);
            hs::mbar_init(&B.pfull[i], 1);
            hs::mbar_init(&B.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            hs::mbar_init(&B.s_full[i], 1);
            hs::mbar_init(&B.pv_done[i], 1);
            hs::mbar_init(&B.flag_full[i], 1);
        }
        hs::mbar_init(&B.p_full, 1);
        hs::mbar_init(&B.p_peer, 1);
        hs::mbar_init(&B.l_full, 1);
        hs::mbar_init(&B.drain, 1);
        hs::mbar_init(&B.q_full, kThreads);
        for (int i = 0; i < kHeads; ++i) B.mref[0][i] = -CUDART_INF_F;
        B.abort = 0;
        hs::fence_mbar_init();
    }
    if (warp == kCtlWarp) {
        pr::tmem_alloc2(&B.tmem_base, kTmemCols);
        pr::tmem_relinquish2();
    }
    __syncthreads();  // barriers initialised before the query's copies arrive on q_full
    // This CTA's 64 heads of the query -> 9 swizzled K-major blocks, landing
    // while the first tile's rows are gathered (q_full).
    {
        const __nv_bfloat16* qg = a.q + (int64_t(row) * kHeads + kHalfHeads * rank) * 576;
        for (int e = tid; e < kHalfHeads * 72; e += kThreads) {
            const int h = e / 72, c = e % 72;
            const int b = c >> 3, cc = c & 7;
            hs::tc::cp_async16(q_base + b * kQBlk + h * 128 + ((cc ^ (h & 7)) << 4),
                               qg + int64_t(h) * 576 + c * 8, 16u);
        }
        hs::tc::cp_async_arrive_noinc(&B.q_full);
    }
    hs::tc::fence_before_sync();
    __syncthreads();
    pr::cluster_sync();  // barriers of both CTAs initialised
    hs::tc::fence_after_sync();
    hs::pdl_wait();
    const uint32_t tmem = B.tmem_base;
    const int n = a.count ? min(max(a.count[row], 0), a.cap) : a.cap;
    const int ntiles = (n + kPairTok - 1) / kPairTok;
    const int per = (ntiles + a.splits - 1) / a.splits;
    const int t_begin = min(ntiles, split * per);
    const int T = min(ntiles, t_begin + per) - t_begin;

    if (warp >= kSoftWarps && warp < kCtlWarp) {
        // ------------------------------ loaders ------------------------------
        const int lt = tid - kSoftThreads;
        constexpr int kRowStep = kLoaderThreads / 8;
        const int c = lt & 7;
        const int r0 = lt >> 3;
        const uint32_t swz = uint32_t((c ^ (r0 & 7)) << 4);
        bool bad = false;
        // Row ids of both token halves of tiles t and t + 1.
        int32_t cur[2][kLoadRows], nxt[2][kLoadRows];
        auto fetch = [&](int t, int32_t (&id)[2][kLoadRows]) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int i = 0; i < kLoadRows; ++i) {
                    const int j = (t_begin + t) * kPairTok + h * kTok + r0 + kRowStep * i;
                    id[h][i] = (t < T && j < n) ? __ldg(kv_rows + j) : -1;
                }
            }
        };
        // Rows of token half `h` (a run-time value: selected per element, so
        // that the id arrays stay in registers).
        auto fill = [&](int k, const int32_t (&id)[2][kLoadRows], int h, int b0, int b1) -> bool {
            const int slot = k % kNU;
            if (!pr::mbar_wait(&B.empty[slot], ((k / kNU) & 1) ^ 1, tmo, abort_flag)) return false;
            const uint32_t dst = ring_base + slot * kUnit + r0 * 128 + swz;
#pragma unroll
            for (int i = 0; i < kLoadRows; ++i) {
                const int32_t x = h ? id[1][i] : id[0][i];
                const bool v = x >= 0 && int64_t(x) < a.num_kv_rows;
                const char* src = reinterpret_cast<const char*>(a.kv) +
                                  (v ? int64_t(x) : 0) * a.row_stride * 2 + c * 16;
                hs::tc::cp_async16(dst + i * kRowStep * 128, src + b0 * 128, v ? 16u : 0u);
                if (b1 >= 0)
                    hs::tc::cp_async16(dst + kBlk + i * kRowStep * 128, src + b1 * 128,
                                       v ? 16u : 0u);
            }
            hs::tc::cp_async_arrive_noinc(&B.full[slot][0]);
            hs::tc::cp_async_arrive_noinc(&B.full[slot][1]);
            return true;
        };
        auto load_qk = [&](int t, const int32_t (&id)[2][kLoadRows], int u0, int u1) -> bool {
            if (u0 == 0) {
#pragma unroll
                for (int i = 0; i < kLoadRows; ++i)
                    if (int64_t(rank ? id[1][i] : id[0][i]) >= a.num_kv_rows) bad = true;
            }
            for (int u = u0; u < u1; ++u)
                if (!fill(unit_seq(t, 0, u, T), id, int(rank), u < 4 ? 2 * u : 8,
                          u < 4 ? 2 * u + 1 : -1))
                    return false;
            return true;
        };
        // PV unit u = (d pair j = u / 2, token half h = u % 2): V columns
        // [256 j + 128 r, + 128) = blocks 4 j + 2 r, 4 j + 2 r + 1.
        auto load_pv = [&](int t, const int32_t (&id)[2][kLoadRows]) -> bool {
            const int k0 = unit_seq(t, 1, 0, T);
            for (int u = 0; u < kPvUnits; ++u) {
                const int b0 = 4 * (u >> 1) + 2 * int(rank);
                if (!fill(k0 + u, id, u & 1, b0, b0 + 1)) return false;
            }
            return true;
        };
        fetch(0, cur);
        fetch(1, nxt);
        bool ok = T == 0 || load_qk(0, cur, 0, kQkUnits);
        for (int t = 0; t < T && ok; ++t) {
            if (t + 1 < T) ok = load_qk(t + 1, nxt, 0, kQkSplit);
            if (ok) ok = load_pv(t, cur);
            if (ok && t + 1 < T) ok = load_qk(t + 1, nxt, kQkSplit, kQkUnits);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < kLoadRows; ++i) cur[h][i] = nxt[h][i];
            fetch(t + 2, nxt);
        }
        if (!ok) fail();
        if (bad) hs::set_status(a.status, HS_ERR_BAD_INDEX);
        hs::tc::cp_async_wait_all();
    } else if (warp == kCtlWarp) {
        if (lane == 0 && rank == 0) {
            // -------------------- MMA issuer (even CTA) ----------------------
            constexpr uint32_t idesc_qk = hs::tc::idesc_bf16(256, kHeads, 0, 0);
            constexpr uint32_t idesc_pv = hs::tc::idesc_bf16(256, kHeads, 1, 0);
            auto wait_local = [&](int k, int b) -> bool {
                return pr::mbar_wait(&B.full[k % kNU][b], (k / kNU) & 1, tmo, abort_flag);
            };
            auto wait_peer = [&](int k) -> bool {
                return pr::mbar_wait(&B.pfull[k % kNU], (k / kNU) & 1, tmo, abort_flag);
            };
            // Blocks [2 u0, min(2 u1, 9)) of QK(t); the last part commits S.
            auto issue_qk = [&](int t, int u0, int u1) -> bool {
                const int sb = t & 1;
                if (t == 0 && u0 == 0) {
                    if (!pr::mbar_wait(&B.q_full, 0, tmo, abort_flag)) return false;
                    hs::fence_proxy_async_shared();
                }
                for (int b = 2 * u0; b < min(2 * u1, kNB); ++b) {
                    const int k = unit_seq(t, 0, b >> 1, T);
                    if ((b & 1) == 0 && !wait_peer(k)) return false;
                    if (!wait_local(k, b & 1)) return false;
                    if (b == kNB - 1 && !wait_local(k, 1)) return false;
                    hs::tc::fence_after_sync();
                    const uint32_t abase = ring_base + (k % kNU) * kUnit + (b & 1) * kBlk;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = hs::tc::sdesc_sw128(abase + kk * 32, 16, 1024);
                        const uint64_t bd = hs::tc::sdesc_sw128(q_base + b * kQBlk + kk * 32, 16, 1024);
                        pr::mma2_bf16(tmem + kS + sb * kHeads, ad, bd, idesc_qk, (b | kk) ? 1u : 0u);
                    }
                    if ((b & 1) || b == kNB - 1) pr::commit2_both(&B.empty[k % kNU], pmask);
                }
                if (u1 == kQkUnits && u0 < u1) pr::commit2_both(&B.s_full[sb], pmask);
                return true;
            };
            auto issue_pv = [&](int t) -> bool {
                if (!pr::mbar_wait(&B.p_full, t & 1, tmo, abort_flag)) return false;
                if (!pr::mbar_wait(&B.p_peer, t & 1, tmo, abort_flag)) return false;
                hs::tc::fence_after_sync();
                const int k0 = unit_seq(t, 1, 0, T);
#pragma unroll 1
                for (int u = 0; u < kPvUnits; ++u) {
                    const int j = u >> 1, h = u & 1;
                    const int k = k0 + u;
                    if (!wait_peer(k) || !wait_local(k, 0) || !wait_local(k, 1)) return false;
                    hs::tc::fence_after_sync();
                    const uint32_t vbase = ring_base + (k % kNU) * kUnit;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = hs::tc::sdesc_sw128(vbase + kk * 2048, kBlk, 1024);
                        const uint64_t bd = hs::tc::sdesc_sw128(
                            p_base + (2 * h + (kk >> 2)) * kPBlk + (kk & 3) * 32, 16, 1024);
                        pr::mma2_bf16(tmem + kO + j * kHeads, ad, bd, idesc_pv,
                                      (t > 0 || h > 0 || kk > 0) ? 1u : 0u);
                    }
                    pr::commit2_both(&B.empty[k % kNU], pmask);
                }
                pr::commit2_both(&B.pv_done[t & 1], pmask);
                return true;
            };
            bool ok = T == 0 || issue_qk(0, 0, kQkUnits);
            for (int t = 0; t < T && ok; ++t) {
                if (t + 1 < T) ok = issue_qk(t + 1, 0, kQkSplit);
                if (ok) ok = issue_pv(t);
                if (ok && t + 1 < T && kQkSplit < kQkUnits) ok = issue_qk(t + 1, kQkSplit, kQkUnits);
            }
            if (!ok) fail();
            // Drain: every pair MMA has completed before tensor memory is freed.
            pr::commit2_both(&B.drain, pmask);
            pr::mbar_wait(&B.drain, 0, tmo, nullptr);
        } else if (lane == 0) {
            // ---------- relay (odd CTA): this CTA's units and P^T ready -------
            const uint32_t r_pfull = pr::mapa(hs::smem_u32(&B.pfull[0]), pair_base);
            const uint32_t r_ppeer = pr::mapa(hs::smem_u32(&B.p_peer), pair_base);
            auto relay = [&](int k) -> bool {
                const int slot = k % kNU;
                if (!pr::mbar_wait(&B.full[slot][0], (k / kNU) & 1, tmo, abort_flag)) return false;
                if (!pr::mbar_wait(&B.full[slot][1], (k / kNU) & 1, tmo, abort_flag)) return false;
                hs::fence_proxy_async_shared();
                pr::mbar_arrive_remote(r_pfull + slot * 8);
                return true;
            };
            bool ok = true;
            if (T > 0) {
                // The first unit also tells the even CTA that this CTA's query landed.
                ok = pr::mbar_wait(&B.q_full, 0, tmo, abort_flag);
                hs::fence_proxy_async_shared();
            }
            for (int u = 0; u < kQkUnits && ok && T > 0; ++u) ok = relay(u);
            for (int t = 0; t < T && ok; ++t) {
                if (t + 1 < T)
                    for (int u = 0; u < kQkSplit && ok; ++u) ok = relay(unit_seq(t + 1, 0, u, T));
                if (!ok) break;
                if (!pr::mbar_wait(&B.p_full, t & 1, tmo, abort_flag)) { ok = false; break; }
                hs::tc::fence_after_sync();
                hs::fence_proxy_async_shared();
                pr::mbar_arrive_remote(r_ppeer);
                for (int u = 0; u < kPvUnits && ok; ++u) ok = relay(unit_seq(t, 1, u, T));
                if (t + 1 < T)
                    for (int u = kQkSplit; u < kQkUnits && ok; ++u) ok = relay(unit_seq(t + 1, 0, u, T));
            }
            if (!ok) fail();
        }
        __syncwarp();
    } else {
        // ----------------------- softmax / epilogue (warps 0-7) ---------------
        const int qd = warp & 3;             // TMEM lane quarter
        const int hf = warp >> 2;            // head half handled by this thread
        const int st = tid;                  // 0 .. 255
        const int tl = qd * 32 + lane;       // TMEM lane: own token (S^T) or d row (O^T)
        const uint32_t lane_base = uint32_t(qd * 32) << 16;
        float l_part[kHalfHeads];
#pragma unroll
        for (int h = 0; h < kHalfHeads; ++h) l_part[h] = 0.f;
        int msel = 0;
        bool ok = true;
        auto token_id = [&](int t) -> int32_t {
            const int j = (t_begin + t) * kPairTok + int(rank) * kTok + tl;
            return (t < T && j < n) ? __ldg(kv_rows + j) : -1;
        };
        int32_t id_next = token_id(0);
        for (int t = 0; t < T && ok; ++t) {
            const int sb = t & 1;
            const int32_t id_t = id_next;
            id_next = token_id(t + 1);
            const bool valid = id_t >= 0 && int64_t(id_t) < a.num_kv_rows;
            const uint32_t s_addr = tmem + lane_base + kS + sb * kHeads + hf * kHalfHeads;
            if (!pr::mbar_wait(&B.s_full[sb], (t >> 1) & 1, tmo, abort_flag)) { ok = false; break; }
            hs::tc::fence_after_sync();
            // Pass 1: heads whose logit exceeds the reference by more than
            // 2^8 in this warp's 32 tokens, and their warp maxima.
            {
                const float* mr = B.mref[msel] + hf * kHalfHeads;
#pragma unroll 1
                for (int c = 0; c < kHalfHeads; c += 16) {
                    float v[16];
                    hs::tc::tmem_ld16(s_addr + c, v);
                    hs::tc::tmem_wait_ld();
                    uint32_t f = 0;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        v[i] = valid ? v[i] * a.scale_log2 : -CUDART_INF_F;
                        if (v[i] > mr[c + i] + kThresh) f |= 1u << i;
                    }
                    f = __reduce_or_sync(0xffffffffu, f);
                    // Lanes 2 i (i < 16) write the warp maximum of value index
                    // i, or -inf when the warp did not flag that head.
                    float wm = -CUDART_INF_F;
                    if (f != 0u) wm = warp_max16_scatter(v, lane);
                    if ((lane & 1) == 0) {
                        const int vi = lane >> 1;
                        B.red[qd][hf * kHalfHeads + c + vi] = ((f >> vi) & 1u) ? wm : -CUDART_INF_F;
                    }
                }
            }
            // The previous tile's outgoing copies have read their sources.
            if (st == 0) pr::bulk_wait_read();
            pr::named_sync(kSoftBar, kSoftThreads);
            // This CTA's tile maxima of the flagged heads (-inf: not flagged),
            // exchanged with the partner in one 512-byte copy each way.
            if (st < kHeads)
                B.tmax_out[sb][st] = fmaxf(fmaxf(B.red[0][st], B.red[1][st]),
                                           fmaxf(B.red[2][st], B.red[3][st]));
            hs::fence_proxy_async_shared();
            pr::named_sync(kSoftBar, kSoftThreads);
            if (st == 0) {
                pr::mbar_arrive_expect_tx_cluster(&B.flag_full[sb], kHeads * 4);
                pr::bulk_s2s(pr::mapa(hs::smem_u32(B.tmax_in[sb]), peer),
                             hs::smem_u32(B.tmax_out[sb]), kHeads * 4,
                             pr::mapa(hs::smem_u32(&B.flag_full[sb]), peer));
                pr::bulk_commit();
            }
            if (!pr::mbar_wait(&B.flag_full[sb], (t >> 1) & 1, tmo, abort_flag)) { ok = false; break; }
            // New reference maxima (identical in both CTAs).  A CTA's logits
            // of a head it did not flag are at most 2^8 above the old
            // reference, hence above the new one; so only flagged maxima
            // enter it.
            bool resc = false;
            if (st < kHeads) {
                const float mo = B.mref[msel][st];
                const float tm = fmaxf(B.tmax_out[sb][st], B.tmax_in[sb][st]);
                float mn = mo, al = 1.f;
                if (tm != -CUDART_INF_F) {
                    resc = true;
                    mn = fmaxf(mo, tm);
                    al = mo == -CUDART_INF_F ? 0.f : exp2f(mo - mn);
                }
                B.mref[msel ^ 1][st] = mn;
                B.alpha[st] = al;
            }
            const bool any = pr::named_sync_or(kSoftBar, kSoftThreads, resc);
            msel ^= 1;
            bool pv_prev_done = t == 0;
            if (any) {
                const float* al = B.alpha + hf * kHalfHeads;
#pragma unroll
                for (int h = 0; h < kHalfHeads; ++h) l_part[h] *= al[h];
                if (t > 0) {
                    // O holds PV(0 .. t-1): wait for PV(t-1), rescale in TMEM.
                    if (!pr::mbar_wait(&B.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, tmo,
                                       abort_flag)) { ok = false; break; }
                    pv_prev_done = true;
                    hs::tc::fence_after_sync();
#pragma unroll 1
                    for (int j = 0; j < 2; ++j) {
#pragma unroll 1
                        for (int c = 0; c < kHalfHeads; c += 16) {
                            float o[16];
                            const uint32_t ta = tmem + lane_base + kO + j * kHeads + hf * kHalfHeads + c;
                            hs::tc::tmem_ld16(ta, o);
                            hs::tc::tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) o[i] *= al[c + i];
                            hs::tc::tmem_st16(ta, o);
                        }
                    }
                    hs::tc::tmem_wait_st();
                }
            }
            // The single P^T buffer: PV(t-1) must have read it (in both CTAs).
            if (!pv_prev_done) {
                if (!pr::mbar_wait(&B.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, tmo, abort_flag)) {
                    ok = false;
                    break;
                }
            }
            // Pass 2: P^T, bf16, K-major [head][token]: this CTA's heads in
            // place (token block 2 r + tl / 64), the partner's heads into the
            // outgoing half.
            {
                const float* mr = B.mref[msel] + hf * kHalfHeads;
                unsigned char* prow =
                    hf == int(rank) ? smem + kPOff + (2 * int(rank) + (tl >> 6)) * kPBlk
                                    : smem + kStageOff + (tl >> 6) * kPBlk;
                const int tcol = (tl & 63) * 2;
#pragma unroll
                for (int c = 0; c < kHalfHeads; c += 16) {
                    float v[16];
                    hs::tc::tmem_ld16(s_addr + c, v);
                    // The reference maxima in registers before the P stores
                    // (read through the shared-memory pointer inside the loop,
                    // each load would wait for the stores before it).
                    float mreg[16];
#pragma unroll
                    for (int i = 0; i < 16; i += 4) {
                        const float4 m4 = *reinterpret_cast<const float4*>(mr + c + i);
                        mreg[i] = m4.x;
                        mreg[i + 1] = m4.y;
                        mreg[i + 2] = m4.z;
                        mreg[i + 3] = m4.w;
                    }
                    hs::tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        const int h = c + i;
                        float p[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float m = mreg[i + e];
                            p[e] = (valid && m != -CUDART_INF_F)
                                       ? ex2_approx(fmaf(v[i + e], a.scale_log2, -m)) : 0.f;
                        }
                        // Two heads' P rounded to bf16 in one conversion; each
                        // goes to its own row of P^T.
                        const __nv_bfloat162 pb = __floats2bfloat162_rn(p[0], p[1]);
                        const uint32_t pu = *reinterpret_cast<const uint32_t*>(&pb);
                        l_part[h] += __uint_as_float(pu << 16);
                        l_part[h + 1] += __uint_as_float(pu & 0xffff0000u);
                        *reinterpret_cast<uint16_t*>(
                            prow + h * 128 + ((((tcol >> 4) ^ (h & 7)) << 4) | (tcol & 15))) =
                            uint16_t(pu & 0xffffu);
                        *reinterpret_cast<uint16_t*>(
                            prow + (h + 1) * 128 + ((((tcol >> 4) ^ ((h + 1) & 7)) << 4) | (tcol & 15))) =
                            uint16_t(pu >> 16);
                    }
                }
            }
            hs::fence_proxy_async_shared();
            hs::tc::fence_before_sync();
            pr::named_sync(kSoftBar, kSoftThreads);
            if (st == 0) {
                pr::mbar_arrive_expect_tx_cluster(&B.p_full, 2 * kPBlk);
                pr::bulk_s2s(pr::mapa(p_base + 2 * rank * kPBlk, peer), s_base + kStageOff,
                             2 * kPBlk, pr::mapa(hs::smem_u32(&B.p_full), peer));
                pr::bulk_commit();
            }
        }
        // ------------------------------ epilogue ------------------------------
        if (ok && T > 0) {
            ok = pr::mbar_wait(&B.pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, tmo, abort_flag);
            hs::tc::fence_after_sync();
        }
        if (ok) {
            // Exponent sums of this CTA's tokens per head, then the pair's.
            {
                float s0, s1;
                warp_sum64_scatter(l_part, lane, s0, s1);
                B.red[qd][hf * kHalfHeads + 2 * lane] = s0;
                B.red[qd][hf * kHalfHeads + 2 * lane + 1] = s1;
            }
            if (st == 0) pr::bulk_wait_read();
            pr::named_sync(kSoftBar, kSoftThreads);
            if (st < kHeads)
                B.l_out[st] = B.red[0][st] + B.red[1][st] + B.red[2][st] + B.red[3][st];
            hs::fence_proxy_async_shared();
            pr::named_sync(kSoftBar, kSoftThreads);
            if (st == 0) {
                pr::mbar_arrive_expect_tx_cluster(&B.l_full, kHeads * 4);
                pr::bulk_s2s(pr::mapa(hs::smem_u32(B.l_in), peer), hs::smem_u32(B.l_out),
                             kHeads * 4, pr::mapa(hs::smem_u32(&B.l_full), peer));
                pr::bulk_commit();
            }
            ok = pr::mbar_wait(&B.l_full, 0, tmo, abort_flag);
        }
        if constexpr (kClusterMerge) {
            // The row's two splits are the two pairs of this cluster: every CTA
            // parks its unnormalised O (its 256 d rows, all heads, [head][d
            // row] in the idle ring and query space) and its pair's (m, l);
            // after a cluster barrier that every thread of the cluster passes
            // once here (the other warps at their end), CTA (s, r) merges
            // heads [64 s, 64 s + 64) of its d rows from both splits with
            // eq. (7), split 0's part first.
            float* os = reinterpret_cast<float*>(smem + kRingOff);
            const int64_t qh0 = int64_t(row) * kHeads;
            if (!ok) {
                fail();
            } else {
#pragma unroll 1
                for (int j = 0; j < 2; ++j) {
#pragma unroll 1
                    for (int c = 0; c < kHalfHeads; c += 16) {
                        float o[16];
                        if (T > 0) {
                            hs::tc::tmem_ld16(tmem + lane_base + kO + j * kHeads + hf * kHalfHeads + c, o);
                            hs::tc::tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) o[i] = 0.f;
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            os[(hf * kHalfHeads + c + i) * 256 + j * 128 + tl] = o[i];
                    }
                }
                if (st < kHeads) {
                    const float L = B.l_out[st] + B.l_in[st];
                    B.mlc[0][st] = L > 0.f ? B.mref[msel][st] : -CUDART_INF_F;
                    B.mlc[1][st] = L;
                }
            }
            pr::cluster_sync();
            const uint32_t other = crank ^ 2u;  // the other split's CTA of this rank
            const bool merge_ok =
                *abort_flag == 0 && pr::ld_remote_s32(pr::mapa(hs::smem_u32(&B.abort), other)) == 0;
            if (merge_ok) {
                const int sp = split;  // 0 or 1
                if (st < kHalfHeads) {
                    const int h = kHalfHeads * sp + st;
                    const float mo = B.mlc[0][h], lo = B.mlc[1][h];
                    const float mr = pr::ld_remote_f32(pr::mapa(hs::smem_u32(&B.mlc[0][h]), other));
                    const float lr = pr::ld_remote_f32(pr::mapa(hs::smem_u32(&B.mlc[1][h]), other));
                    const float m0 = sp == 0 ? mo : mr, l0 = sp == 0 ? lo : lr;
                    const float m1 = sp == 0 ? mr : mo, l1 = sp == 0 ? lr : lo;
                    float M = l0 > 0.f ? m0 : -CUDART_INF_F;
                    if (l1 > 0.f) M = fmaxf(M, m1);
                    float Lt = 0.f, w0 = 0.f, w1 = 0.f;
                    if (M != -CUDART_INF_F) {
                        if (l0 > 0.f) {
                            w0 = exp2f(m0 - M);
                            Lt = fmaf(w0, l0, Lt);
                        }
                        if (l1 > 0.f) {
                            w1 = exp2f(m1 - M);
                            Lt = fmaf(w1, l1, Lt);
                        }
                    }
                    B.cwc[st][0] = w0;
                    B.cwc[st][1] = w1;
                    B.cwc[st][2] = Lt > 0.f ? 1.f / Lt : 0.f;
                    if (rank == 0 && a.lse != nullptr)
                        a.lse[qh0 + h] = Lt > 0.f ? (M + log2f(Lt)) * 0.6931471805599453f
                                                  : -CUDART_INF_F;
                }
                pr::named_sync(kSoftBar, kSoftThreads);
                // 64 heads x 256 d rows = 4096 16-byte chunks, 16 per thread,
                // four at a time from each split.
                const uint32_t os_l = hs::smem_u32(os);
                const uint32_t os_r = pr::mapa(os_l, other);
#pragma unroll 1
                for (int i0 = 0; i0 < 16; i0 += 4) {
                    float4 vl[4], vr[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int e = st + kSoftThreads * (i0 + k);
                        const uint32_t off = uint32_t(((kHalfHeads * sp + (e >> 6)) * 256 + (e & 63) * 4) * 4);
                        vl[k] = *reinterpret_cast<const float4*>(smem + kRingOff + off);
                        vr[k] = pr::ld_remote_v4(os_r + off);
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int e = st + kSoftThreads * (i0 + k);
                        const int hl = e >> 6, dl = (e & 63) * 4;
                        const float w0 = B.cwc[hl][0], w1 = B.cwc[hl][1], inv = B.cwc[hl][2];
                        const float4 p0 = sp == 0 ? vl[k] : vr[k];
                        const float4 p1 = sp == 0 ? vr[k] : vl[k];
                        const float x = fmaf(w1, p1.x, w0 * p0.x) * inv;
                        const float y = fmaf(w1, p1.y, w0 * p0.y) * inv;
                        const float z = fmaf(w1, p1.z, w0 * p0.z) * inv;
                        const float w = fmaf(w1, p1.w, w0 * p0.w) * inv;
                        __nv_bfloat162 lo2 = __floats2bfloat162_rn(x, y);
                        __nv_bfloat162 hi2 = __floats2bfloat162_rn(z, w);
                        uint2 pk;
                        pk.x = *reinterpret_cast<uint32_t*>(&lo2);
                        pk.y = *reinterpret_cast<uint32_t*>(&hi2);
                        const int d = 256 * (dl >> 7) + 128 * int(rank) + (dl & 127);
                        *reinterpret_cast<uint2*>(a.out + (qh0 + kHalfHeads * sp + hl) * 512 + d) = pk;
                    }
                }
            } else {
                hs::set_status(a.status, HS_ERR_TIMEOUT);
            }
        } else if (!ok) {
            fail();
        } else {
            float* cw = reinterpret_cast<float*>(smem + kRingOff);  // [128][splits] + inv[128]
            float* cinv = cw + kHeads * kMlaPairMaxSplits;
            const int64_t qh0 = int64_t(row) * kHeads;
            int last = 1;
            int32_t* ctr = a.sync != nullptr ? a.sync + (int64_t(row) * 2 + rank) * 2 : nullptr;
            if (a.splits > 1) {
                if (st == 0) {
                    const int old = atomicAdd(ctr, 1);
                    B.last = old == a.splits - 1 ? 1 : 0;
                }
                pr::named_sync(kSoftBar, kSoftThreads);
                last = B.last;
            }
            if (!last) {
                // Partial state (unnormalised O for this CTA's d rows; m, l per head).
#pragma unroll 1
                for (int j = 0; j < 2; ++j) {
                    const int d = 256 * j + 128 * int(rank) + tl;
#pragma unroll 1
                    for (int c = 0; c < kHalfHeads; c += 16) {
                        float o[16];
                        if (T > 0) {
                            hs::tc::tmem_ld16(tmem + lane_base + kO + j * kHeads + hf * kHalfHeads + c, o);
                            hs::tc::tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) o[i] = 0.f;
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int64_t qh = qh0 + hf * kHalfHeads + c + i;
                            a.part_o[(qh * a.splits + split) * 512 + d] = o[i];
                        }
                    }
                }
                if (st < kHeads) {
                    const float L = B.l_out[st] + B.l_in[st];
                    float* ml = a.part_m + ((int64_t(rank) * a.rows * kHeads + qh0 + st) * a.splits + split) * 2;
                    ml[0] = L > 0.f ? B.mref[msel][st] : -CUDART_INF_F;
                    ml[1] = L;
                }
                __threadfence();
                pr::named_sync(kSoftBar, kSoftThreads);
                if (st == 0) atomicAdd(ctr + 1, 1);
            } else {
                bool merged_ok = true;
                if (a.splits > 1) {
                    // The others have counted themselves in: wait until their
                    // partial states are written (they wait on nothing).
                    if (st == 0) {
                        const uint64_t t0 = hs::global_timer_ns();
                        int seen = 0;
                        for (uint32_t it = 0;; ++it) {
                            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(seen) : "l"(ctr + 1) : "memory");
                            if (seen >= a.splits - 1) break;
                            if ((it & 63u) == 0 && hs::global_timer_ns() - t0 > tmo) break;
                        }
                        B.last = seen >= a.splits - 1 ? 1 : 0;
                        // Every split has arrived and written: reset for the next call.
                        ctr[0] = 0;
                        ctr[1] = 0;
                    }
                    pr::named_sync(kSoftBar, kSoftThreads);
                    merged_ok = B.last != 0;
                    __threadfence();
                }
                if (!merged_ok) {
                    fail();
                } else {
                    if (st < kHeads) {
                        const int64_t qh = qh0 + st;
                        const float Lown = B.l_out[st] + B.l_in[st];
                        const float Mown = B.mref[msel][st];
                        const float* ml = a.part_m + (int64_t(rank) * a.rows * kHeads + qh) * a.splits * 2;
                        // Every split's (m, l) in one round of loads.
                        float msp[kMlaPairMaxSplits], lsp[kMlaPairMaxSplits];
#pragma unroll
                        for (int sp = 0; sp < kMlaPairMaxSplits; ++sp) {
                            const bool other = sp < a.splits && sp != split;
                            const float2 v = other ? __ldcg(reinterpret_cast<const float2*>(ml + sp * 2))
                                                   : make_float2(Mown, Lown);
                            msp[sp] = v.x;
                            lsp[sp] = sp < a.splits ? v.y : 0.f;
                        }
                        float M = Lown > 0.f ? Mown : -CUDART_INF_F;
#pragma unroll
                        for (int sp = 0; sp < kMlaPairMaxSplits; ++sp)
                            if (sp < a.splits && sp != split && lsp[sp] > 0.f) M = fmaxf(M, msp[sp]);
                        float Lt = 0.f;
#pragma unroll
                        for (int sp = 0; sp < kMlaPairMaxSplits; ++sp) {
                            if (sp >= a.splits) break;
                            float wsp = 0.f;
                            if (M != -CUDART_INF_F && lsp[sp] > 0.f) {
                                wsp = exp2f(msp[sp] - M);
                                Lt = fmaf(wsp, lsp[sp], Lt);
                            }
                            cw[st * kMlaPairMaxSplits + sp] = wsp;
                        }
                        cinv[st] = Lt > 0.f ? 1.f / Lt : 0.f;
                        if (rank == 0 && a.lse != nullptr)
                            a.lse[qh] = Lt > 0.f ? (M + log2f(Lt)) * 0.6931471805599453f : -CUDART_INF_F;
                    }
                    pr::named_sync(kSoftBar, kSoftThreads);
#pragma unroll 1
                    for (int j = 0; j < 2; ++j) {
                        const int d = 256 * j + 128 * int(rank) + tl;
#pragma unroll 1
                        for (int c = 0; c < kHalfHeads; c += 32) {
                            float o[32];
                            if (T > 0) {
                                hs::tc::tmem_ld16(tmem + lane_base + kO + j * kHeads + hf * kHalfHeads + c,
                                                  *reinterpret_cast<float(*)[16]>(o));
                                hs::tc::tmem_ld16(tmem + lane_base + kO + j * kHeads + hf * kHalfHeads + c + 16,
                                                  *reinterpret_cast<float(*)[16]>(o + 16));
                                hs::tc::tmem_wait_ld();
                            } else {
#pragma unroll
                                for (int i = 0; i < 32; ++i) o[i] = 0.f;
                            }
                            float acc[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                acc[i] = cw[(hf * kHalfHeads + c + i) * kMlaPairMaxSplits + split] * o[i];
                            // The other splits' partial outputs: 32 independent
                            // loads per split in flight.
                            for (int sp = 0; sp < a.splits; ++sp) {
                                if (sp == split) continue;
                                float po[32];
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    po[i] = __ldcg(a.part_o + ((qh0 + hf * kHalfHeads + c + i) * a.splits + sp) * 512 + d);
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    acc[i] = fmaf(cw[(hf * kHalfHeads + c + i) * kMlaPairMaxSplits + sp], po[i], acc[i]);
                            }
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int g = hf * kHalfHeads + c + i;
                                a.out[(qh0 + g) * 512 + d] = __float2bfloat16_rn(acc[i] * cinv[g]);
                            }
                        }
                    }
                }
            }
        }
        if (st == 0) pr::bulk_wait();
        hs::tc::fence_before_sync();
    }
    if constexpr (kClusterMerge) {
        // The cluster merge's barrier, passed by the softmax warps in their
        // epilogue and by the other warps here.
        if (warp >= kSoftWarps) pr::cluster_sync();
    }
    __syncthreads();
    pr::cluster_sync();  // no copy into the partner and no pair MMA is in flight past here
    if (warp == kCtlWarp) {
        hs::tc::fence_after_sync();
        pr::tmem_dealloc2(tmem, kTmemCols);
    }
}

}  // namespace

namespace {
int g_smem_set2[64] = {};
int g_smem_set4[64] = {};
int g_clusters4[64];
bool g_clusters4_init = false;
}  // namespace

bool mla_pair_cluster_merge(int rows, int splits) {
    if (splits != 2 || rows <= 0) return false;
    // Only when every row's cluster of four is resident at once (the merge
    // waits for the other pair of the cluster).
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!g_clusters4_init) {
        for (int i = 0; i < 64; ++i) g_clusters4[i] = -1;
        g_clusters4_init = true;
    }
    if (g_clusters4[dev] < 0) {
        int n = 0;
        if (hs_host::ensure_dynamic_smem(reinterpret_cast<const void*>(mla_pair_kernel<4>),
                                         size_t(kSmemBytes), g_smem_set4) == HS_OK) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(4);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = size_t(kSmemBytes);
            if (cudaOccupancyMaxActiveClusters(&n, mla_pair_kernel<4>, &cfg) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
        }
        g_clusters4[dev] = n;
    }
    return rows <= g_clusters4[dev];
}

int launch_mla_pair(const MlaArgs& a, int pairs, hs_stream_t stream) {
    if (mla_pair_cluster_merge(a.rows, a.splits)) {
        const int rc = hs_host::ensure_dynamic_smem(
            reinterpret_cast<const void*>(mla_pair_kernel<4>), size_t(kSmemBytes), g_smem_set4);
        if (rc != HS_OK) return rc;
        return hs_host::launch_pdl(mla_pair_kernel<4>, dim3(2 * pairs), dim3(kThreads),
                                   size_t(kSmemBytes), stream, a);
    }
    const int rc = hs_host::ensure_dynamic_smem(reinterpret_cast<const void*>(mla_pair_kernel<2>),
                                                size_t(kSmemBytes), g_smem_set2);
    if (rc != HS_OK) return rc;
    return hs_host::launch_pdl(mla_pair_kernel<2>, dim3(2 * pairs), dim3(kThreads),
                               size_t(kSmemBytes), stream, a);
}

}  // namespace hs_attn
