// hs_attention.cu -- S4, sparse decode attention on CUDA cores, and the
// split-KV merge.
//
// PaperTrace 5.1.1 "从索引到 Kernel": section 3.1 eqs. (4)-(6) (per-tile max,
// exponent sums and rescaled accumulators), section 3.2 (mask before the
// exponent; an empty candidate set gives a zero output and LSE = -inf) and
// eq. (7) (exact split-KV merge of unnormalised partial states).
// "PagedAttention 与 RadixAttention：上游机制与海光实现对照" section 1.4: the
// exp2 form with scale * log2(e) folded in, the v2 combine, and the GQA grid
// over KV heads so that one work unit serves its whole query-head group and
// reads each K/V row once.
//
// GB300 design (HBM-bound: ~4 FLOP/byte for GQA): one CTA of 8 warps per
// (index row, KV head, head chunk, split).  Each warp streams its share of
// candidate rows straight from the paged cache (no gather copy: PaperTrace
// section 2.1 eq. (3)), every lane holding one 4-byte bf16 pair of each 64-
// element block, so a warp-wide load of a row is one coalesced 128-byte line.
// Warps keep private online-softmax states (eqs. 5-6 in the exp2 domain);
// the 8 states are merged by eq. (7) through shared memory, and the splits by
// merge_kernel (eq. 7 again) when a row is split.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>
#include <atomic>

#include "hs_attention_internal.cuh"
#include "hs_common.cuh"

namespace hs_attn {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    int64_t row_stride, head_stride, num_kv_rows;
    const int32_t* kv_rows;
    const int32_t* count;
    int32_t rows, cap, heads, kv_heads, d_qk, d_v;
    float scale_log2;  // scale * log2(e)
    __nv_bfloat16* out;
    float* lse;
    float* part_m;  // [rows*heads, splits]
    float* part_l;
    float* part_o;  // [rows*heads, part_stride, d_v]
    int32_t splits, chunks_per_kvh;
    int32_t* status;
    int32_t part_stride, part_base, force_partial;
    int32_t* sync;  // GQA: one arrival counter per unit (zeroed), the last split merges; or null
};

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
    float2 r;
    r.x = __uint_as_float(u << 16);
    r.y = __uint_as_float(u & 0xffff0000u);
    return r;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// G query heads of one KV head, rows of DQK (K) / DV (V) bf16 elements.
template <int DQK, int DV, int G, bool SHARED_KV, int U>
__global__ void __launch_bounds__(kThreads) attn_cc_kernel(const AttnArgs a) {
    hs::pdl_trigger();
    constexpr int NQ = DQK / 64;
    constexpr int NV = DV / 64;
    extern __shared__ __align__(16) float red[];  // [kWarps][G][DV] + m,l [kWarps][G]

    const int unit = blockIdx.x;
    const int split = blockIdx.y;
    const int chunk = unit % a.chunks_per_kvh;
    const int kvh = (unit / a.chunks_per_kvh) % a.kv_heads;
    const int row = unit / (a.chunks_per_kvh * a.kv_heads);
    const int group = a.heads / a.kv_heads;
    const int h0 = kvh * group + chunk * G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Query registers, pre-scaled into the exp2 domain.
    float2 q[G][NQ];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint32_t* qr =
            reinterpret_cast<const uint32_t*>(a.q + (int64_t(row) * a.heads + h0 + h) * DQK);
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            float2 f = bf2_to_f2(__ldg(qr + 32 * i + lane));
            q[h][i] = make_float2(f.x * a.scale_log2, f.y * a.scale_log2);
        }
    }
    float2 o[G][NV];
    float m[G], l[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -CUDART_INF_F;
        l[h] = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) o[h][i] = make_float2(0.f, 0.f);
    }

    const int64_t idx_base = (int64_t(row) * a.kv_heads + kvh) * a.cap;
    const int n = a.count ? min(max(a.count[int64_t(row) * a.kv_heads + kvh], 0), a.cap) : a.cap;
    const int per = (n + a.splits - 1) / a.splits;
    const int t0 = min(n, split * per), t1 = min(n, t0 + per);
    const char* kb = reinterpret_cast<const char*>(a.k) + int64_t(kvh) * a.head_stride * 2;
    const char* vb = reinterpret_cast<const char*>(a.v) + int64_t(kvh) * a.head_stride * 2;
    bool bad = false;

    // Software pipeline per warp: the row ids of iteration it+2 and the K/V
    // rows of iteration it+1 are in flight while iteration it is computed.
    constexpr int kStep = kWarps * U;
    int32_t id_n2[U];   // ids two iterations ahead
    int64_t rs_n[U];    // rows one iteration ahead
    uint32_t kr_n[U][NQ];
    uint32_t vr_n[U][SHARED_KV ? 1 : NV];
    auto load_ids = [&](int j0, int32_t (&id)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u;
            id[u] = j < t1 ? __ldg(a.kv_rows + idx_base + j) : -1;
        }
    };
    auto load_rows = [&](const int32_t (&id)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            int64_t r = id[u];
            if (r >= a.num_kv_rows) { bad = true; r = -1; }
            if (r < 0) r = -1;
            rs_n[u] = r;
            if (r >= 0) {  // warp-uniform branch
                const uint32_t* kp = reinterpret_cast<const uint32_t*>(kb + r * a.row_stride * 2);
#pragma unroll
                for (int i = 0; i < NQ; ++i) kr_n[u][i] = __ldg(kp + 32 * i + lane);
                if constexpr (!SHARED_KV) {
                    const uint32_t* vp =
                        reinterpret_cast<const uint32_t*>(vb + r * a.row_stride * 2);
#pragma unroll
                    for (int i = 0; i < NV; ++i) vr_n[u][i] = __ldg(vp + 32 * i + lane);
                }
            } else {
#pragma unroll
                for (int i = 0; i < NQ; ++i) kr_n[u][i] = 0u;
                if constexpr (!SHARED_KV) {
#pragma unroll
                    for (int i = 0; i < NV; ++i) vr_n[u][i] = 0u;
                }
            }
        }
    };
    {
        int32_t id0[U];
        load_ids(t0 + warp * U, id0);
        load_ids(t0 + warp * U + kStep, id_n2);
        load_rows(id0);
    }
    for (int j0 = t0 + warp * U; j0 < t1; j0 += kStep) {
        // Current iteration's rows, then start the next iteration's loads.
        int64_t rowsel[U];
        uint32_t kr[U][NQ];
        uint32_t vr[U][SHARED_KV ? 1 : NV];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            rowsel[u] = rs_n[u];
#pragma unroll
            for (int i = 0; i < NQ; ++i) kr[u][i] = kr_n[u][i];
            if constexpr (!SHARED_KV) {
#pragma unroll
                for (int i = 0; i < NV; ++i) vr[u][i] = vr_n[u][i];
            }
        }
        if (j0 + kStep < t1) {
            int32_t id1[U];
#pragma unroll
            for (int u = 0; u < U; ++u) id1[u] = id_n2[u];
            load_ids(j0 + 2 * kStep, id_n2);
            load_rows(id1);
        }
        float s[U][G];
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    const float2 kf = bf2_to_f2(kr[u][i]);
                    acc = fmaf(q[h][i].x, kf.x, acc);
                    acc = fmaf(q[h][i].y, kf.y, acc);
                }
                acc = warp_sum(acc);
                s[u][h] = rowsel[u] >= 0 ? acc : -CUDART_INF_F;
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float mb = s[0][h];
#pragma unroll
            for (int u = 1; u < U; ++u) mb = fmaxf(mb, s[u][h]);
            const float mn = fmaxf(m[h], mb);
            if (mn == -CUDART_INF_F) continue;  // nothing valid yet: skip the empty tile
            const float alpha = exp2f(m[h] - mn);
            float p[U];
            float ps = 0.f;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                p[u] = exp2f(s[u][h] - mn);
                ps += p[u];
            }
            l[h] = l[h] * alpha + ps;
            m[h] = mn;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                float2 acc = make_float2(o[h][i].x * alpha, o[h][i].y * alpha);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float2 vf = bf2_to_f2(SHARED_KV ? kr[u][i] : vr[u][SHARED_KV ? 0 : i]);
                    acc.x = fmaf(p[u], vf.x, acc.x);
                    acc.y = fmaf(p[u], vf.y, acc.y);
                }
                o[h][i] = acc;
            }
        }
    }
    if (bad) hs::set_status(a.status, HS_ERR_BAD_INDEX);

    // Merge the warps' states (eq. 7) through shared memory.
    float* so = red;                           // [kWarps][G][DV]
    float* sm = red + kWarps * G * DV;         // [kWarps][G]
    float* sl = sm + kWarps * G;               // [kWarps][G]
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float2* dst = reinterpret_cast<float2*>(so + (warp * G + h) * DV + 64 * i) + lane;
            *dst = o[h][i];
        }
        if (lane == 0) {
            sm[warp * G + h] = m[h];
            sl[warp * G + h] = l[h];
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < G * DV; e += kThreads) {
        const int h = e / DV, d = e % DV;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            if (sl[w * G + h] > 0.f) M = fmaxf(M, sm[w * G + h]);
        float L = 0.f, O = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float lw = sl[w * G + h];
                if (!(lw > 0.f)) continue;
                const float sc = exp2f(sm[w * G + h] - M);
                L = fmaf(sc, lw, L);
                O = fmaf(sc, so[(w * G + h) * DV + d], O);
            }
        }
        const int64_t qh = int64_t(row) * a.heads + h0 + h;
        if (a.splits == 1 && !a.force_partial) {
            a.out[qh * DV + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
            if (d == 0 && a.lse != nullptr)
                a.lse[qh] = L > 0.f ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
        } else {
            const int64_t pi = qh * a.part_stride + a.part_base + split;
            a.part_o[pi * DV + d] = O;
            if (d == 0) {
                a.part_m[pi] = M;
                a.part_l[pi] = L;
            }
        }
    }
}

// Eq. (7) over `parts` partial states per output row; m in log2 units.
__global__ void merge_kernel(const float* __restrict__ pm, const float* __restrict__ pl,
                             const float* __restrict__ po, int32_t parts, int32_t d_v,
                             __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                             int32_t stride) {
    hs::pdl_trigger();
    const int64_t n = blockIdx.x;
    const float* m = pm + n * stride;
    const float* l = pl + n * stride;
    float M = -CUDART_INF_F;
    for (int p = 0; p < parts; ++p)
        if (l[p] > 0.f) M = fmaxf(M, m[p]);
    float L = 0.f;
    if (M != -CUDART_INF_F)
        for (int p = 0; p < parts; ++p)
            if (l[p] > 0.f) L = fmaf(exp2f(m[p] - M), l[p], L);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int d = threadIdx.x; d < d_v; d += blockDim.x) {
        float O = 0.f;
        if (M != -CUDART_INF_F)
            for (int p = 0; p < parts; ++p)
                if (l[p] > 0.f) O = fmaf(exp2f(m[p] - M), po[(n * stride + p) * d_v + d], O);
        out[n * d_v + d] = __float2bfloat16_rn(O * inv);
    }
    if (threadIdx.x == 0 && lse != nullptr)
        lse[n] = L > 0.f ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
}

// ----------------------------------------------------------------------------
// Host side: kernel choice and split policy.

struct Plan {
    int kind;  // 0 unsupported, 1 MLA on CUDA cores, 2 GQA d=128, 3 MLA on tcgen05,
               // 4 MLA with 128 heads on tcgen05 CTA pairs
    int G;     // heads per CTA
    int chunks_per_kvh;
    int splits;
    int kv_heads;
};

// pair_ok: the one-call decode (no caller-held partial columns) may use the
// CTA-pair kernel for 128 heads.
Plan make_plan(int rows, int heads, int kv_heads, int cap, int d_qk, int d_v, bool shared,
               bool pair_ok) {
    Plan p{0, 0, 0, 1, kv_heads};
    if (rows <= 0 || heads <= 0 || kv_heads <= 0 || heads % kv_heads) return p;
    const int group = heads / kv_heads;
    const bool mla = d_qk == 576 && d_v == 512 && kv_heads == 1 && shared;
    if (mla && heads == 128 && pair_ok) {
        // One CTA pair per (row, split): every row of a 256-row pair tile is
        // gathered once for all 128 heads; splits fill the SM pairs once.
        p.kind = 4;
        p.G = 128;
        p.chunks_per_kvh = 1;
        const int64_t pairs = hs::max64(1, hs_host::num_sms() / 2);
        int64_t s = rows >= pairs ? 1 : pairs / rows;
        s = hs::min64(s, hs::max64(1, (cap + 255) / 256));
        p.splits = int(hs::max64(1, hs::min64(s, kMlaPairMaxSplits)));
        return p;
    }
    if (mla && mla_tc_head_group(heads) > 0) {
        // Tensor-core kernel: one CTA per SM (about 220 KB of shared memory);
        // split the candidate list so that the grid fills the SMs once.
        p.kind = 3;
        p.G = mla_tc_head_group(heads);
        p.chunks_per_kvh = heads / p.G;
        const int64_t units = int64_t(rows) * p.chunks_per_kvh;
        const int64_t sms = hs_host::num_sms();
        int64_t s = units >= sms ? 1 : sms / units;
        s = hs::min64(s, hs::max64(1, (cap + 127) / 128));
        p.splits = int(hs::max64(1, hs::min64(s, 64)));
        return p;
    }
    if (mla && heads % 4 == 0) {
        p.kind = 1;
        p.G = 4;
    } else if (d_qk == 128 && d_v == 128 && (group == 1 || group == 2 || group == 4 || group == 8)) {
        p.kind = 2;
        p.G = group;
    } else {
        return p;
    }
    p.chunks_per_kvh = group / p.G;
    const int64_t units = int64_t(rows) * kv_heads * p.chunks_per_kvh;
    // GQA: one resident wave (one CTA per SM), so that longer CTAs amortise
    // the Q load, the epilogue and the merge.  MLA on CUDA cores: up to four
    // CTAs per SM.
    const int64_t per_sm = p.kind == 2 ? 1 : 4;
    const int64_t target = per_sm * hs_host::num_sms();
    int64_t s = hs::max64(1, target / units);
    s = hs::min64(s, std::max(1, cap / 32));
    s = hs::max64(1, hs::min64(s, 64));
    p.splits = int(s);
    return p;
}

// Bytes of the partial states; the tcgen05 MLA and the GQA kernels also keep
// one arrival counter per work unit behind them, 16-byte aligned.
int64_t partial_bytes(const Plan& p, int rows, int heads, int d_v) {
    const int64_t n = int64_t(rows) * heads;
    return n * p.splits * (2 + int64_t(d_v)) * int64_t(sizeof(float));
}

int64_t sync_words(const Plan& p, int rows) {
    return int64_t(rows) * p.kv_heads * p.chunks_per_kvh;
}

// CTA-pair kernel: partial O, then (m, l) per CTA rank, then counters.
int64_t pair_part_o_bytes(const Plan& p, int rows) {
    return int64_t(rows) * 128 * p.splits * 512 * int64_t(sizeof(float));
}
int64_t pair_part_ml_bytes(const Plan& p, int rows) {
    return 2 * int64_t(rows) * 128 * p.splits * 2 * int64_t(sizeof(float));
}

int64_t workspace_bytes(const Plan& p, int rows, int heads, int d_v) {
    if (p.kind == 0 || p.splits <= 1) return 0;
    if (p.kind == 4) {
        // A row's two splits merged inside one cluster need no scratch.
        if (mla_pair_cluster_merge(rows, p.splits)) return 0;
        return pair_part_o_bytes(p, rows) + pair_part_ml_bytes(p, rows) +
               (int64_t(rows) * 4 * 4 + 15) / 16 * 16;
    }
    int64_t b = partial_bytes(p, rows, heads, d_v);
    if (p.kind == 3 || p.kind == 2) b += (sync_words(p, rows) * 4 + 15) / 16 * 16;
    return b;
}

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Warp-level bf16 tensor-core helpers (mma.sync m16n8k16 and ldmatrix; PTX
// ISA "Warp-level matrix instructions").  Fragment ownership, g = lane / 4,
// t = lane % 4: A (16 x 16, row-major) a0 = (g, 2t..2t+1), a1 = (g + 8, 2t..),
// a2 = (g, 2t + 8..), a3 = (g + 8, 2t + 8..); B (16 x 8, k x n) b0 = (2t..2t+1,
// g), b1 = (2t + 8.., g); C (16 x 8) c0, c1 = (g, 2t..2t+1), c2, c3 = (g + 8,
// 2t..).
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a2,
                                               uint32_t b0, uint32_t b1) {
    // Rows 8..15 of A are zero (a head group has at most 8 query heads).
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&d)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&d)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// GQA rows of 128 bf16 with K and V in separate caches, on the warp-level
// tensor cores.  A head group (G <= 8 query heads of one KV head) is the M
// dimension of both products, padded to 16: per block of 16 candidates a warp
// computes S = Q K^T (8 k-steps of 16 dims, two n-tiles of 8 candidates) and
// O += P V (16 n-tiles of 8 dims, one k-step of 16 candidates), and the S
// accumulators are the A fragment of P V in place, so the online softmax
// (eqs. 4-6, exp2 domain) runs on registers between the two: four scores a
// lane, two shuffles for the row maximum, and the row sum kept per lane until
// the end.  The contraction is only G wide, so the kernel is HBM-bound; the
// tensor cores are there to take the dot products off the issue slots.
//
// Loads: the CTA's candidate ids are staged in shared memory (one coalesced
// read per chunk of kIdChunk); each warp streams its blocks (every W-th block
// of 16) through a private S-stage cp.async ring of [16 x 256 B] K and V tiles
// whose 16-byte chunks are XOR-swizzled by (candidate mod 8), so that every
// 8 x 8 ldmatrix touches 8 distinct bank groups.  Absent candidates are zero-
// filled and masked.  Each warp keeps its own state; the W states are merged
// with eq. (7) through shared memory, the splits by merge_kernel.
constexpr int kIdChunk = 2048;
constexpr int kGqaMaxSplits = 64;             // splits of one unit (the plan's limit)
constexpr int kGqaBlock = 16;                 // candidates per warp step
constexpr int kGqaTile = kGqaBlock * 256;     // bytes of one K (or V) tile

template <int G, int W, int S>
constexpr size_t gqa_smem_bytes() {
    constexpr size_t ring = size_t(W) * S * 2 * kGqaTile;
    constexpr size_t reduce = size_t(W) * G * (128 + 2) * sizeof(float);
    return kIdChunk * sizeof(int32_t) + (ring > reduce ? ring : reduce);
}

template <int G, int W, int S>
__global__ void __launch_bounds__(W * 32) attn_gqa_kernel(const AttnArgs a) {
    hs::pdl_trigger();
    static_assert(G >= 1 && G <= 8, "a head group fills at most half of the MMA rows");
    constexpr int D = 128;
    extern __shared__ __align__(128) unsigned char gsm[];
    int32_t* ids = reinterpret_cast<int32_t*>(gsm);                    // [kIdChunk]
    unsigned char* ring = gsm + kIdChunk * sizeof(int32_t);            // [W][S][K, V tile]
    float* red = reinterpret_cast<float*>(ring);  // after the loop: [W][G][D] + m, l [W][G]

    const int unit = blockIdx.x;
    const int split = blockIdx.y;
    const int chunk = unit % a.chunks_per_kvh;
    const int kvh = (unit / a.chunks_per_kvh) % a.kv_heads;
    const int row = unit / (a.chunks_per_kvh * a.kv_heads);
    const int group = a.heads / a.kv_heads;
    const int h0 = kvh * group + chunk * G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;

    // Q as the A fragment of 8 k-steps (rows g < G; the other rows are 0).
    uint32_t qa[8][2];
    {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            a.q + (int64_t(row) * a.heads + h0 + min(g, G - 1)) * D);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qa[ks][0] = g < G ? __ldg(qrow + ks * 8 + t) : 0u;
            qa[ks][1] = g < G ? __ldg(qrow + ks * 8 + 4 + t) : 0u;
        }
    }
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m = -CUDART_INF_F, l = 0.f;  // state of head row g (l: this lane's columns)

    const int64_t idx_base = (int64_t(row) * a.kv_heads + kvh) * a.cap;
    const int n = a.count ? min(max(a.count[int64_t(row) * a.kv_heads + kvh], 0), a.cap) : a.cap;
    const int per = (n + a.splits - 1) / a.splits;
    const int t0 = min(n, split * per), t1 = min(n, t0 + per);
    const char* kb = reinterpret_cast<const char*>(a.k) + int64_t(kvh) * a.head_stride * 2;
    const char* vb = reinterpret_cast<const char*>(a.v) + int64_t(kvh) * a.head_stride * 2;
    const uint32_t ring_w = hs::smem_u32(ring) + uint32_t(warp) * (S * 2 * kGqaTile);
    bool bad = false;

    // Copy lanes: 16-byte chunk cc = lane % 16 of candidates 2 i + lane / 16,
    // i = 0..7, so that one warp-wide copy moves two whole rows.
    const int cc = lane & 15, ch = lane >> 4;
    // ldmatrix lanes: matrix mi = lane / 8, row r = lane % 8 of it.
    const int mi = lane >> 3, r8 = lane & 7;

    for (int c0 = t0; c0 < t1; c0 += kIdChunk) {
        const int cn = min(kIdChunk, t1 - c0);
        __syncthreads();  // the previous chunk's ids are no longer read
        for (int i = threadIdx.x; i < cn; i += W * 32) {
            const int32_t r = __ldg(a.kv_rows + idx_base + c0 + i);
            if (r >= a.num_kv_rows) bad = true;
            ids[i] = r < a.num_kv_rows ? r : -1;
        }
        __syncthreads();
        const int nblk = (cn + kGqaBlock - 1) / kGqaBlock;
        const int niter = nblk > warp ? (nblk - warp + W - 1) / W : 0;  // warp-uniform
        auto issue = [&](int it) {
            const int jb = (it * W + warp) * kGqaBlock;
            const uint32_t st = ring_w + uint32_t(it % S) * (2 * kGqaTile);
#pragma unroll
            for (int i = 0; i < kGqaBlock / 2; ++i) {
                const int key = 2 * i + ch;
                const int j = jb + key;
                const int32_t r = j < cn ? ids[j] : -1;
                const int64_t off = r >= 0 ? int64_t(r) * a.row_stride * 2 + cc * 16 : 0;
                const uint32_t nb = r >= 0 ? 16u : 0u;  // 0: zero-fill, nothing read
                const uint32_t dst = st + key * 256 + uint32_t((cc ^ (key & 7)) * 16);
                cp_async16_zfill(dst, kb + off, nb);
                cp_async16_zfill(dst + kGqaTile, vb + off, nb);
            }
        };
#pragma unroll
        for (int it = 0; it < S - 1; ++it) {
            if (it < niter) issue(it);
            cp_async_commit();
        }
        for (int it = 0; it < niter; ++it) {
            if (it + S - 1 < niter) issue(it + S - 1);
            cp_async_commit();
            cp_async_wait<S - 1>();
            __syncwarp();
            const uint32_t kt = ring_w + uint32_t(it % S) * (2 * kGqaTile);
            const uint32_t vt = kt + kGqaTile;

            // S = Q K^T: n-tile 0 = candidates 0..7, n-tile 1 = 8..15.
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
            {
                const int key = r8 + (mi >> 1) * 8;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int c = 2 * ks + (mi & 1);
                    uint32_t b[4];
                    ldsm_x4(kt + key * 256 + ((c ^ r8) * 16), b);
                    mma_bf16_16816(s0, qa[ks][0], qa[ks][1], b[0], b[1]);
                    mma_bf16_16816(s1, qa[ks][0], qa[ks][1], b[2], b[3]);
                }
            }
            // Online softmax of head row g over this lane's four candidates.
            const int jb = (it * W + warp) * kGqaBlock;
            float x[4] = {s0[0], s0[1], s1[0], s1[1]};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = jb + (i >> 1) * 8 + 2 * t + (i & 1);
                const bool live = j < cn && ids[j] >= 0;
                x[i] = live ? x[i] * a.scale_log2 : -CUDART_INF_F;
            }
            float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m, mx);
            float alpha = 1.f;
            uint32_t pa0 = 0u, pa2 = 0u;
            if (mn != -CUDART_INF_F) {
                alpha = exp2f(m - mn);
                // P is rounded to bf16 for the MMA; the row sum uses the
                // rounded weights so that numerator and denominator agree.
                pa0 = pack_bf16x2(exp2f(x[0] - mn), exp2f(x[1] - mn));
                pa2 = pack_bf16x2(exp2f(x[2] - mn), exp2f(x[3] - mn));
                const float2 p01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pa0));
                const float2 p23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pa2));
                l = l * alpha + ((p01.x + p01.y) + (p23.x + p23.y));
                m = mn;
            }
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    o[nt][0] *= alpha;
                    o[nt][1] *= alpha;
                }
            }
            // O += P V: n-tiles 2 np and 2 np + 1 (dims 16 np .. 16 np + 15).
            {
                const int key = r8 + (mi & 1) * 8;
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    const int c = 2 * np + (mi >> 1);
                    uint32_t b[4];
                    ldsm_x4_trans(vt + key * 256 + ((c ^ r8) * 16), b);
                    mma_bf16_16816(o[2 * np], pa0, pa2, b[0], b[1]);
                    mma_bf16_16816(o[2 * np + 1], pa0, pa2, b[2], b[3]);
                }
            }
            __syncwarp();  // every lane's reads of this stage precede its refill
        }
    }
    cp_async_wait<0>();
    if (bad) hs::set_status(a.status, HS_ERR_BAD_INDEX);
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    __syncthreads();  // the ring is reused for the reduction below

    // Merge the W warps' states (eq. 7) through shared memory.
    float* so = red;                     // [W][G][D]
    float* sm = red + W * G * D;         // [W][G]
    float* sl = sm + W * G;              // [W][G]
    if (g < G) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
            *reinterpret_cast<float2*>(so + (warp * G + g) * D + nt * 8 + 2 * t) =
                make_float2(o[nt][0], o[nt][1]);
        if (t == 0) {
            sm[warp * G + g] = m;
            sl[warp * G + g] = l;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < G * D; e += W * 32) {
        const int h = e / D, d = e % D;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < W; ++w)
            if (sl[w * G + h] > 0.f) M = fmaxf(M, sm[w * G + h]);
        float L = 0.f, O = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float lw = sl[w * G + h];
                if (!(lw > 0.f)) continue;
                const float sc = exp2f(sm[w * G + h] - M);
                L = fmaf(sc, lw, L);
                O = fmaf(sc, so[(w * G + h) * D + d], O);
            }
        }
        const int64_t qh = int64_t(row) * a.heads + h0 + h;
        if (a.splits == 1 && !a.force_partial) {
            a.out[qh * D + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
            if (d == 0 && a.lse != nullptr)
                a.lse[qh] = L > 0.f ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
        } else {
            const int64_t pi = qh * a.part_stride + a.part_base + split;
            a.part_o[pi * D + d] = O;
            if (d == 0) {
                a.part_m[pi] = M;
                a.part_l[pi] = L;
            }
        }
    }
    if (a.sync == nullptr) return;

    // Split merge (eq. 7) by the split of this unit that finishes last: every
    // split publishes its partial state, then counts itself in; the one that
    // sees splits - 1 earlier arrivals reads all of them back from L2, in
    // three dependent steps: the (m, l) pairs into shared memory, the weights
    // of each head, then the partial outputs with independent loads.
    __shared__ int last_split;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        last_split = atomicAdd(a.sync + unit, 1) == a.splits - 1;
        if (last_split) a.sync[unit] = 0;  // every split has arrived: reset for the next call
    }
    __syncthreads();
    if (!last_split) return;
    __threadfence();
    float* wm = red;                              // [G][kGqaMaxSplits] m, then weights
    float* wl = red + G * kGqaMaxSplits;          // [G][kGqaMaxSplits] l
    float* winv = wl + G * kGqaMaxSplits;         // [G] 1 / L and [G] lse
    const int64_t qh0 = int64_t(row) * a.heads + h0;
    for (int e = threadIdx.x; e < G * a.splits; e += W * 32) {
        const int h = e / a.splits, sp = e % a.splits;
        wm[h * kGqaMaxSplits + sp] = __ldcg(a.part_m + (qh0 + h) * a.part_stride + sp);
        wl[h * kGqaMaxSplits + sp] = __ldcg(a.part_l + (qh0 + h) * a.part_stride + sp);
    }
    __syncthreads();
    if (threadIdx.x < G) {
        const int h = threadIdx.x;
        float M = -CUDART_INF_F;
        for (int sp = 0; sp < a.splits; ++sp)
            if (wl[h * kGqaMaxSplits + sp] > 0.f) M = fmaxf(M, wm[h * kGqaMaxSplits + sp]);
        float L = 0.f;
        for (int sp = 0; sp < a.splits; ++sp) {
            const float lw = wl[h * kGqaMaxSplits + sp];
            const float sc = (M != -CUDART_INF_F && lw > 0.f)
                                 ? exp2f(wm[h * kGqaMaxSplits + sp] - M) : 0.f;
            L = fmaf(sc, lw, L);
            wm[h * kGqaMaxSplits + sp] = sc;
        }
        winv[h] = L > 0.f ? 1.f / L : 0.f;
        winv[G + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < G * D; e += W * 32) {
        const int h = e / D, d = e % D;
        const float* po = a.part_o + (qh0 + h) * a.part_stride * D + d;
        float O = 0.f;
#pragma unroll 8
        for (int sp = 0; sp < a.splits; ++sp)
            O = fmaf(wm[h * kGqaMaxSplits + sp], __ldcg(po + int64_t(sp) * D), O);
        a.out[(qh0 + h) * D + d] = __float2bfloat16_rn(O * winv[h]);
        if (d == 0 && a.lse != nullptr) a.lse[qh0 + h] = winv[G + h];
    }
}

// Warps per CTA and ring stages of the GQA kernel: one CTA per SM (about
// 200 KB of shared memory), 8 warps x 2 blocks of 8 KB in flight.
constexpr int kGqaWarps = 8;
constexpr int kGqaStages = 3;

template <int G>
int launch_gqa(const AttnArgs& a, int units, hs_stream_t stream) {
    auto kern = attn_gqa_kernel<G, kGqaWarps, kGqaStages>;
    constexpr size_t smem = gqa_smem_bytes<G, kGqaWarps, kGqaStages>();
    static int smem_set[64] = {};
    const int rc = hs_host::ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem,
                                                smem_set);
    if (rc != HS_OK) return rc;
    dim3 grid(units, a.splits);
    kern<<<grid, kGqaWarps * 32, smem, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    return hs_host::launch_status();
}

template <int DQK, int DV, int G, bool SHARED, int U>
int launch(const AttnArgs& a, int units, hs_stream_t stream) {
    auto kern = attn_cc_kernel<DQK, DV, G, SHARED, U>;
    const size_t smem = size_t(kWarps) * G * (DV + 2) * sizeof(float);
    static int smem_set[64] = {};
    const int rc = hs_host::ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem,
                                                smem_set);
    if (rc != HS_OK) return rc;
    dim3 grid(units, a.splits);
    kern<<<grid, kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    return hs_host::launch_status();
}

}  // namespace hs_attn

using namespace hs_attn;

extern "C" int64_t hs_sparse_decode_workspace_bytes(int32_t rows, int32_t heads,
                                                    int32_t kv_heads, int32_t cap,
                                                    int32_t d_qk, int32_t d_v) {
    const Plan p =
        make_plan(rows, heads, kv_heads, cap, d_qk, d_v, kv_heads == 1 && d_qk == 576, true);
    return workspace_bytes(p, rows, heads, d_v);
}

namespace {

struct PartialOut {
    float* m;
    float* l;
    float* o;
    int32_t parts_total;
    int32_t part_base;
    int32_t finish;  // 1: merge with columns [0, part_base) and write out / lse
    int32_t* sync;   // finish: arrival counters (rows * heads int32) for the last-CTA merge, or null
};

int decode_impl(const void* q, const void* k_base, const void* v_base, int64_t row_stride,
                int64_t kv_head_stride, int64_t num_kv_rows, const int32_t* kv_rows,
                const int32_t* count, int32_t rows, int32_t cap, int32_t heads, int32_t kv_heads,
                int32_t d_qk, int32_t d_v, float scale, void* out, float* lse, void* workspace,
                int64_t workspace_bytes_given, const PartialOut* po, int32_t* status,
                hs_stream_t stream) {
    if (rows < 0 || cap < 0 || heads <= 0 || kv_heads <= 0 || d_qk <= 0 || d_v <= 0 ||
        row_stride <= 0 || kv_head_stride < 0 || num_kv_rows < 0)
        return HS_ERR_INVALID_ARG;
    if (rows == 0) return HS_OK;
    if (q == nullptr || k_base == nullptr || v_base == nullptr ||
        (po == nullptr && out == nullptr) || (cap > 0 && kv_rows == nullptr))
        return HS_ERR_INVALID_ARG;
    const auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(q) || !al(k_base) || !al(v_base) || (out != nullptr && !al(out)) ||
        row_stride % 8 || kv_head_stride % 8)
        return HS_ERR_MISALIGNED;
    const bool shared = k_base == v_base;
    const Plan p = make_plan(rows, heads, kv_heads, cap, d_qk, d_v, shared, po == nullptr);
    if (p.kind == 0) return HS_ERR_UNSUPPORTED;
    const int64_t n = int64_t(rows) * heads;
    AttnArgs a{};
    int combine = 0;
    int32_t* sync = nullptr;
    int merge_total = 0;
    Plan pl = p;
    if (po != nullptr) {
        if (po->m == nullptr || po->l == nullptr || po->o == nullptr || po->part_base < 0 ||
            po->part_base > po->parts_total)
            return HS_ERR_INVALID_ARG;
        // The last-CTA merge reads part_o in 16-byte vectors.
        if (po->finish && pl.kind == 3 && po->sync != nullptr && p.splits > 1 &&
            (reinterpret_cast<uintptr_t>(po->o) & 15u) == 0 &&
            po->part_base + p.splits <= std::min(po->parts_total, kMlaMaxMerge)) {
            // Several CTAs per row and head group; the last to finish merges.
            if (out == nullptr) return HS_ERR_INVALID_ARG;
            sync = po->sync;
            merge_total = po->part_base + p.splits;
        } else if (po->finish && pl.kind == 3 && po->part_base <= 4) {
            // One CTA per row and head group; its epilogue merges.
            pl.splits = 1;
            combine = po->part_base;
            if (out == nullptr) return HS_ERR_INVALID_ARG;
        } else if (po->part_base + p.splits > po->parts_total) {
            return HS_ERR_INVALID_ARG;
        }
        a.part_m = po->m;
        a.part_l = po->l;
        a.part_o = po->o;
        a.part_stride = po->parts_total;
        a.part_base = po->part_base;
        const bool fused = po->finish && pl.kind == 3 && po->part_base <= 4 && sync == nullptr;
        a.force_partial = fused ? 0 : 1;
    } else {
        const int64_t ws = workspace_bytes(p, rows, heads, d_v);
        if (ws > 0 && (workspace == nullptr || workspace_bytes_given < ws)) return HS_ERR_CAPACITY;
        if (p.kind == 4) {
            MlaArgs m{};
            m.q = static_cast<const __nv_bfloat16*>(q);
            m.kv = static_cast<const __nv_bfloat16*>(k_base);
            m.row_stride = row_stride;
            m.num_kv_rows = num_kv_rows;
            m.kv_rows = kv_rows;
            m.count = count;
            m.rows = rows;
            m.cap = cap;
            m.heads = heads;
            m.scale_log2 = scale * kLog2e;
            m.out = static_cast<__nv_bfloat16*>(out);
            m.lse = lse;
            m.splits = p.splits;
            m.status = status;
            m.timeout_ns = hs::kWaitTimeoutNs;
            if (p.splits > 1 && !mla_pair_cluster_merge(rows, p.splits)) {
                unsigned char* w = static_cast<unsigned char*>(workspace);
                m.part_o = reinterpret_cast<float*>(w);
                m.part_m = reinterpret_cast<float*>(w + pair_part_o_bytes(p, rows));
                m.sync = reinterpret_cast<int32_t*>(w + pair_part_o_bytes(p, rows) +
                                                    pair_part_ml_bytes(p, rows));
                if (cudaMemsetAsync(m.sync, 0, size_t(rows) * 4 * sizeof(int32_t),
                                    reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
                    return HS_ERR_CUDA;
            }
            return launch_mla_pair(m, rows * p.splits, stream);
        }
        if (p.splits > 1) {
            float* w = static_cast<float*>(workspace);
            a.part_m = w;
            a.part_l = w + n * p.splits;
            a.part_o = w + 2 * n * p.splits;
            if ((p.kind == 3 && p.splits <= kMlaMaxMerge && al(a.part_o)) || p.kind == 2) {
                sync = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) +
                                                  partial_bytes(p, rows, heads, d_v));
                merge_total = p.splits;
            }
        }
        a.part_stride = p.splits;
        a.part_base = 0;
        a.force_partial = 0;
    }
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k_base);
    a.v = static_cast<const __nv_bfloat16*>(v_base);
    a.row_stride = row_stride;
    a.head_stride = kv_head_stride;
    a.num_kv_rows = num_kv_rows;
    a.kv_rows = kv_rows;
    a.count = count;
    a.rows = rows;
    a.cap = cap;
    a.heads = heads;
    a.kv_heads = kv_heads;
    a.d_qk = d_qk;
    a.d_v = d_v;
    a.scale_log2 = scale * kLog2e;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.splits = pl.splits;
    a.chunks_per_kvh = p.chunks_per_kvh;
    a.status = status;
    const int units = rows * kv_heads * p.chunks_per_kvh;
    a.sync = sync;
    // Counters in the workspace are zeroed here; the caller's counters of the
    // finishing pass are zero on entry, and every launch leaves them zero
    // (the last split resets its counter), so no memset node separates that
    // launch from its stream predecessor.
    if (sync != nullptr && po == nullptr &&
        cudaMemsetAsync(sync, 0, size_t(units) * sizeof(int32_t),
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return HS_ERR_CUDA;
    int rc;
    if (p.kind == 3) {
        MlaArgs m{};
        m.q = a.q;
        m.kv = a.k;
        m.row_stride = row_stride;
        m.num_kv_rows = num_kv_rows;
        m.kv_rows = kv_rows;
        m.count = count;
        m.rows = rows;
        m.cap = cap;
        m.heads = heads;
        m.scale_log2 = a.scale_log2;
        m.out = a.out;
        m.lse = lse;
        m.part_m = a.part_m;
        m.part_l = a.part_l;
        m.part_o = a.part_o;
        m.splits = pl.splits;
        m.part_stride = a.part_stride;
        m.part_base = a.part_base;
        m.force_partial = a.force_partial;
        m.combine_parts = combine;
        m.sync = sync;
        m.merge_total = merge_total;
        m.status = status;
        m.timeout_ns = hs::kWaitTimeoutNs;
        rc = launch_mla_tc(m, p.G, dim3(units, pl.splits), stream);
    } else if (p.kind == 1) {
        rc = launch<576, 512, 4, true, 2>(a, units, stream);
    } else {
        switch (p.G) {
            case 1: rc = launch_gqa<1>(a, units, stream); break;
            case 2: rc = launch_gqa<2>(a, units, stream); break;
            case 4: rc = launch_gqa<4>(a, units, stream); break;
            default: rc = launch_gqa<8>(a, units, stream); break;
        }
    }
    if (rc != HS_OK) return rc;
    if (sync != nullptr) return rc;  // merged by the last CTA of each (row, head group)
    if (po != nullptr) {
        if (!po->finish || (pl.kind == 3 && po->part_base <= 4)) return rc;
        // Finish on the other kernels: merge every column written so far.
        merge_kernel<<<int(n), 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
            a.part_m, a.part_l, a.part_o, po->part_base + p.splits, d_v,
            static_cast<__nv_bfloat16*>(out), lse, po->parts_total);
        return hs_host::launch_status();
    }
    if (p.splits == 1) return rc;
    merge_kernel<<<int(n), 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        a.part_m, a.part_l, a.part_o, p.splits, d_v, a.out, lse, p.splits);
    return hs_host::launch_status();
}

}  // namespace

extern "C" int hs_sparse_decode(const void* q, const void* k_base, const void* v_base,
                                int64_t row_stride, int64_t kv_head_stride, int64_t num_kv_rows,
                                const int32_t* kv_rows, const int32_t* count, int32_t rows,
                                int32_t cap, int32_t heads, int32_t kv_heads, int32_t d_qk,
                                int32_t d_v, float scale, void* out, float* lse,
                                void* workspace, int64_t workspace_bytes_given, int32_t* status,
                                hs_stream_t stream) {
    return decode_impl(q, k_base, v_base, row_stride, kv_head_stride, num_kv_rows, kv_rows, count,
                       rows, cap, heads, kv_heads, d_qk, d_v, scale, out, lse, workspace,
                       workspace_bytes_given, nullptr, status, stream);
}

extern "C" int32_t hs_sparse_decode_partial_splits(int32_t rows, int32_t heads, int32_t kv_heads,
                                                   int32_t cap, int32_t d_qk, int32_t d_v) {
    const Plan p =
        make_plan(rows, heads, kv_heads, cap, d_qk, d_v, kv_heads == 1 && d_qk == 576, false);
    return p.kind == 0 ? 0 : p.splits;
}

extern "C" int hs_sparse_decode_partial(const void* q, const void* k_base, const void* v_base,
                                        int64_t row_stride, int64_t kv_head_stride,
                                        int64_t num_kv_rows, const int32_t* kv_rows,
                                        const int32_t* count, int32_t rows, int32_t cap,
                                        int32_t heads, int32_t kv_heads, int32_t d_qk,
                                        int32_t d_v, float scale, float* part_m, float* part_l,
                                        float* part_o, int32_t parts_total, int32_t part_base,
                                        int32_t* status, hs_stream_t stream) {
    const PartialOut po{part_m, part_l, part_o, parts_total, part_base, 0, nullptr};
    return decode_impl(q, k_base, v_base, row_stride, kv_head_stride, num_kv_rows, kv_rows, count,
                       rows, cap, heads, kv_heads, d_qk, d_v, scale, nullptr, nullptr, nullptr, 0,
                       &po, status, stream);
}

extern "C" int hs_sparse_decode_finish(const void* q, const void* k_base, const void* v_base,
                                       int64_t row_stride, int64_t kv_head_stride,
                                       int64_t num_kv_rows, const int32_t* kv_rows,
                                       const int32_t* count, int32_t rows, int32_t cap,
                                       int32_t heads, int32_t kv_heads, int32_t d_qk,
                                       int32_t d_v, float scale, float* part_m, float* part_l,
                                       float* part_o, int32_t parts_total, int32_t parts_used,
                                       int32_t* sync, void* out, float* lse, int32_t* status,
                                       hs_stream_t stream) {
    const PartialOut po{part_m, part_l, part_o, parts_total, parts_used, 1, sync};
    return decode_impl(q, k_base, v_base, row_stride, kv_head_stride, num_kv_rows, kv_rows, count,
                       rows, cap, heads, kv_heads, d_qk, d_v, scale, out, lse, nullptr, 0, &po,
                       status, stream);
}

extern "C" int hs_merge_states(const float* m, const float* l, const float* o, int32_t n,
                               int32_t parts, int32_t d_v, void* out, float* lse,
                               hs_stream_t stream) {
    if (n < 0 || parts <= 0 || d_v <= 0) return HS_ERR_INVALID_ARG;
    if (n == 0) return HS_OK;
    if (m == nullptr || l == nullptr || o == nullptr || out == nullptr) return HS_ERR_INVALID_ARG;
    merge_kernel<<<n, 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        m, l, o, parts, d_v, static_cast<__nv_bfloat16*>(out), lse, parts);
    return hs_host::launch_status();
}

// ----------------------------------------------------------------------------
// Allocation-free variant of hs_sparse_decode: the split-KV partial states
// live in a scratch array compiled into the library, for callers that may
// not allocate device memory on the decode path.  The array's device address
// is looked up once per device (cudaGetSymbolAddress, with that device
// current) on the first call there; the host-side name of the array is only
// a stand-in and is never passed to a kernel.
namespace {
__device__ __align__(256) unsigned char g_noalloc_workspace[HS_NOALLOC_WORKSPACE_BYTES];
// Device address of the array per device, looked up once per process.  Two
// host threads making their first call at once may both look it up; they
// store the same value, and the atomic makes that well defined.
std::atomic<void*> g_noalloc_workspace_dev[64];
}  // namespace

extern "C" int hs_sparse_decode_noalloc(const void* q, const void* k_base, const void* v_base,
                                        int64_t row_stride, int64_t kv_head_stride,
                                        int64_t num_kv_rows, const int32_t* kv_rows,
                                        const int32_t* count, int32_t rows, int32_t cap,
                                        int32_t heads, int32_t kv_heads, int32_t d_qk,
                                        int32_t d_v, float scale, void* out, float* lse,
                                        int32_t* status, hs_stream_t stream) {
    const int64_t need =
        hs_sparse_decode_workspace_bytes(rows, heads, kv_heads, cap, d_qk, d_v);
    if (need > int64_t(HS_NOALLOC_WORKSPACE_BYTES)) return HS_ERR_CAPACITY;
    void* ws = nullptr;
    if (need > 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
        if (dev < 0 || dev >= 64) return HS_ERR_UNSUPPORTED;
        ws = g_noalloc_workspace_dev[dev].load(std::memory_order_acquire);
        if (ws == nullptr) {
            if (cudaGetSymbolAddress(&ws, g_noalloc_workspace) != cudaSuccess || ws == nullptr) {
                cudaGetLastError();
                return HS_ERR_CUDA;
            }
            g_noalloc_workspace_dev[dev].store(ws, std::memory_order_release);
        }
    }
    return hs_sparse_decode(q, k_base, v_base, row_stride, kv_head_stride, num_kv_rows, kv_rows,
                            count, rows, cap, heads, kv_heads, d_qk, d_v, scale, out, lse, ws,
                            need, status, stream);
}
