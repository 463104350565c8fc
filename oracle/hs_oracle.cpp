// hs_oracle.cpp -- the oracle: a plain, slow, single-threaded CPU statement of
// what each stage of the HiSparse sparse-decode step computes.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
// bench's CPU-baseline leg may load this library.  It shares no code, header,
// table or helper with the CUDA path under sparse_top_kv_gb300/csrc, and it
// never calls into it.  Floating point is fp64 throughout.
//
// Sources (web pages, cited by title and section):
//  [HS]  vLLM HiSparse walkthrough (devpress.csdn.net, "HiSparse hot-buffer
//        decode"): sections "triton_convert_req_index_to_global_index",
//        "调用核心 Swap-In 内核", Phase 1 .. Phase 5 of hisparse_swap_in_kernel.
//  [PT]  PaperTrace 5.1.1 "从索引到 Kernel" (From indices to kernel):
//        section 1.1 eq. (1), section 1.2 eq. (2) and the two worked examples,
//        section 3.1 eqs. (4)-(6), section 3.2 eq. (7), section 7.3 eq. (16)
//        and eq. (17), section 7.3 "空集合和非法集合必须有唯一含义".
//  [PA]  "PagedAttention 与 RadixAttention：上游机制与海光实现对照",
//        section 1.3 (addressing) and 1.4 (split-KV combine).
//
// Every function returns 0 on success or a non-zero code for arguments the
// definition does not cover; nothing here is tuned for speed.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <map>
#include <set>
#include <vector>

namespace {

// bf16 bit pattern -> exact double (bf16 is the top half of an IEEE binary32).
double bf16_to_double(uint16_t bits) {
    uint32_t u = static_cast<uint32_t>(bits) << 16;
    float f;
    std::memcpy(&f, &u, sizeof(f));
    return static_cast<double>(f);
}

enum Reject { kValid = -1, kRange = 0, kCausal = 1, kOwner = 2 };

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// S1 -- candidate normalisation ([PT] 1.1 eq. (1), 1.2 eq. (2), 7.3 eq. (16);
// [HS] triton_convert_req_index_to_global_index).
//
// For index row r with request q = row_req[r] and context length T = seq_lens[q]:
//   D = the n_cand dynamic candidates (the value -1 is padding and is skipped),
//   W = [max(0, T - window), T),  A = [0, min(num_sinks, T)),
//   S = unique(D u W u A) restricted to valid positions.
// A position t is valid when, checked in this order,
//   t >= 0                      (else: range error),
//   t <  T                      (else: causal error),
//   b = floor(t / B) < max_blocks (else: range error),
//   p = table[q][b] in [0, num_pages) (else: range error),
//   page_owner == NULL or page_owner[p] == q (else: owner error).
// Rejected positions are counted and dropped.  W and A are inserted first,
// then D in order; a valid D entry already present in S counts as a duplicate.
// Output: S ascending in t, slot = p * B + t mod B, -1 padding up to cap.
// err_counts[r] = {range, causal, owner, duplicate}.
int hso_normalize_indices(const int32_t* cand, int32_t rows, int32_t n_cand, int32_t window,
                          int32_t num_sinks, const int32_t* row_req, const int32_t* seq_lens,
                          const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                          const int32_t* page_owner, int32_t num_reqs, int32_t num_pages,
                          int32_t page_size, int32_t cap, int32_t* out_tok, int32_t* out_slot,
                          int32_t* out_count, int32_t* err_counts) {
    if (rows < 0 || n_cand < 0 || window < 0 || num_sinks < 0 || page_size <= 0 || cap < 0)
        return 1;
    if (static_cast<int64_t>(cap) < static_cast<int64_t>(n_cand) + window + num_sinks) return 3;
    for (int32_t r = 0; r < rows; ++r) {
        int32_t* tok = out_tok + static_cast<int64_t>(r) * cap;
        int32_t* slot = out_slot + static_cast<int64_t>(r) * cap;
        int32_t* err = err_counts + static_cast<int64_t>(r) * 4;
        for (int k = 0; k < 4; ++k) err[k] = 0;
        for (int32_t j = 0; j < cap; ++j) tok[j] = slot[j] = -1;
        out_count[r] = 0;
        const int32_t* row = cand + static_cast<int64_t>(r) * n_cand;
        const int32_t q = row_req[r];
        if (q < 0 || q >= num_reqs) {
            // The row has no request: none of its dynamic candidates can be
            // resolved, each one is a range error.
            for (int32_t i = 0; i < n_cand; ++i)
                if (row[i] != -1) err[kRange] += 1;
            continue;
        }
        const int64_t T = seq_lens[q] > 0 ? seq_lens[q] : 0;
        const int32_t* table = block_table + static_cast<int64_t>(q) * bt_stride;
        auto check = [&](int64_t t) -> int {
            if (t < 0) return kRange;
            if (t >= T) return kCausal;
            const int64_t b = t / page_size;
            if (b >= max_blocks) return kRange;
            const int64_t p = table[b];
            if (p < 0 || p >= num_pages) return kRange;
            if (page_owner != nullptr && page_owner[p] != q) return kOwner;
            return kValid;
        };
        std::set<int64_t> S;
        // Structural candidates: sinks, then the window (their overlap is one set).
        std::set<int64_t> WA;
        for (int64_t t = 0; t < std::min<int64_t>(num_sinks, T); ++t) WA.insert(t);
        for (int64_t t = std::max<int64_t>(0, T - window); t < T; ++t) WA.insert(t);
        for (int64_t t : WA) {
            const int c = check(t);
            if (c == kValid) S.insert(t); else err[c] += 1;
        }
        for (int32_t i = 0; i < n_cand; ++i) {
            const int64_t t = row[i];
            if (t == -1) continue;  // padding
            const int c = check(t);
            if (c != kValid) { err[c] += 1; continue; }
            if (!S.insert(t).second) err[3] += 1;
        }
        int32_t j = 0;
        for (int64_t t : S) {
            const int64_t p = table[t / page_size];
            tok[j] = static_cast<int32_t>(t);
            slot[j] = static_cast<int32_t>(p * page_size + t % page_size);
            ++j;
        }
        out_count[r] = j;
    }
    return 0;
}

// ---------------------------------------------------------------------------
// S2 -- hot-buffer lookup and LRU slot assignment ([HS] Phase 1 .. Phase 4),
// written as the sequential definition.
//
// Row r owns hot rows [r*region_stride, r*region_stride + hot_size] (the last
// one is reserved for the newest token), dgi[r][0..hot_size) (global slot held
// by each hot slot, -1 = empty) and lru[r][0..hot_size) (hot slots from least
// to most recently used; a permutation of 0..hot_size-1).
// Phase 1: entry i with g < 0 (or i >= count) -> -1; g == newest -> reserved
//          row; otherwise pending.  A repeat of an earlier pending g -> -1 and
//          counts in err[r] (only the first occurrence resolves).
// Phase 2: walk lru oldest->newest; slot s is a hit when dgi[s] is pending;
//          hits H and evictables E both keep LRU order.
// Phase 3: the pending entries that did not hit, in row order m = 0,1,..,
//          take E[m]: dgi[E[m]] = g, miss_mask = 1, (miss_src, miss_dst)[m].
// Phase 4: lru = E[M:] ++ E[:M] ++ H.   stats += {|H|, M}.
// Rows r >= num_real_rows output -1 and leave their state untouched.
int hso_hot_lookup_assign(const int32_t* slot, const int32_t* count, int32_t rows, int32_t cap,
                          int32_t num_real_rows, const int32_t* newest_slot, int32_t* dgi,
                          int16_t* lru, int32_t hot_size, int64_t region_stride,
                          int32_t* hot_idx, uint8_t* miss_mask, int32_t* miss_src,
                          int64_t* miss_dst, int32_t* miss_count, int64_t* stats, int32_t* err) {
    if (rows < 0 || cap < 0 || hot_size <= 0 || hot_size > 32767) return 1;
    if (region_stride < static_cast<int64_t>(hot_size) + 1) return 1;
    if (cap > hot_size) return 3;
    for (int32_t r = 0; r < rows; ++r) {
        const int32_t* g_row = slot + static_cast<int64_t>(r) * cap;
        int32_t* out = hot_idx + static_cast<int64_t>(r) * cap;
        uint8_t* mm = miss_mask ? miss_mask + static_cast<int64_t>(r) * cap : nullptr;
        int32_t* msrc = miss_src + static_cast<int64_t>(r) * cap;
        int64_t* mdst = miss_dst + static_cast<int64_t>(r) * cap;
        for (int32_t i = 0; i < cap; ++i) {
            out[i] = -1;
            if (mm) mm[i] = 0;
            msrc[i] = -1;
            mdst[i] = -1;
        }
        miss_count[r] = 0;
        err[r] = 0;
        if (r >= num_real_rows) continue;
        int32_t* d = dgi + static_cast<int64_t>(r) * hot_size;
        int16_t* L = lru + static_cast<int64_t>(r) * hot_size;
        const int64_t hot_base = static_cast<int64_t>(r) * region_stride;
        const int32_t n = count ? std::min(std::max(count[r], 0), cap) : cap;
        const int32_t newest = newest_slot ? newest_slot[r] : -1;

        // Phase 1.  pending: g -> the row position i of its first occurrence.
        std::map<int32_t, int32_t> pending;
        for (int32_t i = 0; i < n; ++i) {
            const int32_t g = g_row[i];
            if (g < 0) continue;
            if (newest >= 0 && g == newest) {
                out[i] = static_cast<int32_t>(hot_base + hot_size);
                continue;
            }
            if (!pending.emplace(g, i).second) err[r] += 1;
        }
        // Phase 2.
        std::vector<int16_t> H, E;
        for (int32_t pos = 0; pos < hot_size; ++pos) {
            const int16_t s = L[pos];
            bool hit = false;
            if (s >= 0 && s < hot_size && d[s] >= 0) {
                auto it = pending.find(d[s]);
                if (it != pending.end()) {
                    out[it->second] = static_cast<int32_t>(hot_base + s);
                    pending.erase(it);
                    hit = true;
                }
            }
            (hit ? H : E).push_back(s);
        }
        // Phase 3: the remaining pending entries, in row order.
        std::vector<int32_t> misses;
        for (const auto& kv : pending) misses.push_back(kv.second);
        std::sort(misses.begin(), misses.end());
        int32_t M = 0;
        for (int32_t i : misses) {
            const int16_t s = E[M];
            d[s] = g_row[i];
            out[i] = static_cast<int32_t>(hot_base + s);
            if (mm) mm[i] = 1;
            msrc[M] = g_row[i];
            mdst[M] = hot_base + s;
            ++M;
        }
        // Phase 4.
        std::vector<int16_t> nl;
        for (size_t k = M; k < E.size(); ++k) nl.push_back(E[k]);
        for (int32_t k = 0; k < M; ++k) nl.push_back(E[k]);
        for (int16_t s : H) nl.push_back(s);
        for (int32_t pos = 0; pos < hot_size; ++pos) L[pos] = nl[pos];
        miss_count[r] = M;
        stats[0] += static_cast<int64_t>(H.size());
        stats[1] += M;
    }
    return 0;
}

// ---------------------------------------------------------------------------
// S3 -- SwapIn ([HS] Phase 5): for each miss m of row r, copy row_bytes from
// host_pool[g] to hot[dst]; when g is outside [0, host_rows) the hot row is
// zeroed and, when dgi is given, its slot's ownership is revoked (dgi = -1).
int hso_swap_in(const uint8_t* host_pool, int64_t host_rows, uint8_t* hot, int64_t row_bytes,
                const int32_t* miss_src, const int64_t* miss_dst, const int32_t* miss_count,
                int32_t rows, int32_t cap, int32_t* dgi, int32_t hot_size,
                int64_t region_stride) {
    if (row_bytes <= 0 || row_bytes % 16 != 0) return 2;
    for (int32_t r = 0; r < rows; ++r) {
        for (int32_t m = 0; m < miss_count[r]; ++m) {
            const int64_t g = miss_src[static_cast<int64_t>(r) * cap + m];
            const int64_t dst = miss_dst[static_cast<int64_t>(r) * cap + m];
            uint8_t* to = hot + dst * row_bytes;
            if (g >= 0 && g < host_rows) {
                std::memcpy(to, host_pool + g * row_bytes, static_cast<size_t>(row_bytes));
            } else {
                std::memset(to, 0, static_cast<size_t>(row_bytes));
                if (dgi != nullptr) {
                    const int64_t s = dst - static_cast<int64_t>(r) * region_stride;
                    if (s >= 0 && s < hot_size) dgi[static_cast<int64_t>(r) * hot_size + s] = -1;
                }
            }
        }
    }
    return 0;
}

// BackUp ([HS] overview: "BackUp" copies each step's new KV row to host
// memory): host_pool[dst_slots[i]] = src[src_rows[i]].  A destination of -1
// is padding (an inactive request of a fixed-size batch) and is skipped; any
// other destination outside [0, host_rows) is not written either, and the
// number of those rows is returned in *bad.
int hso_backup(const uint8_t* src, const int64_t* src_rows, uint8_t* host_pool,
               const int32_t* dst_slots, int32_t n, int64_t row_bytes, int64_t host_rows,
               int32_t* bad) {
    if (row_bytes <= 0 || row_bytes % 16 != 0) return 2;
    *bad = 0;
    for (int32_t i = 0; i < n; ++i) {
        const int64_t g = dst_slots[i];
        if (g == -1) continue;
        if (g < 0 || g >= host_rows) { *bad += 1; continue; }
        std::memcpy(host_pool + g * row_bytes, src + src_rows[i] * row_bytes,
                    static_cast<size_t>(row_bytes));
    }
    return 0;
}

// ---------------------------------------------------------------------------
// Layer transfer (SGLang PR "[HiCache] TMA-staged host<->device KV transfer
// kernel (sm_90+)", Motivation and Modifications): HiCache moves the rows of
// cached tokens between the pinned host pool and the device's per-layer
// pools.  For every buffer b < nbuf (K and V, or one buffer for MLA), every
// layer l < layers and every i < n, the row of token src_idx[i] is copied to
// the row of token dst_idx[i].  Row addresses, in bytes:
//   device pool (one array per buffer and layer): dev[b * layers + l] + t * rb
//   host, layer-first:  host + b * host_buf_bytes + (l * host_tokens + t) * rb
//   host, page-first:   host + b * host_buf_bytes
//                       + ((t / P) * layers * P + l * P + t % P) * rb
// direction 0 copies host -> device (src on the host), 1 device -> host.
// Indices are int32 (index_bytes = 4) or int64 (8).  A source or destination
// index outside its pool ([0, host_tokens) on the host, [0, dev_tokens) on the
// device) skips the row; the number of skipped (buffer, layer, row) copies is
// returned in *bad.
int hso_layer_transfer(uint8_t* const* dev, uint8_t* host, int64_t host_tokens,
                       int64_t host_buf_bytes, int32_t nbuf, int32_t layers, int32_t page_size,
                       int32_t page_first, int64_t dev_tokens, int64_t row_bytes,
                       const void* src_idx, const void* dst_idx, int32_t index_bytes, int64_t n,
                       int32_t direction, int64_t* bad) {
    if (row_bytes <= 0 || row_bytes % 16 != 0 || page_size <= 0) return 2;
    if (index_bytes != 4 && index_bytes != 8) return 1;
    const auto idx = [&](const void* p, int64_t i) -> int64_t {
        return index_bytes == 4 ? static_cast<const int32_t*>(p)[i]
                                : static_cast<const int64_t*>(p)[i];
    };
    const auto host_row = [&](int32_t b, int32_t l, int64_t t) -> uint8_t* {
        int64_t r;
        if (page_first) {
            r = (t / page_size) * layers * page_size + static_cast<int64_t>(l) * page_size +
                t % page_size;
        } else {
            r = static_cast<int64_t>(l) * host_tokens + t;
        }
        return host + b * host_buf_bytes + r * row_bytes;
    };
    *bad = 0;
    for (int32_t b = 0; b < nbuf; ++b) {
        for (int32_t l = 0; l < layers; ++l) {
            uint8_t* dbase = dev[static_cast<int64_t>(b) * layers + l];
            for (int64_t i = 0; i < n; ++i) {
                const int64_t s = idx(src_idx, i), d = idx(dst_idx, i);
                const int64_t s_lim = direction == 0 ? host_tokens : dev_tokens;
                const int64_t d_lim = direction == 0 ? dev_tokens : host_tokens;
                if (s < 0 || s >= s_lim || d < 0 || d >= d_lim) {
                    *bad += 1;
                    continue;
                }
                const uint8_t* from = direction == 0 ? host_row(b, l, s) : dbase + s * row_bytes;
                uint8_t* to = direction == 0 ? dbase + d * row_bytes : host_row(b, l, d);
                std::memcpy(to, from, static_cast<size_t>(row_bytes));
            }
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// S4 -- sparse decode attention over the candidate rows ([PT] 3.1, 3.2, and
// 7.3 "空集合": an empty set gives a zero output and LSE = -inf).
//
// For row r and query head h (KV head g = h / (heads / kv_heads)), with
// J = { kv_rows[r][g][j] : j < count[r][g], kv_rows[r][g][j] >= 0 } taken as
// given (a repeated row would count twice; the caller passes a set):
//   s_j = scale * sum_d q[r][h][d] * K_j[g][d]       (d < d_qk)
//   m   = max_j s_j,  p_j = exp(s_j - m),  L = sum_j p_j
//   out = sum_j p_j V_j[g] / L                       (d < d_v)
//   lse = m + ln L
// K_j[g][d] = k_base[j * row_stride + g * kv_head_stride + d], the same for V.
// q, K and V are bf16 bit patterns, converted to double exactly.  A direct
// two-pass softmax over the whole set: no tiling, no online rescaling.
int hso_sparse_decode(const uint16_t* q, const uint16_t* k_base, const uint16_t* v_base,
                      int64_t row_stride, int64_t kv_head_stride, const int32_t* kv_rows,
                      const int32_t* count, int32_t rows, int32_t cap, int32_t heads,
                      int32_t kv_heads, int32_t d_qk, int32_t d_v, double scale, double* out,
                      double* lse) {
    if (rows < 0 || cap < 0 || heads <= 0 || kv_heads <= 0 || heads % kv_heads != 0) return 1;
    const int32_t group = heads / kv_heads;
    std::vector<double> s;
    for (int32_t r = 0; r < rows; ++r) {
        for (int32_t h = 0; h < heads; ++h) {
            const int32_t g = h / group;
            const int64_t idx_row = (static_cast<int64_t>(r) * kv_heads + g) * cap;
            const int32_t n = count ? std::min(std::max(count[static_cast<int64_t>(r) * kv_heads + g], 0), cap) : cap;
            const uint16_t* qv = q + (static_cast<int64_t>(r) * heads + h) * d_qk;
            double* o = out + (static_cast<int64_t>(r) * heads + h) * d_v;
            std::vector<int64_t> J;
            for (int32_t j = 0; j < n; ++j)
                if (kv_rows[idx_row + j] >= 0) J.push_back(kv_rows[idx_row + j]);
            for (int32_t d = 0; d < d_v; ++d) o[d] = 0.0;
            if (J.empty()) {
                lse[static_cast<int64_t>(r) * heads + h] = -std::numeric_limits<double>::infinity();
                continue;
            }
            s.assign(J.size(), 0.0);
            double m = -std::numeric_limits<double>::infinity();
            for (size_t j = 0; j < J.size(); ++j) {
                const uint16_t* kr = k_base + J[j] * row_stride + g * kv_head_stride;
                double acc = 0.0;
                for (int32_t d = 0; d < d_qk; ++d) acc += bf16_to_double(qv[d]) * bf16_to_double(kr[d]);
                s[j] = scale * acc;
                if (s[j] > m) m = s[j];
            }
            double L = 0.0;
            for (size_t j = 0; j < J.size(); ++j) {
                const double p = std::exp(s[j] - m);
                L += p;
                const uint16_t* vr = v_base + J[j] * row_stride + g * kv_head_stride;
                for (int32_t d = 0; d < d_v; ++d) o[d] += p * bf16_to_double(vr[d]);
            }
            for (int32_t d = 0; d < d_v; ++d) o[d] /= L;
            lse[static_cast<int64_t>(r) * heads + h] = m + std::log(L);
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// Split-KV merge of unnormalised partial states, [PT] 3.2 eq. (7):
//   m = max(m_1, .., m_P),  l = sum_p e^{m_p - m} l_p,  o = sum_p e^{m_p - m} o_p.
// A part with l_p == 0 (no valid candidate) is skipped, so its m_p never
// enters the maximum ([PT] 7.1 after eq. (14)).  n states, P parts each, d_v
// wide: m[n][P], l[n][P], o[n][P][d_v] -> m_out[n], l_out[n], o_out[n][d_v].
int hso_merge(const double* m, const double* l, const double* o, int32_t n, int32_t parts,
              int32_t d_v, double* m_out, double* l_out, double* o_out) {
    for (int32_t i = 0; i < n; ++i) {
        double M = -std::numeric_limits<double>::infinity();
        for (int32_t p = 0; p < parts; ++p) {
            const int64_t k = static_cast<int64_t>(i) * parts + p;
            if (l[k] > 0.0 && m[k] > M) M = m[k];
        }
        double L = 0.0;
        double* oo = o_out + static_cast<int64_t>(i) * d_v;
        for (int32_t d = 0; d < d_v; ++d) oo[d] = 0.0;
        if (M != -std::numeric_limits<double>::infinity()) {
            for (int32_t p = 0; p < parts; ++p) {
                const int64_t k = static_cast<int64_t>(i) * parts + p;
                if (!(l[k] > 0.0)) continue;
                const double w = std::exp(m[k] - M);
                L += w * l[k];
                for (int32_t d = 0; d < d_v; ++d) oo[d] += w * o[k * d_v + d];
            }
        }
        m_out[i] = M;
        l_out[i] = L;
    }
    return 0;
}


// ---------------------------------------------------------------------------
// fp8_ds_mla KV rows ([HS] the FlashMLASparseBackend cache shape, the
// FP8_DS_MLA_ROW_BYTES constant and the 656-byte copy walk-through of
// Phase 5; [PT] 7.2 "量化 KV 与内核特化": the scale is applied to the stored
// codes to reconstruct the values the attention computes with).
//
// One row is 656 bytes: bytes [0, 512) are the 512 latent (NoPE) columns as
// OCP FP8 E4M3 codes, bytes [512, 528) are four IEEE binary32 scales
// (little-endian), bytes [528, 656) are the 64 RoPE columns as bf16
// (little-endian).  Readings: the 16 bytes of scales are four fp32 values and
// scale g multiplies latent columns [128 g, 128 g + 128) (512 / 4); the value
// of a latent column is code x scale, formed in binary32 (the scale's own
// precision) and rounded to bf16, the operand precision of the attention
// products (both roundings to nearest, ties to even).
//
// E4M3 from its definition: sign bit 7, exponent bits 6..3 (bias 7), mantissa
// bits 2..0.  Exponent 0 is subnormal (m / 8 * 2^-6); exponent 15 with
// mantissa 7 is NaN; there is no infinity (1111.110 = 448 is the largest).
static double e4m3_to_double(uint8_t c) {
    const int sgn = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
    if (e == 0)
        v = std::ldexp(static_cast<double>(m) / 8.0, -6);
    else
        v = std::ldexp(1.0 + static_cast<double>(m) / 8.0, e - 7);
    return sgn ? -v : v;
}

// binary32 -> bf16 bits, round to nearest, ties to even (NaN stays a quiet NaN).
static uint16_t float_to_bf16_rne(float f) {
    uint32_t u;
    std::memcpy(&u, &f, sizeof(u));
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return static_cast<uint16_t>((u >> 16) | 0x0040u);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return static_cast<uint16_t>(u >> 16);
}

int hso_e4m3_decode(const uint8_t* codes, int64_t n, double* out) {
    if (n < 0) return 1;
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_double(codes[i]);
    return 0;
}

// One 656-byte row -> 576 bf16 bits: latent columns reconstructed as above,
// RoPE columns copied.
static void fp8ds_row(const uint8_t* r, uint16_t* o) {
    float scale[4];
    for (int g = 0; g < 4; ++g) {
        uint32_t u = 0;
        for (int b = 0; b < 4; ++b) u |= static_cast<uint32_t>(r[512 + 4 * g + b]) << (8 * b);
        std::memcpy(&scale[g], &u, sizeof(float));
    }
    for (int d = 0; d < 512; ++d) {
        // The code's value is exact in binary32 (4 significant bits).
        const float code = static_cast<float>(e4m3_to_double(r[d]));
        const float v = code * scale[d / 128];
        o[d] = float_to_bf16_rne(v);
    }
    for (int d = 0; d < 64; ++d)
        o[512 + d] = static_cast<uint16_t>(r[528 + 2 * d] | (r[528 + 2 * d + 1] << 8));
}

// Rows ids[i] of `rows8` (row_bytes apart, row_bytes >= 656) -> out[i][576].
int hso_fp8ds_dequant(const uint8_t* rows8, int64_t row_bytes, const int64_t* ids, int64_t n,
                      uint16_t* out) {
    if (row_bytes < 656 || n < 0) return 1;
    for (int64_t i = 0; i < n; ++i) fp8ds_row(rows8 + ids[i] * row_bytes, out + i * 576);
    return 0;
}

// SwapIn from a pool of fp8_ds_mla rows into a hot buffer of bf16 rows
// (576 columns): the hso_swap_in walk, with each copied row reconstructed by
// fp8ds_row.  A source outside the pool zeroes the hot row and revokes its
// slot, as in hso_swap_in.
int hso_swap_in_fp8ds(const uint8_t* host_pool8, int64_t host_rows, int64_t host_row_bytes,
                      uint16_t* hot, const int32_t* miss_src, const int64_t* miss_dst,
                      const int32_t* miss_count, int32_t rows, int32_t cap, int32_t* dgi,
                      int32_t hot_size, int64_t region_stride) {
    if (host_row_bytes < 656) return 1;
    for (int32_t r = 0; r < rows; ++r) {
        for (int32_t m = 0; m < miss_count[r]; ++m) {
            const int64_t g = miss_src[static_cast<int64_t>(r) * cap + m];
            const int64_t dst = miss_dst[static_cast<int64_t>(r) * cap + m];
            uint16_t* to = hot + dst * 576;
            if (g >= 0 && g < host_rows) {
                fp8ds_row(host_pool8 + g * host_row_bytes, to);
            } else {
                for (int d = 0; d < 576; ++d) to[d] = 0;
                if (dgi != nullptr) {
                    const int64_t s = dst - static_cast<int64_t>(r) * region_stride;
                    if (s >= 0 && s < hot_size) dgi[static_cast<int64_t>(r) * hot_size + s] = -1;
                }
            }
        }
    }
    return 0;
}

}  // extern "C"
