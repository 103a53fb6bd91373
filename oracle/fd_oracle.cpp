// fd_oracle.cpp -- the oracle for split-KV decode attention.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously correct
// CPU statement of what the decode hot path computes.  It is compiled into its
// own shared library (liboracle) and is used only by the test-suite, by the
// smoke check and by the bench's CPU-baseline leg.  The product library never
// links, loads or calls it, and it shares no code, header or constant with the
// CUDA path.
//
// Everything is IEEE double.  std::exp / std::log / std::sqrt are called, never
// re-implemented.  Inputs in fp16 / bf16 are converted exactly to double from
// the bit-level definition of those formats.
//
// Sources (web pages on Flash-Decoding / split-KV decode attention):
//  [FD]   "Flash-Decoding: Split-KV Attention for Long-Context Decode"
//         (kanthi.in), sections 1, 2, 6 and 9.
//  [DKV]  "Decode 专项 Attention：把长KV拆开算，再正确合并" (xuujii.github.io),
//         sections 03, 04 and 06.
//  [TV]   tinyvolt.com Flash-decoding article, "Combine kernel" section.
//
// Parity pins (all in tests/, run with -m "not gpu"):
//  fdo_attend / fdo_decode : [DKV] §03 worked example (4.9), closed forms
//                            (L=1, equal scores, one dominant score), scipy
//                            logsumexp/softmax on tiny inputs, GQA / paged /
//                            strided address maps against hand-built caches.
//  fdo_merge               : [DKV] §04 state example (ell=2.5, u=12.25),
//                            [FD] §3 merge-trap printed values, split
//                            invariance of attend-then-merge.
//  fdo_plan                : [FD] §6 printed split table (132 SMs) and the
//                            FA3 efficiency comment quoted in the vatshank
//                            split-KV post (0.89 / 0.67).
//  fdo_half_to_double /
//  fdo_bf16_to_double      : every finite bit pattern against numpy's own
//                            float16 conversion and bf16 = top half of f32.
// No function here is "parity unpinned".
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

// IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double half_bits_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = std::ldexp(static_cast<double>(frac), -24);          // subnormal / zero
    } else if (expo == 31) {
        mag = frac ? std::numeric_limits<double>::quiet_NaN()
                   : std::numeric_limits<double>::infinity();
    } else {
        mag = std::ldexp(1024.0 + frac, expo - 25);                 // (1 + f/2^10) 2^(e-15)
    }
    return sign ? -mag : mag;
}

// bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
double bf16_bits_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 7) & 0xff;
    const int frac = h & 0x7f;
    double mag;
    if (expo == 0) {
        mag = std::ldexp(static_cast<double>(frac), -133);          // f/2^7 * 2^-126
    } else if (expo == 255) {
        mag = frac ? std::numeric_limits<double>::quiet_NaN()
                   : std::numeric_limits<double>::infinity();
    } else {
        mag = std::ldexp(128.0 + frac, expo - 134);                 // (1 + f/2^7) 2^(e-127)
    }
    return sign ? -mag : mag;
}

// OCP FP8 E4M3 ("fn": no infinities): 1 sign bit, 4 exponent bits (bias 7),
// 3 fraction bits; exponent 15 with fraction 7 is NaN, the rest is finite
// (largest 448).
double e4m3_bits_to_double(uint8_t x) {
    const int sign = (x >> 7) & 1;
    const int expo = (x >> 3) & 0xf;
    const int frac = x & 0x7;
    double mag;
    if (expo == 0) {
        mag = std::ldexp(static_cast<double>(frac), -9);            // f/2^3 * 2^-6
    } else if (expo == 15 && frac == 7) {
        mag = std::numeric_limits<double>::quiet_NaN();
    } else {
        mag = std::ldexp(8.0 + frac, expo - 10);                     // (1 + f/2^3) 2^(e-7)
    }
    return sign ? -mag : mag;
}

double to_double(uint16_t bits, int dtype) {
    return dtype == 0 ? half_bits_to_double(bits) : bf16_bits_to_double(bits);
}

// Element e of a cache of dtype 0 (fp16), 1 (bf16) or 2 (fp8 e4m3).
double cache_elem(const void* base, int64_t e, int dtype) {
    if (dtype == 2) return e4m3_bits_to_double(static_cast<const uint8_t*>(base)[e]);
    return to_double(static_cast<const uint16_t*>(base)[e], dtype);
}

// Attention of one query row over L keys, [FD] §1 and §2:
//   s_j = q.k_j / sqrt(d),  o = sum_j softmax(s)_j v_j,  LSE = log sum_j e^{s_j}.
// Written with the maximum taken out first so that e^{s} cannot overflow:
//   M = max s,  Z = sum e^{s_j - M},  o = sum e^{s_j - M} v_j / Z,  LSE = M + log Z.
// L = 0 (no visible key): o = 0, LSE = -inf ([DKV] §06 leaves the convention to
// the caller; this library fixes it so).
// key(j, d) / val(j, d) return element d of key / value j as a double.
template <class KeyAt, class ValAt>
void attend_row(int64_t L, int D, const double* q, KeyAt key, ValAt val, double scale,
                double* out, double* lse, std::vector<double>& s, std::vector<double>& acc) {
    if (L <= 0) {
        for (int d = 0; d < D; ++d) out[d] = 0.0;
        *lse = kNegInf;
        return;
    }
    s.resize(static_cast<size_t>(L));
    double M = kNegInf;
    for (int64_t j = 0; j < L; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * key(j, d);
        s[j] = dot * scale;
        M = std::max(M, s[j]);
    }
    double Z = 0.0;
    acc.assign(static_cast<size_t>(D), 0.0);
    for (int64_t j = 0; j < L; ++j) {
        const double w = std::exp(s[j] - M);
        Z += w;
        for (int d = 0; d < D; ++d) acc[d] += w * val(j, d);
    }
    for (int d = 0; d < D; ++d) out[d] = acc[d] / Z;
    *lse = M + std::log(Z);
}

}  // namespace

extern "C" {

int fdo_abi_version(void) { return 1; }

double fdo_half_to_double(uint16_t bits) { return half_bits_to_double(bits); }
double fdo_e4m3_to_double(uint8_t bits) { return e4m3_bits_to_double(bits); }
double fdo_bf16_to_double(uint16_t bits) { return bf16_bits_to_double(bits); }

// Plain attention of one query over L keys in double.  q[D], K[L][D], V[L][D]
// row-major; scale multiplies q.k (1/sqrt(D) for the decode path).
int fdo_attend(int64_t L, int D, const double* q, const double* K, const double* V,
               double scale, double* out, double* lse) {
    if (D <= 0 || L < 0 || !q || !out || !lse || (L > 0 && (!K || !V))) return -1;
    std::vector<double> s, acc;
    attend_row(L, D, q, [&](int64_t j, int d) { return K[j * D + d]; },
               [&](int64_t j, int d) { return V[j * D + d]; }, scale, out, lse, s, acc);
    return 0;
}

// Partial state of one key segment, [DKV] §04: m = max s, ell = sum e^{s-m},
// u = sum e^{s-m} v.  An empty segment is (m=-inf, ell=0, u=0) ([FD] §4 bullet
// on ragged batches; [DKV] §06).
int fdo_segment_state(int64_t L, int D, const double* q, const double* K, const double* V,
                      double scale, double* m, double* ell, double* u) {
    if (D <= 0 || L < 0 || !q || !m || !ell || !u || (L > 0 && (!K || !V))) return -1;
    for (int d = 0; d < D; ++d) u[d] = 0.0;
    if (L == 0) { *m = kNegInf; *ell = 0.0; return 0; }
    std::vector<double> s(static_cast<size_t>(L));
    double M = kNegInf;
    for (int64_t j = 0; j < L; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * K[j * D + d];
        s[j] = dot * scale;
        M = std::max(M, s[j]);
    }
    double l = 0.0;
    for (int64_t j = 0; j < L; ++j) {
        const double w = std::exp(s[j] - M);
        l += w;
        for (int d = 0; d < D; ++d) u[d] += w * V[j * D + d];
    }
    *m = M;
    *ell = l;
    return 0;
}

// Exact merge of n partial states ([DKV] §04; [TV] combine kernel; [FD] §2
// stable form): m = max_i m_i over non-empty states, alpha_i = e^{m_i - m}
// (0 for an empty state, never e^{-inf - (-inf)}), ell = sum alpha_i ell_i,
// u = sum alpha_i u_i.  All states empty -> (-inf, 0, 0).
int fdo_merge(int n, int D, const double* m, const double* ell, const double* u,
              double* m_out, double* ell_out, double* u_out) {
    if (n < 0 || D <= 0 || !m_out || !ell_out || !u_out || (n > 0 && (!m || !ell || !u))) return -1;
    double M = kNegInf;
    for (int i = 0; i < n; ++i)
        if (m[i] != kNegInf) M = std::max(M, m[i]);
    for (int d = 0; d < D; ++d) u_out[d] = 0.0;
    if (M == kNegInf) { *m_out = kNegInf; *ell_out = 0.0; return 0; }
    double l = 0.0;
    for (int i = 0; i < n; ++i) {
        if (m[i] == kNegInf) continue;
        const double alpha = std::exp(m[i] - M);
        l += alpha * ell[i];
        for (int d = 0; d < D; ++d) u_out[d] += alpha * u[static_cast<size_t>(i) * D + d];
    }
    *m_out = M;
    *ell_out = l;
    return 0;
}

// Output and natural-log LSE of a state: o = u / ell, LSE = m + log ell.
// An empty state gives o = 0, LSE = -inf.
int fdo_finalize(int D, double m, double ell, const double* u, double* out, double* lse) {
    if (D <= 0 || !u || !out || !lse) return -1;
    if (m == kNegInf || ell == 0.0) {
        for (int d = 0; d < D; ++d) out[d] = 0.0;
        *lse = kNegInf;
        return 0;
    }
    for (int d = 0; d < D; ++d) out[d] = u[d] / ell;
    *lse = m + std::log(ell);
    return 0;
}

// Split-count heuristic, [FD] §6 ("How many splits?"), steps in the page's order:
//  1. a launch of work_items CTAs that already covers 80% of the slots is not split;
//  2. candidate split counts run from 1 to min(max_splits, slots, n_kv_blocks);
//  3. a count whose blocks-per-split equals that of the next smaller count is
//     skipped (it adds a combine and no parallelism);
//  4. each remaining count s has waves = work*s/slots and efficiency
//     waves / ceil(waves) (how full the last wave is);
//  5. the answer is the smallest remaining s whose efficiency reaches 85% of the best.
// n_kv_blocks = 0 (every sequence empty) has no candidate; the answer is then 1.
// eff_out (nullable, max_splits+1 doubles) receives each candidate's efficiency
// and -1 for skipped counts.
int fdo_plan(int64_t work_items, int64_t slots, int64_t n_kv_blocks, int max_splits,
             double* eff_out) {
    if (work_items <= 0 || slots <= 0 || n_kv_blocks < 0 || max_splits <= 0) return -1;
    if (eff_out)
        for (int s = 0; s <= max_splits; ++s) eff_out[s] = -1.0;
    if (static_cast<double>(work_items) >= 0.8 * static_cast<double>(slots)) return 1;
    const int64_t cap = std::min<int64_t>(std::min<int64_t>(max_splits, slots), n_kv_blocks);
    if (cap < 1) return 1;
    auto blocks_per_split = [&](int64_t s) { return (n_kv_blocks + s - 1) / s; };
    std::vector<double> eff(static_cast<size_t>(cap) + 1, -1.0);
    double best = -1.0;
    for (int64_t s = 1; s <= cap; ++s) {
        if (s > 1 && blocks_per_split(s) == blocks_per_split(s - 1)) continue;
        const double waves = static_cast<double>(work_items * s) / static_cast<double>(slots);
        eff[s] = waves / std::ceil(waves);
        best = std::max(best, eff[s]);
        if (eff_out) eff_out[s] = eff[s];
    }
    for (int64_t s = 1; s <= cap; ++s)
        if (eff[s] >= 0.0 && eff[s] >= 0.85 * best) return static_cast<int>(s);
    return 1;
}

// Decode attention for a batch: q_len query rows per sequence (1 for plain
// decode; 2-8 for the short query blocks of speculative verification,
// "Flash-Decoding ..." §7 and §9), each with its own visibility ([DKV] §06):
//  * query position i (0 <= i < q_len) of sequence b sees keys
//    0 .. L_b - q_len + i, i.e. the first L_b - q_len + 1 + i keys (the
//    block's own tokens are already in the cache, causally ordered); none if
//    that count is <= 0;
//  * query head h reads KV head h / (n_q_heads / n_kv_heads)  (grouped-query
//    attention with consecutive query heads sharing a KV head; [FD] §1 GQA note);
//  * sequence b sees keys 0 .. seqlens[b]-1;
//  * key j of (b, kv head g) is read at
//      contiguous (page_size == 0): k + b*k_sb + g*k_sh + j*k_st
//      paged      (page_size  > 0): k + P*k_sb + g*k_sh + (j % page_size)*k_st,
//                                   P = block_table[b*max_pages_per_seq + j/page_size]
//    ([FD] §7 paged row; [DKV] §02: splits are logical ranges resolved through
//    the block table), and the same for v;
//  * s_j = q.k_j / sqrt(head_dim); out = softmax(s) V, lse = natural-log LSE.
// q is read at q + b*q_sb + i*q_st + h*q_sh.  dtype 0 = fp16, 1 = bf16 (raw
// bits) is the type of q and, when kv_dtype < 0, of the cache; kv_dtype 2 is
// an fp8 e4m3 cache whose key / value j is k_scale / v_scale times the stored
// value (one scale per tensor; 16-bit caches use the same scales, normally
// 1).  Strides are in elements of each tensor's own type.
// Rows are numbered r = (b*q_len + i)*n_q_heads + h; rows (nullable)
// lists the rows to evaluate, and out/lse then hold n_rows results in that
// order.  Rows run on n_threads host threads (<= 0: all hardware threads).
int fdo_decode(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
               int32_t dtype, int32_t kv_dtype, double k_scale, double v_scale, int32_t q_len,
               const uint16_t* q, int64_t q_sb, int64_t q_st, int64_t q_sh,
               const void* k, int64_t k_sb, int64_t k_sh, int64_t k_st,
               const void* v, int64_t v_sb, int64_t v_sh, int64_t v_st,
               const int32_t* seqlens,
               int32_t page_size, const int32_t* block_table, int32_t max_pages_per_seq,
               const int64_t* rows, int64_t n_rows,
               double* out, double* lse, int32_t n_threads) {
    if (batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || q_len <= 0) return -1;
    if (n_q_heads % n_kv_heads != 0) return -1;
    if (dtype != 0 && dtype != 1) return -1;
    const int cdt = kv_dtype < 0 ? dtype : kv_dtype;
    if (cdt != 0 && cdt != 1 && cdt != 2) return -1;
    if (!q || !k || !v || !seqlens || !out || !lse) return -1;
    if (page_size < 0 || (page_size > 0 && (!block_table || max_pages_per_seq <= 0))) return -1;
    const int64_t total = static_cast<int64_t>(batch) * q_len * n_q_heads;
    const int64_t count = rows ? n_rows : total;
    if (count < 0) return -1;
    for (int64_t r = 0; rows && r < count; ++r)
        if (rows[r] < 0 || rows[r] >= total) return -1;
    const int group = n_q_heads / n_kv_heads;
    const int D = head_dim;
    const double scale = 1.0 / std::sqrt(static_cast<double>(D));

    auto work = [&](int64_t first, int64_t last) {
        std::vector<double> qd(D), s, acc;
        for (int64_t r = first; r < last; ++r) {
            const int64_t row = rows ? rows[r] : r;
            const int64_t h = row % n_q_heads;
            const int64_t i = (row / n_q_heads) % q_len;
            const int64_t b = row / (static_cast<int64_t>(n_q_heads) * q_len);
            const int64_t g = h / group;
            const int64_t L = std::max<int64_t>(static_cast<int64_t>(seqlens[b]) - q_len + 1 + i, 0);
            for (int d = 0; d < D; ++d)
                qd[d] = to_double(q[b * q_sb + i * q_st + h * q_sh + d], dtype);
            // element offset of key / value j of (b, g), before the head-dim index
            auto k_off = [&](int64_t j) -> int64_t {
                if (page_size == 0) return b * k_sb + g * k_sh + j * k_st;
                const int64_t P = block_table[b * max_pages_per_seq + j / page_size];
                return P * k_sb + g * k_sh + (j % page_size) * k_st;
            };
            auto v_off = [&](int64_t j) -> int64_t {
                if (page_size == 0) return b * v_sb + g * v_sh + j * v_st;
                const int64_t P = block_table[b * max_pages_per_seq + j / page_size];
                return P * v_sb + g * v_sh + (j % page_size) * v_st;
            };
            attend_row(L, D, qd.data(),
                       [&](int64_t j, int d) { return k_scale * cache_elem(k, k_off(j) + d, cdt); },
                       [&](int64_t j, int d) { return v_scale * cache_elem(v, v_off(j) + d, cdt); },
                       scale, out + r * D, lse + r, s, acc);
        }
    };

    int nt = n_threads > 0 ? n_threads : static_cast<int>(std::thread::hardware_concurrency());
    if (nt < 1) nt = 1;
    if (nt > count) nt = static_cast<int>(std::max<int64_t>(count, 1));
    if (nt == 1) {
        work(0, count);
        return 0;
    }
    std::vector<std::thread> pool;
    const int64_t per = (count + nt - 1) / nt;
    for (int t = 0; t < nt; ++t) {
        const int64_t a = t * per, e = std::min(count, a + per);
        if (a >= e) break;
        pool.emplace_back(work, a, e);
    }
    for (auto& th : pool) th.join();
    return 0;
}

int fdo_hardware_threads(void) {
    const unsigned n = std::thread::hardware_concurrency();
    return n ? static_cast<int>(n) : 1;
}

}  // extern "C"
