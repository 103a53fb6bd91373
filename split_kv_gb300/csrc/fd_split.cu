// fd_split.cu -- the split kernel of split-KV decode attention on sm_103a.
//
// One CTA per (KV split, KV head, sequence).  It streams the split's K/V
// rows once, for all G query heads of the KV head's group, and leaves the
// group's unnormalised partial states (u, m, l) in the workspace:
//   m = max_j s_j,  l = sum_j exp(s_j - m),  u = sum_j exp(s_j - m) v_j
// over the split's keys j ("Decode 专项 Attention：把长KV拆开算，再正确合并",
// §04; the tinyvolt Flash-decoding article's fd_split, which also stores the
// undivided O with m and l).  Inside the split the online-softmax recurrence
// of "Flash-Decoding: Split-KV Attention for Long-Context Decode" §4 runs tile
// by tile; an empty split leaves (u=0, m=-inf, l=0) (same page, §4 bullet on
// ragged batches).
//
// GB300 structure
//  - The last warp is a TMA producer.  16-bit caches: per 64-token stage it
//    issues four 2-D boxes [64 tokens x 64 dims] (K low/high half, V low/high
//    half) with 128-byte swizzle into a 3-stage ring, completing on the
//    stage's "full" mbarrier.  fp8 caches: two boxes of 128-byte rows (K, V)
//    per stage.  Contiguous caches use one box per tensor (or half); paged
//    caches 16-row boxes (8 for 8-token pages) resolved through the block
//    table a stage ahead.  Geo<KIND> below holds each variant's geometry.
//  - The other warps consume.  Each owns 16 of a stage's rows and keeps its
//    own running (m, l, acc) per column; the warp states are merged exactly at
//    the end of the split (the same max-subtracted rule).  Three consumers:
//    consume_tc (default) runs QK^T and PV as warp MMAs fed by ldmatrix;
//    consume_f8 builds the same MMAs' fragments from e4m3 bytes in registers;
//    consume_simt (FD_FLAG_CUDA_CORES) uses FP32 FMAs, a half-warp per K row.
//  - Query blocks of 17-128 columns on a 16-bit cache run instead on 5th-
//    generation tensor cores (fd_split_umma64_kernel, fd_split_umma_kernel):
//    one CTA per split holds every column as the M rows of tcgen05 MMAs with
//    S and O accumulated in tensor memory, fed by the same TMA stages.
//  - Scores are kept in base 2: t = (q.k) * log2(e)/sqrt(D), p = 2^(t - m).
//    The workspace m is converted back to natural units of s.
//  - Every mbarrier wait is bounded (2 s of wall time); on timeout the kernel
//    records kStatusTimeout in the device status word, drains its own copies
//    (bounded) and returns without writing states.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>

#include "fd_device.cuh"
#include "fd_internal.h"

namespace fdk {

// Per-device status word: sticky error bits read by fd_device_status().
__device__ unsigned int g_fd_status = 0;

namespace {

__device__ __forceinline__ void raise_status(unsigned bits) { atomicOr(&g_fd_status, bits); }

// mbar_wait that records a timeout in the status word.
__device__ __forceinline__ bool wait_or_flag(uint32_t bar, uint32_t parity) {
    if (mbar_wait(bar, parity)) return true;
    raise_status(kStatusTimeoutBit);
    return false;
}

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLn2 = 0.693147180559945309f;

template <typename T>
struct Cvt;

template <>
struct Cvt<__half> {
    static __device__ __forceinline__ float2 pair(uint32_t w) {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    }
};

template <>
struct Cvt<__nv_bfloat16> {
    // a bf16 pattern is the upper half of the f32 pattern of the same value
    static __device__ __forceinline__ float2 pair(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
};

template <typename T>
__device__ __forceinline__ void cvt8(const uint4& r, float (&f)[8]) {
    float2 a = Cvt<T>::pair(r.x), b = Cvt<T>::pair(r.y), c = Cvt<T>::pair(r.z),
           d = Cvt<T>::pair(r.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

template <typename T>
__device__ __forceinline__ void cvt4(const uint2& r, float (&f)[4]) {
    float2 a = Cvt<T>::pair(r.x), b = Cvt<T>::pair(r.y);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

// One reduce-scatter level over lanes `lane ^ MASK`: of N values per lane,
// the lane keeps the lower half (MASK bit clear) or the upper half (set),
// summed with the partner's copy of the same half.
template <int N, int MASK>
__device__ __forceinline__ void reduce_scatter(float* v, int lane) {
    const bool up = (lane & MASK) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = up ? v[i] : v[i + N / 2];
        const float keep = up ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(kFull, send, MASK);
    }
}

template <int G>
struct GroupShape {
    static constexpr int kLog = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
    // lanes whose all-reduced bits are zero own one (row, head) result
    static constexpr int kOwnerMask = (16 >> kLog) - 1;
};

// Sums G per-lane partial dot products over the 16 lanes of a half-warp.
// Afterwards lane l holds the full dot product of head head_of_lane<G>(l).
template <int G>
__device__ __forceinline__ float reduce16(float (&v)[G], int lane) {
    constexpr int LG = GroupShape<G>::kLog;
    if constexpr (LG >= 1) reduce_scatter<G, 8>(v, lane);
    if constexpr (LG >= 2) reduce_scatter<G / 2, 4>(v, lane);
    if constexpr (LG >= 3) reduce_scatter<G / 4, 2>(v, lane);
#pragma unroll
    for (int mask = 8 >> LG; mask >= 1; mask >>= 1) v[0] += __shfl_xor_sync(kFull, v[0], mask);
    return v[0];
}

template <int G>
__device__ __forceinline__ int head_of_lane(int lane) {
    constexpr int LG = GroupShape<G>::kLog;
    int g = 0;
#pragma unroll
    for (int k = 0; k < LG; ++k)
        if (lane & (8 >> k)) g += G >> (k + 1);
    return g;
}

// Shared-memory map (dynamic, 1024-byte aligned base for the 128B swizzle).
constexpr int kOffBars = kStages * kStageBytes;                   // full[kStages], empty[kStages]
constexpr int kOffP = kOffBars + 128;                             // [warps][16 rows][8 heads] f32
constexpr int kOffAlpha = kOffP + kConsumerWarps * 16 * 8 * 4;    // [warps][8] f32
constexpr int kOffFlag = kOffAlpha + kConsumerWarps * 8 * 4;      // abort flag
constexpr int kSmemUsed = kOffFlag + 16;
// end-of-split merge area (reuses stage memory once every stage is consumed)
constexpr int kCols = 16;                                         // (query, head) columns per CTA
constexpr int kOffWAcc = 0;                                       // [warps][16][128] f32
constexpr int kOffWM = kConsumerWarps * kCols * kHeadDim * 4;     // [warps][16]
constexpr int kOffWL = kOffWM + kConsumerWarps * kCols * 4;       // [warps][16]
static_assert(kOffWL + kConsumerWarps * kCols * 4 <= kOffBars, "merge area must fit in the stages");

}  // namespace

// Geometry of each kernel variant (KIND, see Consumer below).  16-bit caches:
// four consumer warps, 3 stages of 64 tokens, each stage four [64 x 64-dim]
// boxes (the map above).  fp8 caches: two [rows x 128-dim] e4m3 boxes (K, V)
// per stage, read by the consumers straight into registers; with at most 8
// columns per CTA (KIND 21) six consumer warps take 96-token stages, 4 deep,
// otherwise (KIND 22) four take 64-token stages, 6 deep.  Either way the ring
// holds 96 KB, and two CTAs fit on an SM.
template <int KIND>
struct Geo {
    static constexpr bool kUmma = KIND == 31 || KIND == 32;    // tcgen05 consumers, see below
    static constexpr bool kF8 = KIND >= 20 && !kUmma;
    static constexpr int kWarps = KIND == 21 ? kConsumerWarpsF8 : kUmma ? 8 : kConsumerWarps;
    static constexpr int kSub = kUmma ? 64 : 16 * kWarps;      // tokens per stage
    static constexpr int kRing = KIND == 21 ? 4 : KIND == 22 ? 6 : KIND == 31 ? 5 : KIND == 32 ? 4 : kStages;
    static constexpr int kTile = kSub * 128;                   // one box of 128-byte rows
    static constexpr int kStageBytes = (kF8 ? 2 : 4) * kTile;
    static constexpr int kOffExtra = kRing * kStageBytes;      // tcgen05: Q tile (and P, KIND 32)
    // + the softmax exchange and the tcgen05 barriers (4 KB)
    static constexpr int kExtraBytes = KIND == 31 ? 2 * 16384 + 4096 : KIND == 32 ? 4 * 16384 + 4096 : 0;
    static constexpr int kOffBars = kOffExtra + kExtraBytes;   // full[kRing], empty[kRing]
    static constexpr bool kOwnMap = kF8 || kUmma;
    static_assert(!kUmma || kSub == fdk::kSub, "the tcgen05 variant streams the 16-bit stages");
    static constexpr int kOffFlag = (kOwnMap ? kOffBars + 128 : fdk::kOffFlag);
    static constexpr int kSmem = (kOwnMap ? kOffFlag + 16 : kSmemUsed) + 1024;   // + alignment slack
    // + one TMA producer warp (+ one MMA-issuing warp for tcgen05)
    static constexpr int kThreads = (kWarps + (kUmma ? 2 : 1)) * 32;
    static constexpr int kEmptyArrivals = kUmma ? 1 : kWarps;  // tcgen05: the MMA commit
    // end-of-split merge area in stage memory: acc [warps][16][128], m, l [warps][16]
    static constexpr int kOffWM = kWarps * kCols * kHeadDim * 4;
    static constexpr int kOffWL = kOffWM + kWarps * kCols * 4;
    static_assert(2 * kRing * 8 <= 128, "barriers must fit");
    static_assert(kOffWL + kWarps * kCols * 4 <= kOffBars, "merge area must fit in the stages");
    static_assert(kOwnMap || (kSub == fdk::kSub && kStageBytes == fdk::kStageBytes &&
                              kOffBars == fdk::kOffBars), "16-bit variants use the map above");
};

// Everything a CTA knows about its split, shared by the producer and consumers.
struct SplitCtx {
    const SplitParams* p;
    uint8_t* smem;
    uint32_t bar0;
    int stages;                 // ring depth (the empty barriers follow the full ones)
    volatile int* abort_flag;   // any warp gave up
    volatile int* cons_abort;   // a consumer warp gave up
    int b, kvh, split;
    int cb;                     // block of 16 (query, head) columns this CTA serves
    int L;                      // the sequence's length (keys in the cache)
    int tok0, tok1, n_sub;

    __device__ __forceinline__ uint32_t full_bar(int s) const { return bar0 + 8u * s; }
    __device__ __forceinline__ uint32_t empty_bar(int s) const { return bar0 + 8u * (stages + s); }
};

// ---------------------------------------------------------------------------
// Producer warp: streams the split's K/V stages with TMA.  16-bit caches: four
// [rows x 64 dims] boxes per stage (K, V low and high halves); fp8 caches
// (F8): two [rows x 128 dims] boxes (K, V).
// ---------------------------------------------------------------------------
template <int KIND>
__device__ __forceinline__ void produce(const SplitCtx& c, const CUtensorMap* tmK,
                                        const CUtensorMap* tmV, int lane) {
    using Gm = Geo<KIND>;
    constexpr bool F8 = Gm::kF8;
    constexpr int kStages = Gm::kRing;
    constexpr int kStageBytes = Gm::kStageBytes;
    constexpr int kSub = Gm::kSub;
    const SplitParams& p = *c.p;
    // K/V are read once (evict first), or once per column block of the split
    // (kept at normal priority for the sibling CTAs that read them next)
    const uint64_t policy = p.col_blocks > 1 ? policy_evict_normal() : policy_evict_first();
    const bool paged = p.page_size != 0;
    const int rows = paged ? min(kPagedBoxRows, p.page_size) : kSub;   // tokens per box
    const int nbox = kSub / rows;                                        // boxes per half per stage
    // physical page of box `lane` of sub-tile i (paged); -1 reads zeros
    auto page_of = [&](int i) -> int {
        const int t = c.tok0 + i * kSub + lane * rows;
        if (lane >= nbox || i >= c.n_sub || t >= c.tok1) return -1;
        const int pg = __ldg(p.block_table + static_cast<size_t>(c.b) * p.max_pages +
                             (t >> p.page_shift));
        if (pg < 0 || pg >= p.n_pages) {
            raise_status(kStatusPageBit);
            return -1;
        }
        return pg;
    };
    int page_next = paged ? page_of(0) : 0;
    int issued = 0;
    const int first = p.drop_first_stage ? 1 : 0;   // test hook: stage 0 is never requested
#pragma unroll 1
    for (int i = 0; i < c.n_sub; ++i) {
        const int st = i % kStages;
        if (i >= kStages) {
            const bool ok = wait_or_flag(c.empty_bar(st), ((i / kStages) - 1) & 1);
            if (!__all_sync(kFull, ok)) *c.abort_flag = 1;
        }
        if (*c.abort_flag) break;
        const int page = page_next;
        const int tok = c.tok0 + i * kSub;
        const uint32_t dst = smem_u32(c.smem + st * kStageBytes);
        const uint32_t bar = c.full_bar(st);
        if (i < first) {
            if (paged) page_next = page_of(i + 1);
            continue;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar, kStageBytes);
        __syncwarp();
        if (F8) {
            if (lane < (paged ? nbox : 1)) {
                const int row = paged ? (tok + lane * rows) & (p.page_size - 1) : tok;
                const int outer = paged ? page : c.b;
                const uint32_t off = static_cast<uint32_t>(lane * rows * 128);
                tma_load_4d_hint(dst + off, tmK, bar, 0, row, c.kvh, outer, policy);
                tma_load_4d_hint(dst + Gm::kTile + off, tmV, bar, 0, row, c.kvh, outer, policy);
            }
        } else if (!paged) {
            if (lane == 0) {
                tma_load_4d_hint(dst + 0 * kHalfBytes, tmK, bar, 0, tok, c.kvh, c.b, policy);
                tma_load_4d_hint(dst + 1 * kHalfBytes, tmK, bar, 64, tok, c.kvh, c.b, policy);
                tma_load_4d_hint(dst + 2 * kHalfBytes, tmV, bar, 0, tok, c.kvh, c.b, policy);
                tma_load_4d_hint(dst + 3 * kHalfBytes, tmV, bar, 64, tok, c.kvh, c.b, policy);
            }
        } else if (lane < nbox) {
            const int in_page = (tok + lane * rows) & (p.page_size - 1);
            const uint32_t off = static_cast<uint32_t>(lane * rows * 128);
            tma_load_4d_hint(dst + 0 * kHalfBytes + off, tmK, bar, 0, in_page, c.kvh, page, policy);
            tma_load_4d_hint(dst + 1 * kHalfBytes + off, tmK, bar, 64, in_page, c.kvh, page, policy);
            tma_load_4d_hint(dst + 2 * kHalfBytes + off, tmV, bar, 0, in_page, c.kvh, page, policy);
            tma_load_4d_hint(dst + 3 * kHalfBytes + off, tmV, bar, 64, in_page, c.kvh, page, policy);
        }
        issued = i + 1;
        if (paged) page_next = page_of(i + 1);   // block-table read overlaps the next wait
    }
    // Drain: the last sub-tile issued into each stage must have landed before
    // this CTA may exit (a no-op unless a consumer gave up).
    if (lane == 0) {
        for (int i = max(first, issued - kStages); i < issued; ++i)
            wait_or_flag(c.full_bar(i % kStages), (i / kStages) & 1);
    }
}

// ---------------------------------------------------------------------------
// Consumer, CUDA-core path: QK^T and PV as FP32 FMAs.
// Writes the warp's (m, l, acc) into the merge area; false after a timeout.
// ---------------------------------------------------------------------------
template <typename T, int G>
__device__ __forceinline__ bool consume_simt(const SplitCtx& c, int cw, int lane) {
    const SplitParams& p = *c.p;
    const int hw = lane >> 4;                   // which of the two rows of a QK step
    const int c16 = lane & 15;                  // QK: dims 8*c16 .. 8*c16+7
    const int qk_half = c16 >> 3, qk_chunk = c16 & 7;
    const int pv_half = lane >> 4;              // PV: dims 4*lane .. 4*lane+3
    const int pv_chunk = (lane & 15) >> 1, pv_sub = (lane & 1) * 8;
    const int g_lane = head_of_lane<G>(lane);
    const bool owner = (lane & GroupShape<G>::kOwnerMask) == 0;   // per half-warp

    float qf[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const T* qrow = static_cast<const T*>(p.q) + static_cast<int64_t>(c.b) * p.q_sb +
                        static_cast<int64_t>(c.kvh * G + g) * p.q_sh + 8 * c16;
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qrow));
        cvt8<T>(raw, qf[g]);
    }

    float m_run = -INFINITY;   // base-2 running max of this warp's scores for head g_lane
    float l_run = 0.f;
    float acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[g][j] = 0.f;

    float* pw = reinterpret_cast<float*>(c.smem + kOffP) + cw * 16 * 8;
    float* aw = reinterpret_cast<float*>(c.smem + kOffAlpha) + cw * 8;

#pragma unroll 1
    for (int i = 0; i < c.n_sub; ++i) {
        const int st = i % kStages;
        const bool ok = wait_or_flag(c.full_bar(st), (i / kStages) & 1);
        if (!__all_sync(kFull, ok)) {
            *c.cons_abort = 1;
            *c.abort_flag = 1;
            break;
        }
        const uint8_t* sb = c.smem + st * kStageBytes;
        const int nvalid = min(kSub, c.tok1 - (c.tok0 + i * kSub));

        // ---- scores of this warp's 16 rows (two rows per step)
        float sc[8];
#pragma unroll
        for (int step = 0; step < 8; ++step) {
            const int r = cw * 16 + 2 * step + hw;
            const uint4 raw = *reinterpret_cast<const uint4*>(
                sb + qk_half * kHalfBytes + r * 128 + ((qk_chunk ^ (r & 7)) << 4));
            float kf[8];
            cvt8<T>(raw, kf);
            float part[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float a = qf[g][0] * kf[0];
#pragma unroll
                for (int j = 1; j < 8; ++j) a = fmaf(qf[g][j], kf[j], a);
                part[g] = a;
            }
            const float dot = reduce16<G>(part, lane);
            sc[step] = r < nvalid ? dot * p.score_scale_log2 : -INFINITY;
        }

        // ---- online softmax for head g_lane over the warp's 16 rows
        float mx = sc[0];
#pragma unroll
        for (int step = 1; step < 8; ++step) mx = fmaxf(mx, sc[step]);
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
        const float m_new = fmaxf(m_run, mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;   // never -inf - -inf
        const float alpha = fast_exp2(m_run - m_use);
        float psum = 0.f;
#pragma unroll
        for (int step = 0; step < 8; ++step) {
            const float pv = fast_exp2(sc[step] - m_use);
            psum += pv;
            if (owner) pw[(2 * step + hw) * 8 + g_lane] = pv;
        }
        psum += __shfl_xor_sync(kFull, psum, 16);
        l_run = fmaf(alpha, l_run, psum);
        m_run = m_new;
        if (owner && hw == 0) aw[g_lane] = alpha;
        __syncwarp();

        // ---- PV: acc[g][dims] = alpha_g acc + sum_r p[r][g] v[r][dims]
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float a = aw[g];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[g][j] *= a;
        }
        const int nrows = min(16, max(0, nvalid - cw * 16));
        const uint8_t* vb = sb + (2 + pv_half) * kHalfBytes;
        auto pv_row = [&](int r16) {
            const int r = cw * 16 + r16;
            const uint2 raw = *reinterpret_cast<const uint2*>(
                vb + r * 128 + (((pv_chunk ^ (r & 7)) << 4) | pv_sub));
            float vf[4];
            cvt4<T>(raw, vf);
            float pg[G];
            const float* pr = pw + r16 * 8;
            if constexpr (G >= 4) {
#pragma unroll
                for (int g = 0; g < G; g += 4) {
                    const float4 t4 = *reinterpret_cast<const float4*>(pr + g);
                    pg[g] = t4.x; pg[g + 1] = t4.y; pg[g + 2] = t4.z; pg[g + 3] = t4.w;
                }
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g) pg[g] = pr[g];
            }
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[g][j] = fmaf(pg[g], vf[j], acc[g][j]);
        };
        if (nrows == 16) {
#pragma unroll
            for (int r16 = 0; r16 < 16; ++r16) pv_row(r16);
        } else {
#pragma unroll 1
            for (int r16 = 0; r16 < nrows; ++r16) pv_row(r16);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(c.empty_bar(st));
    }

    // Only consumers write cons_abort, and only before this barrier, so every
    // consumer warp takes the same branch below.
    named_sync(1, kConsumerWarps * 32);
    if (*c.cons_abort) return false;   // states are not written after a timeout
    float* wacc = reinterpret_cast<float*>(c.smem + kOffWAcc);
    float* wm = reinterpret_cast<float*>(c.smem + kOffWM);
    float* wl = reinterpret_cast<float*>(c.smem + kOffWL);
    if (owner && hw == 0) {
        wm[cw * kCols + g_lane] = m_run;
        wl[cw * kCols + g_lane] = l_run;
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
        *reinterpret_cast<float4*>(wacc + (cw * kCols + g) * kHeadDim + 4 * lane) =
            make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
    return true;
}

// ---------------------------------------------------------------------------
// Consumer, tensor-core path: the packed group's QK^T and PV on warp-level
// MMAs (m16n8k16, f32 accumulate), "swap-AB": 16 tokens are the M rows and up
// to 8 * NB (query position, head) columns of the group are N:
//   S^T[16 tok x 8]  = K[16 tok x 128]   . Q^T[128 x 8]        (8 MMAs per N block)
//   O^T[128 x 8]    += V^T[128 x 16 tok] . P^T[16 tok x 8]     (8 x 2 MMAs per N block)
// Column n of the CTA's block cb is query position i = (16 cb + n) / G and
// head g = (16 cb + n) % G of the group; it sees the first L - q_len + 1 + i
// keys.  One query per sequence (q_len = 1) is the plain decode step.
// K and V^T fragments come straight from the swizzled stage with ldmatrix
// (no conversion instructions); P^T is the transposed S^T accumulator
// (movmatrix), carried as hi + lo 16-bit parts so that PV keeps ~2^-18
// relative precision in P even for bf16.
// Lane (gid = lane/4, tig = lane%4) holds columns 8j + 2tig, 8j + 2tig + 1 of
// tokens gid, gid+8 in S^T and dims 16mb+gid(+8) of the same columns in O^T.
// ---------------------------------------------------------------------------
template <typename T>
struct Mma;

template <>
struct Mma<__half> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // (lo, hi) -> one 32-bit register of two 16-bit values; also returns what was kept
    static __device__ __forceinline__ uint32_t pack(float lo, float hi, float& lo_kept, float& hi_kept) {
        const __half2 h = __floats2half2_rn(lo, hi);
        const float2 f = __half22float2(h);
        lo_kept = f.x;
        hi_kept = f.y;
        uint32_t r;
        memcpy(&r, &h, 4);
        return r;
    }
};

template <>
struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi, float& lo_kept, float& hi_kept) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        uint32_t r;
        memcpy(&r, &h, 4);
        lo_kept = __uint_as_float(r << 16);
        hi_kept = __uint_as_float(r & 0xffff0000u);
        return r;
    }
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Online softmax (base 2) of TILES 16-token tiles for up to 8 * NB columns,
// and P^T of each tile as hi + lo B fragments of the PV MMAs.  s[t] holds tile
// t's S^T (C fragments); csc[j][e] is the base-2 score scale of the lane's
// column 8j + 2tig + e, which sees the keys before vis[j][e]; tile t starts at
// key tok[t] and has nvalid[t] rows.  Without `masked` every row is taken as
// visible to every column (a full tile and one query per sequence).  The
// running max moves once per call.
// Returns whether any running max moved (the accumulators then take al).
template <typename MT, int NB, int TILES>
__device__ __forceinline__ bool softmax_tiles(const float (&s)[TILES][NB][4], const float (&csc)[NB][2],
                                              const int (&vis)[NB][2], const int (&nvalid)[TILES],
                                              const int (&tok)[TILES], int row0, int row1,
                                              bool masked, float (&m)[NB][2], float (&l)[NB][2],
                                              float (&al)[NB][2], uint32_t (&bh)[TILES][NB][2],
                                              uint32_t (&bl)[TILES][NB][2]) {
    bool rescale = false;
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        float t[TILES][4];
#pragma unroll
        for (int x = 0; x < TILES; ++x)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                t[x][e] = s[x][j][e] * csc[j][e];           // token gid
                t[x][e + 2] = s[x][j][e + 2] * csc[j][e];   // token gid + 8
            }
        if (masked) {   // warp-uniform: a partial tile, or columns with their own prefix
#pragma unroll
            for (int x = 0; x < TILES; ++x)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int lim = min(nvalid[x], vis[j][e] - tok[x]);
                    if (row0 >= lim) t[x][e] = -INFINITY;
                    if (row1 >= lim) t[x][e + 2] = -INFINITY;
                }
        }
        float pr[TILES][4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float mx = -INFINITY;
#pragma unroll
            for (int x = 0; x < TILES; ++x) mx = fmaxf(mx, fmaxf(t[x][e], t[x][e + 2]));
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
            const float mn = fmaxf(m[j][e], mx);
            const float mu = mn == -INFINITY ? 0.f : mn;   // never -inf - -inf
            al[j][e] = fast_exp2(m[j][e] - mu);
            float sum = 0.f;
#pragma unroll
            for (int x = 0; x < TILES; ++x) {
                pr[x][e] = fast_exp2(t[x][e] - mu);
                pr[x][e + 2] = fast_exp2(t[x][e + 2] - mu);
                sum += pr[x][e] + pr[x][e + 2];
            }
            l[j][e] = fmaf(al[j][e], l[j][e], sum);
            m[j][e] = mn;
            rescale |= al[j][e] != 1.f;
        }
        // P^T as B fragments: hi + lo parts, transposed in registers
#pragma unroll
        for (int x = 0; x < TILES; ++x) {
            float k0, k1, k2, k3, d0, d1, d2, d3;
            const uint32_t hi01 = Mma<MT>::pack(pr[x][0], pr[x][1], k0, k1);
            const uint32_t hi23 = Mma<MT>::pack(pr[x][2], pr[x][3], k2, k3);
            const uint32_t lo01 = Mma<MT>::pack(pr[x][0] - k0, pr[x][1] - k1, d0, d1);
            const uint32_t lo23 = Mma<MT>::pack(pr[x][2] - k2, pr[x][3] - k3, d2, d3);
            bh[x][j][0] = movmatrix_trans(hi01);
            bh[x][j][1] = movmatrix_trans(hi23);
            bl[x][j][0] = movmatrix_trans(lo01);
            bl[x][j][1] = movmatrix_trans(lo23);
        }
    }
    return __any_sync(kFull, rescale);
}

template <int NB>
__device__ __forceinline__ void rescale_acc(float (&acc)[8][NB][4], const float (&al)[NB][2]) {
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            acc[mb][j][0] *= al[j][0];
            acc[mb][j][1] *= al[j][1];
            acc[mb][j][2] *= al[j][0];
            acc[mb][j][3] *= al[j][1];
        }
}

// Keys visible to the lane's C columns: column n is query position n / G and
// sees the first L - q_len + 1 + n / G keys.
template <int NB>
__device__ __forceinline__ void visible_keys(const SplitCtx& c, int tig, int (&vis)[NB][2]) {
    const SplitParams& p = *c.p;
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = c.cb * kCols + 8 * j + 2 * tig + e;
            vis[j][e] = n < p.cols ? c.L - p.q_len + 1 + n / p.group : c.L;
        }
}

// Start of the row of q for column n of the CTA's block (row 0 for padding columns).
template <typename T>
__device__ __forceinline__ const T* q_row(const SplitCtx& c, int n, bool& real) {
    const SplitParams& p = *c.p;
    real = n < p.cols;
    const int i = real ? n / p.group : 0, g = real ? n % p.group : 0;
    return static_cast<const T*>(p.q) + static_cast<int64_t>(c.b) * p.q_sb +
           static_cast<int64_t>(i) * p.q_st + static_cast<int64_t>(c.kvh * p.group + g) * p.q_sh;
}

template <typename T, int NB>
__device__ __forceinline__ bool consume_tc(const SplitCtx& c, int cw, int lane) {
    const SplitParams& p = *c.p;
    const int gid = lane >> 2, tig = lane & 3;
    const int r0 = cw * 16;                      // the warp's 16 rows of each stage

    // Q^T as the B operand of N block j: column 8j + gid,
    // b0 = q[.][16kb + 2tig .. +1], b1 = q[.][16kb + 8 + 2tig .. +1]
    uint32_t qb[NB][8][2];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        bool real;
        const T* qrow = q_row<T>(c, c.cb * kCols + 8 * j + gid, real);
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
            const uint32_t lo = __ldg(reinterpret_cast<const unsigned int*>(qrow + 16 * kb + 2 * tig));
            const uint32_t hi = __ldg(reinterpret_cast<const unsigned int*>(qrow + 16 * kb + 8 + 2 * tig));
            qb[j][kb][0] = real ? lo : 0u;
            qb[j][kb][1] = real ? hi : 0u;
        }
    }
    int vis[NB][2];
    visible_keys<NB>(c, tig, vis);
    float csc[NB][2];
#pragma unroll
    for (int j = 0; j < NB; ++j) csc[j][0] = csc[j][1] = p.score_scale_log2;

    float m[NB][2], l[NB][2];               // base-2 running max; this lane's share of the sums
    float acc[8][NB][4];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        m[j][0] = m[j][1] = -INFINITY;
        l[j][0] = l[j][1] = 0.f;
#pragma unroll
        for (int mb = 0; mb < 8; ++mb)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mb][j][e] = 0.f;
    }

    // ldmatrix row addresses (bytes within a half box, before the stage base)
    // K (A operand, not transposed): matrix j = lane/8 holds tokens +0/+8 and dims +0/+8
    const int k_row = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int k_csel = lane >> 4;
    // V^T (A operand via .trans): matrix j holds tokens +0/+8 (j/2) and dims +0/+8 (j%2)
    const int v_row = r0 + (lane & 7) + ((lane >> 4) & 1) * 8;
    const int v_csel = (lane >> 3) & 1;

#pragma unroll 1
    for (int it = 0; it < c.n_sub; ++it) {
        const int st = it % kStages;
        const bool ok = wait_or_flag(c.full_bar(st), (it / kStages) & 1);
        if (!__all_sync(kFull, ok)) {
            *c.cons_abort = 1;
            *c.abort_flag = 1;
            break;
        }
        uint8_t* sb = c.smem + st * kStageBytes;
        const int stage_tok = c.tok0 + it * kSub;
        const int nvalid = min(kSub, c.tok1 - stage_tok);
        const uint32_t kbase = smem_u32(sb);
        const uint32_t vbase = smem_u32(sb + 2 * kHalfBytes);

        // Rows past the sequence end hold whatever the cache holds there; P is
        // 0 for them, but 0 * NaN would still poison PV, so zero those V rows.
        if (nvalid < r0 + 16) {
            uint8_t* vb = sb + 2 * kHalfBytes;
#pragma unroll
            for (int idx = lane; idx < 16 * 16; idx += 32) {
                const int rr = r0 + (idx >> 4);
                const int ch = idx & 15;
                if (rr >= nvalid)
                    *reinterpret_cast<uint4*>(vb + (ch >> 3) * kHalfBytes + rr * 128 + ((ch & 7) << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();   // ordered before the next TMA write of this stage
            __syncwarp();
        }

        // ---- S^T = K . Q^T for the warp's 16 tokens
        float s[1][NB][4];
#pragma unroll
        for (int j = 0; j < NB; ++j) s[0][j][0] = s[0][j][1] = s[0][j][2] = s[0][j][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
            const int chunk = 2 * kb + k_csel;                     // 16-byte chunk of the row
            const uint32_t addr = kbase + (chunk >> 3) * kHalfBytes + k_row * 128 +
                                  (((chunk & 7) ^ (k_row & 7)) << 4);
            uint32_t a[4];
            ldsm_x4(a, addr);
#pragma unroll
            for (int j = 0; j < NB; ++j) Mma<T>::run(s[0][j], a, qb[j][kb][0], qb[j][kb][1]);
        }

        // ---- online softmax per column over the 16 tokens
        float al[NB][2];
        uint32_t bh[1][NB][2], bl[1][NB][2];
        const int nv[1] = {nvalid}, tk[1] = {stage_tok};
        if (softmax_tiles<T, NB, 1>(s, csc, vis, nv, tk, r0 + gid, r0 + gid + 8,
                                    nvalid < kSub || stage_tok + kSub > c.L - p.q_len + 1, m, l,
                                    al, bh, bl))
            rescale_acc<NB>(acc, al);

        // ---- O^T += V^T . P^T
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
            const int chunk = 2 * mb + v_csel;
            const uint32_t addr = vbase + (chunk >> 3) * kHalfBytes + v_row * 128 +
                                  (((chunk & 7) ^ (v_row & 7)) << 4);
            uint32_t a[4];
            ldsm_x4_trans(a, addr);
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                Mma<T>::run(acc[mb][j], a, bh[0][j][0], bh[0][j][1]);
                Mma<T>::run(acc[mb][j], a, bl[0][j][0], bl[0][j][1]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(c.empty_bar(st));
    }

    // lane sums -> column sums over the 8 token rows (lanes with equal tig)
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) l[j][e] += __shfl_xor_sync(kFull, l[j][e], o);

    named_sync(1, kConsumerWarps * 32);
    if (*c.cons_abort) return false;   // states are not written after a timeout
    float* wacc = reinterpret_cast<float*>(c.smem + kOffWAcc);
    float* wm = reinterpret_cast<float*>(c.smem + kOffWM);
    float* wl = reinterpret_cast<float*>(c.smem + kOffWL);
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int col = 8 * j + 2 * tig + e;
            if (gid == 0) {
                wm[cw * kCols + col] = m[j][e];
                wl[cw * kCols + col] = l[j][e];
            }
#pragma unroll
            for (int mb = 0; mb < 8; ++mb) {
                wacc[(cw * kCols + col) * kHeadDim + 16 * mb + gid] = acc[mb][j][e];
                wacc[(cw * kCols + col) * kHeadDim + 16 * mb + gid + 8] = acc[mb][j][e + 2];
            }
        }
    return true;
}

// ---------------------------------------------------------------------------
// Consumer for an fp8 (E4M3) cache: the same swap-AB tile as f16 MMAs, with
// the A fragments built in registers from the e4m3 stage (no ldmatrix, no
// staging copy).  Each MMA's contraction index is permuted so that every lane
// reads whole 16-byte chunks of the swizzled stage:
//  - QK: lane (gid, tig) reads K bytes 32tig .. 32tig+31 of tokens gid and
//    gid + 8.  Block kb takes dims 32tig + 4kb + {0,1} as its k = 2tig + {0,1}
//    and dims 32tig + 4kb + {2,3} as k = 2tig + 8 + {0,1}; Q^T's fragments
//    follow the same order, so each score is still the full dot product.
//  - PV: lane (gid, tig) reads V bytes 16gid .. 16gid+15 of tokens 2tig,
//    2tig+1, 2tig+8 and 2tig+9; output row gid (gid + 8) of block mb is dim
//    16gid + 2mb (+1).  Token order is the plain one, as P^T expects.
// e4m3 -> f16 is exact (one cvt per pair).  A bf16 Q enters as f16 after a
// per-column power of two that puts the column's largest |q| in [2^14, 2^15)
// (every element within 2^31 of it converts exactly); that column's score
// scale takes the inverse power.  P goes to f16 as hi + lo parts.
// The warp's 8 chunk loads are its only reads of a stage, so it hands the
// stage back to the producer right after them.  An e4m3 stage carries half
// the bytes of a 16-bit one, so the same arithmetic per token has half the
// time: the narrow variant (KIND 21) runs six consumer warps per CTA to hide
// the instruction latencies that bound this consumer.
// ---------------------------------------------------------------------------
// four e4m3 bytes -> two f16 pairs: (b0, b1) and (b2, b3), low byte in the low half
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 x, y;\n\tmov.b32 {x, y}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, x;\n\tcvt.rn.f16x2.e4m3x2 %1, y;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ void unpack4(const uint4& r, uint32_t* w) {
    w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
}

template <typename T, int KIND>
__device__ __forceinline__ bool consume_f8(const SplitCtx& c, int cw, int lane) {
    using Gm = Geo<KIND>;
    constexpr int NB = KIND == 21 ? 1 : 2;
    constexpr int kSub = Gm::kSub;
    constexpr int kRing = Gm::kRing;
    const SplitParams& p = *c.p;
    const int gid = lane >> 2, tig = lane & 3;
    const int r0 = cw * 16;                      // the warp's 16 rows of each stage

    // Q^T of N block j (column 8j + gid) in the permuted order: b0 of block kb
    // is q[32tig + 4kb .. +1], b1 is q[32tig + 4kb + 2 .. +3]
    uint32_t qb[NB][8][2];
    int qexp[NB];                                // the column's power of two
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        bool real;
        const T* qrow = q_row<T>(c, c.cb * kCols + 8 * j + gid, real);
        uint32_t w[16];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const uint4 r = real ? __ldg(reinterpret_cast<const uint4*>(qrow + 32 * tig) + x)
                                 : make_uint4(0u, 0u, 0u, 0u);
            unpack4(r, w + 4 * x);
        }
        int k = 0;
        if constexpr (!std::is_same<T, __half>::value) {
            float mx = 0.f;
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const float2 f = Cvt<T>::pair(w[x]);
                mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));   // the column's 4 lanes
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
            const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127;
            k = (mx > 0.f && mx <= 3.402823466e38f) ? min(14 - ex, 126) : 0;
            const float qm = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const float2 f = Cvt<T>::pair(w[x]);
                const __half2 h = __floats2half2_rn(f.x * qm, f.y * qm);
                memcpy(&w[x], &h, 4);
            }
        }
        qexp[j] = k;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
            qb[j][kb][0] = w[2 * kb];
            qb[j][kb][1] = w[2 * kb + 1];
        }
    }
    // score scale of the lane's C columns 8j + 2tig + e (held by lanes gid = 2tig + e)
    float csc[NB][2];
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int k = __shfl_sync(kFull, qexp[j], (2 * tig + e) * 4);
            csc[j][e] = p.score_scale_log2 * __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
        }
    int vis[NB][2];
    visible_keys<NB>(c, tig, vis);

    float m[NB][2], l[NB][2];
    float acc[8][NB][4];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        m[j][0] = m[j][1] = -INFINITY;
        l[j][0] = l[j][1] = 0.f;
#pragma unroll
        for (int mb = 0; mb < 8; ++mb)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mb][j][e] = 0.f;
    }

    // byte offsets of the lane's chunks in a stage (128-byte rows, 128B swizzle:
    // chunk ch of row r sits at chunk ch ^ (r & 7)); rows r and r + 8 share the phase
    const int krow = r0 + gid;
    const int k_off0 = krow * 128 + (((2 * tig) ^ (krow & 7)) << 4);
    const int k_off1 = krow * 128 + (((2 * tig + 1) ^ (krow & 7)) << 4);
    int v_row[4], v_off[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        v_row[x] = r0 + 2 * tig + (x & 1) + (x >> 1) * 8;
        v_off[x] = Gm::kTile + v_row[x] * 128 + ((gid ^ (v_row[x] & 7)) << 4);
    }

#pragma unroll 1
    for (int it = 0; it < c.n_sub; ++it) {
        const int st = it % kRing;
        const bool ok = wait_or_flag(c.full_bar(st), (it / kRing) & 1);
        if (!__all_sync(kFull, ok)) {
            *c.cons_abort = 1;
            *c.abort_flag = 1;
            break;
        }
        const uint8_t* sb = c.smem + st * Gm::kStageBytes;
        const int tok = c.tok0 + it * kSub;
        const int nvalid = min(kSub, c.tok1 - tok);

        uint32_t kw[16], vw[4][4];
        unpack4(*reinterpret_cast<const uint4*>(sb + k_off0), kw);
        unpack4(*reinterpret_cast<const uint4*>(sb + k_off1), kw + 4);
        unpack4(*reinterpret_cast<const uint4*>(sb + k_off0 + 8 * 128), kw + 8);
        unpack4(*reinterpret_cast<const uint4*>(sb + k_off1 + 8 * 128), kw + 12);
#pragma unroll
        for (int x = 0; x < 4; ++x) unpack4(*reinterpret_cast<const uint4*>(sb + v_off[x]), vw[x]);
        __syncwarp();
        if (lane == 0) mbar_arrive(c.empty_bar(st));   // the stage is in registers
        const bool partial = nvalid < kSub;            // the split's last stage
        if (partial) {
            // Rows past the end hold whatever the cache holds there; P is 0 for
            // them, but 0 * NaN would still poison PV, so those V rows are 0.
#pragma unroll
            for (int x = 0; x < 4; ++x)
                if (v_row[x] >= nvalid) vw[x][0] = vw[x][1] = vw[x][2] = vw[x][3] = 0u;
        }

        // ---- S^T = K . Q^T (permuted dims); with one N block, even and odd k
        // blocks go to separate accumulators: two MMA chains of four
        constexpr bool kTwoChains = NB == 1;
        float s[1][NB][4], s2[NB][4];
#pragma unroll
        for (int j = 0; j < NB; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[0][j][e] = s2[j][e] = 0.f;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
            uint32_t a[4];
            e4m3x4_to_f16(kw[kb], a[0], a[2]);        // token gid
            e4m3x4_to_f16(kw[8 + kb], a[1], a[3]);    // token gid + 8
#pragma unroll
            for (int j = 0; j < NB; ++j)
                Mma<__half>::run((kTwoChains && (kb & 1)) ? s2[j] : s[0][j], a, qb[j][kb][0],
                                 qb[j][kb][1]);
        }
        if constexpr (kTwoChains) {
#pragma unroll
            for (int j = 0; j < NB; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[0][j][e] += s2[j][e];
        }

        float al[NB][2];
        uint32_t bh[1][NB][2], bl[1][NB][2];
        const int nv[1] = {nvalid}, tk[1] = {tok};
        if (softmax_tiles<__half, NB, 1>(s, csc, vis, nv, tk, r0 + gid, r0 + gid + 8,
                                         partial || tok + kSub > c.L - p.q_len + 1, m, l, al, bh,
                                         bl))
            rescale_acc<NB>(acc, al);

        // ---- O^T += V^T . P^T (permuted dims)
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
            // bytes 2mb, 2mb+1 of tokens (2tig, 2tig+1) and (2tig+8, 2tig+9), interleaved
            const uint32_t sel = (mb & 1) ? 0x7362u : 0x5140u;
            uint32_t a[4];
            e4m3x4_to_f16(__byte_perm(vw[0][mb >> 1], vw[1][mb >> 1], sel), a[0], a[1]);
            e4m3x4_to_f16(__byte_perm(vw[2][mb >> 1], vw[3][mb >> 1], sel), a[2], a[3]);
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                Mma<__half>::run(acc[mb][j], a, bh[0][j][0], bh[0][j][1]);
                Mma<__half>::run(acc[mb][j], a, bl[0][j][0], bl[0][j][1]);
            }
        }
    }

#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) l[j][e] += __shfl_xor_sync(kFull, l[j][e], o);

    named_sync(1, Gm::kWarps * 32);
    if (*c.cons_abort) return false;   // states are not written after a timeout
    float* wacc = reinterpret_cast<float*>(c.smem);
    float* wm = reinterpret_cast<float*>(c.smem + Gm::kOffWM);
    float* wl = reinterpret_cast<float*>(c.smem + Gm::kOffWL);
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int col = 8 * j + 2 * tig + e;
            if (gid == 0) {
                wm[cw * kCols + col] = m[j][e];
                wl[cw * kCols + col] = l[j][e];
            }
#pragma unroll
            for (int mb = 0; mb < 8; ++mb)
                *reinterpret_cast<float2*>(wacc + (cw * kCols + col) * kHeadDim + 16 * gid + 2 * mb) =
                    make_float2(acc[mb][j][e], acc[mb][j][e + 2]);
        }
    return true;
}

// ---------------------------------------------------------------------------
// The split kernel.  The consumer is consume_tc<T, NB> (default), consume_f8<T, KIND> or
// consume_simt<T, G>; both leave per-warp states of up to 16 columns for the
// final merge.
// ---------------------------------------------------------------------------
template <typename T, int KIND>
struct Consumer;
// KIND 1, 2: tensor cores with 8 or 16 columns; 21, 22: the same on an fp8
// cache; KIND 10 + G: CUDA cores, group G
template <typename T> struct Consumer<T, 1> {
    static __device__ bool run(const SplitCtx& c, int w, int l) { return consume_tc<T, 1>(c, w, l); }
};
template <typename T> struct Consumer<T, 2> {
    static __device__ bool run(const SplitCtx& c, int w, int l) { return consume_tc<T, 2>(c, w, l); }
};
template <typename T> struct Consumer<T, 21> {
    static __device__ bool run(const SplitCtx& c, int w, int l) { return consume_f8<T, 21>(c, w, l); }
};
template <typename T> struct Consumer<T, 22> {
    static __device__ bool run(const SplitCtx& c, int w, int l) { return consume_f8<T, 22>(c, w, l); }
};
template <typename T> struct Consumer<T, 11> {
    static __device__ bool run(const SplitCtx& c, int w, int l) { return consume_simt<T, 1>(c, w, l); }
};
template <typename T> struct Consumer<T, 12> {
    static __device__ bool run(const SplitCtx& c, int w, int l) { return consume_simt<T, 2>(c, w, l); }
};
template <typename T> struct Consumer<T, 14> {
    static __device__ bool run(const SplitCtx& c, int w, int l) { return consume_simt<T, 4>(c, w, l); }
};
template <typename T> struct Consumer<T, 18> {
    static __device__ bool run(const SplitCtx& c, int w, int l) { return consume_simt<T, 8>(c, w, l); }
};

// The start every split kernel shares: the context, the ring's barriers, the
// programmatic-dependent-launch wait, and the split's token range.
template <int KIND>
__device__ __forceinline__ void split_begin(SplitCtx& c, uint8_t* smem, const SplitParams& p,
                                            const CUtensorMap* tmK, const CUtensorMap* tmV) {
    using Gm = Geo<KIND>;
    constexpr int kRing = Gm::kRing;
    c.stages = kRing;
    c.p = &p;
    c.smem = smem;
    // grid (n_splits * col_blocks, n_kv_heads, batch): the column blocks of
    // one split are adjacent, so they run together and the later readers of
    // the split's K/V find it in L2
    c.split = blockIdx.x / p.col_blocks;
    c.cb = blockIdx.x % p.col_blocks;
    c.kvh = blockIdx.y;
    c.b = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.n_splits;

    c.bar0 = smem_u32(smem + Gm::kOffBars);
    c.abort_flag = reinterpret_cast<volatile int*>(smem + Gm::kOffFlag);
    c.cons_abort = reinterpret_cast<volatile int*>(smem + Gm::kOffFlag + 4);
    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < kRing; ++s) {
            mbar_init(c.full_bar(s), 1);
            mbar_init(c.empty_bar(s), Gm::kEmptyArrivals);
        }
        *c.abort_flag = 0;
        *c.cons_abort = 0;
        fence_barrier_init();
    }
    if (warp == Gm::kWarps && lane == 0) {
        prefetch_tensormap(tmK);
        prefetch_tensormap(tmV);
    }
    // Programmatic dependent launch: let the combine kernel that follows get
    // resident now, and wait for whatever preceded this kernel in the stream
    // to finish (and its writes to land) before reading any input.
    grid_dependency_trigger();
    grid_dependency_wait();

    // ---- this split's token range: the sequence cut into S balanced ranges
    // of whole 16-token units (8 for 8-token pages), so no TMA box straddles
    // a page and a paged cache splits exactly like a contiguous one
    int L = __ldg(p.seqlens + c.b);
    if (L < 0 || L > p.capacity) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_status(kStatusSeqlenBit);
        L = L < 0 ? 0 : p.capacity;
    }
    c.L = L;
    const int unit = p.split_unit;
    const int n_units = (L + unit - 1) / unit;
    const int base = n_units / S, rem = n_units % S;
    const int u_begin = c.split * base + (c.split < rem ? c.split : rem);
    const int u_count = base + (c.split < rem ? 1 : 0);
    c.tok0 = u_begin * unit;
    c.tok1 = min((u_begin + u_count) * unit, L);
    c.n_sub = c.tok1 > c.tok0 ? (c.tok1 - c.tok0 + Gm::kSub - 1) / Gm::kSub : 0;
}

template <typename T, int KIND>
__global__ void __launch_bounds__(Geo<KIND>::kThreads, 2)
    fd_split_kernel(const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
    using Gm = Geo<KIND>;
    constexpr int kWarps = Gm::kWarps;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    SplitCtx c;
    split_begin<KIND>(c, smem, p, &tmK, &tmV);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.n_splits;
    __syncthreads();

    if (warp == kWarps) {
        produce<KIND>(c, &tmK, &tmV, lane);
        return;
    }

    if (!Consumer<T, KIND>::run(c, warp, lane)) return;
    named_sync(1, kWarps * 32);
    if (threadIdx.x >= kHeadDim) return;   // one thread per dim below

    // ---- merge the consumer warps' states of each column and write the split's state
    const float* wacc = reinterpret_cast<const float*>(smem);
    const float* wm = reinterpret_cast<const float*>(smem + Gm::kOffWM);
    const float* wl = reinterpret_cast<const float*>(smem + Gm::kOffWL);
    const int d = threadIdx.x;   // 0 .. 127
    const int ncols = min(kCols, p.cols - c.cb * kCols);
    for (int col = 0; col < ncols; ++col) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kCols + col]);
        float u = 0.f, l = 0.f, m_out = -INFINITY;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float mw = wm[w * kCols + col];
                const float e = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
                u = fmaf(e, wacc[(w * kCols + col) * kHeadDim + d], u);
                l = fmaf(e, wl[w * kCols + col], l);
            }
            m_out = M * kLn2;
        }
        const int n = c.cb * kCols + col;
        const int i = n / p.group, g = n % p.group;
        const int64_t row = (static_cast<int64_t>(c.b) * p.q_len + i) * p.n_q_heads +
                            c.kvh * p.group + g;
        const int64_t idx = row * S + c.split;
        const float us = u * p.v_scale;   // values are v_scale x the stored ones
        if (p.direct) {
            // One split: the merge of a single state (weight exp(0) = 1) is
            // out = u / l, lse = m + log l; the same operations here give the
            // combine kernel's bits without its launch.
            const bool empty = m_out == -INFINITY || !(l > 0.f);
            const float o = empty ? 0.f : us / l;
            const int64_t oi = row * kHeadDim + d;
            if (p.out_dtype == 2)
                static_cast<float*>(p.out)[oi] = o;
            else if (p.out_dtype == 0)
                static_cast<__half*>(p.out)[oi] = __float2half_rn(o);
            else
                static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
            if (d == 0 && p.lse != nullptr) p.lse[row] = empty ? -INFINITY : m_out + logf(l);
            continue;
        }
        p.ws_u[idx * kHeadDim + d] = us;
        if (d == 0) {
            p.ws_m[idx] = m_out;
            p.ws_l[idx] = l;
        }
    }
}

// ---------------------------------------------------------------------------
// tcgen05 variant (KIND 31) for query blocks of 65-128 columns (16-bit
// caches; KIND 32 below takes 17-64): one CTA serves all G * q_len
// (position, head) columns of a KV head as the M rows of 5th-generation
// tensor-core MMAs with the accumulators in tensor memory, instead of one CTA
// per 16 columns each repeating the split's arithmetic on warp MMAs.
//   S[col][tok]  = Q[col][:] . K[tok][:]        M = 128 columns, N = 64 tokens, K = 128 dims
//   O[col][dim] += P[col][tok] . V[tok][dim]    M = 128, N = 128 dims, K = 64 tokens (V read MN-major)
// Q (K-major, 128-byte swizzle) is staged once in shared memory; K and V come
// from the TMA ring exactly as for the 16-bit consumer.  P never leaves the
// tensor memory: the softmax stores it there (hi + lo 16-bit parts, two per
// 32-bit column) and PV takes it as its A operand.  Tensor memory holds two S
// buffers and two P buffers (64 columns each) and O (128 columns), so the
// softmax of stage i + 1 overlaps PV of stage i.
// Warps 0-7 run the online softmax (base 2): warp w reaches tensor-memory
// lanes 32 (w % 4) .. +31, i.e. columns 32 (w % 4) .. +31, and takes tokens
// 32 (w / 4) .. +31 of each stage, so the two warps of a lane quarter split a
// stage's tokens and exchange their maxima through shared memory.  Warp 8 is
// the TMA producer; one thread of warp 9 issues every MMA.  A column's running
// max moves only when a stage's max exceeds it by more than 8 (log2 units),
// so p stays below 2^8 and O is rescaled in tensor memory only then.  The
// states written at the end are the same (u, m, l) as the other consumers'.
// Shared memory: 5-stage ring (160 KB), Q (32 KB), the softmax pairs'
// exchange and the tcgen05 barriers (4 KB).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(Geo<31>::kThreads, 1)
    fd_split_umma_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
    using Gm = Geo<31>;
    constexpr int kRing = Gm::kRing;
    constexpr int kSoftmaxThreads = Gm::kWarps * 32;   // 256
    // S [0, 128) and P [128, 256) double-buffered by stage parity, O [256, 384)
    constexpr uint32_t kTmemCols = 512;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    SplitCtx c;
    split_begin<31>(c, smem, p, &tmK, &tmV);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.n_splits;
    const int n_sub = c.n_sub;
    uint8_t* sQ = smem + Gm::kOffExtra;       // two halves [128 x 64 dims]
    // the softmax pairs' exchange: stage maxima [stage parity][token half][column],
    // final sums [token half][column]
    float* xmax = reinterpret_cast<float*>(sQ + 2 * 16384);
    float* xsum = xmax + 512;
    // mbarriers, each [2] by stage parity except drain and the pairs'
    const uint32_t b_pair0 = smem_u32(xsum + 256);   // [4], one per lane quarter: one arrival per warp of the pair
    const uint32_t b_s_full = b_pair0 + 32;   // one arrival (MMA commit): S written
    const uint32_t b_p_full = b_pair0 + 64;   // one arrival per softmax warp: P written (and O rescaled)
    const uint32_t b_o_done = b_pair0 + 80;   // one arrival (MMA commit): PV done
    const uint32_t b_drain = b_pair0 + 96;    // one arrival (MMA commit): every MMA done
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(xsum + 256 + 26);   // b_pair0 + 104
    if (threadIdx.x == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) mbar_init(b_pair0 + 8u * q, 2);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            mbar_init(b_s_full + 8u * b, 1);
            mbar_init(b_p_full + 8u * b, Gm::kWarps);
            mbar_init(b_o_done + 8u * b, 1);
        }
        mbar_init(b_drain, 1);
        fence_barrier_init();
    }
    __syncthreads();   // every barrier is initialised
    if (warp == Gm::kWarps) {   // the producer streams at once; Q and tensor memory follow
        produce<31>(c, &tmK, &tmV, lane);
        return;
    }
    if (threadIdx.x < 128) {
        // Q tile: row r is column r of the group (zeros past the columns)
        const int r = threadIdx.x;
        bool real;
        const T* qrow = q_row<T>(c, r, real);
        const uint4* src = reinterpret_cast<const uint4*>(qrow);
#pragma unroll 4
        for (int ch = 0; ch < 16; ++ch) {
            const uint4 v = real ? __ldg(src + ch) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(sQ + (ch >> 3) * 16384 + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
    }
    if (warp == 0) tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    tc_fence_before();
    named_sync(3, kSoftmaxThreads + 32);   // the softmax warps and the MMA warp
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_p = tmem + 128;
    const uint32_t tmem_o = tmem + 256;

    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;

    if (warp == Gm::kWarps + 1) {
        // ---- MMA issue: S of stage i + 1 goes out before PV of stage i, so
        // the softmax of one stage overlaps the tensor cores' work on the next
        // Buffer reuse needs no waits of its own: S of stage i + 1 overwrites
        // the scores of stage i - 1, which the softmax read before it handed
        // over P of stage i - 1 (waited for before PV of stage i - 1); and the
        // commit that signals S of stage i completes only after every earlier
        // MMA, PV of stage i - 2 included, so the softmax may then overwrite
        // that stage's P buffer.
        if (lane == 0) {
            // Issue cost bounds this thread: each descriptor is built once and
            // offset by constants (the start address is the low field, in
            // 16-byte units, and no operand crosses 256 KB, so adding never carries).
            const uint32_t id_s = umma_idesc_f16(128, 64, kBf16, false);
            const uint32_t id_o = umma_idesc_f16(128, 128, kBf16, true);
            const uint64_t dq = umma_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dk0 = umma_desc_sw128(smem_u32(c.smem), 16, 1024);
            const uint64_t dv0 = umma_desc_sw128(smem_u32(c.smem + 2 * kHalfBytes), static_cast<uint32_t>(kHalfBytes), 1024);
            constexpr uint32_t kStageUnits = Gm::kStageBytes >> 4;
            auto issue_s = [&](int i) {
                const uint64_t dk = dk0 + static_cast<uint32_t>(i % kRing) * kStageUnits;
                const uint32_t d = tmem + 64u * static_cast<uint32_t>(i & 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {   // 16 dims per MMA: 32 bytes inside a 128-byte row
                    const uint32_t q_off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                    const uint32_t k_off = ((kk >> 2) * static_cast<uint32_t>(kHalfBytes) + (kk & 3) * 32u) >> 4;
                    umma_f16(d, dq + q_off, dk + k_off, id_s, kk > 0);
                }
                umma_commit(b_s_full + 8u * static_cast<uint32_t>(i & 1));
            };
            bool ok = true;
            if (n_sub > 0) {
                ok = wait_or_flag(c.full_bar(0), 0);
                if (ok) {
                    tc_fence_after();
                    issue_s(0);
                }
            }
            for (int i = 0; ok && i < n_sub; ++i) {
                if (i + 1 < n_sub) {
                    const int j = i + 1;
                    ok = wait_or_flag(c.full_bar(j % kRing), (j / kRing) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(j);
                }
                ok = wait_or_flag(b_p_full + 8u * (i & 1), (i >> 1) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dv = dv0 + static_cast<uint32_t>(i % kRing) * kStageUnits;
                const uint32_t pa = tmem_p + 64u * static_cast<uint32_t>(i & 1);
#pragma unroll
                for (int part = 0; part < 2; ++part) {   // P hi, then P lo
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {     // 16 tokens (two 8-row groups) per MMA
                        // tokens 16 kk .. +15 were written by the warps of token half kk / 2:
                        // hi at columns 32 (kk / 2) + 8 (kk % 2), lo 16 columns further
                        const uint32_t a = pa + 32u * (kk >> 1) + 16u * part + 8u * (kk & 1);
                        umma_f16_ta(tmem_o, a, dv + ((kk * 2048u) >> 4), id_o, i > 0 || part > 0 || kk > 0);
                    }
                }
                umma_commit(b_o_done + 8u * static_cast<uint32_t>(i & 1));
                umma_commit(c.empty_bar(i % kRing));
            }
            if (!ok) {
                *c.cons_abort = 1;
                *c.abort_flag = 1;
            }
            umma_commit(b_drain);              // tensor memory is freed only after this
            wait_or_flag(b_drain, 0);
        }
        __syncwarp();
    } else {
        // ---- softmax warps: thread (w, lane) owns column r = 32 (w % 4) + lane
        // (tensor-memory lane r) and tokens 32 h .. 32 h + 31 of each stage, h = w / 4
        const int quarter = warp & 3, h = warp >> 2;
        const int r = quarter * 32 + lane;
        const bool quarter_active = quarter * 32 < p.cols;   // the pair's columns hold queries
        const bool real = r < p.cols;
        const int vis = real ? c.L - p.q_len + 1 + r / p.group : c.L;
        // scores stay raw until the exponent: sc (log2(e) / sqrt(d), a 16-bit
        // cache) is positive, so maxima of raw scores scale to maxima of scaled ones
        const float sc = p.score_scale_log2;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t b_pair = b_pair0 + 8u * quarter;   // warps quarter and quarter + 4
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int i = 0; i < n_sub; ++i) {
            const int buf = i & 1;
            ok = __all_sync(kFull, wait_or_flag(b_s_full + 8u * buf, (i >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
            float t[32];
            if (quarter_active) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t v[16];
                    tmem_ld16(tmem + lane_base + 64u * buf + 32u * h + 16u * q, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) t[16 * q + e] = __uint_as_float(v[e]);
                }
            }
            const int tok = c.tok0 + i * Gm::kSub;
            const int nvalid = min(Gm::kSub, c.tok1 - tok);
            const bool partial = nvalid < Gm::kSub;
            float alpha = 1.f;
            bool need = false;
            uint32_t hi[16], lo[16];
            if (quarter_active) {
                if (partial || tok + Gm::kSub > c.L - p.q_len + 1) {
                    const int lim = min(nvalid, vis - tok) - 32 * h;   // in this warp's tokens
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (e >= lim) t[e] = -INFINITY;
                }
                float mx = -INFINITY;
#pragma unroll
                for (int e = 0; e < 32; ++e) mx = fmaxf(mx, t[e]);
                // the stage's max over both token halves, identical in both warps
                // (double-buffered by stage parity: the partner has read the
                // previous use of a slot before this warp passes the next exchange)
                float* xm = xmax + (i & 1) * 256;
                xm[h * 128 + r] = mx;
                __syncwarp();
                if (lane == 0) mbar_arrive(b_pair);
                ok = __all_sync(kFull, wait_or_flag(b_pair, i & 1));
                if (!ok) break;
                mx = fmaxf(mx, xm[(h ^ 1) * 128 + r]) * sc;   // raw scores: sc > 0 keeps the max
                need = mx > m_run + 8.f;       // also true for the first finite max
                if (need) {
                    alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - mx);
                    l_run *= alpha;
                    m_run = mx;
                }
                const float mu = m_run == -INFINITY ? 0.f : m_run;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float p0 = fast_exp2(fmaf(t[2 * e], sc, -mu));
                    const float p1 = fast_exp2(fmaf(t[2 * e + 1], sc, -mu));
                    l_run += p0 + p1;
                    float k0, k1, d0, d1;
                    hi[e] = Mma<T>::pack(p0, p1, k0, k1);
                    lo[e] = Mma<T>::pack(p0 - k0, p1 - k1, d0, d1);
                }
            }
            if (quarter_active) {
                // this warp's 32 tokens: hi in its first 16 columns, lo in the next 16
                const uint32_t pa = tmem_p + lane_base + 64u * buf + 32u * h;
                tmem_st16(pa, hi);
                tmem_st16(pa + 16u, lo);
            }
            if (i > 0 && quarter_active && __any_sync(kFull, need)) {
                // O is rescaled once PV of stage i - 1 is done with it
                const bool done = __all_sync(kFull, wait_or_flag(b_o_done + 8u * (buf ^ 1), ((i - 1) >> 1) & 1));
                if (done) {
                    tc_fence_after();
                    // this warp's half of the column's O row
#pragma unroll 1
                    for (int q = 0; q < 4; ++q) {
                        uint32_t v[16];
                        const uint32_t ta = tmem_o + lane_base + 64u * h + 16u * q;
                        tmem_ld16(ta, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st16(ta, v);
                    }
                }
                ok = done;
            }
            tmem_wait_st();
            if (!ok) break;
            if (partial) {
                // V rows past the end hold whatever the cache holds there; P is 0
                // for them, but 0 * NaN would still poison PV
                uint8_t* vb = c.smem + (i % kRing) * Gm::kStageBytes + 2 * kHalfBytes;
                for (int idx = threadIdx.x; idx < (Gm::kSub - nvalid) * 16; idx += kSoftmaxThreads) {
                    const int row = nvalid + (idx >> 4), ch = idx & 15;
                    *reinterpret_cast<uint4*>(vb + (ch >> 3) * kHalfBytes + row * 128 + ((ch & 7) << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_p_full + 8u * buf);
        }
        if (ok && n_sub > 0) {   // the last PV done (it completes after every earlier one)
            ok = __all_sync(kFull, wait_or_flag(b_o_done + 8u * ((n_sub - 1) & 1), ((n_sub - 1) >> 1) & 1));
            tc_fence_after();
        }
        if (!ok) *c.cons_abort = 1;
        xsum[h * 128 + r] = l_run;
        named_sync(1, kSoftmaxThreads);
        if (*c.cons_abort == 0 && quarter_active) {
            // the column's state (u, m, l), or out / lse directly with one split;
            // this warp writes dims 64 h .. 64 h + 63
            const float l_col = xsum[r] + xsum[128 + r];
            const int64_t row = real ? (static_cast<int64_t>(c.b) * p.q_len + r / p.group) * p.n_q_heads +
                                           c.kvh * p.group + r % p.group
                                     : 0;
            const float m_out = m_run == -INFINITY ? -INFINITY : m_run * kLn2;
            const bool empty = m_out == -INFINITY || !(l_col > 0.f);
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t v[16];
                if (n_sub > 0) {
                    tmem_ld16(tmem_o + lane_base + 64u * h + 16u * q, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = 0u;
                }
                if (!real) continue;
                const int d0 = 64 * h + 16 * q;
                if (p.direct) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float o = empty ? 0.f : (__uint_as_float(v[e]) * p.v_scale) / l_col;
                        const int64_t oi = row * kHeadDim + d0 + e;
                        if (p.out_dtype == 2)
                            static_cast<float*>(p.out)[oi] = o;
                        else if (p.out_dtype == 0)
                            static_cast<__half*>(p.out)[oi] = __float2half_rn(o);
                        else
                            static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
                    }
                } else {
                    float4* dst = reinterpret_cast<float4*>(p.ws_u + (row * S + c.split) * kHeadDim + d0);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_float4(__uint_as_float(v[4 * e]) * p.v_scale, __uint_as_float(v[4 * e + 1]) * p.v_scale,
                                             __uint_as_float(v[4 * e + 2]) * p.v_scale, __uint_as_float(v[4 * e + 3]) * p.v_scale);
                }
            }
            if (real && h == 0) {
                if (p.direct) {
                    if (p.lse != nullptr) p.lse[row] = empty ? -INFINITY : m_out + logf(l_col);
                } else {
                    p.ws_m[row * S + c.split] = m_out;
                    p.ws_l[row * S + c.split] = l_col;
                }
            }
        }
    }
    // every tensor-memory user is done (the MMA thread waited for its last commit)
    tc_fence_before();
    named_sync(2, kSoftmaxThreads + 32);
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// tcgen05 variant for 17-64 columns (KIND 32).  Every tcgen05.mma costs the
// tensor pipe about the same time up to N = 128, so this variant fills the
// M = 128 rows twice over instead of leaving half of them empty:
//   Q rows 64 + c repeat rows c, so S lanes 64 + c repeat the scores of column c;
//   P rows 0..63 hold the hi parts of the columns' weights, rows 64..127 the lo parts,
//   and one MMA per 16 tokens accumulates O rows c (hi) and 64 + c (lo) together.
// PV takes 4 MMAs per stage instead of 8, and the result is O[c] = O[c] + O[64 + c]
// at the end.  Each column is served by four softmax warps (both lane quarters
// that hold its scores, two warps each), each taking 16 of a stage's 64 tokens;
// the four exchange their maxima every stage, so all four track the same
// running max and each rescales its own O rows when it moves.  P is written to
// shared memory (K-major, 128-byte swizzle), double-buffered by stage parity.
// Shared memory: 4-stage ring (128 KB), Q (32 KB), P (2 x 16 KB), the
// exchange and the tcgen05 barriers (4 KB).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(Geo<32>::kThreads, 1)
    fd_split_umma64_kernel(const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
    using Gm = Geo<32>;
    constexpr int kRing = Gm::kRing;
    constexpr int kSoftmaxThreads = Gm::kWarps * 32;   // 256
    constexpr uint32_t kTmemCols = 256;       // S [0, 128) double-buffered by stage parity, O [128, 256)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    SplitCtx c;
    split_begin<32>(c, smem, p, &tmK, &tmV);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.n_splits;
    const int n_sub = c.n_sub;
    uint8_t* sQ = smem + Gm::kOffExtra;       // two halves [128 x 64 dims]
    uint8_t* sP = sQ + 2 * 16384;             // [stage parity][128 rows x 64 tokens]
    // the exchange: stage maxima [stage parity][token quarter][column], sums [token quarter][column]
    float* xmax = reinterpret_cast<float*>(sP + 2 * 16384);
    float* xsum = xmax + 512;
    // mbarriers, [2] by stage parity unless noted
    const uint32_t b_grp0 = smem_u32(xsum + 256);   // [2], one per column group: one arrival per warp of its four
    const uint32_t b_s_full = b_grp0 + 16;    // one arrival (MMA commit): S written
    const uint32_t b_p_full = b_grp0 + 48;    // one arrival per softmax warp: P written (and O rescaled)
    const uint32_t b_o_done = b_grp0 + 64;    // one arrival (MMA commit): PV done
    const uint32_t b_drain = b_grp0 + 80;     // single, one arrival (MMA commit): every MMA done
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(xsum + 256 + 22);   // b_grp0 + 88
    if (threadIdx.x == 0) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            mbar_init(b_grp0 + 8u * b, 4);
            mbar_init(b_s_full + 8u * b, 1);
            mbar_init(b_p_full + 8u * b, Gm::kWarps);
            mbar_init(b_o_done + 8u * b, 1);
        }
        mbar_init(b_drain, 1);
        fence_barrier_init();
    }
    __syncthreads();   // every barrier is initialised
    if (warp == Gm::kWarps) {   // the producer streams at once; Q and tensor memory follow
        produce<32>(c, &tmK, &tmV, lane);
        return;
    }
    if (threadIdx.x < 128) {
        // Q tile: rows r and 64 + r are column r of the group (zeros past the columns)
        const int r = threadIdx.x;
        bool real;
        const T* qrow = q_row<T>(c, r & 63, real);
        const uint4* src = reinterpret_cast<const uint4*>(qrow);
#pragma unroll 4
        for (int ch = 0; ch < 16; ++ch) {
            const uint4 v = real ? __ldg(src + ch) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(sQ + (ch >> 3) * 16384 + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
    }
    if (warp == 0) tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    tc_fence_before();
    named_sync(3, kSoftmaxThreads + 32);   // the softmax warps and the MMA warp
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_o = tmem + 128;

    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;

    if (warp == Gm::kWarps + 1) {
        // ---- MMA issue (one thread): S of stage i + 1 goes out before PV of stage i.
        // Each descriptor is built once and offset by constants (the start address
        // is the low field, in 16-byte units, and no operand crosses 256 KB).
        // Buffer reuse needs no waits of its own: S of stage i + 1 overwrites
        // the scores of stage i - 1, which the softmax read before it handed
        // over P of stage i - 1 (waited for before PV of stage i - 1); and the
        // commit that signals S of stage i completes only after every earlier
        // MMA, PV of stage i - 2 included, so the softmax may then overwrite
        // that stage's P buffer.
        if (lane == 0) {
            const uint32_t id_s = umma_idesc_f16(128, 64, kBf16, false);
            const uint32_t id_o = umma_idesc_f16(128, 128, kBf16, true);
            const uint64_t dq = umma_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dp0 = umma_desc_sw128(smem_u32(sP), 16, 1024);
            const uint64_t dk0 = umma_desc_sw128(smem_u32(c.smem), 16, 1024);
            const uint64_t dv0 = umma_desc_sw128(smem_u32(c.smem + 2 * kHalfBytes), static_cast<uint32_t>(kHalfBytes), 1024);
            constexpr uint32_t kStageUnits = Gm::kStageBytes >> 4;
            auto issue_s = [&](int i) {
                const uint64_t dk = dk0 + static_cast<uint32_t>(i % kRing) * kStageUnits;
                const uint32_t d = tmem + 64u * static_cast<uint32_t>(i & 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {   // 16 dims per MMA: 32 bytes inside a 128-byte row
                    const uint32_t q_off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                    const uint32_t k_off = ((kk >> 2) * static_cast<uint32_t>(kHalfBytes) + (kk & 3) * 32u) >> 4;
                    umma_f16(d, dq + q_off, dk + k_off, id_s, kk > 0);
                }
                umma_commit(b_s_full + 8u * static_cast<uint32_t>(i & 1));
            };
            bool ok = true;
            if (n_sub > 0) {
                ok = wait_or_flag(c.full_bar(0), 0);
                if (ok) {
                    tc_fence_after();
                    issue_s(0);
                }
            }
            for (int i = 0; ok && i < n_sub; ++i) {
                if (i + 1 < n_sub) {
                    const int j = i + 1;
                    ok = wait_or_flag(c.full_bar(j % kRing), (j / kRing) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(j);
                }
                ok = wait_or_flag(b_p_full + 8u * (i & 1), (i >> 1) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dv = dv0 + static_cast<uint32_t>(i % kRing) * kStageUnits;
                const uint64_t dp = dp0 + static_cast<uint32_t>(i & 1) * (16384u >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)   // 16 tokens per MMA: hi and lo rows together
                    umma_f16(tmem_o, dp + ((kk * 32u) >> 4), dv + ((kk * 2048u) >> 4), id_o, i > 0 || kk > 0);
                umma_commit(b_o_done + 8u * static_cast<uint32_t>(i & 1));
                umma_commit(c.empty_bar(i % kRing));
            }
            if (!ok) {
                *c.cons_abort = 1;
                *c.abort_flag = 1;
            }
            umma_commit(b_drain);              // tensor memory is freed only after this
            wait_or_flag(b_drain, 0);
        }
        __syncwarp();
    } else {
        // ---- softmax warps.  Warp w reaches tensor-memory lanes 32 q .. +31,
        // q = w % 4: the scores (and O rows) of columns col = 32 (q % 2) + lane,
        // the hi rows for q < 2 and the lo rows for q >= 2.  Its tokens are
        // 16 tq .. 16 tq + 15 of each stage, tq = 2 (q / 2) + w / 4, and its O
        // dims are 64 (w / 4) .. +63.  Column group g = q % 2 has the four warps
        // g, g + 2, g + 4, g + 6.
        const int q = warp & 3, hw = warp >> 2;
        const int g = q & 1, side = q >> 1;
        const int col = 32 * g + lane;
        const int tq = 2 * side + hw;
        const bool group_active = 32 * g < p.cols;
        const bool real = col < p.cols;
        const int vis = real ? c.L - p.q_len + 1 + col / p.group : c.L;
        // scores stay raw until the exponent: sc (log2(e) / sqrt(d), a 16-bit
        // cache) is positive, so maxima of raw scores scale to maxima of scaled ones
        const float sc = p.score_scale_log2;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t b_grp = b_grp0 + 8u * g;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int i = 0; i < n_sub; ++i) {
            const int buf = i & 1;
            ok = __all_sync(kFull, wait_or_flag(b_s_full + 8u * buf, (i >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
            float t[16];
            if (group_active) {
                uint32_t v[16];
                tmem_ld16(tmem + lane_base + 64u * buf + 16u * tq, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) t[e] = __uint_as_float(v[e]);
            }
            const int tok = c.tok0 + i * Gm::kSub;
            const int nvalid = min(Gm::kSub, c.tok1 - tok);
            const bool partial = nvalid < Gm::kSub;
            float alpha = 1.f;
            bool need = false;
            uint32_t hi[8], lo[8];
            if (group_active) {
                if (partial || tok + Gm::kSub > c.L - p.q_len + 1) {
                    const int lim = min(nvalid, vis - tok) - 16 * tq;   // in this warp's tokens
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (e >= lim) t[e] = -INFINITY;
                }
                float mx = -INFINITY;
#pragma unroll
                for (int e = 0; e < 16; ++e) mx = fmaxf(mx, t[e]);
                // the stage's max over the four token quarters, identical in the
                // group's four warps (double-buffered by stage parity: every warp
                // has read a slot before the group passes its next exchange)
                float* xm = xmax + (i & 1) * 256;
                xm[tq * 64 + col] = mx;
                __syncwarp();
                if (lane == 0) mbar_arrive(b_grp);
                ok = __all_sync(kFull, wait_or_flag(b_grp, i & 1));
                if (!ok) break;
                mx = fmaxf(fmaxf(xm[col], xm[64 + col]), fmaxf(xm[128 + col], xm[192 + col])) * sc;
                need = mx > m_run + 8.f;       // also true for the first finite max
                if (need) {
                    alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - mx);
                    l_run *= alpha;
                    m_run = mx;
                }
                const float mu = m_run == -INFINITY ? 0.f : m_run;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float p0 = fast_exp2(fmaf(t[2 * e], sc, -mu));
                    const float p1 = fast_exp2(fmaf(t[2 * e + 1], sc, -mu));
                    l_run += p0 + p1;
                    float k0, k1, d0, d1;
                    hi[e] = Mma<T>::pack(p0, p1, k0, k1);
                    lo[e] = Mma<T>::pack(p0 - k0, p1 - k1, d0, d1);
                }
            }
            if (group_active) {
                // tokens 16 tq .. +15 = chunks 2 tq, 2 tq + 1 of rows col (hi) and 64 + col (lo)
                uint8_t* pb = sP + buf * 16384;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int chunk = 2 * tq + h2;
                    const int rh = col, rl = 64 + col;
                    *reinterpret_cast<uint4*>(pb + rh * 128 + ((chunk ^ (rh & 7)) << 4)) =
                        make_uint4(hi[4 * h2], hi[4 * h2 + 1], hi[4 * h2 + 2], hi[4 * h2 + 3]);
                    *reinterpret_cast<uint4*>(pb + rl * 128 + ((chunk ^ (rl & 7)) << 4)) =
                        make_uint4(lo[4 * h2], lo[4 * h2 + 1], lo[4 * h2 + 2], lo[4 * h2 + 3]);
                }
            }
            if (i > 0 && group_active && __any_sync(kFull, need)) {
                // O is rescaled once PV of stage i - 1 is done with it: this warp's
                // 32 O rows, dims 64 hw .. +63
                ok = __all_sync(kFull, wait_or_flag(b_o_done + 8u * (buf ^ 1), ((i - 1) >> 1) & 1));
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int qq = 0; qq < 4; ++qq) {
                    uint32_t v[16];
                    const uint32_t ta = tmem_o + lane_base + 64u * hw + 16u * qq;
                    tmem_ld16(ta, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st16(ta, v);
                }
                tmem_wait_st();
            }
            if (partial) {
                // V rows past the end hold whatever the cache holds there; P is 0
                // for them, but 0 * NaN would still poison PV
                uint8_t* vb = c.smem + (i % kRing) * Gm::kStageBytes + 2 * kHalfBytes;
                for (int idx = threadIdx.x; idx < (Gm::kSub - nvalid) * 16; idx += kSoftmaxThreads) {
                    const int row = nvalid + (idx >> 4), ch = idx & 15;
                    *reinterpret_cast<uint4*>(vb + (ch >> 3) * kHalfBytes + row * 128 + ((ch & 7) << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_p_full + 8u * buf);
        }
        if (ok && n_sub > 0) {   // the last PV done (it completes after every earlier one)
            ok = __all_sync(kFull, wait_or_flag(b_o_done + 8u * ((n_sub - 1) & 1), ((n_sub - 1) >> 1) & 1));
            tc_fence_after();
        }
        if (!ok) *c.cons_abort = 1;
        xsum[tq * 64 + col] = l_run;
        // the lo rows of O go through shared memory (ring stage 0, idle now):
        // [64 columns][128 dims] fp32
        float* olo = reinterpret_cast<float*>(c.smem);
        if (ok && side == 1 && group_active && n_sub > 0) {
#pragma unroll 1
            for (int qq = 0; qq < 4; ++qq) {
                uint32_t v[16];
                tmem_ld16(tmem_o + lane_base + 64u * hw + 16u * qq, v);
                tmem_wait_ld();
                float4* dst = reinterpret_cast<float4*>(olo + col * kHeadDim + 64 * hw + 16 * qq);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                         __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
            }
        }
        named_sync(1, kSoftmaxThreads);
        if (*c.cons_abort == 0 && side == 0 && group_active) {
            // the column's state (u, m, l), or out / lse directly with one split;
            // this warp writes dims 64 hw .. 64 hw + 63
            const float l_col = (xsum[col] + xsum[64 + col]) + (xsum[128 + col] + xsum[192 + col]);
            const int64_t row = real ? (static_cast<int64_t>(c.b) * p.q_len + col / p.group) * p.n_q_heads +
                                           c.kvh * p.group + col % p.group
                                     : 0;
            const float m_out = m_run == -INFINITY ? -INFINITY : m_run * kLn2;
            const bool empty = m_out == -INFINITY || !(l_col > 0.f);
#pragma unroll 1
            for (int qq = 0; qq < 4; ++qq) {
                uint32_t v[16];
                if (n_sub > 0) {
                    tmem_ld16(tmem_o + lane_base + 64u * hw + 16u * qq, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = 0u;
                }
                if (!real) continue;
                const int d0 = 64 * hw + 16 * qq;
                float o[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    o[e] = n_sub > 0 ? (__uint_as_float(v[e]) + olo[col * kHeadDim + d0 + e]) * p.v_scale : 0.f;
                if (p.direct) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float y = empty ? 0.f : o[e] / l_col;
                        const int64_t oi = row * kHeadDim + d0 + e;
                        if (p.out_dtype == 2)
                            static_cast<float*>(p.out)[oi] = y;
                        else if (p.out_dtype == 0)
                            static_cast<__half*>(p.out)[oi] = __float2half_rn(y);
                        else
                            static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(y);
                    }
                } else {
                    float4* dst = reinterpret_cast<float4*>(p.ws_u + (row * S + c.split) * kHeadDim + d0);
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
                }
            }
            if (real && hw == 0) {
                if (p.direct) {
                    if (p.lse != nullptr) p.lse[row] = empty ? -INFINITY : m_out + logf(l_col);
                } else {
                    p.ws_m[row * S + c.split] = m_out;
                    p.ws_l[row * S + c.split] = l_col;
                }
            }
        }
    }
    // every tensor-memory user is done (the MMA thread waited for its last commit)
    tc_fence_before();
    named_sync(2, kSoftmaxThreads + 32);
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Raises the dynamic shared-memory limit of `kern` to `smem`, once per CUDA
// context (the attribute belongs to the context's copy of the kernel).  With
// no readable context id it is set on every launch; the call is idempotent.
template <typename Kern>
static cudaError_t allow_smem(Kern kern, size_t smem, std::atomic<unsigned long long>& configured_ctx) {
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && configured_ctx.load(std::memory_order_acquire) == ctx) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess && ctx != 0) configured_ctx.store(ctx, std::memory_order_release);
    return e;
}

template <typename T, int KIND>
static cudaError_t launch_split_t(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                  const SplitParams& p, int batch, int n_kv_heads,
                                  cudaStream_t stream) {
    auto kern = fd_split_kernel<T, KIND>;
    const size_t smem = Geo<KIND>::kSmem;
    static std::atomic<unsigned long long> configured_ctx{0};
    cudaError_t e = allow_smem(kern, smem, configured_ctx);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(p.n_splits * p.col_blocks, n_kv_heads, batch),
                      dim3(Geo<KIND>::kThreads), smem, stream, tmK, tmV, p);
}

template <typename T, int KIND>
static cudaError_t launch_split_umma(const CUtensorMap& tmK, const CUtensorMap& tmV, const SplitParams& p,
                                    int batch, int n_kv_heads, cudaStream_t stream);

template <typename T>
static cudaError_t launch_split_dt(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                   const SplitParams& p, bool fp8, bool cuda_cores, int batch,
                                   int n_kv_heads, cudaStream_t stream) {
    if (use_umma(fp8, cuda_cores, p.cols))
        return p.cols <= 64 ? launch_split_umma<T, 32>(tmK, tmV, p, batch, n_kv_heads, stream)
                            : launch_split_umma<T, 31>(tmK, tmV, p, batch, n_kv_heads, stream);
    if (fp8)
        return p.cols <= 8 ? launch_split_t<T, 21>(tmK, tmV, p, batch, n_kv_heads, stream)
                           : launch_split_t<T, 22>(tmK, tmV, p, batch, n_kv_heads, stream);
    if (cuda_cores) {
        switch (p.group) {
            case 1: return launch_split_t<T, 11>(tmK, tmV, p, batch, n_kv_heads, stream);
            case 2: return launch_split_t<T, 12>(tmK, tmV, p, batch, n_kv_heads, stream);
            case 4: return launch_split_t<T, 14>(tmK, tmV, p, batch, n_kv_heads, stream);
            case 8: return launch_split_t<T, 18>(tmK, tmV, p, batch, n_kv_heads, stream);
        }
        return cudaErrorInvalidValue;
    }
    return p.cols <= 8 ? launch_split_t<T, 1>(tmK, tmV, p, batch, n_kv_heads, stream)
                       : launch_split_t<T, 2>(tmK, tmV, p, batch, n_kv_heads, stream);
}

template <typename T, int KIND>
static cudaError_t launch_split_umma(const CUtensorMap& tmK, const CUtensorMap& tmV, const SplitParams& p,
                                    int batch, int n_kv_heads, cudaStream_t stream) {
    auto kern = KIND == 32 ? fd_split_umma64_kernel<T> : fd_split_umma_kernel<T>;
    const size_t smem = Geo<KIND>::kSmem;
    static std::atomic<unsigned long long> configured_ctx{0};
    cudaError_t e = allow_smem(kern, smem, configured_ctx);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(p.n_splits * p.col_blocks, n_kv_heads, batch),
                      dim3(Geo<KIND>::kThreads), smem, stream, tmK, tmV, p);
}

cudaError_t launch_split(const CUtensorMap& tmK, const CUtensorMap& tmV, const SplitParams& p,
                         int q_dtype, bool fp8, bool cuda_cores, int batch, int n_kv_heads,
                         cudaStream_t stream) {
    if (q_dtype == 0)
        return launch_split_dt<__half>(tmK, tmV, p, fp8, cuda_cores, batch, n_kv_heads, stream);
    return launch_split_dt<__nv_bfloat16>(tmK, tmV, p, fp8, cuda_cores, batch, n_kv_heads, stream);
}

cudaError_t read_status(unsigned* value, cudaStream_t stream, bool clear) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_fd_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    if (clear) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_fd_status, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace fdk
