// fd_split.cu -- the split kernel of split-KV decode attention on sm_103a.
//
// One CTA per (KV split, KV head, sequence) (the fp8 kernel with up to 8
// columns: two per CTA once splits outnumber SMs).  It streams the split's K/V
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
//    generation tensor cores (fd_split_umma_kernel): a persistent grid of at
//    most one CTA per SM serves the splits in turn, each holding every column
//    as the M rows of tcgen05 MMAs with S and O accumulated in tensor memory,
//    fed by the same TMA stages laid out in pairs.
//  - Before its launch wait, a CTA of the warp-MMA kernels prefetches the
//    first tokens of its split into L2, so its first stages overlap the tail
//    of the kernel before it in the stream.
//  - Scores are kept in base 2: t = (q.k) * log2(e)/sqrt(D), p = 2^(t - m).
//    The workspace m is converted back to natural units of s.
//  - Every mbarrier wait is bounded (2 s of wall time); on timeout the kernel
//    records kStatusTimeout in the device status word, drains its own copies
//    (bounded) and returns without writing states.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>

#include "../../include/fd.h"
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
// end-of-split merge area (reuses stage memory once every stage is consumed):
// a row of kAccStride floats per (warp, column), dims d at d + skew * (d / 32)
// (skew 2 for the tensor-core consumers, 0 for the CUDA-core one), so that the
// warps' fragment stores meet distinct banks (rows of 128 put the lanes of a
// store on 4-8 banks) while the merge still reads each row contiguously
constexpr int kCols = 16;                                         // (query, head) columns per CTA
constexpr int kAccStride = 164;                                   // 128 dims + 6 of skew, = 4 mod 32
constexpr int kOffWAcc = 0;                                       // [warps][16][kAccStride] f32
constexpr int kOffWM = kConsumerWarps * kCols * kAccStride * 4;   // [warps][16]
constexpr int kOffWL = kOffWM + kConsumerWarps * kCols * 4;       // [warps][16]
static_assert(kOffWL + kConsumerWarps * kCols * 4 <= kOffBars, "merge area must fit in the stages");

}  // namespace

// Geometry of each kernel variant (KIND, see Consumer below).  16-bit caches:
// four consumer warps, 3 stages of 64 tokens, each stage four [64 x 64-dim]
// boxes (the map above).  fp8 caches: two [rows x 128-dim] e4m3 boxes (K, V)
// per stage, read by the consumers straight into registers; with at most 8
// columns per CTA (KIND 21) six consumer warps take 96-token stages, 4 deep,
// otherwise (KIND 22) four take 64-token stages, 6 deep.  Either way the ring
// holds 96 KB, and two CTAs (or the two halves of a KIND 21 CTA that serves
// two splits) fit on an SM.
template <int KIND>
struct Geo {
    static constexpr bool kUmma = KIND == 31 || KIND == 32;    // tcgen05 consumers, see below
    static constexpr bool kF8 = KIND >= 20 && !kUmma;
    static constexpr int kWarps = KIND == 21 ? kConsumerWarpsF8 : kUmma ? 8 : kConsumerWarps;
    static constexpr int kSub = kUmma ? 64 : 16 * kWarps;      // tokens per stage
    static constexpr int kRing = KIND == 21 ? 4 : KIND == 22 ? 6 : kUmma ? 6 : kStages;
    static constexpr int kTile = kSub * 128;                   // one box of 128-byte rows
    static constexpr int kStageBytes = (kF8 ? 2 : 4) * kTile;
    // tcgen05: consecutive stages land side by side in pairs, so that one MMA
    // spans 128 tokens -- pair p holds four 16 KB regions (K low half, K high
    // half, V low, V high), each [128 tokens x 64 dims]; stage 2p writes rows
    // 0-63 of each region and stage 2p + 1 rows 64-127
    static constexpr bool kPairs = kUmma;
    static constexpr int kBoxStride = kPairs ? 2 * kTile : kTile;   // K lo -> K hi -> V lo -> V hi
    static __device__ __forceinline__ uint32_t stage_off(int st) {
        return kPairs ? static_cast<uint32_t>((st >> 1) * 4 * kBoxStride + (st & 1) * kTile)
                      : static_cast<uint32_t>(st * kStageBytes);
    }
    static constexpr int kOffExtra = kRing * kStageBytes;
    // tcgen05: KIND 32's exchange of O's lo rows (17 KB), then the softmax
    // exchange and the tcgen05 barriers (4 KB)
    static constexpr int kOloBytes = KIND == 32 ? 64 * 68 * 4 : 0;
    // + KIND 31's per-warp staging of states in the epilogue ([16][36] floats)
    static constexpr int kStgBytes = KIND == 31 ? 8 * 16 * 36 * 4 : 0;
    static constexpr int kExtraBytes = kUmma ? kOloBytes + kStgBytes + 4096 : 0;
    static constexpr int kOffBars = kOffExtra + kExtraBytes;   // full[kRing], empty[kRing]
    static constexpr bool kOwnMap = kF8 || kUmma;
    static_assert(!kUmma || kSub == fdk::kSub, "the tcgen05 variant streams the 16-bit stages");
    static constexpr int kOffFlag = (kOwnMap ? kOffBars + 128 : fdk::kOffFlag);
    static constexpr int kSmem = (kOwnMap ? kOffFlag + 16 : kSmemUsed) + 1024;   // + alignment slack
    // a CTA that serves two splits at once (see fd_split_kernel) gives each this much
    static constexpr int kSmemHalf = (kSmem - 1024 + 1023) / 1024 * 1024;
    // + one TMA producer warp (+ one MMA-issuing warp for tcgen05)
    static constexpr int kThreads = (kWarps + (kUmma ? 2 : 1)) * 32;
    static constexpr int kEmptyArrivals = kUmma ? 1 : kWarps;  // tcgen05: the MMA commit
    // end-of-split merge area in stage memory: acc [warps][16][128], m, l [warps][16]
    static constexpr int kOffWM = kWarps * kCols * kAccStride * 4;
    static constexpr int kOffWL = kOffWM + kWarps * kCols * 4;
    // per column, from the merge's first phase: state row, warp weights, m, l
    static constexpr int kOffCRow = (kOffWL + kWarps * kCols * 4 + 7) / 8 * 8;   // int64 [kCols]
    static constexpr int kOffCW = kOffCRow + kCols * 8;                          // [kCols][kWarps]
    static constexpr int kOffCM = kOffCW + kCols * kWarps * 4;                   // [kCols]
    static constexpr int kOffCL = kOffCM + kCols * 4;                            // [kCols]
    static constexpr int kAccSkew = KIND >= 11 && KIND <= 18 ? 0 : 2;   // see the merge area above
    static_assert(2 * kRing * 8 <= 128, "barriers must fit");
    static_assert(kOffCL + kCols * 4 <= kOffBars, "merge area must fit in the stages");
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
    int bar_id;                 // the consumer warps' named barrier (1, or 2 for a CTA's second half)

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
        const uint32_t dst = smem_u32(c.smem) + Gm::stage_off(st);
        const uint32_t bar = c.full_bar(st);
        constexpr uint32_t kBox = Gm::kBoxStride;
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
                tma_load_4d_hint(dst + 0 * kBox, tmK, bar, 0, tok, c.kvh, c.b, policy);
                tma_load_4d_hint(dst + 1 * kBox, tmK, bar, 64, tok, c.kvh, c.b, policy);
                tma_load_4d_hint(dst + 2 * kBox, tmV, bar, 0, tok, c.kvh, c.b, policy);
                tma_load_4d_hint(dst + 3 * kBox, tmV, bar, 64, tok, c.kvh, c.b, policy);
            }
        } else if (lane < nbox) {
            const int in_page = (tok + lane * rows) & (p.page_size - 1);
            const uint32_t off = static_cast<uint32_t>(lane * rows * 128);
            tma_load_4d_hint(dst + 0 * kBox + off, tmK, bar, 0, in_page, c.kvh, page, policy);
            tma_load_4d_hint(dst + 1 * kBox + off, tmK, bar, 64, in_page, c.kvh, page, policy);
            tma_load_4d_hint(dst + 2 * kBox + off, tmV, bar, 0, in_page, c.kvh, page, policy);
            tma_load_4d_hint(dst + 3 * kBox + off, tmV, bar, 64, in_page, c.kvh, page, policy);
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
    named_sync(c.bar_id, kConsumerWarps * 32);
    if (*c.cons_abort) return false;   // states are not written after a timeout
    float* wacc = reinterpret_cast<float*>(c.smem + kOffWAcc);
    float* wm = reinterpret_cast<float*>(c.smem + kOffWM);
    float* wl = reinterpret_cast<float*>(c.smem + kOffWL);
    if (owner && hw == 0) {
        wm[cw * kCols + g_lane] = m_run;
        wl[cw * kCols + g_lane] = l_run;
    }
#pragma unroll
    for (int g = 0; g < G; ++g)   // (no skew: whole rows of float4s)
        *reinterpret_cast<float4*>(wacc + (cw * kCols + g) * kAccStride + 4 * lane) =
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

// Margin of the lazy running max (log2 units): weights stay below 2^8.
constexpr float kLazyMax = 8.f;

// Online softmax (base 2) of TILES 16-token tiles for up to 8 * NB columns,
// and P^T of each tile as hi + lo B fragments of the PV MMAs.  s[t] holds tile
// t's S^T (C fragments); csc[j][e] is the base-2 score scale of the lane's
// column 8j + 2tig + e, which sees the keys before vis[j][e]; tile t starts at
// key tok[t] and has nvalid[t] rows.  Without `masked` every row is taken as
// visible to every column (a full tile and one query per sequence).  The
// running max moves at most once per call.
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
        // Lazy running max: it moves only when some score exceeds it by more
        // than kLazyMax (log2 units), so p stays below 2^kLazyMax; until then the
        // tile needs no max reduction across the lanes, only one vote.  Any
        // reference point gives the same state (u, m, l) up to rounding.
        float lmx[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            lmx[e] = -INFINITY;
#pragma unroll
            for (int x = 0; x < TILES; ++x) lmx[e] = fmaxf(lmx[e], fmaxf(t[x][e], t[x][e + 2]));
        }
        const bool move = __any_sync(kFull, lmx[0] > m[j][0] + kLazyMax || lmx[1] > m[j][1] + kLazyMax);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float mn = m[j][e];
            if (move) {   // warp-uniform
                float mx = lmx[e];
#pragma unroll
                for (int o = 4; o <= 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
                mn = fmaxf(mn, mx);
            }
            const float mu = mn == -INFINITY ? 0.f : mn;   // never -inf - -inf
            al[j][e] = move ? fast_exp2(m[j][e] - mu) : 1.f;
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

    named_sync(c.bar_id, kConsumerWarps * 32);
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
            for (int mb = 0; mb < 8; ++mb) {   // dims 16 mb + gid (+8): skew 2 * (mb / 2)
                float* row = wacc + (cw * kCols + col) * kAccStride + 16 * mb + 2 * (mb >> 1);
                row[gid] = acc[mb][j][e];
                row[gid + 8] = acc[mb][j][e + 2];
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

    named_sync(c.bar_id, Gm::kWarps * 32);
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
            for (int mb = 0; mb < 8; ++mb)   // dims 16 gid + 2 mb (+1): skew 2 * (gid / 2)
                *reinterpret_cast<float2*>(wacc + (cw * kCols + col) * kAccStride + 16 * gid + 2 * (gid >> 1) +
                                           2 * mb) = make_float2(acc[mb][j][e], acc[mb][j][e + 2]);
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

// Split `split` of S over L tokens: the tokens [tok0, tok1) of its share of
// the ceil(L / unit) units, the first L mod S shares one unit longer.
__device__ __forceinline__ void split_tokens(int L, int S, int unit, int split, int& tok0, int& tok1) {
    const int n_units = (L + unit - 1) / unit;
    const int base = n_units / S, rem = n_units % S;
    const int u_begin = split * base + (split < rem ? split : rem);
    const int u_count = base + (split < rem ? 1 : 0);
    tok0 = u_begin * unit;
    tok1 = min((u_begin + u_count) * unit, L);
}

// The token range of split `split` of sequence b (KV head kvh): the sequence
// cut into S balanced ranges of whole 16-token units (8 for 8-token pages), so
// no TMA box straddles a page and a paged cache splits exactly like a
// contiguous one.  `report`: this thread records an out-of-range length.
template <int KIND>
__device__ __forceinline__ void split_range(SplitCtx& c, int b, int kvh, int split, bool report) {
    const SplitParams& p = *c.p;
    c.b = b;
    c.kvh = kvh;
    c.split = split;
    int L = __ldg(p.seqlens + b);
    if (L < 0 || L > p.capacity) {
        if (report) raise_status(kStatusSeqlenBit);
        L = L < 0 ? 0 : p.capacity;
    }
    c.L = L;
    split_tokens(L, p.n_splits, p.split_unit, split, c.tok0, c.tok1);
    c.n_sub = c.tok1 > c.tok0 ? (c.tok1 - c.tok0 + Geo<KIND>::kSub - 1) / Geo<KIND>::kSub : 0;
}

// Tokens the L2 prefetch ahead of the launch wait covers per CTA: half the
// split, at most this many (measured: more delays the first stages).
constexpr int kPrefetchTokens = 256;

// Ahead of the launch wait: the first tokens of one split into L2, so that
// its first stages are served from L2 once the wait ends.  The length comes
// from a relaxed load, since the kernel before this one may still be writing
// it; a stale length only misplaces the prefetch, never a result (every load
// after the wait reads the length again).  Contiguous caches only: a block
// table is read only after the wait.
template <int KIND>
__device__ __forceinline__ void prefetch_split(const SplitParams& p, const CUtensorMap* tmK,
                                               const CUtensorMap* tmV, int b, int kvh, int split) {
    using Gm = Geo<KIND>;
    if (p.page_size != 0) return;
    int L = ld_relaxed_s32(p.seqlens + b);
    L = L < 0 ? 0 : (L > p.capacity ? p.capacity : L);
    int t0, t1;
    split_tokens(L, p.n_splits, p.split_unit, split, t0, t1);
    t1 = min(t1, t0 + min(kPrefetchTokens, max(Gm::kSub, (t1 - t0) / 2)));
#pragma unroll 1
    for (int t = t0; t < t1; t += Gm::kSub) {
        if (Gm::kF8) {
            tma_prefetch_4d(tmK, 0, t, kvh, b);
            tma_prefetch_4d(tmV, 0, t, kvh, b);
        } else {
            tma_prefetch_4d(tmK, 0, t, kvh, b);
            tma_prefetch_4d(tmK, 64, t, kvh, b);
            tma_prefetch_4d(tmV, 0, t, kvh, b);
            tma_prefetch_4d(tmV, 64, t, kvh, b);
        }
    }
}

// The start every split kernel shares: the context, the ring's barriers and
// the programmatic-dependent-launch wait.
template <int KIND>
__device__ __forceinline__ void split_setup(SplitCtx& c, uint8_t* smem, const SplitParams& p,
                                            const CUtensorMap* tmK, const CUtensorMap* tmV,
                                            int pf_b, int pf_kvh, int pf_split, int tid = threadIdx.x,
                                            int half = 0) {
    using Gm = Geo<KIND>;
    constexpr int kRing = Gm::kRing;
    c.stages = kRing;
    c.p = &p;
    c.smem = smem;
    c.cb = 0;
    c.bar_id = 1 + half;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    c.bar0 = smem_u32(smem + Gm::kOffBars);
    c.abort_flag = reinterpret_cast<volatile int*>(smem + Gm::kOffFlag);
    c.cons_abort = reinterpret_cast<volatile int*>(smem + Gm::kOffFlag + 4);
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < kRing; ++s) {
            mbar_init(c.full_bar(s), 1);
            mbar_init(c.empty_bar(s), Gm::kEmptyArrivals);
        }
        *c.abort_flag = 0;
        *c.cons_abort = 0;
        *reinterpret_cast<volatile int*>(smem + Gm::kOffFlag + 8) = 0;   // the tcgen05 softmax's own flag
        fence_barrier_init();
    }
    if (warp == Gm::kWarps && lane == 0) {
        prefetch_tensormap(tmK);
        prefetch_tensormap(tmV);
        // (pf_b < 0: a column block after the first, whose sibling prefetches)
        if (pf_b >= 0) prefetch_split<KIND>(p, tmK, tmV, pf_b, pf_kvh, pf_split);
    }
    // Programmatic dependent launch: let the combine kernel that follows get
    // resident now, and wait for whatever preceded this kernel in the stream
    // to finish (and its writes to land) before reading any input.
    grid_dependency_trigger();
    grid_dependency_wait();
}

// split_setup and the token range of the split of virtual block vx (x index
// of the grid (n_splits * col_blocks, n_kv_heads, batch); vx < 0: none), the
// column blocks of one split adjacent, so they run together and the later
// readers of the split's K/V find it in L2.
template <int KIND>
__device__ __forceinline__ void split_begin(SplitCtx& c, uint8_t* smem, const SplitParams& p,
                                            const CUtensorMap* tmK, const CUtensorMap* tmV, int tid,
                                            int half, int vx) {
    split_setup<KIND>(c, smem, p, tmK, tmV, vx >= 0 && vx % p.col_blocks == 0 ? static_cast<int>(blockIdx.z) : -1,
                      blockIdx.y, vx / p.col_blocks, tid, half);
    if (vx < 0) return;
    split_range<KIND>(c, blockIdx.z, blockIdx.y, vx / p.col_blocks, tid == 0 && vx == 0 && blockIdx.y == 0);
    c.cb = vx % p.col_blocks;
}

// HALVES = 2: the CTA serves two splits at once, each with its own half of
// the threads, shared memory, barriers and named barrier, so that every SM
// holding work holds two splits (splits are otherwise placed one per SM
// first, and where the consumers cannot keep up with HBM alone, the SMs left
// with one split finish early while those with two set the kernel's time).
template <typename T, int KIND, int HALVES>
__global__ void __launch_bounds__(Geo<KIND>::kThreads * HALVES, HALVES == 1 ? 2 : 1)
    fd_split_kernel(const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
    using Gm = Geo<KIND>;
    constexpr int kWarps = Gm::kWarps;
    extern __shared__ uint8_t smem_raw[];
    const int half = HALVES == 1 ? 0 : static_cast<int>(threadIdx.x) / Gm::kThreads;
    const int tid = static_cast<int>(threadIdx.x) - half * Gm::kThreads;
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023)) + half * Gm::kSmemHalf;
    const int vx = static_cast<int>(blockIdx.x) * HALVES + half;
    const bool idle = vx >= p.n_splits * p.col_blocks;   // the second half of the last CTA
    SplitCtx c;
    split_begin<KIND>(c, smem, p, &tmK, &tmV, tid, half, idle ? -1 : vx);
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int S = p.n_splits;
    __syncthreads();
    if (idle) return;

    if (warp == kWarps) {
        produce<KIND>(c, &tmK, &tmV, lane);
        return;
    }

    if (!Consumer<T, KIND>::run(c, warp, lane)) return;
    named_sync(c.bar_id, kWarps * 32);

    // ---- merge the consumer warps' states of each column and write the split's
    // state, in two phases so that the columns' dependent chains run side by
    // side: one thread per column takes the max, the warps' weights and l
    // (and the state row), then one thread per dim sums its u over the warps
    const float* wacc = reinterpret_cast<const float*>(smem);
    const float* wm = reinterpret_cast<const float*>(smem + Gm::kOffWM);
    const float* wl = reinterpret_cast<const float*>(smem + Gm::kOffWL);
    int64_t* crow = reinterpret_cast<int64_t*>(smem + Gm::kOffCRow);
    float* cw = reinterpret_cast<float*>(smem + Gm::kOffCW);
    float* cm = reinterpret_cast<float*>(smem + Gm::kOffCM);
    float* cl = reinterpret_cast<float*>(smem + Gm::kOffCL);
    const int ncols = min(kCols, p.cols - c.cb * kCols);
    if (tid < ncols) {
        const int col = tid;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kCols + col]);
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float mw = wm[w * kCols + col];
            const float e = (M == -INFINITY || mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
            cw[col * kWarps + w] = e;
            l = fmaf(e, wl[w * kCols + col], l);
        }
        cm[col] = M == -INFINITY ? -INFINITY : M * kLn2;
        cl[col] = l;
        const int n = c.cb * kCols + col;
        const int i = n / p.group, g = n % p.group;
        crow[col] = (static_cast<int64_t>(c.b) * p.q_len + i) * p.n_q_heads + c.kvh * p.group + g;
    }
    named_sync(c.bar_id, kWarps * 32);
    if (tid >= kHeadDim) return;   // one thread per dim below
    const int d = tid;   // 0 .. 127
    const int dd = d + Gm::kAccSkew * (d >> 5);
#pragma unroll 1
    for (int col = 0; col < ncols; ++col) {
        float u = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) u = fmaf(cw[col * kWarps + w], wacc[(w * kCols + col) * kAccStride + dd], u);
        const float m_out = cm[col], l = cl[col];
        const int64_t row = crow[col];
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

// Work item `item` of the tcgen05 kernel: split item % S of KV head
// (item / S) % n_kv_heads of sequence item / (S n_kv_heads) -- the order of
// the other split kernels' grid.
template <int KIND>
__device__ __forceinline__ void set_item(SplitCtx& c, int item, bool report) {
    const SplitParams& p = *c.p;
    const int S = p.n_splits;
    const int rest = item / S;
    split_range<KIND>(c, rest / p.n_kv_heads, rest % p.n_kv_heads, item - rest * S, report);
}

// ---------------------------------------------------------------------------
// Producer of the tcgen05 kernel: streams the stages of every work item
// (split) the CTA serves, back to back, into the ring in pairs of slots.  An
// item with an odd number of stages leaves the second slot of its last pair
// unfilled (its full barrier gets a plain arrival), so every pair starts on an
// even slot and each slot's barrier phases stay in step.
// ---------------------------------------------------------------------------
template <int KIND>
__device__ __forceinline__ void produce_pairs(const SplitCtx& c0, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV, int lane, int n_items) {
    using Gm = Geo<KIND>;
    constexpr int kRing = Gm::kRing;
    constexpr uint32_t kBox = Gm::kBoxStride;
    const SplitParams& p = *c0.p;
    const uint64_t policy = policy_evict_first();   // K/V are read once
    const bool paged = p.page_size != 0;
    const int rows = paged ? min(kPagedBoxRows, p.page_size) : kSub;   // tokens per box
    const int nbox = kSub / rows;                                        // boxes per half per stage
    const int first = p.drop_first_stage ? 1 : 0;   // test hook: slot 0 is never filled
    int gs = 0;                                     // slots used so far, over all items
    bool stop = false;
    for (int item = blockIdx.x; item < n_items && !stop; item += gridDim.x) {
        SplitCtx c = c0;
        set_item<KIND>(c, item, false);
        const int n_slots = 2 * ((c.n_sub + 1) >> 1);
        // physical page of box `lane` of stage i (paged); -1 reads zeros
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
#pragma unroll 1
        for (int i = 0; i < n_slots; ++i, ++gs) {
            const int st = gs % kRing;
            if (gs >= kRing) {
                const bool ok = wait_or_flag(c.empty_bar(st), ((gs / kRing) - 1) & 1);
                if (!__all_sync(kFull, ok)) *c.abort_flag = 1;
            }
            if (*c.abort_flag) {
                stop = true;
                break;
            }
            const int page = page_next;
            if (paged) page_next = page_of(i + 1);
            if (gs < first) continue;
            const uint32_t bar = c.full_bar(st);
            if (i >= c.n_sub) {   // the unfilled half of an odd item's last pair
                if (lane == 0) mbar_arrive(bar);
                __syncwarp();
                continue;
            }
            const int tok = c.tok0 + i * kSub;
            const uint32_t dst = smem_u32(c.smem) + Gm::stage_off(st);
            if (lane == 0) mbar_arrive_expect_tx(bar, Gm::kStageBytes);
            __syncwarp();
            if (!paged) {
                if (lane == 0) {
                    tma_load_4d_hint(dst + 0 * kBox, tmK, bar, 0, tok, c.kvh, c.b, policy);
                    tma_load_4d_hint(dst + 1 * kBox, tmK, bar, 64, tok, c.kvh, c.b, policy);
                    tma_load_4d_hint(dst + 2 * kBox, tmV, bar, 0, tok, c.kvh, c.b, policy);
                    tma_load_4d_hint(dst + 3 * kBox, tmV, bar, 64, tok, c.kvh, c.b, policy);
                }
            } else if (lane < nbox) {
                const int in_page = (tok + lane * rows) & (p.page_size - 1);
                const uint32_t off = static_cast<uint32_t>(lane * rows * 128);
                tma_load_4d_hint(dst + 0 * kBox + off, tmK, bar, 0, in_page, c.kvh, page, policy);
                tma_load_4d_hint(dst + 1 * kBox + off, tmK, bar, 64, in_page, c.kvh, page, policy);
                tma_load_4d_hint(dst + 2 * kBox + off, tmV, bar, 0, in_page, c.kvh, page, policy);
                tma_load_4d_hint(dst + 3 * kBox + off, tmV, bar, 64, in_page, c.kvh, page, policy);
            }
        }
    }
    // Drain: the last fill of each slot must have landed before this CTA may
    // exit (a no-op unless a consumer gave up).
    if (lane == 0) {
        for (int g = max(first, gs - kRing); g < gs; ++g) wait_or_flag(c0.full_bar(g % kRing), (g / kRing) & 1);
    }
}

// Walks the pairs of stages of a persistent CTA's items in order, skipping
// items with no keys; kq counts the non-empty items before the current one.
template <int KIND>
struct PairWalk {
    SplitCtx c;        // the current item's range
    int item, n_items;
    int j, n_pairs, kq;
    bool done;

    __device__ __forceinline__ void seek() {   // from `item` on, the first non-empty item
        for (; item < n_items; item += gridDim.x) {
            set_item<KIND>(c, item, false);
            n_pairs = (c.n_sub + 1) >> 1;
            if (n_pairs > 0) return;
        }
        done = true;
    }
    __device__ __forceinline__ void start(const SplitCtx& c0, int n) {
        c = c0;
        item = blockIdx.x;
        n_items = n;
        j = 0;
        kq = 0;
        done = false;
        seek();
    }
    __device__ __forceinline__ void next() {
        if (++j < n_pairs) return;
        j = 0;
        ++kq;
        item += gridDim.x;
        seek();
    }
};

// ---------------------------------------------------------------------------
// tcgen05 kernel for query blocks of 17-128 columns (16-bit caches): one CTA
// serves all G * q_len (position, head) columns of a KV head as the M rows of
// 5th-generation tensor-core MMAs with the accumulators in tensor memory,
// instead of one CTA per 16 columns each repeating the split's arithmetic on
// warp MMAs.  Per pair of 64-token stages (128 tokens, side by side in shared
// memory, see Geo):
//   S[col][tok]  = Q[col][:] . K[tok][:]        M = 128, N = 128 tokens, K = 128 dims (8 MMAs)
//   O[col][dim] += P[col][tok] . V[tok][dim]    M = 128, N = 128 dims, 16 tokens per MMA
// A tcgen05.mma costs its issuing thread about the same time whatever N up to
// 128, so S over a whole pair (N = 128) halves the S MMAs of 64-token stages.
// Q is staged into tensor memory (the A operand of S); P (hi + lo 16-bit parts
// of the weights, two per 32-bit column) is written by the softmax over the
// columns that held its scores and read by PV as its A operand.  The next S
// into that buffer is issued after PV, and tcgen05 MMAs of one thread run in
// issue order, so PV has read P before S overwrites it.
//   KIND 31 (65-128 columns): lane r is column r; PV takes P's hi and lo
//     parts as two MMAs per 16 tokens (16 per pair).
//   KIND 32 (17-64 columns): Q rows 64 + c repeat rows c, so lanes 64 + c
//     hold column c's scores again; lanes 0-63 of P hold the hi parts and
//     lanes 64-127 the lo parts, so one MMA per 16 tokens accumulates both
//     (8 per pair), and O[c] + O[64 + c] is the result.
// Persistent: the grid is at most one CTA per SM, as many as give every CTA
// the same number of work items (one fewer for some), and CTA
// c serves the work items (split, KV head, sequence) c, c + gridDim.x, ...
// back to back -- the producer streams the next item's stages without a
// break, the next item's Q goes to the second Q buffer while the current item
// runs, and an item's epilogue (O read out, state written) overlaps the next
// item's first S MMAs; PV of the next item waits for it to release O.
// Warps 0-7 run the online softmax (base 2): warp w reaches tensor-memory
// lanes 32 (w % 4) .. +31 and takes tokens 64 (w / 4) .. +63 of each pair;
// the warps that share a column exchange their maxima once per pair (two
// warps, or four for KIND 32, whose hi and lo lanes must move their maxima
// together).  Warp 8 is the TMA producer; one thread of warp 9 issues every
// MMA.  A column's running max moves only when a pair's max exceeds it by
// more than 8 (log2 units), so p stays below 2^8 and O is rescaled in tensor
// memory only then.  The states written are the same (u, m, l) as the other
// consumers'.
// Tensor memory (512 columns): S/P [0, 128) and [128, 256) by pair parity,
// O [256, 384), Q [384, 448) and [448, 512) by item parity.  Shared memory:
// the 3-pair ring (192 KB), KIND 32's exchange of O's lo rows (17 KB), the
// epilogue's per-warp staging of states (2.3 KB a warp), the
// softmax exchange and the tcgen05 barriers (4 KB).
// ---------------------------------------------------------------------------
template <typename T, int KIND>
__global__ void __launch_bounds__(Geo<KIND>::kThreads, 1)
    fd_split_umma_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
    using Gm = Geo<KIND>;
    constexpr bool kStack = KIND == 32;
    constexpr int kRing = Gm::kRing;
    constexpr int kPairSlots = kRing / 2;
    constexpr int kSoftmaxThreads = Gm::kWarps * 32;   // 256
    constexpr uint32_t kTmemCols = 512;
    constexpr uint32_t kColO = 256, kColQ = 384;
    constexpr uint32_t kRegion = Gm::kBoxStride;       // 16 KB: [128 tokens x 64 dims]
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    SplitCtx c;
    const int S = p.n_splits;
    const int n_items = S * p.n_kv_heads * p.batch;
    // (no L2 prefetch ahead of the launch wait: measured slower here, by 1.7 us
    // at 64 columns with 256 tokens of K and V, by 10 us at 128 with the first
    // pair's K alone)
    split_setup<KIND>(c, smem, p, &tmK, &tmV, -1, 0, 0);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // KIND 32: O's lo rows pass through shared memory, [64 columns][68 words] of bf16 pairs
    uint32_t* olo_w = reinterpret_cast<uint32_t*>(smem + Gm::kOffExtra);
    // the epilogue's staging of a warp's 16 rows x 32 dims, rows padded to 36
    // floats (each 8-lane phase of a 16-byte access meets distinct banks)
    constexpr int kStgRow = 36;
    constexpr int kStgWarp = 16 * kStgRow;
    constexpr int kOloRow = 68;   // KIND 32: words per column of the lo exchange (64 + 4 padding)
    static_assert(!kStack || 64 * kOloRow * 4 <= Gm::kOloBytes, "the lo exchange must fit");
    float* stg = reinterpret_cast<float*>(smem + Gm::kOffExtra + Gm::kOloBytes);
    // the softmax exchange: pair maxima [pair parity][256], final sums [256]
    float* xmax = reinterpret_cast<float*>(smem + Gm::kOffExtra + Gm::kOloBytes + Gm::kStgBytes);
    float* xsum = xmax + 512;
    // mbarriers, [2] by pair parity (q_full: by item parity) unless noted
    const uint32_t b_x0 = smem_u32(xsum + 256);   // [4] exchange, one per group of warps sharing columns
    const uint32_t b_s_full = b_x0 + 32;          // one arrival (MMA commit): S written
    const uint32_t b_p_full = b_x0 + 48;          // one arrival per softmax warp: P written (and O rescaled)
    const uint32_t b_o_done = b_x0 + 64;          // one arrival (MMA commit): PV done
    const uint32_t b_q_full = b_x0 + 80;          // one arrival per softmax warp: an item's Q staged
    const uint32_t b_o_free = b_x0 + 96;          // single, one arrival per softmax warp: O read out
    const uint32_t b_drain = b_x0 + 104;          // single, one arrival (MMA commit): every MMA done
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(xsum + 256 + 28);   // b_x0 + 112
    if (threadIdx.x == 0) {
#pragma unroll
        for (int g = 0; g < 4; ++g) mbar_init(b_x0 + 8u * g, kStack ? 4 : 2);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            mbar_init(b_s_full + 8u * b, 1);
            mbar_init(b_p_full + 8u * b, Gm::kWarps);
            mbar_init(b_o_done + 8u * b, 1);
            mbar_init(b_q_full + 8u * b, Gm::kWarps);
        }
        mbar_init(b_o_free, Gm::kWarps);
        mbar_init(b_drain, 1);
        fence_barrier_init();
    }
    __syncthreads();   // every barrier is initialised
    if (warp == Gm::kWarps) {   // the producer streams at once; Q and tensor memory follow
        produce_pairs<KIND>(c, &tmK, &tmV, lane, n_items);
        return;
    }
    if (warp == 0) tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    tc_fence_before();
    named_sync(3, kSoftmaxThreads + 32);   // the softmax warps and the MMA warp
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_o = tmem + kColO;

    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;

    if (warp == Gm::kWarps + 1) {
        // ---- MMA issue: S of the next pair goes out before PV of the current
        // one, so the softmax of one pair overlaps the tensor cores' work on
        // the next (also across items).  The scores of pair g - 1, which S of
        // pair g + 1 overwrites, were read before the softmax handed over P of
        // pair g - 1, which PV of pair g - 1 (issued earlier) reads first.
        // Each descriptor is built once and offset by constants (the start
        // address is the low field, in 16-byte units, and no operand crosses
        // 256 KB).
        if (lane == 0) {
            const uint32_t id_s = umma_idesc_f16(128, 128, kBf16, false);
            const uint32_t id_s64 = umma_idesc_f16(128, 64, kBf16, false);   // a pair's lone stage
            const uint32_t id_o = umma_idesc_f16(128, 128, kBf16, true);
            const uint64_t dk0 = umma_desc_sw128(smem_u32(c.smem), 16, 1024);
            const uint64_t dv0 = umma_desc_sw128(smem_u32(c.smem + 2 * kRegion), kRegion, 1024);
            constexpr uint32_t kPairUnits = (4 * kRegion) >> 4;
            // S of pair gp: the item's Q (ready), both stages landed (a last pair may have one)
            auto issue_s = [&](const PairWalk<KIND>& w, int gp) -> bool {
                if (w.j == 0 && !wait_or_flag(b_q_full + 8u * (w.kq & 1), (w.kq >> 1) & 1)) return false;
                const int s0 = 2 * gp;
                const bool two = 2 * w.j + 1 < w.c.n_sub;
                if (!wait_or_flag(c.full_bar(s0 % kRing), (s0 / kRing) & 1)) return false;
                if (two && !wait_or_flag(c.full_bar((s0 + 1) % kRing), ((s0 + 1) / kRing) & 1)) return false;
                tc_fence_after();
                const uint64_t dk = dk0 + static_cast<uint32_t>(gp % kPairSlots) * kPairUnits;
                const uint32_t d = tmem + 128u * static_cast<uint32_t>(gp & 1);
                const uint32_t tq = tmem + kColQ + 64u * static_cast<uint32_t>(w.kq & 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {   // 16 dims per MMA: 32 bytes inside a 128-byte row
                    const uint32_t k_off = ((kk >> 2) * kRegion + (kk & 3) * 32u) >> 4;
                    umma_f16_ta(d, tq + 8u * kk, dk + k_off, two ? id_s : id_s64, kk > 0);
                }
                umma_commit(b_s_full + 8u * static_cast<uint32_t>(gp & 1));
                return true;
            };
            PairWalk<KIND> ws, wv;   // the pair S is issued for next, the pair PV is
            ws.start(c, n_items);
            wv = ws;
            int gps = 0, gpv = 0;
            bool ok = true;
            if (!ws.done) ok = issue_s(ws, gps);
            while (ok && !wv.done) {
                ws.next();
                ++gps;
                // at an item boundary PV of the item's last pair goes first, so that
                // the item's epilogue can start sooner
                const bool boundary = !ws.done && ws.j == 0;
                if (!ws.done && !boundary) {
                    ok = issue_s(ws, gps);
                    if (!ok) break;
                }
                ok = wait_or_flag(b_p_full + 8u * (gpv & 1), (gpv >> 1) & 1);
                if (!ok) break;
                if (wv.j == 0 && wv.kq > 0) {   // the last item's epilogue has read O
                    ok = wait_or_flag(b_o_free, (wv.kq - 1) & 1);
                    if (!ok) break;
                }
                tc_fence_after();
                const uint64_t dv = dv0 + static_cast<uint32_t>(gpv % kPairSlots) * kPairUnits;
                const uint32_t pa = tmem + 128u * static_cast<uint32_t>(gpv & 1);
                const bool two = 2 * wv.j + 1 < wv.c.n_sub;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {   // 16 tokens per MMA
                    if (kk == 4 && !two) break;
                    // 17-64 columns: the pair's first stage is read by the MMAs so far, so
                    // its slot refills while the second stage's MMAs run (with 65-128
                    // columns the earlier refill measured slower)
                    if (kStack && kk == 4) umma_commit(c.empty_bar((2 * gpv) % kRing));
                    // tokens 16 kk .. +15 were written by the warps of token half kk / 4:
                    // hi at columns 64 (kk / 4) + 8 (kk % 4), lo 32 columns further
                    const uint32_t a = pa + 64u * (kk >> 2) + 8u * (kk & 3);
                    const uint64_t b = dv + ((kk * 2048u) >> 4);
                    umma_f16_ta(tmem_o, a, b, id_o, wv.j > 0 || kk > 0);
                    if (!kStack) umma_f16_ta(tmem_o, a + 32u, b, id_o, true);
                }
                umma_commit(b_o_done + 8u * static_cast<uint32_t>(gpv & 1));
                if (!kStack || !two) umma_commit(c.empty_bar((2 * gpv) % kRing));
                umma_commit(c.empty_bar((2 * gpv + 1) % kRing));    // filled or not
                wv.next();
                ++gpv;
                if (boundary) {
                    ok = issue_s(ws, gps);
                    if (!ok) break;
                }
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
        // ---- softmax warps: thread (w, lane) owns column `col` (tensor-memory
        // lane r) and tokens 64 h .. 64 h + 63 of each pair; for KIND 32 side
        // 0 holds the hi lanes and side 1 the lo lanes
        const int q = warp & 3, h = (warp >> 2) & 1;
        const int r = q * 32 + lane;
        const int col = kStack ? (r & 63) : r;
        const int side = kStack ? (q >> 1) : 0;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const bool active = kStack ? 32 * (q & 1) < p.cols : 32 * q < p.cols;   // warp-uniform
        const bool real = col < p.cols;
        // scores stay raw until the exponent: sc (log2(e) / sqrt(d), a 16-bit
        // cache) is positive, so maxima of raw scores scale to maxima of scaled ones
        const float sc = p.score_scale_log2;
        const uint32_t b_x = b_x0 + 8u * static_cast<uint32_t>(kStack ? (q & 1) : q);
        const int xslot = kStack ? (side * 2 + h) * 64 + col : h * 128 + r;
        // Q of a non-empty item into buffer kb: this lane's row, dims 64 h .. +63
        // (d, d + 1 share column d / 2); every softmax warp arrives on q_full
        auto stage_q = [&](const SplitCtx& ci, int kb) {
            bool rl;
            const T* qrow = q_row<T>(ci, col, rl);
            const uint4* src = reinterpret_cast<const uint4*>(qrow + 64 * h);
            uint32_t qw[32];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const uint4 v = rl ? __ldg(src + x) : make_uint4(0u, 0u, 0u, 0u);
                qw[4 * x] = v.x;
                qw[4 * x + 1] = v.y;
                qw[4 * x + 2] = v.z;
                qw[4 * x + 3] = v.w;
            }
            const uint32_t qa = tmem + lane_base + kColQ + 64u * static_cast<uint32_t>(kb & 1) + 32u * h;
            tmem_st16(qa, *reinterpret_cast<const uint32_t(*)[16]>(qw));
            tmem_st16(qa + 16u, *reinterpret_cast<const uint32_t(*)[16]>(qw + 16));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_q_full + 8u * static_cast<uint32_t>(kb & 1));
        };
        // the state of an item's column: (u, m, l), or out / lse with one split;
        // o: 16 dims d0 .. d0 + 15 of u (unscaled by v), this thread's row
        auto write_state = [&](const SplitCtx& ci, int d0, const float (&o)[16], float m_out, float l_col,
                               bool with_ml) {
            const int64_t row = (static_cast<int64_t>(ci.b) * p.q_len + col / p.group) * p.n_q_heads +
                                ci.kvh * p.group + col % p.group;
            const bool empty = m_out == -INFINITY || !(l_col > 0.f);
            if (p.direct) {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float y = empty ? 0.f : (o[e] * p.v_scale) / l_col;
                    const int64_t oi = row * kHeadDim + d0 + e;
                    if (p.out_dtype == 2)
                        static_cast<float*>(p.out)[oi] = y;
                    else if (p.out_dtype == 0)
                        static_cast<__half*>(p.out)[oi] = __float2half_rn(y);
                    else
                        static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(y);
                }
                if (with_ml && p.lse != nullptr) p.lse[row] = empty ? -INFINITY : m_out + logf(l_col);
            } else {
                float4* dst = reinterpret_cast<float4*>(p.ws_u + (row * S + ci.split) * kHeadDim + d0);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_float4(o[4 * e] * p.v_scale, o[4 * e + 1] * p.v_scale,
                                         o[4 * e + 2] * p.v_scale, o[4 * e + 3] * p.v_scale);
                if (with_ml) {
                    p.ws_m[row * S + ci.split] = m_out;
                    p.ws_l[row * S + ci.split] = l_col;
                }
            }
        };

        // set by softmax warps only, read by all of them between two barriers
        volatile int* sm_abort = reinterpret_cast<volatile int*>(smem + Gm::kOffFlag + 8);
        PairWalk<KIND> wq;   // the next non-empty item whose Q is to be staged
        wq.start(c, n_items);
        if (!wq.done) stage_q(wq.c, 0);
        int gp = 0, kq = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            SplitCtx ci = c;
            set_item<KIND>(ci, item, threadIdx.x == 0);
            const int n_pairs = (ci.n_sub + 1) >> 1;
            if (n_pairs == 0) {   // no keys: u = 0, m = -inf, l = 0
                if (side == 0 && active && real) {
                    const float zero[16] = {};
#pragma unroll 1
                    for (int qq = 0; qq < 4; ++qq) write_state(ci, 64 * h + 16 * qq, zero, -INFINITY, 0.f, h == 0 && qq == 0);
                }
                continue;
            }
            const int vis = real ? ci.L - p.q_len + 1 + col / p.group : ci.L;
            float m_run = -INFINITY, l_run = 0.f;
#pragma unroll 1
            for (int j = 0; j < n_pairs; ++j, ++gp) {
                const int buf = gp & 1;
                ok = __all_sync(kFull, wait_or_flag(b_s_full + 8u * buf, (gp >> 1) & 1));
                if (!ok) break;
                tc_fence_after();
                const uint32_t sa = tmem + lane_base + 128u * buf + 64u * h;   // this warp's 64 columns
                const int tok = ci.tok0 + 128 * j + 64 * h;
                const int nvalid = min(64, ci.tok1 - tok);   // <= 0: this half of a short last pair
                float alpha = 1.f;
                bool need = false;
                if (active) {
                    uint32_t t[64];
                    tmem_ld64(sa, t);
                    tmem_wait_ld();
                    if (nvalid < 64 || tok + 64 > ci.L - p.q_len + 1) {
                        const int lim = min(nvalid, vis - tok);   // in this warp's tokens
#pragma unroll
                        for (int e = 0; e < 64; ++e)
                            if (e >= lim) t[e] = __float_as_uint(-INFINITY);
                    }
                    float mx = -INFINITY;
#pragma unroll
                    for (int e = 0; e < 64; ++e) mx = fmaxf(mx, __uint_as_float(t[e]));
                    // the pair's max over every warp holding the column, the same in
                    // each (double-buffered by pair parity: every warp of the group has
                    // read a slot before the group passes its next exchange)
                    float* xm = xmax + buf * 256;
                    xm[xslot] = mx;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_x);
                    ok = __all_sync(kFull, wait_or_flag(b_x, gp & 1));
                    if (!ok) break;
                    if (kStack)
                        mx = fmaxf(fmaxf(xm[col], xm[64 + col]), fmaxf(xm[128 + col], xm[192 + col]));
                    else
                        mx = fmaxf(xm[r], xm[128 + r]);
                    mx *= sc;                      // raw scores: sc > 0 keeps the max
                    need = mx > m_run + 8.f;       // also true for the first finite max
                    if (need) {
                        alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - mx);
                        l_run *= alpha;
                        m_run = mx;
                    }
                    const float mu = m_run == -INFINITY ? 0.f : m_run;
                    // P over the scores' columns, 32 tokens at a time: hi parts at
                    // columns 0-31 of the warp's 64, lo parts at 32-63 (KIND 32: each
                    // side keeps its own part at 0-31)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t hi[16], lo[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float p0 = fast_exp2(fmaf(__uint_as_float(t[32 * hf + 2 * e]), sc, -mu));
                            const float p1 = fast_exp2(fmaf(__uint_as_float(t[32 * hf + 2 * e + 1]), sc, -mu));
                            l_run += p0 + p1;
                            float k0, k1, d0, d1;
                            hi[e] = Mma<T>::pack(p0, p1, k0, k1);
                            lo[e] = Mma<T>::pack(p0 - k0, p1 - k1, d0, d1);
                        }
                        if (kStack) {
                            if (side == 0)
                                tmem_st16(sa + 16u * hf, hi);
                            else
                                tmem_st16(sa + 16u * hf, lo);
                        } else {
                            tmem_st16(sa + 16u * hf, hi);
                            tmem_st16(sa + 32u + 16u * hf, lo);
                        }
                    }
                }
                if (j > 0 && active && __any_sync(kFull, need)) {
                    // O is rescaled once PV of the previous pair is done with it:
                    // this lane's O row, dims 64 h .. 64 h + 63
                    ok = __all_sync(kFull, wait_or_flag(b_o_done + 8u * (buf ^ 1), ((gp - 1) >> 1) & 1));
                    if (ok) {
                        tc_fence_after();
#pragma unroll 1
                        for (int qq = 0; qq < 4; ++qq) {
                            uint32_t v[16];
                            const uint32_t ta = tmem_o + lane_base + 64u * h + 16u * qq;
                            tmem_ld16(ta, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                            tmem_st16(ta, v);
                        }
                    }
                }
                tmem_wait_st();
                if (!ok) break;
                // V rows past the end of a loaded stage hold whatever the cache holds
                // there; P is 0 for them, but 0 * NaN would still poison PV
                const int slot_base = (gp % kPairSlots) * 4 * static_cast<int>(kRegion);
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    if (2 * j + hh >= ci.n_sub) break;
                    const int nv = min(64, ci.tok1 - (ci.tok0 + 128 * j + 64 * hh));
                    if (nv >= 64) continue;
                    for (int idx = threadIdx.x; idx < (64 - nv) * 16; idx += kSoftmaxThreads) {
                        const int row = 64 * hh + nv + (idx >> 4), ch = idx & 15;
                        *reinterpret_cast<uint4*>(c.smem + slot_base + (2 + (ch >> 3)) * kRegion + row * 128 +
                                                  (((ch & 7) ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(b_p_full + 8u * buf);
                // the next non-empty item's Q goes to the other buffer, whose last
                // reader (S of the item before this one) completed before this
                // item's first scores
                if (j == min(1, n_pairs - 1)) {
                    wq.next();               // from this item's pairs ...
                    while (!wq.done && wq.j != 0) wq.next();   // ... to the next item
                    if (!wq.done) stage_q(wq.c, kq + 1);
                }
            }
            // ---- the item's epilogue: once the last PV is done, O read out and
            // the column states written; O is then handed back to PV
            if (ok) {
                ok = __all_sync(kFull, wait_or_flag(b_o_done + 8u * ((gp - 1) & 1), ((gp - 1) >> 1) & 1));
                tc_fence_after();
            }
            if (!ok) *sm_abort = 1;
            xsum[xslot] = l_run;
            named_sync(1, kSoftmaxThreads);
            if (*sm_abort != 0) break;   // every softmax warp leaves together
            const float m_out = m_run == -INFINITY ? -INFINITY : m_run * kLn2;
            const float l_col = kStack ? xsum[col] + xsum[64 + col] : xsum[r] + xsum[128 + r];
            const bool empty = m_out == -INFINITY || !(l_col > 0.f);
            const int64_t my_row = real ? (static_cast<int64_t>(ci.b) * p.q_len + col / p.group) * p.n_q_heads +
                                              ci.kvh * p.group + col % p.group
                                        : 0;
            if (kStack) {
                // O's lo rows (at most 2^-9 of the result) pass to the hi side as
                // bf16 pairs, [column][dim pair] with rows padded to 68 words, so
                // that each 8-lane phase of a 16-byte access meets distinct banks
                if (side == 1 && active) {
                    uint32_t v[64];
                    tmem_ld64(tmem_o + lane_base + 64u * h, v);
                    tmem_wait_ld();
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const __nv_bfloat162 w = __floats2bfloat162_rn(__uint_as_float(v[2 * e]),
                                                                       __uint_as_float(v[2 * e + 1]));
                        memcpy(&pk[e], &w, 4);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(olo_w + col * kOloRow + 32 * h);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
                named_sync(1, kSoftmaxThreads);
            }
            // tcgen05.ld is warp-wide: every lane loads; lanes past the columns
            // stage values nobody stores
            if (side == 0 && active) {
                if constexpr (kStack) {
                    // each lane writes its own row's 64 dims: 16 independent 16-byte
                    // stores from registers (the row's 256 bytes are contiguous)
                    uint32_t v[64];
                    tmem_ld64(tmem_o + lane_base + 64u * h, v);
                    tmem_wait_ld();
                    if (real) {
                        float o[64];
#pragma unroll
                        for (int e = 0; e < 64; ++e) o[e] = __uint_as_float(v[e]);
                        if (kStack) {
                            const uint4* lw = reinterpret_cast<const uint4*>(olo_w + col * kOloRow + 32 * h);
#pragma unroll
                            for (int x = 0; x < 8; ++x) {
                                const uint4 w4 = lw[x];
                                const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                                for (int t = 0; t < 4; ++t) {
                                    o[8 * x + 2 * t] += __uint_as_float(w[t] << 16);
                                    o[8 * x + 2 * t + 1] += __uint_as_float(w[t] & 0xffff0000u);
                                }
                            }
                        }
                        if (!p.direct) {
                            // 32-byte stores: each writes whole sectors of the row's 256 bytes
                            float* dst = p.ws_u + (my_row * S + ci.split) * kHeadDim + 64 * h;
#pragma unroll
                            for (int x = 0; x < 8; ++x)
                                st_global_v8(dst + 8 * x, o[8 * x] * p.v_scale, o[8 * x + 1] * p.v_scale,
                                             o[8 * x + 2] * p.v_scale, o[8 * x + 3] * p.v_scale,
                                             o[8 * x + 4] * p.v_scale, o[8 * x + 5] * p.v_scale,
                                             o[8 * x + 6] * p.v_scale, o[8 * x + 7] * p.v_scale);
                        } else {   // out carries only its element alignment: scalar stores
                            const int64_t oi = my_row * kHeadDim + 64 * h;
#pragma unroll
                            for (int e = 0; e < 64; ++e) {
                                const float y = empty ? 0.f : (o[e] * p.v_scale) / l_col;
                                if (p.out_dtype == 2)
                                    static_cast<float*>(p.out)[oi + e] = y;
                                else if (p.out_dtype == 0)
                                    static_cast<__half*>(p.out)[oi + e] = __float2half_rn(y);
                                else
                                    static_cast<__nv_bfloat16*>(p.out)[oi + e] = __float2bfloat16_rn(y);
                            }
                        }
                    }
                } else {
                    // 65-128 columns: all eight warps write, so whole 128-byte lines pay off
                    float* sg = stg + warp * kStgWarp;   // [16 rows][36]
                    // four steps of 16 rows x 32 dims: the rows' lanes stage their values,
                    // then lane l stores dims 4 (l % 8) .. +3 of row l / 8 + 4 k, so a
                    // store covers four whole 128-byte lines.  The loop stays rolled: it
                    // runs once per item, and its code is fetched cold each time.
#pragma unroll 1
                    for (int step = 0; step < 4; ++step) {
                        const int rh = step >> 1, dh = step & 1;
                        uint32_t v[32];
                        tmem_ld32(tmem_o + lane_base + 64u * h + 32u * dh, v);
                        tmem_wait_ld();
                        if ((lane >> 4) == rh) {
                            // this row's 32 values: the state's u (values are v_scale x the
                            // stored ones), or out with one split
                            float o[32];
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(v[e]);
                            // (a uniform branch: the division is only paid for with one split)
                            if (!p.direct) {
#pragma unroll
                                for (int e = 0; e < 32; ++e) o[e] *= p.v_scale;
                            } else {
#pragma unroll
                                for (int e = 0; e < 32; ++e) o[e] = empty ? 0.f : (o[e] * p.v_scale) / l_col;
                            }
                            float4* sr = reinterpret_cast<float4*>(sg + (lane & 15) * kStgRow);
#pragma unroll
                            for (int x = 0; x < 8; ++x) sr[x] = make_float4(o[4 * x], o[4 * x + 1], o[4 * x + 2], o[4 * x + 3]);
                        }
                        __syncwarp();
                        // every row and value is read before any store is issued (the
                        // compiler cannot move shared loads above a global store)
                        const int f = lane & 7, d0 = 64 * h + 32 * dh + 4 * f;
                        int64_t rows[4];
                        bool rreal[4];
                        float y[4][4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int rr = (lane >> 3) + 4 * k;     // row within the step's 16
                            rows[k] = __shfl_sync(kFull, my_row, 16 * rh + rr);
                            rreal[k] = __shfl_sync(kFull, real ? 1 : 0, 16 * rh + rr) != 0;
                            const float4 y4 = *reinterpret_cast<const float4*>(sg + rr * kStgRow + 4 * f);
                            y[k][0] = y4.x;
                            y[k][1] = y4.y;
                            y[k][2] = y4.z;
                            y[k][3] = y4.w;
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if (!rreal[k]) continue;
                            if (!p.direct) {
                                *reinterpret_cast<float4*>(p.ws_u + (rows[k] * S + ci.split) * kHeadDim + d0) =
                                    make_float4(y[k][0], y[k][1], y[k][2], y[k][3]);
                            } else {   // out carries only its element alignment: scalar stores
                                const int64_t oi = rows[k] * kHeadDim + d0;
                                if (p.out_dtype == 2) {
                                    float* o = static_cast<float*>(p.out) + oi;
#pragma unroll
                                    for (int t = 0; t < 4; ++t) o[t] = y[k][t];
                                } else if (p.out_dtype == 0) {
                                    __half* o = static_cast<__half*>(p.out) + oi;
#pragma unroll
                                    for (int t = 0; t < 4; ++t) o[t] = __float2half_rn(y[k][t]);
                                } else {
                                    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + oi;
#pragma unroll
                                    for (int t = 0; t < 4; ++t) o[t] = __float2bfloat16_rn(y[k][t]);
                                }
                            }
                        }
                        __syncwarp();   // the staging is rewritten by the next step
                    }
                }
                if (real && h == 0) {
                    if (p.direct) {
                        if (p.lse != nullptr) p.lse[my_row] = empty ? -INFINITY : m_out + logf(l_col);
                    } else {
                        p.ws_m[my_row * S + ci.split] = m_out;
                        p.ws_l[my_row * S + ci.split] = l_col;
                    }
                }
            }
            if (kStack) named_sync(1, kSoftmaxThreads);   // olo is rewritten by the next item
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_o_free);
            ++kq;
            named_sync(1, kSoftmaxThreads);   // every warp has read sm_abort before the next item
        }
        if (!ok) *c.cons_abort = 1;
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
    using Gm = Geo<KIND>;
    const int blocks = p.n_splits * p.col_blocks;
    // fp8, up to 8 columns: its consumers do not keep up with HBM on an SM of
    // their own, so once splits outnumber SMs every CTA takes two -- while one
    // wave holds those CTAs (a CTA of two takes a whole SM, and an odd split
    // count leaves a half idle per (sequence, KV head); beyond one wave the
    // CTAs of one, two to an SM, quantise better)
    if constexpr (KIND == 21) {
        const int sms = fd_num_sms(-1);
        const int64_t heads = static_cast<int64_t>(n_kv_heads) * batch;
        if (blocks * heads > sms && ((blocks + 1) / 2) * heads <= sms) {
            auto kern = fd_split_kernel<T, KIND, 2>;
            const size_t smem = 2 * Gm::kSmemHalf + 1024;
            static std::atomic<unsigned long long> configured_ctx2{0};
            cudaError_t e = allow_smem(kern, smem, configured_ctx2);
            if (e != cudaSuccess) return e;
            return launch_pdl(kern, dim3((blocks + 1) / 2, n_kv_heads, batch), dim3(2 * Gm::kThreads), smem,
                              stream, tmK, tmV, p);
        }
    }
    auto kern = fd_split_kernel<T, KIND, 1>;
    const size_t smem = Gm::kSmem;
    static std::atomic<unsigned long long> configured_ctx{0};
    cudaError_t e = allow_smem(kern, smem, configured_ctx);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(blocks, n_kv_heads, batch), dim3(Gm::kThreads), smem, stream, tmK, tmV, p);
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
    auto kern = fd_split_umma_kernel<T, KIND>;
    const size_t smem = Geo<KIND>::kSmem;
    static std::atomic<unsigned long long> configured_ctx{0};
    cudaError_t e = allow_smem(kern, smem, configured_ctx);
    if (e != cudaSuccess) return e;
    // persistent: at most one CTA per SM, and as many CTAs as give every CTA
    // the same number of items (one more for some at most): 288 items on 152
    // SMs run as 144 CTAs of two, rather than 136 of two beside 16 of one
    // that idle through the second half while an SM's own streaming rate
    // holds the other 136 below the memory's
    const int sms = fd_num_sms(-1);
    if (sms < 1) return cudaErrorInvalidDevice;
    const int64_t items = static_cast<int64_t>(p.n_splits) * n_kv_heads * batch;
    const int64_t per_cta = (items + sms - 1) / sms;
    const int ctas = static_cast<int>((items + per_cta - 1) / per_cta);
    return launch_pdl(kern, dim3(ctas), dim3(Geo<KIND>::kThreads), smem, stream, tmK, tmV, p);
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
