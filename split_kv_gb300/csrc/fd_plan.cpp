// fd_plan.cpp -- host split planner of the decode library.
//
// "Flash-Decoding: Split-KV Attention for Long-Context Decode", §6 "How many
// splits?": the split count is chosen by wave efficiency.  A launch of
// work*s CTAs on `slots` concurrent CTA slots runs in ceil(work*s/slots)
// waves, the last of them work*s/slots - (waves-1) full; the efficiency of s
// is (work*s/slots) / ceil(work*s/slots).  Counts that give the same number of
// KV blocks per split as the next smaller count are skipped, the best
// efficiency over the rest is found, and the smallest count within 85% of it
// wins.  Launches that already cover 80% of the slots are not split at all.
// The FlashAttention-3 heuristic comment quoted in the vatshank split-KV post
// ("Benchmarking split-KV against vanilla FA") states the same rule.
//
// All comparisons are made on IEEE doubles exactly as the page's Python makes
// them (int*int is exact, a/b is correctly rounded), so the plan is
// reproducible bit for bit on any host.  Do not build with fast-math.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "../../include/fd.h"
#include "fd_internal.h"

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

int64_t blocks_per_split(int64_t n_blocks, int64_t s) { return (n_blocks + s - 1) / s; }

double wave_efficiency(int64_t work, int64_t slots, int64_t s) {
    const double waves = static_cast<double>(work * s) / static_cast<double>(slots);
    return waves / std::ceil(waves);
}

}  // namespace

extern "C" int32_t fd_plan_splits(int64_t work_items, int64_t slots, int64_t n_kv_blocks,
                                  int32_t max_splits) {
    if (work_items < 1 || slots < 1 || n_kv_blocks < 0 || max_splits < 1) return FD_ERR_INVALID_ARG;
    if (work_items > (int64_t(1) << 40) || slots > (int64_t(1) << 20)) return FD_ERR_INVALID_ARG;
    if (static_cast<double>(work_items) >= 0.8 * static_cast<double>(slots)) return 1;
    const int64_t top = std::min<int64_t>({static_cast<int64_t>(max_splits), slots, n_kv_blocks});
    if (top < 1) return 1;
    auto counts = [&](int64_t s) {
        return s == 1 || blocks_per_split(n_kv_blocks, s) != blocks_per_split(n_kv_blocks, s - 1);
    };
    double best = 0.0;
    for (int64_t s = 1; s <= top; ++s)
        if (counts(s)) best = std::max(best, wave_efficiency(work_items, slots, s));
    const double bar = 0.85 * best;
    for (int64_t s = 1; s <= top; ++s)
        if (counts(s) && wave_efficiency(work_items, slots, s) >= bar) return static_cast<int32_t>(s);
    return 1;
}

extern "C" int32_t fd_num_sms(int32_t device) {
    int dev = device;
    if (dev < 0 && cudaGetDevice(&dev) != cudaSuccess) return FD_ERR_CUDA;
    if (dev >= kMaxDevices) return FD_ERR_INVALID_ARG;
    int cached = g_sm_count[dev].load(std::memory_order_relaxed);
    if (cached > 0) return cached;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return FD_ERR_CUDA;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace fdk {

int32_t plan_launch(int64_t batch, int64_t n_kv_heads, int cols, bool fp8, bool cuda_cores,
                    int64_t max_seqlen, int32_t num_sms) {
    if (batch < 1 || n_kv_heads < 1 || cols < 1 || max_seqlen < 0) return FD_ERR_INVALID_ARG;
    int32_t sms = num_sms;
    if (sms <= 0) {
        sms = fd_num_sms(-1);
        if (sms < 0) return sms;
    }
    // one CTA per split serves the whole group: up to 16 columns on warp MMAs,
    // or 17-128 on the tcgen05 variant, whose shared memory fills an SM;
    // otherwise one CTA per 16 columns, two CTAs per SM
    const bool umma = use_umma(fp8, cuda_cores, cols);
    const int64_t per_split = umma ? 1 : column_blocks(cols);
    const int64_t blocks = (max_seqlen + FD_TILE_TOKENS - 1) / FD_TILE_TOKENS;
    return fd_plan_splits(batch * n_kv_heads * per_split, (umma ? 1 : 2) * static_cast<int64_t>(sms),
                          blocks, FD_MAX_SPLITS);
}

}  // namespace fdk

extern "C" int32_t fd_plan(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                           const int32_t* seqlens_host, const int32_t* block_table_host,
                           int32_t page_size, int32_t max_pages_per_seq, int32_t num_sms) {
    if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || head_dim < 1) return FD_ERR_INVALID_ARG;
    if (n_q_heads % n_kv_heads != 0 || seqlens_host == nullptr) return FD_ERR_INVALID_ARG;
    const int64_t G = n_q_heads / n_kv_heads;
    if (G > 256) return FD_ERR_UNSUPPORTED;
    if (block_table_host != nullptr) {
        if (page_size < 8 || (page_size & (page_size - 1)) != 0 || page_size > (1 << 20))
            return page_size >= 1 && page_size < 8 && (page_size & (page_size - 1)) == 0
                       ? FD_ERR_UNSUPPORTED
                       : FD_ERR_INVALID_ARG;
        if (max_pages_per_seq < 1) return FD_ERR_INVALID_ARG;
    }
    int64_t max_len = 0;
    for (int32_t b = 0; b < batch; ++b) {
        const int32_t L = seqlens_host[b];
        if (L < 0) return FD_ERR_INVALID_ARG;
        max_len = std::max<int64_t>(max_len, L);
        if (block_table_host == nullptr) continue;
        // the table must name a page for every token of the sequence
        const int64_t need = (static_cast<int64_t>(L) + page_size - 1) / page_size;
        if (need > max_pages_per_seq) return FD_ERR_INVALID_ARG;
        const int32_t* row = block_table_host + static_cast<int64_t>(b) * max_pages_per_seq;
        for (int64_t j = 0; j < need; ++j)
            if (row[j] < 0) return FD_ERR_INVALID_ARG;
    }
    // a 16-bit cache on the default (tensor-core) path, one query per sequence
    return fdk::plan_launch(batch, n_kv_heads, static_cast<int>(G), false, false, max_len, num_sms);
}
