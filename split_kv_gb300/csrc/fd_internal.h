// fd_internal.h -- parameters shared by the host ABI (fd_api.cu) and the
// decode kernels (fd_split.cu, fd_combine.cu).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fdk {

constexpr int kHeadDim = 128;     // D
constexpr int kSub = 64;          // tokens per pipeline stage
constexpr int kStages = 3;        // pipeline depth (stages in flight per CTA)
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;   // + one TMA producer warp
constexpr int kHalfBytes = kSub * 128;                // one [kSub tokens x 64 dims] 16-bit box
constexpr int kSplitUnit = 16;                        // split ranges are whole 16-token units
constexpr int kPagedBoxRows = 16;                     // paged boxes: at most one unit of one page
constexpr int kStageBytes = 4 * kHalfBytes;           // K lo, K hi, V lo, V hi
// fp8 caches with at most 8 columns per CTA: six consumer warps, 96-token stages
constexpr int kConsumerWarpsF8 = 6;
constexpr int kSubF8 = 16 * kConsumerWarpsF8;

// Tokens per pipeline stage (the height of a contiguous cache's TMA box) of
// the split-kernel variant that serves `cols` columns per CTA.
inline int stage_tokens(bool fp8, int cols) { return fp8 && cols <= 8 ? kSubF8 : kSub; }

// Device status bits (sticky until fd_device_status(clear)).
constexpr unsigned kStatusTimeoutBit = 1u;   // an mbarrier wait ran past its limit
constexpr unsigned kStatusSeqlenBit = 2u;    // seqlens[b] < 0 or beyond the cache capacity
constexpr unsigned kStatusPageBit = 4u;      // block-table entry outside [0, n_pages)

struct SplitParams {
    const void* q;
    int64_t q_sb, q_sh, q_st;       // elements: sequence, head, query position
    const int32_t* seqlens;
    const int32_t* block_table;     // paged only
    int32_t max_pages;              // block_table row length
    int32_t page_size;              // 0 = contiguous
    int32_t page_shift;             // log2(page_size)
    int32_t capacity;               // tokens a sequence may hold
    int32_t n_pages;                // paged pool size
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t batch;
    int32_t group;                  // G = query heads per KV head
    int32_t q_len;                  // query positions per sequence
    int32_t cols;                   // G * q_len (query position, head) columns per KV head
    int32_t col_blocks;             // CTAs per (split, KV head): ceil(cols / 16), 1 if cols <= 8
    int32_t n_splits;
    int32_t split_unit;             // split ranges are whole units of this many tokens
    int32_t drop_first_stage;       // test hook: never request stage 0 (the wait for it times out)
    float score_scale_log2;         // log2(e) / sqrt(D), times k_scale for an fp8 cache
    float v_scale;                  // values are v_scale x the stored ones (1 unless fp8)
    float* ws_u;                    // [rows][n_splits][D]
    float* ws_m;                    // [rows][n_splits]
    float* ws_l;                    // [rows][n_splits]
    // direct != 0 (one split): each row's state is its result, so the kernel
    // writes out = u / l and lse = m + log l itself instead of the state
    int32_t direct;
    int32_t out_dtype;              // 0 f16, 1 bf16, 2 f32
    void* out;                      // [rows][D]
    float* lse;                     // [rows] or null
};

struct CombineParams {
    const float* ws_u;
    const float* ws_m;
    const float* ws_l;
    void* out;                      // [rows][D], out_dtype
    float* lse;                     // [rows] or null
    int32_t rows;
    int32_t n_splits;
    int32_t out_dtype;              // 0 f16, 1 bf16, 2 f32
};

// Launches `kern` with programmatic stream serialization, so that it may
// start while the previous kernel in the stream finishes; the kernel itself
// waits (griddepcontrol.wait) before touching anything that kernel wrote.
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       const Args&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Launchers return cudaGetLastError() after the launch.
// q_dtype 0 fp16 / 1 bf16; fp8: the cache holds e4m3 (tensor cores only);
// cuda_cores selects the CUDA-core (FP32 FMA) consumer instead of the tensor-core one.
cudaError_t launch_split(const CUtensorMap& tmK, const CUtensorMap& tmV, const SplitParams& p,
                         int q_dtype, bool fp8, bool cuda_cores, int batch, int n_kv_heads,
                         cudaStream_t stream);

// CTAs per (split, KV head) for G * q_len columns.
inline int column_blocks(int cols) { return cols <= 8 ? 1 : (cols + 15) / 16; }

// Query blocks of 17-128 columns (16-bit caches, tensor-core path) run a
// tcgen05 variant (17-64 columns: the hi and lo parts of P stacked in M;
// 65-128: one lane per column): one CTA serves all columns and takes a whole
// SM, so it is one work item per split and the planner counts one slot per SM.
inline bool use_umma(bool fp8, bool cuda_cores, int cols) {
    return !fp8 && !cuda_cores && cols > 16 && cols <= 128;
}

// Split count of one split-kernel launch by the wave-efficiency heuristic
// (fd_plan_splits): work = the launch's CTAs per split (column blocks, or one
// tcgen05 CTA) x n_kv_heads x batch; slots = the CTAs the GPU holds at once,
// two per SM, or one per SM for the tcgen05 variant; n_kv_blocks =
// ceil(max_seqlen / 128).  cols = G * q_len.  num_sms <= 0 queries the
// current device.  Returns s >= 1 or a negative fd_status.
int32_t plan_launch(int64_t batch, int64_t n_kv_heads, int cols, bool fp8, bool cuda_cores,
                    int64_t max_seqlen, int32_t num_sms);

// Identifier of the CUDA context current on the calling thread, unique per
// context creation (a context destroyed and created again gets a new one);
// 0 when no context is current or the driver cannot say.  Per-context state
// (the fixed workspace's address, kernel attributes) is keyed on it.
unsigned long long current_context_id();
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);

// Device status word helpers (fd_split.cu owns the symbol).
cudaError_t read_status(unsigned* value, cudaStream_t stream, bool clear);

}  // namespace fdk
