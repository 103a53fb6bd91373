// fd_api.cu -- the C ABI of the decode library (declared in include/fd.h):
// host-side validation, workspace layout, TMA descriptors and launches.
// Nothing here allocates device memory or synchronises a stream except
// fd_device_status(), which is documented to.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fd.h"
#include "fd_internal.h"

namespace {

using fdk::kHeadDim;

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct WsLayout {
    size_t off_u, off_m, off_l, total;
};

WsLayout ws_layout(int64_t rows, int64_t splits) {
    WsLayout w;
    w.off_u = 0;
    w.off_m = round_up(static_cast<size_t>(rows * splits * kHeadDim) * sizeof(float));
    w.off_l = w.off_m + round_up(static_cast<size_t>(rows * splits) * sizeof(float));
    w.total = w.off_l + round_up(static_cast<size_t>(rows * splits) * sizeof(float));
    return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A stride in elements of `esize` bytes is usable by TMA: a multiple of 16 bytes.
bool stride_ok(int64_t s, int esize = 2) {
    return s >= 0 && (s * esize) % 16 == 0 && s < (int64_t(1) << 38);
}

bool is_fp8(const fd_desc* d) { return d->kv_dtype == FD_E4M3; }
int cache_esize(const fd_desc* d) { return is_fp8(d) ? 1 : 2; }
// the type of q (and of the MMA operands): kv_dtype, or q_dtype for an fp8 cache
int q_type_of(const fd_desc* d) { return is_fp8(d) ? d->q_dtype : d->kv_dtype; }

int q_len_of(const fd_desc* d) { return d->q_len <= 1 ? 1 : d->q_len; }

int64_t rows_of(const fd_desc* d) {
    return static_cast<int64_t>(d->batch) * q_len_of(d) * d->n_q_heads;
}

int cols_of(const fd_desc* d) { return (d->n_q_heads / d->n_kv_heads) * q_len_of(d); }

bool umma_of(const fd_desc* d) {
    return fdk::use_umma(is_fp8(d), (d->flags & FD_FLAG_CUDA_CORES) != 0, cols_of(d));
}

int col_blocks_of(const fd_desc* d) { return umma_of(d) ? 1 : fdk::column_blocks(cols_of(d)); }

// Shape / layout checks shared by every entry point.  Pointer checks are
// done by the callers, which know which pointers they use.
fd_status check_desc(const fd_desc* d) {
    if (d == nullptr) return FD_ERR_INVALID_ARG;
    if ((d->flags & ~(FD_FLAG_CUDA_CORES | FD_FLAG_TEST_DROP_FIRST_STAGE)) != 0)
        return FD_ERR_INVALID_ARG;
    if (d->q_len < 0) return FD_ERR_INVALID_ARG;
    if (d->batch < 0 || d->n_q_heads < 1 || d->n_kv_heads < 1 || d->head_dim < 1)
        return FD_ERR_INVALID_ARG;
    if (d->n_q_heads % d->n_kv_heads != 0) return FD_ERR_INVALID_ARG;
    if (d->kv_dtype != FD_F16 && d->kv_dtype != FD_BF16 && d->kv_dtype != FD_E4M3)
        return d->kv_dtype == FD_F32 ? FD_ERR_UNSUPPORTED : FD_ERR_INVALID_ARG;
    if (d->reserved != 0) return FD_ERR_INVALID_ARG;
    if (is_fp8(d)) {
        if (d->q_dtype != FD_F16 && d->q_dtype != FD_BF16) return FD_ERR_INVALID_ARG;
        if (!std::isfinite(d->k_scale) || !std::isfinite(d->v_scale)) return FD_ERR_INVALID_ARG;
        if ((d->flags & FD_FLAG_CUDA_CORES) != 0) return FD_ERR_UNSUPPORTED;
    }
    if (d->out_dtype != FD_F16 && d->out_dtype != FD_BF16 && d->out_dtype != FD_F32)
        return FD_ERR_INVALID_ARG;
    if (d->head_dim != kHeadDim) return FD_ERR_UNSUPPORTED;
    const int G = d->n_q_heads / d->n_kv_heads;
    const int ql = q_len_of(d);
    if (ql > 16 || static_cast<int64_t>(G) * ql > 256) return FD_ERR_UNSUPPORTED;
    if ((d->flags & FD_FLAG_CUDA_CORES) != 0 && ((G != 1 && G != 2 && G != 4 && G != 8) || ql != 1))
        return FD_ERR_UNSUPPORTED;
    if (ql > 1 && !stride_ok(d->q_stride_t)) return FD_ERR_INVALID_ARG;
    if (d->n_splits > FD_MAX_SPLITS) return FD_ERR_UNSUPPORTED;
    if (d->page_size < 0) return FD_ERR_INVALID_ARG;
    if (d->page_size > 0) {
        if ((d->page_size & (d->page_size - 1)) != 0 || d->page_size > (1 << 20))
            return FD_ERR_INVALID_ARG;
        if (d->page_size < 8) return FD_ERR_UNSUPPORTED;
        if (d->max_pages_per_seq < 1) return FD_ERR_INVALID_ARG;
        if (static_cast<int64_t>(d->max_pages_per_seq) * d->page_size > INT32_MAX)
            return FD_ERR_INVALID_ARG;
    }
    if (d->kv_extent < 1 || d->kv_extent > INT32_MAX) return FD_ERR_INVALID_ARG;
    if (!stride_ok(d->q_stride_b) || !stride_ok(d->q_stride_h)) return FD_ERR_INVALID_ARG;
    const int es = cache_esize(d);
    if (!stride_ok(d->k_stride_b, es) || !stride_ok(d->k_stride_h, es) || !stride_ok(d->k_stride_t, es))
        return FD_ERR_INVALID_ARG;
    if (!stride_ok(d->v_stride_b, es) || !stride_ok(d->v_stride_h, es) || !stride_ok(d->v_stride_t, es))
        return FD_ERR_INVALID_ARG;
    if (d->k_stride_t < kHeadDim || d->v_stride_t < kHeadDim) return FD_ERR_INVALID_ARG;
    if (d->max_seqlen < 0) return FD_ERR_INVALID_ARG;
    return FD_OK;
}

// Split count a call uses: the descriptor's, or the planner's.
int32_t splits_for(const fd_desc* d) {
    if (d->n_splits >= 1) return d->n_splits;
    return fdk::plan_launch(d->batch, d->n_kv_heads, cols_of(d), is_fp8(d),
                            (d->flags & FD_FLAG_CUDA_CORES) != 0, d->max_seqlen, 0);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name, int version) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<Fn>(p);
    return nullptr;
}

// 4-D map over one cache: dims (head_dim, tokens, kv heads, sequences|pages),
// 128-byte swizzle, zero fill outside.  Box: (64 dims, rows, 1, 1) of 16-bit
// elements, or (128 dims, rows, 1, 1) of 8-bit ones -- 128 bytes a row either way.
fd_status make_map(CUtensorMap* map, const fd_desc* d, const void* base, int64_t sb, int64_t sh,
                   int64_t st) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return FD_ERR_CUDA;
    const bool paged = d->page_size > 0;
    const int64_t n_tok = paged ? d->page_size : d->kv_extent;
    const int64_t n_outer = paged ? d->kv_extent : (d->batch > 0 ? d->batch : 1);
    const int cols = (d->n_q_heads / d->n_kv_heads) * q_len_of(d);
    const int rows = paged ? (d->page_size < fdk::kPagedBoxRows ? d->page_size : fdk::kPagedBoxRows)
                           : fdk::stage_tokens(is_fp8(d), cols);
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(n_tok),
                          static_cast<cuuint64_t>(d->n_kv_heads), static_cast<cuuint64_t>(n_outer)};
    // byte strides of dims 1..3; a stride of a size-1 dim is never used, but
    // must still be a valid multiple of 16
    const int es = cache_esize(d);
    auto bs = [es](int64_t s) { return static_cast<cuuint64_t>(s > 0 ? s * es : 16); };
    cuuint64_t strides[3] = {bs(st), bs(sh), bs(sb)};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(rows), 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = is_fp8(d) ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : d->kv_dtype == FD_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FD_OK : FD_ERR_INVALID_ARG;
}

// direct (S = 1 only): the split kernel writes out / lse itself, no combine.
fd_status split_impl(const fd_desc* d, int32_t S, const void* q, const void* k, const void* v,
                     const int32_t* seqlens, const int32_t* block_table, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream, bool direct = false,
                     void* out = nullptr, float* lse = nullptr) {
    // a direct one-split launch given no workspace never touches one
    const bool no_ws = direct && S == 1 && out != nullptr && workspace == nullptr;
    if (q == nullptr || k == nullptr || v == nullptr || seqlens == nullptr ||
        (workspace == nullptr && !no_ws))
        return FD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return FD_ERR_INVALID_ARG;
    const bool paged = d->page_size > 0;
    if (paged != (block_table != nullptr)) return FD_ERR_INVALID_ARG;
    const int64_t rows = rows_of(d);
    const WsLayout w = ws_layout(rows, S);
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return FD_ERR_WORKSPACE;
    if (!no_ws && workspace_bytes < w.total) return FD_ERR_WORKSPACE;
    if (d->batch == 0) return FD_OK;
    if (d->batch > 65535 || d->n_kv_heads > 65535)   // grid (S * col_blocks, n_kv_heads, batch)
        return FD_ERR_UNSUPPORTED;

    CUtensorMap tmK, tmV;
    fd_status st = make_map(&tmK, d, k, d->k_stride_b, d->k_stride_h, d->k_stride_t);
    if (st != FD_OK) return st;
    st = make_map(&tmV, d, v, d->v_stride_b, d->v_stride_h, d->v_stride_t);
    if (st != FD_OK) return st;

    fdk::SplitParams p;
    p.q = q;
    p.q_sb = d->q_stride_b;
    p.q_sh = d->q_stride_h;
    p.q_st = q_len_of(d) > 1 ? d->q_stride_t : 0;
    p.group = d->n_q_heads / d->n_kv_heads;
    p.q_len = q_len_of(d);
    p.cols = p.group * p.q_len;
    p.col_blocks = col_blocks_of(d);
    p.seqlens = seqlens;
    p.block_table = block_table;
    p.max_pages = paged ? d->max_pages_per_seq : 0;
    p.page_size = paged ? d->page_size : 0;
    int shift = 0;
    while (paged && (1 << shift) < d->page_size) ++shift;
    p.page_shift = shift;
    p.capacity = paged ? d->max_pages_per_seq * d->page_size : static_cast<int32_t>(d->kv_extent);
    p.n_pages = paged ? static_cast<int32_t>(d->kv_extent) : 0;
    p.n_q_heads = d->n_q_heads;
    p.n_kv_heads = d->n_kv_heads;
    p.batch = d->batch;
    p.n_splits = S;
    // whole 16-token units (8-token pages: 8), the paged box height, so a
    // TMA box never crosses a page and paged and contiguous caches split alike
    p.split_unit = paged && d->page_size < fdk::kSplitUnit ? d->page_size : fdk::kSplitUnit;
    p.drop_first_stage = (d->flags & FD_FLAG_TEST_DROP_FIRST_STAGE) != 0 ? 1 : 0;
    // fp8 cache: key = k_scale x stored, so the scale folds into the score
    // scale; value = v_scale x stored, applied to the split's u
    p.score_scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kHeadDim)) *
                                            (is_fp8(d) ? static_cast<double>(d->k_scale) : 1.0));
    p.v_scale = is_fp8(d) ? d->v_scale : 1.0f;
    char* ws = static_cast<char*>(workspace);
    p.ws_u = no_ws ? nullptr : reinterpret_cast<float*>(ws + w.off_u);
    p.ws_m = no_ws ? nullptr : reinterpret_cast<float*>(ws + w.off_m);
    p.ws_l = no_ws ? nullptr : reinterpret_cast<float*>(ws + w.off_l);
    p.direct = direct && S == 1 && out != nullptr ? 1 : 0;
    p.out_dtype = d->out_dtype == FD_F16 ? 0 : d->out_dtype == FD_BF16 ? 1 : 2;
    p.out = out;
    p.lse = lse;
    const cudaError_t e = fdk::launch_split(tmK, tmV, p, q_type_of(d), is_fp8(d),
                                            (d->flags & FD_FLAG_CUDA_CORES) != 0, d->batch,
                                            d->n_kv_heads, stream);
    return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

fd_status combine_impl(const fd_desc* d, int32_t S, const void* workspace, size_t workspace_bytes,
                       void* out, float* lse, cudaStream_t stream) {
    if (workspace == nullptr || out == nullptr) return FD_ERR_INVALID_ARG;
    const int64_t rows = rows_of(d);
    const WsLayout w = ws_layout(rows, S);
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return FD_ERR_WORKSPACE;
    if (workspace_bytes < w.total) return FD_ERR_WORKSPACE;
    if (rows == 0) return FD_OK;
    if (rows > INT32_MAX) return FD_ERR_UNSUPPORTED;
    const char* ws = static_cast<const char*>(workspace);
    fdk::CombineParams p;
    p.ws_u = reinterpret_cast<const float*>(ws + w.off_u);
    p.ws_m = reinterpret_cast<const float*>(ws + w.off_m);
    p.ws_l = reinterpret_cast<const float*>(ws + w.off_l);
    p.out = out;
    p.lse = lse;
    p.rows = static_cast<int32_t>(rows);
    p.n_splits = S;
    p.out_dtype = d->out_dtype == FD_F16 ? 0 : d->out_dtype == FD_BF16 ? 1 : 2;
    const cudaError_t e = fdk::launch_combine(p, stream);
    return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

// ---- fixed workspace for fd_decode_static (callers that cannot allocate)
// The split states of fd_decode_static live here instead of in a caller
// buffer.  Every device that loads the library holds this array until exit.
static __device__ __align__(256) unsigned char g_static_workspace[FD_STATIC_WORKSPACE_BYTES];

// The array's device address in each CUDA context that used it, looked up
// once per context: the address belongs to the context, and a context that
// is destroyed and created again (cudaDeviceReset) may place it elsewhere.
// (In host code the symbol is only a host-side stand-in; handing it to a
// kernel would read the wrong memory.)
constexpr int kStaticSlots = 64;
std::mutex g_static_mutex;
unsigned long long g_static_ctx[kStaticSlots] = {};
void* g_static_ptr[kStaticSlots] = {};
int g_static_next = 0;

fd_status static_workspace(void** ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FD_ERR_CUDA;
    const unsigned long long ctx = fdk::current_context_id();
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (ctx != 0) {
        for (int i = 0; i < kStaticSlots; ++i)
            if (g_static_ctx[i] == ctx) {
                *ptr = g_static_ptr[i];
                return FD_OK;
            }
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) return FD_ERR_CUDA;
    if (ctx != 0) {   // without a context id every call looks the address up again
        g_static_ctx[g_static_next] = ctx;
        g_static_ptr[g_static_next] = p;
        g_static_next = (g_static_next + 1) % kStaticSlots;
    }
    *ptr = p;
    return FD_OK;
}

}  // namespace

namespace fdk {

unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
        get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    unsigned long long id = 0;
    return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

}  // namespace fdk

extern "C" {

int32_t fd_abi_version(void) { return FD_ABI_VERSION; }

const char* fd_status_string(int32_t s) {
    switch (s) {
        case FD_OK: return "ok";
        case FD_ERR_INVALID_ARG: return "invalid argument";
        case FD_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case FD_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case FD_ERR_CUDA: return "CUDA error";
        case FD_ERR_DEVICE_TIMEOUT: return "a device wait timed out";
        case FD_ERR_DEVICE_BOUNDS: return "a sequence length or page index was out of range";
        default: return "unknown status";
    }
}

size_t fd_workspace_size(const fd_desc* desc, int32_t n_splits) {
    if (check_desc(desc) != FD_OK) return 0;
    int32_t S = n_splits;
    if (S <= 0) S = splits_for(desc);
    if (S < 1 || S > FD_MAX_SPLITS) return 0;
    return ws_layout(rows_of(desc), S).total;
}

fd_status fd_split_states(const fd_desc* desc, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* seqlens, const int32_t* block_table,
                          void* workspace, size_t workspace_bytes, void* stream) {
    fd_status st = check_desc(desc);
    if (st != FD_OK) return st;
    const int32_t S = splits_for(desc);
    if (S < 1) return static_cast<fd_status>(S < 0 ? S : FD_ERR_INVALID_ARG);
    return split_impl(desc, S, q, k_cache, v_cache, seqlens, block_table, workspace,
                      workspace_bytes, static_cast<cudaStream_t>(stream));
}

fd_status fd_combine_states(const fd_desc* desc, const void* workspace, size_t workspace_bytes,
                            void* out, float* lse, void* stream) {
    fd_status st = check_desc(desc);
    if (st != FD_OK) return st;
    if (desc->n_splits < 1) return FD_ERR_INVALID_ARG;
    return combine_impl(desc, desc->n_splits, workspace, workspace_bytes, out, lse,
                        static_cast<cudaStream_t>(stream));
}

fd_status fd_decode(const fd_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* seqlens, const int32_t* block_table, void* out, float* lse,
                    void* workspace, size_t workspace_bytes, void* stream) {
    fd_status st = check_desc(desc);
    if (st != FD_OK) return st;
    if (out == nullptr) return FD_ERR_INVALID_ARG;
    const int32_t S = splits_for(desc);
    if (S < 1) return static_cast<fd_status>(S < 0 ? S : FD_ERR_INVALID_ARG);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // one split: the split kernel writes the result itself (no combine launch)
    st = split_impl(desc, S, q, k_cache, v_cache, seqlens, block_table, workspace, workspace_bytes, s,
                    S == 1, out, lse);
    if (st != FD_OK || S == 1) return st;
    return combine_impl(desc, S, workspace, workspace_bytes, out, lse, s);
}

fd_status fd_decode_static(const fd_desc* desc, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* seqlens, const int32_t* block_table,
                           void* out, float* lse, void* stream) {
    fd_status st = check_desc(desc);
    if (st != FD_OK) return st;
    if (out == nullptr) return FD_ERR_INVALID_ARG;
    const int32_t S = splits_for(desc);
    if (S < 1) return static_cast<fd_status>(S < 0 ? S : FD_ERR_INVALID_ARG);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (S == 1) {
        // one split: the split kernel writes out and lse itself and uses no
        // workspace, so neither the size limit nor the array applies
        return split_impl(desc, 1, q, k_cache, v_cache, seqlens, block_table, nullptr, 0, s, true,
                          out, lse);
    }
    const size_t need = ws_layout(rows_of(desc), S).total;
    if (need > FD_STATIC_WORKSPACE_BYTES) return FD_ERR_WORKSPACE;
    void* ws = nullptr;
    st = static_workspace(&ws);
    if (st != FD_OK) return st;
    st = split_impl(desc, S, q, k_cache, v_cache, seqlens, block_table, ws,
                    FD_STATIC_WORKSPACE_BYTES, s, false, out, lse);
    if (st != FD_OK) return st;
    return combine_impl(desc, S, ws, FD_STATIC_WORKSPACE_BYTES, out, lse, s);
}

int32_t fd_plan_desc(const fd_desc* desc, const int32_t* seqlens_host, int32_t num_sms) {
    fd_status st = check_desc(desc);
    if (st != FD_OK) return st;
    if (desc->batch < 1 || seqlens_host == nullptr) return FD_ERR_INVALID_ARG;
    int64_t max_len = 0;
    for (int32_t b = 0; b < desc->batch; ++b) {
        if (seqlens_host[b] < 0) return FD_ERR_INVALID_ARG;
        if (seqlens_host[b] > max_len) max_len = seqlens_host[b];
    }
    return fdk::plan_launch(desc->batch, desc->n_kv_heads, cols_of(desc), is_fp8(desc),
                            (desc->flags & FD_FLAG_CUDA_CORES) != 0, max_len, num_sms);
}

fd_status fd_decode_status(void* stream) { return fd_device_status(stream, 1); }

fd_status fd_device_status(void* stream, int32_t clear) {
    unsigned v = 0;
    if (fdk::read_status(&v, static_cast<cudaStream_t>(stream), clear != 0) != cudaSuccess)
        return FD_ERR_CUDA;
    if (v & fdk::kStatusTimeoutBit) return FD_ERR_DEVICE_TIMEOUT;
    if (v != 0) return FD_ERR_DEVICE_BOUNDS;
    return FD_OK;
}

}  // extern "C"
