/* fd.h -- split-KV decode attention (Flash-Decoding) for GB300 / sm_103a.
 *
 * One decode step of attention: for every sequence b and query head h, one
 * query row q[b,h,:] attends over the first seqlens[b] keys/values of its KV
 * head in a long fp16 / bf16 cache:
 *
 *     s_j = q . k_j / sqrt(D),   out = sum_j softmax(s)_j v_j,
 *     lse = log sum_j exp(s_j)                       (natural log)
 *
 * ("Flash-Decoding: Split-KV Attention for Long-Context Decode", §1 and §2).
 * The KV sequence of each (b, KV head) is cut into n_splits ranges; one CTA
 * per (split, KV head, b) streams its range with an online softmax and leaves
 * an unnormalised partial state (u, m, ell) in a caller-owned fp32 workspace;
 * a second kernel merges the states exactly with the max-subtracted rule
 * ("Decode 专项 Attention：把长KV拆开算，再正确合并", §04; the Flash-Decoding
 * page, §2 "Numerically stable form").
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Ownership: every pointer is owned by the caller.  The library never
 *    allocates, frees or synchronises device memory or streams in fd_decode /
 *    fd_split_states / fd_combine_states.
 *  - Device pointers: q, k_cache, v_cache, seqlens, block_table, out, lse and
 *    workspace are device addresses on the current CUDA device.  Host pointers
 *    are marked "host".
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *    default stream).  Work is enqueued asynchronously; nothing waits for it.
 *  - Errors: every entry point returns an fd_status (or a negative fd_status
 *    where it returns a count).  Arguments are validated on the host before
 *    anything is enqueued; a rejected call enqueues nothing.  A failed kernel
 *    launch returns FD_ERR_CUDA.  Conditions only the GPU can see (a wait
 *    that timed out, a length or page index out of range) are recorded in a
 *    per-device status word read by fd_device_status(); the kernels never trap.
 *  - Grouped-query attention: n_kv_heads divides n_q_heads, G = n_q_heads /
 *    n_kv_heads, and query head h reads KV head h / G (consecutive query heads
 *    share a KV head).  The G query rows of a group are packed into one CTA so
 *    each K/V tile is read from HBM once per group ("Flash-Decoding ...", §1
 *    GQA note).
 *  - Query blocks: q_len query positions per sequence (1 for a plain decode
 *    step; 2-16 for the short query blocks of speculative verification,
 *    "Flash-Decoding ...", §7 and §9).  Position i of sequence b sees the
 *    first seqlens[b] - q_len + 1 + i keys (the block's own tokens are
 *    already in the cache, in order); a position that sees no key gets
 *    out = 0 and lse = -inf.  Every (position, head) of a KV head's group is
 *    one column of the CTA's tensor-core tile.  Up to 16 columns: one CTA per
 *    split on warp MMAs (an fp8 cache with up to 8 columns: a CTA serves two
 *    splits once splits outnumber SMs).  17-128 columns with a 16-bit cache
 *    (and no FD_FLAG_CUDA_CORES): one CTA per split on tcgen05 MMAs, all
 *    columns as the M rows of one 128-row tile (launched as a persistent grid
 *    of at most one CTA per SM that serves the splits in turn).  Otherwise
 *    ceil(G*q_len/16) CTAs per split, each reading the split's K/V once.
 *  - Supported shapes: head_dim 128; G = n_q_heads / n_kv_heads and q_len
 *    with G*q_len <= 256 and q_len <= 16 (with FD_FLAG_CUDA_CORES: G in
 *    {1, 2, 4, 8}, q_len = 1 and a 16-bit cache); kv_dtype FD_F16, FD_BF16 or
 *    FD_E4M3;
 *    1 <= n_splits <= 128.  Other shapes return FD_ERR_UNSUPPORTED.
 */
#ifndef FD_H_
#define FD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FD_ABI_VERSION 4
#define FD_MAX_SPLITS 128   /* the split-count heuristic's cap ("Flash-Decoding ...", §6) */
#define FD_TILE_TOKENS 128  /* the planner's KV block: n_kv_blocks = ceil(max seqlen / 128)
                               ("Flash-Decoding ...", §6).  Split ranges themselves are
                               balanced whole 16-token units (8 for 8-token pages). */

typedef enum fd_status {
    FD_OK = 0,
    FD_ERR_INVALID_ARG = -1,      /* null pointer, bad size/stride, inconsistent shape */
    FD_ERR_UNSUPPORTED = -2,      /* valid but not implemented (head_dim, G, dtype, page size) */
    FD_ERR_WORKSPACE = -3,        /* workspace missing, too small or misaligned */
    FD_ERR_CUDA = -4,             /* a CUDA runtime / launch error */
    FD_ERR_DEVICE_TIMEOUT = -5,   /* a kernel wait ran past its limit (device status word) */
    FD_ERR_DEVICE_BOUNDS = -6     /* a seqlen or block-table entry was out of range (device status word) */
} fd_status;

/* FD_E4M3: an 8-bit floating-point cache (OCP FP8 E4M3, "fn": no infinities,
 * largest 448).  With it, key j = k_scale * stored key and value j = v_scale *
 * stored value (one scale per tensor, fd_desc.k_scale / v_scale), q has
 * fd_desc.q_dtype (FD_F16 or FD_BF16), and the tensor-core path is used. */
typedef enum fd_dtype { FD_F16 = 0, FD_BF16 = 1, FD_F32 = 2, FD_E4M3 = 3 } fd_dtype;

/* fd_desc.flags bits.  By default the split kernel computes the packed
 * group's QK^T and PV on the tensor cores (warp-level MMA, f32 accumulate).
 * FD_FLAG_CUDA_CORES computes them as FP32 FMAs on the CUDA cores instead:
 * same memory pipeline, same results within the stated tolerance; kept for
 * comparison and profiling. */
#define FD_FLAG_CUDA_CORES 1
/* Test hook for failure detection, never for production: the split kernel
 * does not request its first K/V stage, so the wait for it runs out after its
 * limit (about 2 s), the kernel records FD_ERR_DEVICE_TIMEOUT in the device
 * status word and returns without a fault; out and lse are then unspecified. */
#define FD_FLAG_TEST_DROP_FIRST_STAGE (1 << 16)

/* Problem descriptor: plain data, filled by the caller, read (never kept) by
 * each call.  Strides are in ELEMENTS; the head dimension is always contiguous.
 *
 * q        [batch, q_len, n_q_heads, head_dim]:
 *          q[b,i,h,d] at q + b*q_stride_b + i*q_stride_t + h*q_stride_h + d
 *          (q_len = 1: [batch, n_q_heads, head_dim], q_stride_t unused).
 * Contiguous cache (page_size == 0): key j of (b, KV head g) at
 *          k_cache + b*k_stride_b + g*k_stride_h + j*k_stride_t, j < kv_extent
 *          (e.g. a dense [batch, n_kv_heads, T_max, head_dim] tensor: kv_extent = T_max).
 * Paged cache (page_size > 0): a pool of kv_extent pages; key j of (b, g) at
 *          k_cache + P*k_stride_b + g*k_stride_h + (j % page_size)*k_stride_t,
 *          P = block_table[b*max_pages_per_seq + j / page_size]
 *          (a pool laid out [n_pages, n_kv_heads, page_size, head_dim] or
 *          [n_pages, page_size, n_kv_heads, head_dim]: only the strides differ).
 *          Splits are logical token ranges resolved through the table
 *          ("Flash-Decoding ...", §7 paged-KV row).
 * v_* strides describe v_cache the same way.
 * Alignment (TMA): cache base addresses 16-byte aligned and every stride a
 * multiple of 16 bytes (8 elements of 16 bits, 16 of FD_E4M3); q rows
 * 16-byte aligned. */
typedef struct fd_desc {
    int32_t batch;              /* B >= 0; B = 0 enqueues nothing */
    int32_t n_q_heads;          /* Hq >= 1 */
    int32_t n_kv_heads;         /* Hkv >= 1, divides Hq */
    int32_t head_dim;           /* D; 128 */
    int32_t kv_dtype;           /* fd_dtype of K and V: FD_F16, FD_BF16 (q too) or FD_E4M3 */
    int32_t out_dtype;          /* fd_dtype of out: FD_F32, FD_F16 or FD_BF16 */
    int64_t q_stride_b, q_stride_h;
    int64_t k_stride_b, k_stride_h, k_stride_t;
    int64_t v_stride_b, v_stride_h, v_stride_t;
    int64_t kv_extent;          /* contiguous: tokens per (b, g) row (T_max); paged: pages in the pool */
    int32_t page_size;          /* 0 = contiguous; else tokens per page, a power of two >= 8 */
    int32_t max_pages_per_seq;  /* paged: row length (stride) of block_table */
    int32_t max_seqlen;         /* host-known upper bound of seqlens[]; used when n_splits <= 0 */
    int32_t n_splits;           /* >= 1: use it; <= 0: plan it with fd_plan's rule from max_seqlen */
    int32_t flags;              /* 0, or FD_FLAG_* bits */
    int32_t q_len;              /* query positions per sequence; 0 or 1 = one (plain decode) */
    int64_t q_stride_t;         /* elements between query positions (q_len > 1) */
    int32_t q_dtype;            /* kv_dtype FD_E4M3: fd_dtype of q (FD_F16 or FD_BF16); else unused */
    int32_t reserved;           /* must be 0 */
    float k_scale;              /* kv_dtype FD_E4M3: key = k_scale * stored value; else unused */
    float v_scale;              /* kv_dtype FD_E4M3: value = v_scale * stored value; else unused */
} fd_desc;

/* ABI version of the loaded library (FD_ABI_VERSION at build time). */
int32_t fd_abi_version(void);

/* Static, human-readable text for a status code; never NULL. */
const char* fd_status_string(int32_t status);

/* Number of SMs of CUDA device `device` (-1: the current device), or a
 * negative fd_status. */
int32_t fd_num_sms(int32_t device);

/* Split-count heuristic, "Flash-Decoding ...", §6 "How many splits?":
 * no split when work_items >= 0.8*slots; otherwise, over split counts
 * s = 1 .. min(max_splits, slots, n_kv_blocks) that change the blocks per
 * split, the wave efficiency e(s) = w/ceil(w), w = work_items*s/slots, is
 * computed in IEEE double and the smallest s with e(s) >= 0.85 * max e is
 * returned.  n_kv_blocks = 0 returns 1.  Pure host code (no CUDA call).
 * Returns s >= 1, or FD_ERR_INVALID_ARG for work_items < 1, slots < 1,
 * n_kv_blocks < 0 or max_splits < 1. */
int32_t fd_plan_splits(int64_t work_items, int64_t slots, int64_t n_kv_blocks,
                       int32_t max_splits);

/* n_splits for one decode step ("Flash-Decoding ...", §6 "How many splits?",
 * and its §9 decode contract, which plans before launch from the host-known
 * lengths and, for a paged cache, the block table).
 * It is the split count fd_decode plans for this shape with a 16-bit cache on
 * the default (tensor-core) path and one query position per sequence:
 *     fd_plan_splits(work, slots, ceil(max_b seqlens_host[b] / 128), 128)
 * with G = n_q_heads / n_kv_heads and
 *   - G <= 16: work = batch*n_kv_heads (a CTA serves the whole GQA group,
 *     "Flash-Decoding ...", §1 GQA note) and slots = 2*num_sms (two CTAs per
 *     SM, as the page's §6 dispatcher passes);
 *   - 16 < G <= 128: the tcgen05 CTA of all G columns fills an SM, so
 *     work = batch*n_kv_heads and slots = num_sms;
 *   - G > 128: one CTA per 16 columns, work = batch*n_kv_heads*ceil(G/16),
 *     slots = 2*num_sms.
 * For an fp8 cache, query blocks or FD_FLAG_CUDA_CORES use fd_plan_desc.
 *  seqlens_host      : host int32[batch], lengths >= 0.
 *  block_table_host  : host int32[batch*max_pages_per_seq] of a paged cache, or
 *                      NULL.  It never changes the plan; when given it is
 *                      validated: page_size a power of two >= 8, and for every
 *                      sequence b, ceil(seqlens[b]/page_size) <= max_pages_per_seq
 *                      and those entries >= 0 (the pool size is not known
 *                      here; the kernel checks the upper bound).
 *  page_size, max_pages_per_seq : the paged layout (fd_desc); ignored when
 *                      block_table_host is NULL.
 *  num_sms           : <= 0 queries the current device.
 * The result depends only on batch, G, n_kv_heads, max seqlen and num_sms;
 * head_dim is validated only.  Returns s in [1, 128], or FD_ERR_INVALID_ARG
 * (bad shape, a negative length, a table that misses a page),
 * FD_ERR_UNSUPPORTED (G > 256, 1 < page_size < 8) or FD_ERR_CUDA (no device
 * to count SMs on). */
int32_t fd_plan(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                const int32_t* seqlens_host, const int32_t* block_table_host,
                int32_t page_size, int32_t max_pages_per_seq, int32_t num_sms);

/* The split count fd_decode uses for `desc` when desc->n_splits <= 0 and
 * desc->max_seqlen = max_b seqlens_host[b]: the rule of fd_plan with the
 * CTAs per split of this descriptor's kernel -- G*q_len columns per KV head;
 * one CTA per split up to 16 columns, or for 17-128 columns on a 16-bit
 * cache without FD_FLAG_CUDA_CORES (then one slot per SM); otherwise
 * ceil(G*q_len/16) CTAs per split, two slots per SM.  desc->n_splits and
 * desc->max_seqlen are ignored.  seqlens_host: host int32[desc->batch] >= 0.
 * Returns s in [1, 128] or a negative fd_status. */
int32_t fd_plan_desc(const fd_desc* desc, const int32_t* seqlens_host, int32_t num_sms);

/* Bytes of workspace fd_decode needs for `n_splits` (<= 0: the split count
 * fd_decode would plan).  Layout (all fp32, each section 256-byte aligned,
 * row r = (b*q_len + i)*n_q_heads + h):
 *     u  [rows][n_splits][head_dim]   unnormalised partial outputs
 *     m  [rows][n_splits]             max score of the split (natural units of s)
 *     l  [rows][n_splits]             sum of exp(s - m) over the split
 * with rows = batch*q_len*n_q_heads.
 * An empty split holds u = 0, m = -inf, l = 0.  Returns 0 for an invalid
 * descriptor. */
size_t fd_workspace_size(const fd_desc* desc, int32_t n_splits);

/* The whole decode step: fd_split_states then fd_combine_states on `stream`.
 * With one split (n_splits = 1, given or planned) a row's state is already
 * its result: the split kernel writes out and lse itself (the combine's
 * arithmetic at one split, so the same bits) and the workspace is not used.
 *  q, k_cache, v_cache : device, layouts in fd_desc.
 *  seqlens             : device int32[batch], 0 <= seqlens[b] <= capacity,
 *                        capacity = kv_extent (contiguous) or
 *                        max_pages_per_seq*page_size (paged).
 *  block_table         : device int32[batch*max_pages_per_seq] (paged), else NULL.
 *  out                 : device [batch, q_len, n_q_heads, head_dim], out_dtype, contiguous.
 *  lse                 : device float[batch*q_len*n_q_heads], natural-log LSE of the
 *                        scaled scores; NULL to skip.  A row with seqlens[b] = 0
 *                        gets out = 0 and lse = -inf.
 *  workspace           : device, >= fd_workspace_size(desc, n_splits) bytes,
 *                        256-byte aligned; contents on entry are ignored.
 * Asynchronous; CUDA-graph capturable (no allocation, no synchronisation). */
fd_status fd_decode(const fd_desc* desc, const void* q, const void* k_cache,
                    const void* v_cache, const int32_t* seqlens, const int32_t* block_table,
                    void* out, float* lse, void* workspace, size_t workspace_bytes,
                    void* stream);

/* First half of fd_decode: one CTA per (split, KV head, b) writes the partial
 * states (u, m, l) of every query row of its GQA group into the workspace. */
fd_status fd_split_states(const fd_desc* desc, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* seqlens,
                          const int32_t* block_table, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Second half of fd_decode: merges the n_splits states of each row exactly,
 *   M = max over non-empty splits of m_i,  w_i = exp(m_i - M) (0 if empty),
 *   L = sum w_i l_i,  out = sum w_i u_i / L,  lse = M + log L,
 * and writes out / lse (out = 0, lse = -inf when every split is empty).  The
 * workspace may hold states written by fd_split_states or by the caller in
 * the documented layout, which makes this the standalone state merge.
 * desc->n_splits must be >= 1 here. */
fd_status fd_combine_states(const fd_desc* desc, const void* workspace, size_t workspace_bytes,
                            void* out, float* lse, void* stream);

/* Reads (and with clear != 0 resets) the current device's status word after
 * synchronising `stream`.  FD_OK, FD_ERR_DEVICE_TIMEOUT, FD_ERR_DEVICE_BOUNDS
 * or FD_ERR_CUDA.  The word is sticky across calls until cleared.  The word
 * belongs to the current CUDA context (one per device in the usual case). */
fd_status fd_device_status(void* stream, int32_t clear);

/* The decode status call of the decode contract: fd_device_status(stream, 1),
 * i.e. reads the conditions only the GPU can see (a timed-out wait, a length
 * or page index out of range) and clears them. */
fd_status fd_decode_status(void* stream);

/* Size of the fixed device workspace behind fd_decode_static: 8 MiB, enough
 * for batch*n_q_heads*n_splits up to 16131 query-row splits at head_dim 128
 * (each needs (head_dim + 2) * 4 bytes). */
#define FD_STATIC_WORKSPACE_BYTES (8u << 20)

/* fd_decode for callers that cannot allocate device memory.  The pages
 * describe no such entry point; it is an addition of this library.
 *
 * Some callers cannot call cudaMalloc or any allocator at the moment they
 * decode: code running under a custom allocator that must not be re-entered,
 * embedders that forbid device allocations after start-up, or runtimes that
 * own every byte of device memory themselves.  For them this entry point
 * takes the same descriptor, inputs and outputs as fd_decode but no
 * workspace: the split states live in a fixed FD_STATIC_WORKSPACE_BYTES
 * array of device memory that the library holds on every GPU that loads it,
 * until the process exits.
 *
 *  - It allocates nothing and frees nothing (no cudaMalloc, cudaFree or other
 *    allocating routine).  The first call in a CUDA context (normally: on a
 *    device) looks up the array's device address (cudaGetSymbolAddress) with
 *    that context current, and keeps it for that context; make that first
 *    call before any stream capture.  A context destroyed and created again
 *    (cudaDeviceReset) counts as a new one and is looked up again.
 *  - Problems with more than one split whose workspace (fd_workspace_size)
 *    exceeds FD_STATIC_WORKSPACE_BYTES are rejected with FD_ERR_WORKSPACE
 *    before anything is enqueued.  With one split (given, or planned) the
 *    split kernel writes out and lse itself and the array is not used, so
 *    no size limit applies.
 *  - Every call on a device shares the one array, and the array keeps what
 *    the last call left in it.  The split kernel overwrites every state the
 *    combine reads, so nothing needs clearing between calls, but calls whose
 *    kernels can overlap on the GPU (other streams, other host threads) race
 *    on the array: order them, e.g. issue them on one stream.
 * Arguments, layouts, errors and results are those of fd_decode. */
fd_status fd_decode_static(const fd_desc* desc, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* seqlens,
                           const int32_t* block_table, void* out, float* lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FD_H_ */
