// fd_combine.cu -- exact merge of the split states of each query row.
//
// For row r with states (u_i, m_i, l_i), i < n_splits:
//   M = max over non-empty splits of m_i,   w_i = exp(m_i - M)   (0 if m_i = -inf)
//   L = sum_i w_i l_i,   out = sum_i w_i u_i / L,   lse = M + log L
// ("Decode 专项 Attention：把长KV拆开算，再正确合并" §04 and §06: an empty split
// contributes zero and exp(-inf - (-inf)) is never evaluated; "Flash-Decoding:
// Split-KV Attention for Long-Context Decode" §2, numerically stable form).
// A row whose splits are all empty (sequence length 0) gets out = 0 and
// lse = -inf.  The loop order over splits is fixed, so results are bitwise
// repeatable from run to run.
//
// One CTA of 128 threads per row.  Launched with programmatic stream
// serialization: it becomes resident while the split kernel runs and waits
// (griddepcontrol.wait) for that kernel's states before reading them.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fd_device.cuh"
#include "fd_internal.h"

namespace fdk {

namespace {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplits = 128;
constexpr int kWarps = kHeadDim / 32;   // 4
constexpr int kPre = 9;                 // splits per thread loaded up front (S <= 36: all, so the
                                        // planner's frequent 33 and 34 take one round trip)

// One CTA (4 warps) per row.  Thread (w, lane) accumulates dims 4*lane..+3
// over splits i = w, w+4, ..., so the row's S x 128 partial outputs are all
// in flight at once (up to 36 splits together with m and l); the four warp
// partials are added in a fixed order.
__global__ void __launch_bounds__(kHeadDim) fd_combine_kernel(const CombineParams p) {
    __shared__ float s_m[kMaxSplits], s_w[kMaxSplits], s_l[kMaxSplits];
    __shared__ float4 s_part[kWarps][32];
    __shared__ float s_M, s_L;
    // let the next kernel in the stream get resident, then wait for the split
    // kernel (programmatic dependent launch) before reading its states
    grid_dependency_trigger();
    grid_dependency_wait();

    const int row = blockIdx.x;
    const int t = threadIdx.x;
    const int w = t >> 5, lane = t & 31;
    const int S = p.n_splits;
    // The partial outputs do not depend on m and l: request the first kPre of
    // this thread's splits now, so that they travel with m and l.
    const float4* urow = reinterpret_cast<const float4*>(p.ws_u + static_cast<int64_t>(row) * S * kHeadDim) + lane;
    float4 pre[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int i = w + kWarps * k;
        pre[k] = i < S ? urow[i * (kHeadDim / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (t < S) {
        s_m[t] = p.ws_m[static_cast<int64_t>(row) * S + t];
        s_l[t] = p.ws_l[static_cast<int64_t>(row) * S + t];
    }
    __syncthreads();
    if (w == 0) {
        float M = -INFINITY;
        for (int i = lane; i < S; i += 32) M = fmaxf(M, s_m[i]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, o));
        float L = 0.f;
        for (int i = lane; i < S; i += 32) {
            const float m = s_m[i];
            const float wt = (m == -INFINITY || M == -INFINITY) ? 0.f : fast_exp2((m - M) * kLog2e);
            s_w[i] = wt;
            L = fmaf(wt, s_l[i], L);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(kFullMask, L, o);
        if (lane == 0) {
            s_M = M;
            s_L = L;
        }
    }
    __syncthreads();

    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int i = w + kWarps * k;
        if (i < S) {
            const float wt = s_w[i];
            a.x = fmaf(wt, pre[k].x, a.x);
            a.y = fmaf(wt, pre[k].y, a.y);
            a.z = fmaf(wt, pre[k].z, a.z);
            a.w = fmaf(wt, pre[k].w, a.w);
        }
    }
#pragma unroll 8
    for (int i = w + kWarps * kPre; i < S; i += kWarps) {
        const float wt = s_w[i];
        const float4 u = urow[i * (kHeadDim / 4)];
        a.x = fmaf(wt, u.x, a.x);
        a.y = fmaf(wt, u.y, a.y);
        a.z = fmaf(wt, u.z, a.z);
        a.w = fmaf(wt, u.w, a.w);
    }
    s_part[w][lane] = a;
    __syncthreads();

    const float M = s_M, L = s_L;
    const bool empty = (M == -INFINITY) || !(L > 0.f);
    // thread t writes dim t: component t % 4 of float4 t / 4
    const int q4 = t >> 2, c = t & 3;
    float u = 0.f;
#pragma unroll
    for (int k = 0; k < kWarps; ++k) u += reinterpret_cast<const float*>(&s_part[k][q4])[c];
    const float o = empty ? 0.f : u / L;
    const int64_t oi = static_cast<int64_t>(row) * kHeadDim + t;
    if (p.out_dtype == 2)
        static_cast<float*>(p.out)[oi] = o;
    else if (p.out_dtype == 0)
        static_cast<__half*>(p.out)[oi] = __float2half_rn(o);
    else
        static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
    if (p.lse != nullptr && t == 0) p.lse[row] = empty ? -INFINITY : M + logf(L);
}

// Many rows (query blocks): one warp per row, 16 rows per CTA, so thousands
// of rows fit in one wave of few CTAs (4 rows per CTA measured 0.3-0.7 us
// slower per call at 1024-4096 rows).  Lane l
// holds dims 4l .. 4l + 3 and the m, l of splits l, l + 32, ...; the partial
// outputs of the first kPreRows splits are requested together with m and l
// (one round trip to memory up to 16 splits), the rest kRestRows at a time, and
// they are added in split order.
constexpr int kRowsPerCta = 16;
constexpr int kPreRows = 16;
constexpr int kRestRows = 8;

__global__ void __launch_bounds__(32 * kRowsPerCta) fd_combine_rows_kernel(const CombineParams p) {
    grid_dependency_trigger();
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
    if (row >= p.rows) return;
    const int S = p.n_splits;
    const int64_t base = static_cast<int64_t>(row) * S;
    const float4* urow = reinterpret_cast<const float4*>(p.ws_u + base * kHeadDim) + lane;
    constexpr int kStride = kHeadDim / 4;   // float4s per split
    float4 pre[kPreRows];
#pragma unroll
    for (int k = 0; k < kPreRows; ++k) pre[k] = k < S ? urow[k * kStride] : make_float4(0.f, 0.f, 0.f, 0.f);
    float mv[kMaxSplits / 32], lv[kMaxSplits / 32];
#pragma unroll
    for (int j = 0; j < kMaxSplits / 32; ++j) {
        const int i = lane + 32 * j;
        mv[j] = i < S ? p.ws_m[base + i] : -INFINITY;
        lv[j] = i < S ? p.ws_l[base + i] : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxSplits / 32; ++j) M = fmaxf(M, mv[j]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, o));
    float L = 0.f, wv[kMaxSplits / 32];
#pragma unroll
    for (int j = 0; j < kMaxSplits / 32; ++j) {
        wv[j] = (mv[j] == -INFINITY || M == -INFINITY) ? 0.f : fast_exp2((mv[j] - M) * kLog2e);
        L = fmaf(wv[j], lv[j], L);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(kFullMask, L, o);
    // the weight of split i, held by lane i % 32 in wv[i / 32]
    auto weight = [&](int i) {
        const int j = i >> 5;
        const float x = j == 0 ? wv[0] : j == 1 ? wv[1] : j == 2 ? wv[2] : wv[3];
        return __shfl_sync(kFullMask, x, i & 31);
    };
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kPreRows; ++k) {
        const float wt = weight(k);
        if (k < S) {
            a.x = fmaf(wt, pre[k].x, a.x);
            a.y = fmaf(wt, pre[k].y, a.y);
            a.z = fmaf(wt, pre[k].z, a.z);
            a.w = fmaf(wt, pre[k].w, a.w);
        }
    }
    for (int i0 = kPreRows; i0 < S; i0 += kRestRows) {
        float4 u[kRestRows];
#pragma unroll
        for (int k = 0; k < kRestRows; ++k)
            u[k] = i0 + k < S ? urow[(i0 + k) * kStride] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kRestRows; ++k) {
            const float wt = weight(i0 + k);
            if (i0 + k < S) {
                a.x = fmaf(wt, u[k].x, a.x);
                a.y = fmaf(wt, u[k].y, a.y);
                a.z = fmaf(wt, u[k].z, a.z);
                a.w = fmaf(wt, u[k].w, a.w);
            }
        }
    }
    const bool empty = (M == -INFINITY) || !(L > 0.f);
    const float4 o = empty ? make_float4(0.f, 0.f, 0.f, 0.f) : make_float4(a.x / L, a.y / L, a.z / L, a.w / L);
    const int64_t oi = static_cast<int64_t>(row) * kHeadDim + 4 * lane;
    if (p.out_dtype == 2) {   // out carries only its element alignment: scalar stores
        float* d = static_cast<float*>(p.out) + oi;
        d[0] = o.x;
        d[1] = o.y;
        d[2] = o.z;
        d[3] = o.w;
    } else if (p.out_dtype == 0) {
        __half* d = static_cast<__half*>(p.out) + oi;
        d[0] = __float2half_rn(o.x);
        d[1] = __float2half_rn(o.y);
        d[2] = __float2half_rn(o.z);
        d[3] = __float2half_rn(o.w);
    } else {
        __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p.out) + oi;
        d[0] = __float2bfloat16_rn(o.x);
        d[1] = __float2bfloat16_rn(o.y);
        d[2] = __float2bfloat16_rn(o.z);
        d[3] = __float2bfloat16_rn(o.w);
    }
    if (p.lse != nullptr && lane == 0) p.lse[row] = empty ? -INFINITY : M + logf(L);
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    // a CTA of four warps per row shortens each row's chain when rows are few
    // (a decode step's query heads); with a thousand rows or more, a warp per
    // row keeps the launch to one wave
    if (p.rows >= 1024)
        return launch_pdl(fd_combine_rows_kernel, dim3((p.rows + kRowsPerCta - 1) / kRowsPerCta),
                          dim3(32 * kRowsPerCta), 0, stream, p);
    return launch_pdl(fd_combine_kernel, dim3(p.rows), dim3(kHeadDim), 0, stream, p);
}

}  // namespace fdk
