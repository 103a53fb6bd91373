// fd_merge.cuh -- the exact merge of a query row's split states, shared by
// the combine kernel and the fused tail of the split kernel so that both give
// the same bits.
//
// For row r with states (u_i, m_i, l_i), i < S:
//   M = max over non-empty splits of m_i,   w_i = exp(m_i - M)   (0 if m_i = -inf)
//   L = sum_i w_i l_i,   out = sum_i w_i u_i / L,   lse = M + log L
// ("Decode 专项 Attention：把长KV拆开算，再正确合并" §04 and §06: an empty split
// contributes zero and exp(-inf - (-inf)) is never evaluated; "Flash-Decoding:
// Split-KV Attention for Long-Context Decode" §2, numerically stable form).
// A row whose splits are all empty (sequence length 0) gets out = 0 and
// lse = -inf.
//
// 128 threads merge one row: thread (w, lane) accumulates dims 4*lane..+3
// over splits i = w, w+4, ... in that order (merge_accumulate), the four warp
// partials are added in warp order (merge_store).  The order is fixed, so
// results are bitwise repeatable.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fd_device.cuh"
#include "fd_internal.h"

namespace fdk {

constexpr int kMergeWarps = kHeadDim / 32;   // 4
constexpr float kMergeLog2e = 1.4426950408889634f;

// Warp-level: M, L and the weights w[0..S) of one row from its m[0..S), l[0..S).
__device__ __forceinline__ void merge_weights(const float* m, const float* l, int S, float* w,
                                              float* M_out, float* L_out, int lane) {
    float M = -INFINITY;
    for (int i = lane; i < S; i += 32) M = fmaxf(M, m[i]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int i = lane; i < S; i += 32) {
        const float mi = m[i];
        const float wt = (mi == -INFINITY || M == -INFINITY) ? 0.f : fast_exp2((mi - M) * kMergeLog2e);
        w[i] = wt;
        L = fmaf(wt, l[i], L);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
        *M_out = M;
        *L_out = L;
    }
}

// a += wt * u, one split's step of thread (w, lane)'s accumulation
__device__ __forceinline__ void merge_step(float4& a, float wt, const float4& u) {
    a.x = fmaf(wt, u.x, a.x);
    a.y = fmaf(wt, u.y, a.y);
    a.z = fmaf(wt, u.z, a.z);
    a.w = fmaf(wt, u.w, a.w);
}

// Thread t = 32w + lane: the sum of its dim over the four warp partials
// part[0..4)[..] divided by L, written to out[row][t] (and lse[row] by t = 0).
__device__ __forceinline__ void merge_store(const float4 (*part)[32], float M, float L, int t,
                                            int64_t row, void* out, int out_dtype, float* lse) {
    const bool empty = (M == -INFINITY) || !(L > 0.f);
    const int q4 = t >> 2, c = t & 3;   // thread t: component t % 4 of float4 t / 4
    float u = 0.f;
#pragma unroll
    for (int k = 0; k < kMergeWarps; ++k) u += reinterpret_cast<const float*>(&part[k][q4])[c];
    const float o = empty ? 0.f : u / L;
    const int64_t oi = row * kHeadDim + t;
    if (out_dtype == 2)
        static_cast<float*>(out)[oi] = o;
    else if (out_dtype == 0)
        static_cast<__half*>(out)[oi] = __float2half_rn(o);
    else
        static_cast<__nv_bfloat16*>(out)[oi] = __float2bfloat16_rn(o);
    if (lse != nullptr && t == 0) lse[row] = empty ? -INFINITY : M + logf(L);
}

}  // namespace fdk
