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
// One CTA of 128 threads per row, thread d owning output dim d; warp 0 first
// reduces the per-split scalars.  The kernel is a few hundred bytes per row.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fd_device.cuh"
#include "fd_internal.h"

namespace fdk {

namespace {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplits = 128;

__global__ void __launch_bounds__(kHeadDim) fd_combine_kernel(const CombineParams p) {
    __shared__ float s_w[kMaxSplits];
    __shared__ float s_M, s_L;
    const int row = blockIdx.x;
    const int t = threadIdx.x;
    const int S = p.n_splits;
    const float* mrow = p.ws_m + static_cast<int64_t>(row) * S;
    const float* lrow = p.ws_l + static_cast<int64_t>(row) * S;

    if (t < 32) {
        float M = -INFINITY;
        for (int i = t; i < S; i += 32) M = fmaxf(M, mrow[i]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, o));
        float L = 0.f;
        for (int i = t; i < S; i += 32) {
            const float m = mrow[i];
            const float w = (m == -INFINITY || M == -INFINITY) ? 0.f : fast_exp2((m - M) * kLog2e);
            s_w[i] = w;
            L = fmaf(w, lrow[i], L);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(kFullMask, L, o);
        if (t == 0) {
            s_M = M;
            s_L = L;
        }
    }
    __syncthreads();
    const float M = s_M, L = s_L;
    const float* urow = p.ws_u + static_cast<int64_t>(row) * S * kHeadDim + t;
    float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;   // four chains, fixed order
    int i = 0;
    for (; i + 4 <= S; i += 4) {
        u0 = fmaf(s_w[i + 0], urow[(i + 0) * kHeadDim], u0);
        u1 = fmaf(s_w[i + 1], urow[(i + 1) * kHeadDim], u1);
        u2 = fmaf(s_w[i + 2], urow[(i + 2) * kHeadDim], u2);
        u3 = fmaf(s_w[i + 3], urow[(i + 3) * kHeadDim], u3);
    }
    for (; i < S; ++i) u0 = fmaf(s_w[i], urow[i * kHeadDim], u0);
    const float u = (u0 + u1) + (u2 + u3);
    const bool empty = (M == -INFINITY) || !(L > 0.f);
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

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    fd_combine_kernel<<<p.rows, kHeadDim, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace fdk
