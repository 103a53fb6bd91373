// fd_combine.cu -- exact merge of the split states of each query row (the
// rule and its citations are in fd_merge.cuh, shared with the fused tail of
// the split kernel).
//
// One CTA of 128 threads per row.  Launched with programmatic stream
// serialization: it becomes resident while the split kernel runs and waits
// (griddepcontrol.wait) for that kernel's states before reading them.
#include "fd_merge.cuh"

namespace fdk {

namespace {

constexpr int kMaxSplits = 128;
constexpr int kPre = 8;                 // splits per thread loaded up front (S <= 32: all)

// Thread (w, lane) accumulates dims 4*lane..+3 over splits i = w, w+4, ...,
// so the row's S x 128 partial outputs are all in flight at once (up to 32
// splits together with m and l); the four warp partials are added in a
// fixed order.
__global__ void __launch_bounds__(kHeadDim) fd_combine_kernel(const CombineParams p) {
    __shared__ float s_m[kMaxSplits], s_w[kMaxSplits], s_l[kMaxSplits];
    __shared__ float4 s_part[kMergeWarps][32];
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
    const float4* urow =
        reinterpret_cast<const float4*>(p.ws_u + static_cast<int64_t>(row) * S * kHeadDim) + lane;
    float4 pre[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int i = w + kMergeWarps * k;
        pre[k] = i < S ? urow[i * (kHeadDim / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (t < S) {
        s_m[t] = p.ws_m[static_cast<int64_t>(row) * S + t];
        s_l[t] = p.ws_l[static_cast<int64_t>(row) * S + t];
    }
    __syncthreads();
    if (w == 0) merge_weights(s_m, s_l, S, s_w, &s_M, &s_L, lane);
    __syncthreads();

    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int i = w + kMergeWarps * k;
        if (i < S) merge_step(a, s_w[i], pre[k]);
    }
#pragma unroll 8
    for (int i = w + kMergeWarps * kPre; i < S; i += kMergeWarps)
        merge_step(a, s_w[i], urow[i * (kHeadDim / 4)]);
    s_part[w][lane] = a;
    __syncthreads();
    merge_store(s_part, s_M, s_L, t, row, p.out, p.out_dtype, p.lse);
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    return launch_pdl(fd_combine_kernel, dim3(p.rows), dim3(kHeadDim), 0, stream, p);
}

}  // namespace fdk
