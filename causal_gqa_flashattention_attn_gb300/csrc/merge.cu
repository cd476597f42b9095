// merge.cu - LSE-weighted merge of split-K partials.
//
// Follows "splitk_kernels.py" (xformers), _splitK_reduce: per output row the
// maximum partial LSE M, weights w_s = exp(LSE_s - M), O = sum w_s O_s / sum w_s,
// LSE = M + log(sum w_s); a row whose partial LSEs are all -inf gives O = 0
// and LSE = -inf.  One warp per row, lanes across D in float4 chunks; splits
// with LSE = -inf are skipped without reading their O.
#include <cuda_bf16.h>

#include "common.cuh"

namespace gb300 {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxChunks = 8;  // D <= 1024

__device__ __forceinline__ void store4(float* o, float4 v) { *reinterpret_cast<float4*>(o) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* o, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(o) = u;
}

template <typename OutT>
__global__ void __launch_bounds__(32 * kWarps) lse_merge_kernel(const float* __restrict__ o_part,
                                                                const float* __restrict__ lse_part, int N, int S,
                                                                int D, OutT* __restrict__ o, float* __restrict__ lse) {
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const float* lp = lse_part + static_cast<size_t>(row) * S;
    float mx = -INFINITY;
    for (int s = lane; s < S; s += 32) mx = fmaxf(mx, lp[s]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));

    float4 acc[kMaxChunks];
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (mx != -INFINITY) {
        const float* op = o_part + static_cast<size_t>(row) * S * D;
        for (int s = 0; s < S; ++s) {
            const float l = lp[s];
            if (l == -INFINITY) continue;
            const float w = expf(l - mx);
            wsum += w;
#pragma unroll
            for (int c = 0; c < kMaxChunks; ++c) {
                const int d = 4 * (lane + 32 * c);
                if (d < D) {
                    const float4 v = *reinterpret_cast<const float4*>(op + static_cast<size_t>(s) * D + d);
                    acc[c].x += w * v.x;
                    acc[c].y += w * v.y;
                    acc[c].z += w * v.z;
                    acc[c].w += w * v.w;
                }
            }
        }
    }
    const bool alive = mx != -INFINITY;
    const float inv = alive ? 1.f / wsum : 0.f;
    OutT* orow = o + static_cast<size_t>(row) * D;
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
        const int d = 4 * (lane + 32 * c);
        if (d < D) store4(orow + d, make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv));
    }
    if (lse != nullptr && lane == 0) lse[row] = alive ? mx + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const float* o_part, const float* lse_part, int N, int S, int D, void* o, float* lse,
                         int o_dtype, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const dim3 grid((N + kWarps - 1) / kWarps);
    if (o_dtype == ATTN_BF16)
        lse_merge_kernel<__nv_bfloat16><<<grid, 32 * kWarps, 0, stream>>>(o_part, lse_part, N, S, D,
                                                                          static_cast<__nv_bfloat16*>(o), lse);
    else
        lse_merge_kernel<float><<<grid, 32 * kWarps, 0, stream>>>(o_part, lse_part, N, S, D,
                                                                  static_cast<float*>(o), lse);
    return cudaGetLastError();
}

}  // namespace gb300
