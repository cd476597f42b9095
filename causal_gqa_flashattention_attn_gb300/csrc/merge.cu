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

// Gradient of the merge ("splitk_kernels.py", _splitK_reduce_varargs_backward):
// with w_s = exp(LSE_s - LSE) the weight of split s,
//   dO_s = w_s * dO,   dLSE_s = w_s * dLSE + sum_d (O_s - O)_d * w_s * dO_d.
// The merged O and LSE are recomputed here from the partials (fp32), so the
// caller needs to keep only the partials.  One warp per row.
__global__ void __launch_bounds__(32 * kWarps) lse_merge_bwd_kernel(
    const float* __restrict__ o_part, const float* __restrict__ lse_part, const float* __restrict__ d_o,
    const float* __restrict__ d_lse, int N, int S, int D, float* __restrict__ d_o_part,
    float* __restrict__ d_lse_part) {
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const float* lp = lse_part + static_cast<size_t>(row) * S;
    const float* op = o_part + static_cast<size_t>(row) * S * D;
    float* dop = d_o_part + static_cast<size_t>(row) * S * D;
    float* dlp = d_lse_part + static_cast<size_t>(row) * S;
    float mx = -INFINITY;
    for (int s = lane; s < S; s += 32) mx = fmaxf(mx, lp[s]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float4 o[kMaxChunks], g[kMaxChunks];
    float wsum = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
        o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        const int d = 4 * (lane + 32 * c);
        g[c] = d < D ? *reinterpret_cast<const float4*>(d_o + static_cast<size_t>(row) * D + d)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const bool alive = mx != -INFINITY;
    if (alive) {
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
                    o[c].x += w * v.x;
                    o[c].y += w * v.y;
                    o[c].z += w * v.z;
                    o[c].w += w * v.w;
                }
            }
        }
        const float inv = 1.f / wsum;
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
            o[c].x *= inv;
            o[c].y *= inv;
            o[c].z *= inv;
            o[c].w *= inv;
        }
    }
    const float lse = alive ? mx + logf(wsum) : -INFINITY;
    const float dl = (d_lse != nullptr) ? d_lse[row] : 0.f;
    for (int s = 0; s < S; ++s) {
        const float l = lp[s];
        const bool live = alive && l != -INFINITY;
        const float w = live ? expf(l - lse) : 0.f;
        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
            const int d = 4 * (lane + 32 * c);
            if (d < D) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (live) {
                    v = *reinterpret_cast<const float4*>(op + static_cast<size_t>(s) * D + d);
                    dot += (v.x - o[c].x) * g[c].x + (v.y - o[c].y) * g[c].y + (v.z - o[c].z) * g[c].z +
                           (v.w - o[c].w) * g[c].w;
                }
                *reinterpret_cast<float4*>(dop + static_cast<size_t>(s) * D + d) =
                    make_float4(w * g[c].x, w * g[c].y, w * g[c].z, w * g[c].w);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        if (lane == 0) dlp[s] = w * (dl + dot);
    }
}

}  // namespace

cudaError_t launch_merge_bwd(const float* o_part, const float* lse_part, const float* d_o, const float* d_lse, int N,
                             int S, int D, float* d_o_part, float* d_lse_part, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const dim3 grid((N + kWarps - 1) / kWarps);
    lse_merge_bwd_kernel<<<grid, 32 * kWarps, 0, stream>>>(o_part, lse_part, d_o, d_lse, N, S, D, d_o_part,
                                                           d_lse_part);
    return cudaGetLastError();
}

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
