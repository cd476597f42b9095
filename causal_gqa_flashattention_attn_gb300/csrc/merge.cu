// merge.cu - LSE-weighted merge of split-K partials.
//
// Follows "splitk_kernels.py" (xformers), _splitK_reduce: per output row the
// maximum partial LSE M, weights w_s = exp(LSE_s - M), O = sum w_s O_s / sum w_s,
// LSE = M + log(sum w_s); a row whose partial LSEs are all -inf gives O = 0
// and LSE = -inf.  One warp per row, lanes across D in float4 chunks; splits
// with LSE = -inf add nothing, whatever bits their O holds (rows of up to 32
// splits and D <= 128 load every partial at once, the rest skip reading them).
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

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Sums over the warp of 16 per-lane values at once: each butterfly step
// halves the values a lane holds (it keeps one half and adds its partner's
// copy of that half), 8 + 4 + 2 + 1 shuffles, and a last one joins the two
// lanes that share a value.  Lanes 2u and 2u + 1 return the sum of value u.
__device__ __forceinline__ float warp_sum16(const float (&v)[16], int lane) {
    float a[8], b[4], c[2];
    const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = (u16 ? v[i + 8] : v[i]) + __shfl_xor_sync(0xffffffffu, u16 ? v[i] : v[i + 8], 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = (u8 ? a[i + 4] : a[i]) + __shfl_xor_sync(0xffffffffu, u8 ? a[i] : a[i + 4], 8);
#pragma unroll
    for (int i = 0; i < 2; ++i) c[i] = (u4 ? b[i + 2] : b[i]) + __shfl_xor_sync(0xffffffffu, u4 ? b[i] : b[i + 2], 4);
    float d = (u2 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, u2 ? c[0] : c[1], 2);
    return d + __shfl_xor_sync(0xffffffffu, d, 1);
}

constexpr int kBatch = 8;   // splits whose loads are in flight together
constexpr int kFastSplits = 16;   // rows of at most this many splits load everything at once

// Weighted sum over the splits of lane chunk `d` of a row: lane j of each
// block of 32 splits holds the weight of split s0 + j; loads of kBatch splits
// are issued together, and splits of weight 0 (LSE = -inf) are not read.
__device__ __forceinline__ float4 weighted_sum(const float* op, const float* lp, int S, int D, int d, float mx,
                                               int lane) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += 32) {
        const int s = s0 + lane;
        const float l = s < S ? lp[s] : -INFINITY;
        const float w = (l == -INFINITY) ? 0.f : expf(l - mx);
        const int n = min(32, S - s0);
        for (int j0 = 0; j0 < n; j0 += kBatch) {
            float wj[kBatch];
            float4 v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                wj[u] = __shfl_sync(0xffffffffu, w, (j0 + u) & 31);
                const bool take = (j0 + u < n) && wj[u] != 0.f && d < D;
                v[u] = take ? ld4(op + static_cast<size_t>(s0 + j0 + u) * D + d) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                acc.x = fmaf(wj[u], v[u].x, acc.x);
                acc.y = fmaf(wj[u], v[u].y, acc.y);
                acc.z = fmaf(wj[u], v[u].z, acc.z);
                acc.w = fmaf(wj[u], v[u].w, acc.w);
            }
        }
    }
    return acc;
}

// max partial LSE and sum of the weights exp(LSE_s - max) of a row
__device__ __forceinline__ void row_weights(const float* lp, int S, int lane, float& mx, float& wsum) {
    mx = -INFINITY;
    for (int s = lane; s < S; s += 32) mx = fmaxf(mx, lp[s]);
    mx = warp_max(mx);
    wsum = 0.f;
    if (mx != -INFINITY)
        for (int s = lane; s < S; s += 32) {
            const float l = lp[s];
            if (l != -INFINITY) wsum += expf(l - mx);
        }
    wsum = warp_sum(wsum);
}

// A row of at most kN splits with D <= 128: the partial LSEs (one per lane)
// and every partial-O chunk are loaded at once, so the row costs one round
// trip; the same weights, sums and order as the general path.
template <int kN, typename OutT>
__device__ __forceinline__ void merge_row_at_once(const float* op, const float* lp, int S, int D, OutT* orow,
                                                  float* lse, int row, int lane) {
    const int d = 4 * lane;
    const float l = lane < S ? lp[lane] : -INFINITY;
    float4 v[kN];
#pragma unroll
    for (int u = 0; u < kN; ++u)
        v[u] = (u < S && d < D) ? ld4(op + static_cast<size_t>(u) * D + d) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float mx = warp_max(l);
    const bool alive = mx != -INFINITY;
    const float w = (l == -INFINITY) ? 0.f : expf(l - mx);
    const float wsum = warp_sum(w);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < kN; ++u) {
        const float wu = __shfl_sync(0xffffffffu, w, u);
        if (wu != 0.f) {   // splits of weight 0 may hold any bits
            acc.x = fmaf(wu, v[u].x, acc.x);
            acc.y = fmaf(wu, v[u].y, acc.y);
            acc.z = fmaf(wu, v[u].z, acc.z);
            acc.w = fmaf(wu, v[u].w, acc.w);
        }
    }
    const float inv = alive ? 1.f / wsum : 0.f;
    if (d < D) store4(orow + d, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    if (lse != nullptr && lane == 0) lse[row] = alive ? mx + logf(wsum) : -INFINITY;
}

template <typename OutT>
__global__ void __launch_bounds__(32 * kWarps) lse_merge_kernel(const float* __restrict__ o_part,
                                                                const float* __restrict__ lse_part, int N, int S,
                                                                int D, OutT* __restrict__ o, float* __restrict__ lse) {
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const float* lp = lse_part + static_cast<size_t>(row) * S;
    const float* op = o_part + static_cast<size_t>(row) * S * D;
    OutT* orow = o + static_cast<size_t>(row) * D;
    if (D <= 128 && S <= kFastSplits) {
        merge_row_at_once<kFastSplits>(op, lp, S, D, orow, lse, row, lane);
        return;
    }
    if (D <= 128 && S <= 32) {
        merge_row_at_once<32>(op, lp, S, D, orow, lse, row, lane);
        return;
    }
    float mx, wsum;
    row_weights(lp, S, lane, mx, wsum);
    const bool alive = mx != -INFINITY;
    const float inv = alive ? 1.f / wsum : 0.f;
    for (int c = 0; c < kMaxChunks && 128 * c < D; ++c) {
        const int d = 4 * (lane + 32 * c);
        const float4 acc = alive ? weighted_sum(op, lp, S, D, d, mx, lane) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (d < D) store4(orow + d, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    }
    if (lse != nullptr && lane == 0) lse[row] = alive ? mx + logf(wsum) : -INFINITY;
}

// Gradient of the merge ("splitk_kernels.py", _splitK_reduce_varargs_backward):
// with w_s = exp(LSE_s - LSE) the weight of split s,
//   dO_s = w_s * dO,   dLSE_s = w_s * dLSE + sum_d (O_s - O)_d * w_s * dO_d.
// The merged O and LSE are recomputed here from the partials (fp32), so the
// caller needs to keep only the partials.  One warp per row.
//
// Rows of up to 16 splits with D <= 128: every partial is loaded once, with
// dO, and kept in registers for both the merged O and the dot products.  This
// kernel is separate from the general one so that its register count is its
// own: four CTAs fit on an SM, and 2048 rows take one wave of 152 SMs.
__global__ void __launch_bounds__(32 * kWarps, 4) lse_merge_bwd_short_kernel(
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
    const int d = 4 * lane;
    const float l = lane < S ? lp[lane] : -INFINITY;
    float4 v[kFastSplits];
#pragma unroll
    for (int u = 0; u < kFastSplits; ++u)
        v[u] = (u < S && d < D) ? ld4(op + static_cast<size_t>(u) * D + d) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 g = d < D ? ld4(d_o + static_cast<size_t>(row) * D + d) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float dl = (d_lse != nullptr) ? d_lse[row] : 0.f;
    const float mx = warp_max(l);
    const bool alive = mx != -INFINITY;
    const float w0 = (l == -INFINITY) ? 0.f : expf(l - mx);
    const float wsum = warp_sum(w0);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < kFastSplits; ++u) {
        const float wu = __shfl_sync(0xffffffffu, w0, u);
        if (wu != 0.f) {
            a.x = fmaf(wu, v[u].x, a.x);
            a.y = fmaf(wu, v[u].y, a.y);
            a.z = fmaf(wu, v[u].z, a.z);
            a.w = fmaf(wu, v[u].w, a.w);
        }
    }
    const float inv = alive ? 1.f / wsum : 0.f;
    const float4 o = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
    const float lse = alive ? mx + logf(wsum) : -INFINITY;
    const float wl = (alive && l != -INFINITY) ? expf(l - lse) : 0.f;   // lane s: weight of split s
    // per split, this lane's share of sum_d (O_s - O)_d dO_d; splits past S
    // (zero O, weight 0) give 0
    float dot[kFastSplits];
#pragma unroll
    for (int u = 0; u < kFastSplits; ++u) {
        const float wu = __shfl_sync(0xffffffffu, wl, u);
        const float4 x = wu != 0.f ? v[u] : o;
        dot[u] = (x.x - o.x) * g.x + (x.y - o.y) * g.y + (x.z - o.z) * g.z + (x.w - o.w) * g.w;
        if (u < S && d < D)
            *reinterpret_cast<float4*>(dop + static_cast<size_t>(u) * D + d) =
                make_float4(wu * g.x, wu * g.y, wu * g.z, wu * g.w);
    }
    static_assert(kFastSplits == 16, "warp_sum16 reduces 16 values");
    const float t = warp_sum16(dot, lane);   // lanes 2u, 2u + 1: split u
    const int u = lane >> 1;
    const float wu = __shfl_sync(0xffffffffu, wl, u);
    if ((lane & 1) == 0 && u < S) dlp[u] = wu * (dl + t);
}

// The general case: longer rows, or D > 128, in batches of splits whose loads
// are in flight together.
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
    float mx, wsum;
    row_weights(lp, S, lane, mx, wsum);
    const bool alive = mx != -INFINITY;
    const float inv = alive ? 1.f / wsum : 0.f;
    float4 o[kMaxChunks], g[kMaxChunks];
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
        const int d = 4 * (lane + 32 * c);
        g[c] = d < D ? ld4(d_o + static_cast<size_t>(row) * D + d) : make_float4(0.f, 0.f, 0.f, 0.f);
        o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (alive && 128 * c < D) {
            const float4 a = weighted_sum(op, lp, S, D, d, mx, lane);
            o[c] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
        }
    }
    const float lse = alive ? mx + logf(wsum) : -INFINITY;
    const float dl = (d_lse != nullptr) ? d_lse[row] : 0.f;
    for (int s0 = 0; s0 < S; s0 += kBatch) {
        float w[kBatch], dot[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int s = s0 + u;
            const float l = s < S ? lp[s] : -INFINITY;
            w[u] = (alive && l != -INFINITY) ? expf(l - lse) : 0.f;
            dot[u] = 0.f;
        }
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
            const int d = 4 * (lane + 32 * c);
            if (128 * c >= D) break;
            float4 v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const bool take = w[u] != 0.f && d < D;
                v[u] = take ? ld4(op + static_cast<size_t>(s0 + u) * D + d) : o[c];
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                dot[u] += (v[u].x - o[c].x) * g[c].x + (v[u].y - o[c].y) * g[c].y + (v[u].z - o[c].z) * g[c].z +
                          (v[u].w - o[c].w) * g[c].w;
                if (s0 + u < S && d < D)
                    *reinterpret_cast<float4*>(dop + static_cast<size_t>(s0 + u) * D + d) =
                        make_float4(w[u] * g[c].x, w[u] * g[c].y, w[u] * g[c].z, w[u] * g[c].w);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const float t = warp_sum(dot[u]);
            if (lane == 0 && s0 + u < S) dlp[s0 + u] = w[u] * (dl + t);
        }
    }
}

}  // namespace

cudaError_t launch_merge_bwd(const float* o_part, const float* lse_part, const float* d_o, const float* d_lse, int N,
                             int S, int D, float* d_o_part, float* d_lse_part, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const dim3 grid((N + kWarps - 1) / kWarps);
    if (S <= kFastSplits && D <= 128)
        lse_merge_bwd_short_kernel<<<grid, 32 * kWarps, 0, stream>>>(o_part, lse_part, d_o, d_lse, N, S, D,
                                                                     d_o_part, d_lse_part);
    else
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
