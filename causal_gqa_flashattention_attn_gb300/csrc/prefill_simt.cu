// prefill_simt.cu - causal GQA prefill on the CUDA cores, exact fp32 arithmetic.
//
// The computation of "causal_forward_kernel.py",
// _flash_attention_forward_gqa_kernel (online softmax over key blocks, GQA
// head map, O = acc / l, an LSE per row) with the bottom-right visibility of
// "gpt-o3 / triton6fd1ef", _gqa_prefill_kernel (key j visible to query i iff
// j < min(kv_len, i + 1 + delta)).  No tensor cores and no TF32: every product
// and sum is an fp32 FMA/add, so fp32 inputs keep fp32 accuracy.  This path
// serves fp32 inputs and the shapes the tensor-core kernel does not take.
//
// One warp per query row.  Keys go in blocks of 32: lane j scores key j of the
// block against the row's q (kept in shared memory), the block max/sum are
// warp reductions, and for the P.V update lane l owns output columns
// l, l+32, ... and reads V rows coalesced.
#include <cuda_bf16.h>

#include "common.cuh"

namespace gb300 {
namespace {

constexpr int kWarps = 4;

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float v) { *p = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T, int D>
__global__ void __launch_bounds__(32 * kWarps) prefill_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                                   const T* __restrict__ v, T* __restrict__ o,
                                                                   float* __restrict__ lse, int B, int Hq, int Hkv,
                                                                   int q_len, int kv_len, float scale) {
    __shared__ float qs[kWarps][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kWarps + warp;  // over B * Hq * q_len
    const long long n_rows = static_cast<long long>(B) * Hq * q_len;
    if (row >= n_rows) return;
    const int i = static_cast<int>(row % q_len);
    const long long bh = row / q_len;
    const int h = static_cast<int>(bh % Hq);
    const int b = static_cast<int>(bh / Hq);
    const int kvh = h / (Hq / Hkv);
    const int delta = kv_len - q_len;
    const int n_vis = max(0, min(kv_len, i + delta + 1));

    const T* qr = q + row * D;
    const T* kb = k + (static_cast<long long>(b) * Hkv + kvh) * kv_len * D;
    const T* vb = v + (static_cast<long long>(b) * Hkv + kvh) * kv_len * D;
    for (int d = lane; d < D; d += 32) qs[warp][d] = ld(qr + d);
    __syncwarp();

    constexpr int C = D / 32;
    float acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.f;
    float m = -INFINITY, l = 0.f;
    for (int j0 = 0; j0 < n_vis; j0 += 32) {
        const int j = j0 + lane;
        float s = -INFINITY;
        if (j < n_vis) {
            const T* kr = kb + static_cast<long long>(j) * D;
            float dot = 0.f;
#pragma unroll 8
            for (int d = 0; d < D; ++d) dot = fmaf(qs[warp][d], ld(kr + d), dot);
            s = dot * scale;
        }
        float mb = s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
        const float m_new = fmaxf(m, mb);
        const float alpha = expf(m - m_new);  // m = -inf on the first block -> 0
        const float p = j < n_vis ? expf(s - m_new) : 0.f;
        float ps = p;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l = l * alpha + ps;
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] *= alpha;
        const int nb = min(32, n_vis - j0);
        for (int jj = 0; jj < nb; ++jj) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            const T* vr = vb + static_cast<long long>(j0 + jj) * D;
#pragma unroll
            for (int c = 0; c < C; ++c) acc[c] = fmaf(pj, ld(vr + lane + 32 * c), acc[c]);
        }
        m = m_new;
    }
    T* orow = o + row * D;
    const bool alive = n_vis > 0;
#pragma unroll
    for (int c = 0; c < C; ++c) st(orow + lane + 32 * c, alive ? acc[c] / l : 0.f);
    if (lse != nullptr && lane == 0) lse[row] = alive ? m + logf(l) : -INFINITY;
}

template <typename T>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t stream) {
    const long long n_rows = static_cast<long long>(a.B) * a.Hq * a.q_len;
    const dim3 grid(static_cast<unsigned>((n_rows + kWarps - 1) / kWarps));
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);
    T* o = static_cast<T*>(a.o);
    if (a.D == 64)
        prefill_simt_kernel<T, 64><<<grid, 32 * kWarps, 0, stream>>>(q, k, v, o, a.lse, a.B, a.Hq, a.Hkv, a.q_len,
                                                                     a.kv_len, a.scale);
    else
        prefill_simt_kernel<T, 128><<<grid, 32 * kWarps, 0, stream>>>(q, k, v, o, a.lse, a.B, a.Hq, a.Hkv,
                                                                      a.q_len, a.kv_len, a.scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream) {
    if (a.dtype == ATTN_F32) return launch_t<float>(a, stream);
    return launch_t<__nv_bfloat16>(a, stream);
}

}  // namespace gb300
