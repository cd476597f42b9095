// split_merge.cuh - the fused decode mode: the split that finishes last
// merges a (sequence, KV head)'s split partials inside the decode launch.
//
// The merge is "splitk_kernels.py", _splitK_reduce: per output row the
// maximum partial LSE M, weights w_s = exp(LSE_s - M), O = sum w_s O_s /
// sum w_s, LSE = M + log(sum w_s); a row whose partial LSEs are all -inf gives
// O = 0 and LSE = -inf, and a split of weight 0 adds nothing whatever its O
// holds.
//
// Arrival protocol (no waits): every CTA (or warp) that has written the
// partials of its rows of a (sequence, KV head) makes them visible device-wide
// (threadfence) and then adds 1 to that head's counter; the one that brings
// the counter to the number of expected arrivals reads everyone's partials
// from L2, writes O and LSE and puts the counter back to 0, so a workspace
// whose counters start at 0 is left at 0 by every call that completes.  A
// counter found past its range is reported as ATTN_DEV_WORKSPACE_STATE.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace gb300 {

// Arrival of a group of `nthreads` threads (whole warps, meeting at named
// barrier `bar_id`, thread `leader` among them) on `counter`; true in every
// one of them when this group arrived last.  `flag` is a shared word.
__device__ __forceinline__ bool split_arrive(int32_t* counter, int expected, int32_t* status, int* flag, int bar_id,
                                             int nthreads, int leader) {
    __threadfence();
    named_barrier_sync(bar_id, nthreads);
    if (threadIdx.x == leader) {
        const int old = atomicAdd(counter, 1);
        if (old >= expected) flag_status(status, ATTN_DEV_WORKSPACE_STATE);
        *flag = old == expected - 1;
    }
    named_barrier_sync(bar_id, nthreads);
    const bool last = *reinterpret_cast<volatile int*>(flag) != 0;
    if (last) __threadfence();
    return last;
}

// The same for one warp (lane 0 takes the ticket).
__device__ __forceinline__ bool split_arrive_warp(int32_t* counter, int expected, int32_t* status, int lane) {
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        const int old = atomicAdd(counter, 1);
        if (old >= expected) flag_status(status, ATTN_DEV_WORKSPACE_STATE);
        last = old == expected - 1;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) __threadfence();
    return last != 0;
}

// One warp merges partial row `row` (D = 128: four elements per lane) of
// o_part [rows][S][128] / lse_part [rows][S] into o [rows][128] (bf16) and lse
// [rows] (may be NULL).  Partials are read through L2 (other SMs wrote them).
__device__ __forceinline__ void merge_row_warp(const float* o_part, const float* lse_part, int S, size_t row,
                                               __nv_bfloat16* o, float* lse, int lane) {
    const float* lp = lse_part + row * S;
    const float* op = o_part + row * S * 128;
    float mx = -INFINITY;
    for (int s = lane; s < S; s += 32) mx = fmaxf(mx, __ldcg(lp + s));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const bool alive = mx != -INFINITY;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (alive) {
        for (int s0 = 0; s0 < S; s0 += 32) {
            const int s = s0 + lane;
            const float l = s < S ? __ldcg(lp + s) : -INFINITY;
            const float w = l == -INFINITY ? 0.f : expf(l - mx);
            wsum += w;
            const int n = min(32, S - s0);
            for (int u = 0; u < n; ++u) {
                const float wu = __shfl_sync(0xffffffffu, w, u);
                if (wu != 0.f) {   // splits of weight 0 may hold any bits
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(op + static_cast<size_t>(s0 + u) * 128) + lane);
                    acc.x = fmaf(wu, v.x, acc.x);
                    acc.y = fmaf(wu, v.y, acc.y);
                    acc.z = fmaf(wu, v.z, acc.z);
                    acc.w = fmaf(wu, v.w, acc.w);
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    }
    const float inv = alive ? 1.f / wsum : 0.f;
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(o + row * 128 + 4 * lane) = u;
    if (lse != nullptr && lane == 0) lse[row] = alive ? mx + logf(wsum) : -INFINITY;
}

// Fused-mode outputs of a decode launch.
struct FusedOut {
    int32_t* counters;     // [B * Hkv], zero when the launch starts; NULL: partials only
    __nv_bfloat16* o;      // [B, Hq, q_len, D]
    float* lse;            // [B, Hq, q_len] or NULL
};

// Rows [row0, row0 + n_rows) of a (sequence, KV head), merged by warps
// warp0, warp0 + n_warps, ... of the caller.
__device__ __forceinline__ void merge_head(const float* o_part, const float* lse_part, int S, size_t row0, int n_rows,
                                           const FusedOut& f, int warp, int n_warps, int lane) {
    for (int r = warp; r < n_rows; r += n_warps) merge_row_warp(o_part, lse_part, S, row0 + r, f.o, f.lse, lane);
}

// Fused tail of a decode CTA whose `nthreads` threads (warps 0.., meeting at
// named barrier `bar_id`) have written their partial rows of (sequence b, KV
// head kvh): arrive, and if last, merge the head's G * q_len rows.
__device__ __forceinline__ void fused_tail_cta(const FusedOut& f, int n_arrivals, int32_t* status,
                                               const float* o_part, const float* lse_part, int S, int b, int kvh,
                                               int Hq, int Hkv, int G, int nq, int bar_id, int nthreads) {
    __shared__ int s_last;
    int32_t* cnt = f.counters + static_cast<size_t>(b) * Hkv + kvh;
    if (split_arrive(cnt, n_arrivals, status, &s_last, bar_id, nthreads, 0)) {
        const size_t row0 = (static_cast<size_t>(b) * Hq + static_cast<size_t>(kvh) * G) * nq;
        merge_head(o_part, lse_part, S, row0, G * nq, f, threadIdx.x >> 5, nthreads >> 5, threadIdx.x & 31);
        if (threadIdx.x == 0) atomicExch(cnt, 0);
    }
}

}  // namespace gb300
