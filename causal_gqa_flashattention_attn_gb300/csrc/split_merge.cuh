// split_merge.cuh - the fused decode mode: the split that finishes last
// merges a (sequence, KV head)'s split partials inside the decode launch.
//
// The merge is "splitk_kernels.py", _splitK_reduce: per output row the
// maximum partial LSE M, weights w_s = exp(LSE_s - M), O = sum w_s O_s /
// sum w_s, LSE = M + log(sum w_s); a row whose partial LSEs are all -inf gives
// O = 0 and LSE = -inf, and a split of weight 0 adds nothing whatever its O
// holds.
//
// Arrival protocol (no waits): every CTA that has written the partials of its
// rows of a (sequence, KV head) makes them visible device-wide (its threads
// meet, then one thread fences) and adds 1 to that head's counter; the one that brings
// the counter to the number of expected arrivals reads everyone's partials
// from L2, writes O and LSE and puts the counter back to 0, so a workspace
// whose counters start at 0 is left at 0 by every call that completes.  A
// counter found past its range is reported as ATTN_DEV_WORKSPACE_STATE.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace gb300 {

// Arrival of a group of `nthreads` threads (whole warps, meeting at named
// barrier `bar_id`, thread `leader` among them) on `counter`; true in every
// one of them when this group arrived last.  `flag` is a shared word.
// Only the leader fences: the barrier orders every thread's partials before
// the leader's fence, a GPU-scope fence is cumulative (it orders what its
// thread has observed through the barrier, not only its own writes), and the
// fence orders them before the counter update that the last arriver reads.
__device__ __forceinline__ bool split_arrive(int32_t* counter, int expected, int32_t* status, int* flag, int bar_id,
                                             int nthreads, int leader) {
    named_barrier_sync(bar_id, nthreads);
    if (threadIdx.x == leader) {
        __threadfence();
        const int old = atomicAdd(counter, 1);
        if (old >= expected) flag_status(status, ATTN_DEV_WORKSPACE_STATE);
        *flag = old == expected - 1;
    }
    named_barrier_sync(bar_id, nthreads);
    const bool last = *reinterpret_cast<volatile int*>(flag) != 0;
    if (last) __threadfence();
    return last;
}

// One row of a warp's merge, S <= 32 splits (lane j holds split j's LSE),
// the partial O loaded kN splits at a time, all in flight together: one
// round trip per kN splits (D = 128: four elements per lane).  Sums in split
// order, as attn_lse_merge's do.
template <int kN>
__device__ __forceinline__ void merge_row_at_once(const float* o_part, const float* lse_part, int S, size_t row,
                                                  __nv_bfloat16* o, float* lse, int lane) {
    const float l = lane < S ? __ldcg(lse_part + row * S + lane) : -INFINITY;
    float4 v[kN];
#pragma unroll
    for (int u = 0; u < kN; ++u)
        v[u] = u < S ? __ldcg(reinterpret_cast<const float4*>(o_part + (row * S + u) * 128) + lane)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    float mx = l;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float w = (l == -INFINITY || mx == -INFINITY) ? 0.f : expf(l - mx);
    float wsum = w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < S; c0 += kN) {
        if (c0 > 0) {
#pragma unroll
            for (int u = 0; u < kN; ++u)
                v[u] = c0 + u < S ? __ldcg(reinterpret_cast<const float4*>(o_part + (row * S + c0 + u) * 128) + lane)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kN; ++u) {
            const float wu = __shfl_sync(0xffffffffu, w, (c0 + u) & 31);
            if (c0 + u < S && wu != 0.f) {   // a split of weight 0 adds nothing, whatever its O holds
                acc.x = fmaf(wu, v[u].x, acc.x);
                acc.y = fmaf(wu, v[u].y, acc.y);
                acc.z = fmaf(wu, v[u].z, acc.z);
                acc.w = fmaf(wu, v[u].w, acc.w);
            }
        }
    }
    const bool alive = mx != -INFINITY;
    const float inv = alive ? 1.f / wsum : 0.f;
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 u2;
    u2.x = *reinterpret_cast<const uint32_t*>(&a);
    u2.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(o + row * 128 + 4 * lane) = u2;
    if (lse != nullptr && lane == 0) lse[row] = alive ? mx + logf(wsum) : -INFINITY;
}

// One warp merges up to 4 partial rows row0 + k * stride (k < nr; D = 128:
// four elements per lane) of o_part [rows][S][128] / lse_part [rows][S] into
// o [rows][128] (bf16) and lse [rows] (may be NULL).  Partials are read through
// L2 (other SMs wrote them).  Up to 24 splits, a row's partials are loaded in
// one round trip, up to 32 in rounds of 16; more splits go in batches of 4
// splits of all the rows, every load of a batch issued before any is used.  Either way the sums run in
// split order as attn_lse_merge's do.  Not inlined: its registers do not add
// to the decode loop's.
static __device__ __noinline__ void merge_rows_warp(const float* o_part, const float* lse_part, int S, size_t row0,
                                                    size_t stride, int nr, __nv_bfloat16* o, float* lse, int lane) {
    if (S <= 24) {
        for (int k = 0; k < nr; ++k) merge_row_at_once<24>(o_part, lse_part, S, row0 + k * stride, o, lse, lane);
        return;
    }
    if (S <= 32) {
        for (int k = 0; k < nr; ++k) merge_row_at_once<16>(o_part, lse_part, S, row0 + k * stride, o, lse, lane);
        return;
    }
    constexpr int kR = 4, kB = 4;
    float mx[kR], wsum[kR];
    float4 acc[kR];
#pragma unroll
    for (int k = 0; k < kR; ++k) {
        mx[k] = -INFINITY;
        wsum[k] = 0.f;
        acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // the maximum partial LSE of each row
    for (int s0 = 0; s0 < S; s0 += 32) {
        float l[kR];
#pragma unroll
        for (int k = 0; k < kR; ++k)
            l[k] = (k < nr && s0 + lane < S) ? __ldcg(lse_part + (row0 + k * stride) * S + s0 + lane) : -INFINITY;
#pragma unroll
        for (int k = 0; k < kR; ++k) mx[k] = fmaxf(mx[k], l[k]);
    }
#pragma unroll
    for (int k = 0; k < kR; ++k)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], off));
    for (int s0 = 0; s0 < S; s0 += 32) {
        // lane j holds the weight of split s0 + j of each row
        float w[kR];
#pragma unroll
        for (int k = 0; k < kR; ++k) {
            const float l = (k < nr && s0 + lane < S) ? __ldcg(lse_part + (row0 + k * stride) * S + s0 + lane)
                                                      : -INFINITY;
            w[k] = (l == -INFINITY || mx[k] == -INFINITY) ? 0.f : expf(l - mx[k]);
            wsum[k] += w[k];
        }
        const int n = min(32, S - s0);
        for (int j0 = 0; j0 < n; j0 += kB) {
            float4 v[kR][kB];
#pragma unroll
            for (int u = 0; u < kB; ++u)
#pragma unroll
                for (int k = 0; k < kR; ++k)
                    v[k][u] = (k < nr && j0 + u < n)
                                  ? __ldcg(reinterpret_cast<const float4*>(
                                               o_part + ((row0 + k * stride) * S + s0 + j0 + u) * 128) + lane)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < kB; ++u)
#pragma unroll
                for (int k = 0; k < kR; ++k) {
                    const float wu = __shfl_sync(0xffffffffu, w[k], (j0 + u) & 31);
                    if (wu != 0.f) {   // a split of weight 0 adds nothing, whatever its O holds
                        acc[k].x = fmaf(wu, v[k][u].x, acc[k].x);
                        acc[k].y = fmaf(wu, v[k][u].y, acc[k].y);
                        acc[k].z = fmaf(wu, v[k][u].z, acc[k].z);
                        acc[k].w = fmaf(wu, v[k][u].w, acc[k].w);
                    }
                }
        }
    }
#pragma unroll
    for (int k = 0; k < kR; ++k) {
        if (k >= nr) break;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wsum[k] += __shfl_xor_sync(0xffffffffu, wsum[k], off);
        const bool alive = mx[k] != -INFINITY;
        const float inv = alive ? 1.f / wsum[k] : 0.f;
        const __nv_bfloat162 a = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&a);
        u.y = *reinterpret_cast<const uint32_t*>(&b);
        const size_t row = row0 + k * stride;
        *reinterpret_cast<uint2*>(o + row * 128 + 4 * lane) = u;
        if (lse != nullptr && lane == 0) lse[row] = alive ? mx[k] + logf(wsum[k]) : -INFINITY;
    }
}

// Fused-mode outputs of a decode launch.
struct FusedOut {
    int32_t* counters;     // [B * Hkv], zero when the launch starts; NULL: partials only
    __nv_bfloat16* o;      // [B, Hq, q_len, D]
    float* lse;            // [B, Hq, q_len] or NULL
};

// Rows [row0, row0 + n_rows) of a (sequence, KV head), merged by warps
// warp, warp + n_warps, ... of the caller, up to four rows per pass.
__device__ __forceinline__ void merge_head(const float* o_part, const float* lse_part, int S, size_t row0, int n_rows,
                                           const FusedOut& f, int warp, int n_warps, int lane) {
    for (int r = warp; r < n_rows; r += 4 * n_warps)
        merge_rows_warp(o_part, lse_part, S, row0 + r, n_warps, min(4, (n_rows - r + n_warps - 1) / n_warps), f.o,
                        f.lse, lane);
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

// Fused mode of a persistent decode whose CTA takes one unit (sequence, split,
// group of KV heads) at a time, one warp per KV head: after a unit the warps
// have written their rows of the unit's (sequence, head group); the CTA counts
// itself in once (on `cnt`) and, if its split is the last to arrive, every warp
// merges its own head's rows.  `ph` is the phase of the CTA's `unit_bar` (all
// of its warps arrive) and `last_bar` (warp 0 arrives) for this unit.  The
// warps' partials are ordered before warp 0's fence by the warp barrier and the
// CTA's mbarrier; that one fence (cumulative) makes them visible device-wide
// before the count.  Kept out of line so the decode loop's registers do not
// carry any of it.
static __device__ __noinline__ bool unit_fused_tail(FusedOut f, const float* o_part, const float* lse_part,
                                                    int n_split, int32_t* status, int32_t* cnt, size_t row0,
                                                    int n_rows, uint32_t ph, uint64_t* unit_bar, uint64_t* last_bar,
                                                    int* s_last, const int* s_abort, int warp, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(unit_bar);
    if (!mbar_wait(unit_bar, ph, s_abort)) return false;
    if (warp == 0 && lane == 0) {
        __threadfence();
        const int old = atomicAdd(cnt, 1);
        if (old >= n_split) flag_status(status, ATTN_DEV_WORKSPACE_STATE);
        const bool last = old == n_split - 1;
        if (last) atomicExch(cnt, 0);
        *s_last = last;
        mbar_arrive(last_bar);
    }
    if (!mbar_wait(last_bar, ph, s_abort)) return false;
    if (*reinterpret_cast<const volatile int*>(s_last) != 0) {
        __threadfence();
        merge_head(o_part, lse_part, n_split, row0, n_rows, f, 0, 1, lane);
    }
    return true;
}

// Cooperative fused mode of a persistent decode (launched with the
// cooperative attribute, so every CTA of the grid is resident at once): after
// its last unit each CTA sends one thread to a grid barrier made of three words
// of the workspace, zero between launches.  w[0] counts arrivals; the last to
// arrive raises w[1] (release); each CTA that passes counts itself out in
// w[2], and the last to leave puts all three back to zero (no CTA reads them
// after it has left).  Every CTA fences its partials before arriving, the
// waiters acquire w[1], so after the barrier every partial of the launch can be
// read.  A count found out of its range (a workspace that was not zeroed)
// sets ATTN_DEV_WORKSPACE_STATE and that CTA gives up the merge; the wait is
// bounded (ATTN_DEV_WAIT_TIMEOUT).  Either leaves words set: the caller must
// zero the workspace again.  Returns whether the barrier was passed.
__device__ __forceinline__ bool grid_barrier_once(int32_t* w, int32_t* status) {
    const int n = static_cast<int>(gridDim.x);
    __threadfence();
    const int a = atomicAdd(&w[0], 1);
    if (a < 0 || a >= n) {
        flag_status(status, ATTN_DEV_WORKSPACE_STATE);
        return false;
    }
    if (a == n - 1) {
        __threadfence();
        if (atomicExch(&w[1], 1) != 0) flag_status(status, ATTN_DEV_WORKSPACE_STATE);
    } else {
        const uint64_t t0 = global_ns();
        while (ld_acquire_gpu(&w[1]) == 0) {
            if (global_ns() - t0 > kWaitLimitNs) {
                flag_status(status, ATTN_DEV_WAIT_TIMEOUT);
                return false;
            }
            __nanosleep(64);
        }
    }
    __threadfence();
    const int d = atomicAdd(&w[2], 1);
    if (d < 0 || d >= n) {
        flag_status(status, ATTN_DEV_WORKSPACE_STATE);
    } else if (d == n - 1) {
        atomicExch(&w[0], 0);
        atomicExch(&w[1], 0);
        atomicExch(&w[2], 0);
    }
    return true;
}

// The merge of every row of the launch, spread over all the grid's warps
// (`warp` of `n_warps` per CTA): rows [0, n_rows) of o_part / lse_part, row r
// to warp r / gridDim.x of CTA r mod gridDim.x, so every SM takes a share.
__device__ __forceinline__ void grid_merge(const float* o_part, const float* lse_part, int S, int n_rows,
                                           const FusedOut& f, int warp, int n_warps, int lane) {
    const int g = static_cast<int>(gridDim.x);
    for (int r = warp * g + static_cast<int>(blockIdx.x); r < n_rows; r += n_warps * g)
        merge_rows_warp(o_part, lse_part, S, static_cast<size_t>(r), 1, 1, f.o, f.lse, lane);
}

}  // namespace gb300
