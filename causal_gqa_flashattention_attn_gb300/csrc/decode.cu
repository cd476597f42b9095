// decode.cu - single-query split-K decode over a paged KV cache.
//
// Follows "splitk_kernels.py" (xformers), _fwd_kernel_splitK: one program per
// (split, sequence, head), a chunk of split_tokens keys per split, the block
// table giving the physical page of each page_size tokens, an online softmax
// in the exp2 domain, and an epilogue that writes the split's O already
// divided by its own l plus the split's natural-log LSE (O = 0, LSE = -inf for
// an empty split).
//
// GB300 design (not the pages' design):
//   * one CTA per (split, kv head, sequence) serves all G = Hq/Hkv query heads
//     of the group, so each K/V byte is read from HBM exactly once; with
//     q_len > 1 queries per sequence (causal multi-query decode, the
//     NUM_QUERIES_CAUSAL mode of _fwd_kernel_splitK) a CTA serves up to 16
//     (query, head) rows and query i sees the tokens t <= len - q_len + i;
//   * a producer warp streams 64-token K/V tiles with TMA (128-byte swizzle)
//     through a ring of shared-memory stages, guided by the block table;
//   * four consumer warps each take 16 tokens of a tile and compute the G
//     score rows and the P.V update with m16n8k16 bf16 tensor-core MMAs
//     (heads padded to 16 rows), keeping the online-softmax state in
//     registers; row max / sum reductions are warp shuffles;
//   * the four warps' partial states are merged through shared memory.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "split_merge.cuh"

namespace gb300 {
namespace {

constexpr int kD = 128;                         // head dim handled here
constexpr int kTileTok = 64;                    // tokens per pipeline stage
constexpr int kConsumers = 4;                   // consumer warps
constexpr int kThreads = 32 * (kConsumers + 1); // + 1 producer warp
constexpr int kHalfBytes = kTileTok * 128;      // one 64-column half of a K or V tile
constexpr int kKVTileBytes = 2 * kHalfBytes;    // 16 KB per K (or V) tile
constexpr int kStageBytes = 2 * kKVTileBytes;   // K + V

struct Params {
    const __nv_bfloat16* q;  // [B, Hq, D]
    const int32_t* block_table;
    const int32_t* seq_lens;
    int max_pages, B, Hq, Hkv, num_pages, page_size, split_tokens, max_kv_len, n_split;
    int G, nq, rpg, n_rg;   // heads per kv head, queries per sequence, rows per CTA, row groups
    float scale_log2;
    float* o_part;    // [B, Hq, S, D]
    float* lse_part;  // [B, Hq, S]
    int32_t* status;
    FusedOut fused;       // fused merge (counters NULL: partials only)
    int n_arrivals;       // CTAs per (sequence, KV head): splits x row groups
};

// Byte offset of 16-byte chunk `c` (0..15 across D) of token row `r` inside a
// K or V tile written by TMA with 128-byte swizzle (two 64-column halves).
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
    return (c >> 3) * kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Row r of a CTA is the (query i, head h) pair rg * rpg + r = i * G + h.

template <int R, int NS, bool kFused>
__global__ void __launch_bounds__(kThreads) decode_bf16_kernel(const __grid_constant__ CUtensorMap k_map,
                                                               const __grid_constant__ CUtensorMap v_map,
                                                               const Params p) {
    static_assert(R == 1 || R == 2 || R == 4 || R == 8 || R == 16, "rows per CTA");
    constexpr bool kTwoRows = (R > 8);  // rows g+8 of the m16 fragment are real
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    __shared__ __align__(8) uint64_t full_bar[NS];
    __shared__ __align__(8) uint64_t empty_bar[NS];
    __shared__ int s_abort;
    __shared__ int s_skip[NS];   // stage holds no tile: its page id was out of range

    const int split = blockIdx.x, kvh = blockIdx.y / p.n_rg, rg = blockIdx.y % p.n_rg, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int first_row = rg * p.rpg;
    const int n_rows = min(p.rpg, p.G * p.nq - first_row);
    // output row of CTA row r: ((b * Hq + kvh * G + h) * nq + i), with first_row + r = i * G + h
    auto out_row = [&](int r) -> size_t {
        const int rr = first_row + r, i = rr / p.G, h = rr % p.G;
        return (static_cast<size_t>(b) * p.Hq + kvh * p.G + h) * p.nq + i;
    };

    int len = p.seq_lens[b];
    const int cap = min(p.max_kv_len, p.max_pages * p.page_size);
    if (len < 0 || len > cap) {
        if (threadIdx.x == 0) flag_status(p.status, ATTN_DEV_SEQ_TOO_LONG);
        len = len < 0 ? 0 : cap;
    }
    const int lo = split * p.split_tokens;
    const int hi = min(lo + p.split_tokens, len);
    if (lo >= hi) {  // empty split: O = 0, LSE = -inf
        for (int i = threadIdx.x; i < n_rows * kD; i += kThreads)
            p.o_part[(out_row(i / kD) * p.n_split + split) * kD + (i % kD)] = 0.f;
        if (threadIdx.x < n_rows) p.lse_part[out_row(threadIdx.x) * p.n_split + split] = -INFINITY;
        if constexpr (kFused)
            fused_tail_cta(p.fused, p.n_arrivals, p.status, p.o_part, p.lse_part, p.n_split, b, kvh, p.Hq, p.Hkv, p.G,
                           p.nq, 2, kThreads);
        return;
    }
    const int n_tiles = (hi - lo + kTileTok - 1) / kTileTok;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kConsumers);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumers) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&k_map);
            tma_prefetch_desc(&v_map);
            const int32_t* table = p.block_table + static_cast<size_t>(b) * p.max_pages;
            for (int t = 0; t < n_tiles; ++t) {
                const int slot = t % NS;
                if (t >= NS && !mbar_wait(&empty_bar[slot], ((t / NS) - 1) & 1)) {
                    flag_status(p.status, ATTN_DEV_WAIT_TIMEOUT);
                    atomicExch(&s_abort, 1);
                    break;
                }
                const int tok = lo + t * kTileTok;
                const int page = table[tok / p.page_size];
                if (page < 0 || page >= p.num_pages) {
                    flag_status(p.status, ATTN_DEV_PAGE_OUT_OF_RANGE);
                    s_skip[slot] = 1;               // the consumers leave the page's tokens out
                    mbar_arrive(&full_bar[slot]);  // release the consumers; the tile is not loaded
                    continue;
                }
                const int row = page * p.page_size + tok % p.page_size;
                uint8_t* st = smem + slot * kStageBytes;
                s_skip[slot] = 0;
                mbar_arrive_expect_tx(&full_bar[slot], kStageBytes);
                tma_load_3d(st, &k_map, &full_bar[slot], 0, kvh, row);
                tma_load_3d(st + kHalfBytes, &k_map, &full_bar[slot], 64, kvh, row);
                tma_load_3d(st + kKVTileBytes, &v_map, &full_bar[slot], 0, kvh, row);
                tma_load_3d(st + kKVTileBytes + kHalfBytes, &v_map, &full_bar[slot], 64, kvh, row);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int g = lane >> 2, t4 = lane & 3;
    // Q fragments (A operand, rows = (query, head) pairs, zero past the valid rows),
    // and each row's last visible token (bottom-right causal, len - q_len + i)
    uint32_t qa[8][4];
    int lim[2];
    {
        const bool ok0 = g < n_rows, ok1 = kTwoRows && g + 8 < n_rows;
        const __nv_bfloat16* q0 = p.q + out_row(ok0 ? g : 0) * kD;
        const __nv_bfloat16* q1 = p.q + out_row(ok1 ? g + 8 : 0) * kD;
        lim[0] = ok0 ? len - p.nq + (first_row + g) / p.G : -1;
        lim[1] = ok1 ? len - p.nq + (first_row + g + 8) / p.G : -1;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int d0 = kk * 16 + 2 * t4;
            qa[kk][0] = ok0 ? *reinterpret_cast<const uint32_t*>(q0 + d0) : 0u;
            qa[kk][2] = ok0 ? *reinterpret_cast<const uint32_t*>(q0 + d0 + 8) : 0u;
            qa[kk][1] = ok1 ? *reinterpret_cast<const uint32_t*>(q1 + d0) : 0u;
            qa[kk][3] = ok1 ? *reinterpret_cast<const uint32_t*>(q1 + d0 + 8) : 0u;
        }
    }
    float o_acc[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_part[2] = {0.f, 0.f};
    const float sl2 = p.scale_log2;

    for (int t = 0; t < n_tiles; ++t) {
        const int slot = t % NS;
        if (!mbar_wait(&full_bar[slot], (t / NS) & 1)) {
            flag_status(p.status, ATTN_DEV_WAIT_TIMEOUT);
            break;
        }
        if (s_abort) break;
        const int tok0 = lo + t * kTileTok + warp * 16;
        const int n_valid = min(max(hi - tok0, 0), 16);
        const uint32_t k_s = smem_u32(smem + slot * kStageBytes);
        const uint32_t v_s = k_s + kKVTileBytes;
        if (n_valid > 0 && !s_skip[slot]) {
            if (n_valid < 16) {
                // rows past the end of the sequence: zero V so 0 * garbage stays 0
                uint8_t* vt = smem + slot * kStageBytes + kKVTileBytes;
                for (int i = lane; i < (16 - n_valid) * 16; i += 32) {
                    const int r = warp * 16 + n_valid + i / 16, c = i % 16;
                    *reinterpret_cast<uint4*>(vt + tile_off(r, c)) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            // S = Q K^T for 16 tokens (two n8 tiles), fp32.
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            {
                const int mi = lane >> 3, r = warp * 16 + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(b0, b1, b2, b3, k_s + tile_off(r, 2 * kk + (mi & 1)));
                    mma_bf16_16816(s[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                    mma_bf16_16816(s[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
                }
            }
            // mask tokens past the end and past each row's causal limit, scale to the log2 domain
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = nt * 8 + 2 * t4 + (e & 1);
                    s[nt][e] = (tok < n_valid && tok0 + tok <= lim[e >> 1]) ? s[nt][e] * sl2 : -INFINITY;
                }
            }
            // online softmax per row (row g: e = 0,1; row g+8: e = 2,3)
            uint32_t pa[4];
            bool need_rescale = false;
            float alpha[2] = {1.f, 1.f};
#pragma unroll
            for (int rr = 0; rr < (kTwoRows ? 2 : 1); ++rr) {
                float mx = fmaxf(fmaxf(s[0][2 * rr], s[0][2 * rr + 1]), fmaxf(s[1][2 * rr], s[1][2 * rr + 1]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                // lazy rescale: keep a stale max unless the new one exceeds it by 2^8
                // (a row that sees none of these 16 tokens keeps mx = -inf and p = 0)
                if (mx > m_run[rr] + 8.f) {
                    alpha[rr] = ex2(m_run[rr] - mx);  // 0 when m_run = -inf
                    m_run[rr] = mx;
                    need_rescale = true;
                }
                const float m_use = m_run[rr] == -INFINITY ? 0.f : m_run[rr];
                const float p0 = ex2(s[0][2 * rr] - m_use), p1 = ex2(s[0][2 * rr + 1] - m_use);
                const float p2 = ex2(s[1][2 * rr] - m_use), p3 = ex2(s[1][2 * rr + 1] - m_use);
                l_part[rr] = l_part[rr] * alpha[rr] + ((p0 + p1) + (p2 + p3));
                pa[rr] = pack_bf16x2(p0, p1);
                pa[rr + 2] = pack_bf16x2(p2, p3);
            }
            if (!kTwoRows) {
                pa[1] = 0u;
                pa[3] = 0u;
            }
            if (__any_sync(0xffffffffu, need_rescale)) {
#pragma unroll
                for (int dn = 0; dn < 16; ++dn) {
                    o_acc[dn][0] *= alpha[0];
                    o_acc[dn][1] *= alpha[0];
                    o_acc[dn][2] *= alpha[1];
                    o_acc[dn][3] *= alpha[1];
                }
            }
            // O += P V (A = P from registers, B = V^T via ldmatrix.trans)
            {
                const int mi = lane >> 3, r = warp * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
                for (int dn = 0; dn < 16; dn += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(b0, b1, b2, b3, v_s + tile_off(r, dn + (mi >> 1)));
                    mma_bf16_16816(o_acc[dn], pa[0], pa[1], pa[2], pa[3], b0, b1);
                    mma_bf16_16816(o_acc[dn + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
                }
            }
            if (n_valid < 16) fence_proxy_async_smem();  // generic writes before the next TMA fill
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }

    // ------------------------------------------------------- merge the 4 warps
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        l_part[rr] += __shfl_xor_sync(0xffffffffu, l_part[rr], 1);
        l_part[rr] += __shfl_xor_sync(0xffffffffu, l_part[rr], 2);
    }
    named_barrier_sync(1, 32 * kConsumers);  // every consumer is done with the stages
    float* red_o = reinterpret_cast<float*>(smem);                 // [warp][R][kD]
    float* red_m = red_o + kConsumers * R * kD;                    // [warp][R]
    float* red_l = red_m + kConsumers * R;                         // [warp][R]
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int row = g + rr * 8;
        if (row < n_rows) {
#pragma unroll
            for (int dn = 0; dn < 16; ++dn) {
                const int d = dn * 8 + 2 * t4;
                red_o[(warp * R + row) * kD + d] = o_acc[dn][2 * rr];
                red_o[(warp * R + row) * kD + d + 1] = o_acc[dn][2 * rr + 1];
            }
            if (t4 == 0) {
                red_m[warp * R + row] = m_run[rr];
                red_l[warp * R + row] = l_part[rr];
            }
        }
    }
    named_barrier_sync(1, 32 * kConsumers);
    const int d = threadIdx.x;  // 0..127
    for (int row = 0; row < n_rows; ++row) {
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) mx = fmaxf(mx, red_m[w * R + row]);
        float acc = 0.f, l = 0.f;
        if (mx != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) {
                const float c = ex2(red_m[w * R + row] - mx);
                l += c * red_l[w * R + row];
                acc += c * red_o[(w * R + row) * kD + d];
            }
        }
        const bool alive = l > 0.f;
        const size_t orow = out_row(row) * p.n_split + split;
        p.o_part[orow * kD + d] = alive ? acc / l : 0.f;
        if (d == 0) p.lse_part[orow] = alive ? (mx * kLn2 + logf(l)) : -INFINITY;
    }
    if constexpr (kFused)
        fused_tail_cta(p.fused, p.n_arrivals, p.status, p.o_part, p.lse_part, p.n_split, b, kvh, p.Hq, p.Hkv, p.G,
                       p.nq, 1, 32 * kConsumers);
}

template <int R>
cudaError_t launch_bf16(const DecodeArgs& a, cudaStream_t stream, int* occ) {
    constexpr int NS = 3;
    const size_t smem = NS * kStageBytes + 1024;
    auto kern = a.counters != nullptr ? decode_bf16_kernel<R, NS, true> : decode_bf16_kernel<R, NS, false>;
    if (occ != nullptr) return ctas_per_sm(kern, kThreads, smem, occ);
    CUtensorMap k_map, v_map;
    const uint64_t rows = static_cast<uint64_t>(a.num_pages) * a.page_size;
    const uint64_t dims[3] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(a.Hkv), rows};
    const uint64_t strides[2] = {static_cast<uint64_t>(a.D) * 2, static_cast<uint64_t>(a.Hkv) * a.D * 2};
    const uint32_t box[3] = {64, 1, kTileTok};
    if (!encode_tiled_map(&k_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.k_cache, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled_map(&v_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.v_cache, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    Params p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.block_table = a.block_table;
    p.seq_lens = a.seq_lens;
    p.max_pages = a.max_pages;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.num_pages = a.num_pages;
    p.page_size = a.page_size;
    p.split_tokens = a.split_tokens;
    p.max_kv_len = a.max_kv_len;
    p.n_split = a.n_split;
    p.G = a.Hq / a.Hkv;
    p.nq = a.q_len;
    p.rpg = R;
    p.n_rg = (p.G * p.nq + R - 1) / R;
    p.scale_log2 = a.scale * kLog2e;
    p.o_part = a.o_part;
    p.lse_part = a.lse_part;
    p.status = a.dev_status;
    p.fused.counters = a.counters;
    p.fused.o = static_cast<__nv_bfloat16*>(a.o_final);
    p.fused.lse = a.lse_final;
    p.n_arrivals = a.n_split * p.n_rg;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // two CTAs per SM: ask for the largest shared-memory carveout
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    dim3 grid(a.n_split, a.Hkv * p.n_rg, a.B);
    kern<<<grid, kThreads, smem, stream>>>(k_map, v_map, p);
    return cudaGetLastError();
}

}  // namespace


// Rows per CTA: the (query, head) pairs of one KV head, at most 16.
int rows_per_cta(const DecodeArgs& a) {
    const int rows = (a.Hq / a.Hkv) * a.q_len;
    int r = 1;
    while (r < rows && r < 16) r *= 2;
    return r;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream, int* occ) {
    if (a.kv_format == 1) return launch_decode_int4(a, stream, occ);
    switch (rows_per_cta(a)) {
        case 1: return launch_bf16<1>(a, stream, occ);
        case 2: return launch_bf16<2>(a, stream, occ);
        case 4: return launch_bf16<4>(a, stream, occ);
        case 8: return launch_bf16<8>(a, stream, occ);
        case 16: return launch_bf16<16>(a, stream, occ);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300
