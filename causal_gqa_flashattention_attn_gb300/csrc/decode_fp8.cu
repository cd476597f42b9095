// decode_fp8.cu - split-K paged decode over an fp8 (e4m3) row-wise quantised KV cache.
//
// Format ("splitk_kernels.py", _fwd_kernel_splitK with FP8_QUANTIZED, the
// K/V_fp8_scale_shift tensors, cast_uint32_to_half2, dequantize): per
// (token, kv head) a row of D e4m3 bytes, and in a separate tensor one
// int32 word per row holding the fp16 scale (low half) and fp16 shift (high
// half); value = fp8 * scale + shift.
//
// e4m3 values are exact in fp16, so the hardware pair conversion
// cvt.rn.f16x2.e4m3x2 feeds fp16 tensor-core MMAs directly and the row's
// affine map is applied outside the MMA, in fp32:
//   s[r,t] = scale(t) * (q_r . x_t) + shift(t) * Qsum_r
//   O[r]   = sum_t (p_rt scale(t)) x_t + sum_t p_rt shift(t)
// Q is converted to fp16 once (|q| must stay below 65504).  The layout of
// work, the TMA ring and the (query, head) rows per CTA are those of the int4
// decode: S = Q K^T with M = rows, O^T = V^T P^T with M = 16 head-dim rows.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "split_merge.cuh"

namespace gb300 {
namespace {

constexpr int kD = 128;
constexpr int kTileTok = 64;
constexpr int kConsumers = 4;
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kCodeBytes = kTileTok * kD;       // 8 KB of e4m3 bytes, 128-byte swizzle
constexpr int kCoefBytes = kTileTok * 16;       // 4 coefficient words per token (this head's at woff)
constexpr int kStageBytes = 2 * kCodeBytes + 2 * kCoefBytes;
constexpr int NS = 4;

struct Params {
    const __nv_bfloat16* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    int max_pages, B, Hq, Hkv, num_pages, page_size, split_tokens, max_kv_len, n_split;
    int G, nq, rpg, n_rg;
    float scale_log2;
    float* o_part;
    float* lse_part;
    int32_t* status;
    FusedOut fused;       // fused merge (counters NULL: partials only)
    int n_arrivals;       // CTAs per (sequence, KV head): splits x row groups
};

__device__ __forceinline__ float lo_half(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
__device__ __forceinline__ float hi_half(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// two e4m3 bytes (low, high of a 16-bit half) -> f16x2
__device__ __forceinline__ uint32_t e4m3x2_lo(uint32_t w) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(w));
    return r;
}
__device__ __forceinline__ uint32_t e4m3x2_hi(uint32_t w) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, hi;\n\t}" : "=r"(r) : "r"(w));
    return r;
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 16-byte chunk c (0..7) of token row r in a 128-byte-swizzled code tile
__device__ __forceinline__ uint32_t code_off(int r, int c) { return r * 128 + (((c ^ (r & 7)) & 7) << 4); }

template <int R, bool kFused>
__global__ void __launch_bounds__(kThreads, (R > 8) ? 1 : 3) decode_fp8_kernel(
    const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
    const __grid_constant__ CUtensorMap kw_map, const __grid_constant__ CUtensorMap vw_map, const Params p) {
    constexpr bool kTwoRows = (R > 8);
    constexpr int kRows = kTwoRows ? 2 : 1;
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
    if (lo >= hi) {
        for (int i = threadIdx.x; i < n_rows * kD; i += kThreads)
            p.o_part[(out_row(i / kD) * p.n_split + split) * kD + (i % kD)] = 0.f;
        if (threadIdx.x < n_rows) p.lse_part[out_row(threadIdx.x) * p.n_split + split] = -INFINITY;
        if constexpr (kFused)
            fused_tail_cta(p.fused, p.n_arrivals, p.status, p.o_part, p.lse_part, p.n_split, b, kvh, p.Hq, p.Hkv, p.G,
                           p.nq, 2, kThreads);
        return;
    }
    const int n_tiles = (hi - lo + kTileTok - 1) / kTileTok;
    const int wx0 = kvh & ~3, woff = kvh & 3;   // 16-byte aligned box of coefficient words

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
        if (lane == 0) {
            tma_prefetch_desc(&k_map);
            tma_prefetch_desc(&v_map);
            tma_prefetch_desc(&kw_map);
            tma_prefetch_desc(&vw_map);
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
                tma_load_3d(st + kCodeBytes, &v_map, &full_bar[slot], 0, kvh, row);
                tma_load_2d(st + 2 * kCodeBytes, &kw_map, &full_bar[slot], wx0, row);
                tma_load_2d(st + 2 * kCodeBytes + kCoefBytes, &vw_map, &full_bar[slot], wx0, row);
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t4 = lane & 3;
    // Q in fp16, in the element order of the K operand: k-step ks, lane t
    // covers bytes 4w .. 4w+3 of word w = 8t + ks of the token row.
    uint32_t qa[8][4];
    float qsum[2];
    int lim[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int row = g + 8 * rr;
        const bool real = (rr == 0 || kTwoRows) && row < n_rows;
        const __nv_bfloat16* qrow = p.q + out_row(real ? row : 0) * kD;
        lim[rr] = real ? len - p.nq + (first_row + row) / p.G : -1;
        // the quad's four lanes hold all D elements between them: the row sum
        // of q is a quad reduction of the fragment values
        float qs = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int e0 = 4 * (8 * t4 + ks);
            uint32_t lo_pair = 0u, hi_pair = 0u;
            if (real) {
                const uint2 x = *reinterpret_cast<const uint2*>(qrow + e0);   // elements e0 .. e0+3
                const float2 f01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
                const float2 f23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
                lo_pair = pack_f16x2(f01.x, f01.y);
                hi_pair = pack_f16x2(f23.x, f23.y);
                qs += (f01.x + f01.y) + (f23.x + f23.y);
            }
            qa[ks][rr] = lo_pair;       // a0 / a1: k = 2t, 2t+1
            qa[ks][rr + 2] = hi_pair;   // a2 / a3: k = 2t+8, 2t+9
        }
        qs += __shfl_xor_sync(0xffffffffu, qs, 1);
        qs += __shfl_xor_sync(0xffffffffu, qs, 2);
        qsum[rr] = qs;
    }
    if (!kTwoRows) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) qa[ks][1] = qa[ks][3] = 0u;
    }
    float o_acc[kRows][8][4];
#pragma unroll
    for (int h = 0; h < kRows; ++h)
#pragma unroll
        for (int i = 0; i < 8; ++i) o_acc[h][i][0] = o_acc[h][i][1] = o_acc[h][i][2] = o_acc[h][i][3] = 0.f;
    float off_acc[2] = {0.f, 0.f};    // sum_t p shift(t), per score row (partial over this lane's tokens)
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
        if (n_valid > 0 && !s_skip[slot]) {
            const uint8_t* kc = smem + slot * kStageBytes;
            const uint8_t* vc = kc + kCodeBytes;
            const uint32_t* kw = reinterpret_cast<const uint32_t*>(kc + 2 * kCodeBytes) + woff;
            const uint32_t* vw = reinterpret_cast<const uint32_t*>(kc + 2 * kCodeBytes + kCoefBytes) + woff;
            const int tk[4] = {2 * t4, 2 * t4 + 1, 8 + 2 * t4, 9 + 2 * t4};
            // ---- scores
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                const int r = warp * 16 + nt * 8 + g;
                const uint4 c0 = *reinterpret_cast<const uint4*>(kc + code_off(r, 2 * t4));
                const uint4 c1 = *reinterpret_cast<const uint4*>(kc + code_off(r, 2 * t4 + 1));
                const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_f16_16816(acc, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], e4m3x2_lo(w[ks]),
                                  e4m3x2_hi(w[ks]));
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = nt * 8 + 2 * t4 + (e & 1);
                    const uint32_t cw = kw[(warp * 16 + tok) * 4];
                    const float v = lo_half(cw) * acc[e] + hi_half(cw) * qsum[e >> 1];
                    s[nt][e] = (tok < n_valid && tok0 + tok <= lim[e >> 1]) ? v * sl2 : -INFINITY;
                }
            }
            // ---- online softmax
            float pv[2][4];
            bool need_rescale = false;
            float alpha[2] = {1.f, 1.f};
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) {
                float mx = fmaxf(fmaxf(s[0][2 * rr], s[0][2 * rr + 1]), fmaxf(s[1][2 * rr], s[1][2 * rr + 1]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                if (mx > m_run[rr] + 8.f) {
                    alpha[rr] = ex2(m_run[rr] - mx);
                    m_run[rr] = mx;
                    need_rescale = true;
                }
                const float m_use = m_run[rr] == -INFINITY ? 0.f : m_run[rr];
                pv[rr][0] = ex2(s[0][2 * rr] - m_use);
                pv[rr][1] = ex2(s[0][2 * rr + 1] - m_use);
                pv[rr][2] = ex2(s[1][2 * rr] - m_use);
                pv[rr][3] = ex2(s[1][2 * rr + 1] - m_use);
                l_part[rr] = l_part[rr] * alpha[rr] + ((pv[rr][0] + pv[rr][1]) + (pv[rr][2] + pv[rr][3]));
                off_acc[rr] *= alpha[rr];
            }
            if (__any_sync(0xffffffffu, need_rescale)) {
#pragma unroll
                for (int h = 0; h < kRows; ++h) {
                    const float a0 = __shfl_sync(0xffffffffu, alpha[h], 8 * t4);
                    const float a1 = __shfl_sync(0xffffffffu, alpha[h], 8 * t4 + 4);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        o_acc[h][i][0] *= a0;
                        o_acc[h][i][1] *= a1;
                        o_acc[h][i][2] *= a0;
                        o_acc[h][i][3] *= a1;
                    }
                }
            }
            // ---- O^T += x^T (P * scale)^T ; shifts summed apart
            float scv[4], shv[4];
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
                const bool ok = tk[e4] < n_valid;   // rows past the end may hold any bits
                const uint32_t cw = vw[(warp * 16 + tk[e4]) * 4];
                scv[e4] = ok ? lo_half(cw) : 0.f;
                shv[e4] = ok ? hi_half(cw) : 0.f;
            }
            uint32_t pb[2][2] = {{0u, 0u}, {0u, 0u}};
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) {
                pb[rr][0] = pack_f16x2(pv[rr][0] * scv[0], pv[rr][1] * scv[1]);
                pb[rr][1] = pack_f16x2(pv[rr][2] * scv[2], pv[rr][3] * scv[3]);
                off_acc[rr] += pv[rr][0] * shv[0] + pv[rr][1] * shv[1] + pv[rr][2] * shv[2] + pv[rr][3] * shv[3];
            }
            // this lane's 16 head-dim elements: chunk g of each token row
            uint4 xv[4];
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
                const int r = warp * 16 + tk[e4];
                xv[e4] = *reinterpret_cast<const uint4*>(vc + code_off(r, g));
                if (tk[e4] >= n_valid) xv[e4] = make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                // rows g, g+8 of m-tile mt are head-dim elements 16g + 2mt and 16g + 2mt + 1
                const int wi = mt >> 1;
                const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
                const uint32_t wa = (&xv[0].x)[wi], wb = (&xv[1].x)[wi], wc = (&xv[2].x)[wi], wd = (&xv[3].x)[wi];
                const uint32_t xab = __byte_perm(wa, wb, sel);   // tokens 2t, 2t+1
                const uint32_t xcd = __byte_perm(wc, wd, sel);   // tokens 2t+8, 2t+9
                const uint32_t a0 = e4m3x2_lo(xab), a1 = e4m3x2_hi(xab);
                const uint32_t a2 = e4m3x2_lo(xcd), a3 = e4m3x2_hi(xcd);
#pragma unroll
                for (int h = 0; h < kRows; ++h) mma_f16_16816(o_acc[h][mt], a0, a1, a2, a3, pb[h][0], pb[h][1]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }

    // ------------------------------------------------------------ warp merge
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        l_part[rr] += __shfl_xor_sync(0xffffffffu, l_part[rr], 1);
        l_part[rr] += __shfl_xor_sync(0xffffffffu, l_part[rr], 2);
        off_acc[rr] += __shfl_xor_sync(0xffffffffu, off_acc[rr], 1);
        off_acc[rr] += __shfl_xor_sync(0xffffffffu, off_acc[rr], 2);
    }
    named_barrier_sync(1, 32 * kConsumers);
    float* red_o = reinterpret_cast<float*>(smem);
    float* red_m = red_o + kConsumers * R * kD;
    float* red_l = red_m + kConsumers * R;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int row = g + rr * 8;
        if (row < n_rows && t4 == 0) {
            red_m[warp * R + row] = m_run[rr];
            red_l[warp * R + row] = l_part[rr];
        }
    }
#pragma unroll
    for (int h = 0; h < kRows; ++h) {
        const float c0 = __shfl_sync(0xffffffffu, off_acc[h], 8 * t4);
        const float c1 = __shfl_sync(0xffffffffu, off_acc[h], 8 * t4 + 4);
        const int row0 = 8 * h + 2 * t4, row1 = row0 + 1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const float* f = o_acc[h][mt];
            const int d_lo = 16 * g + 2 * mt, d_hi = d_lo + 1;
            if (row0 < n_rows) {
                red_o[(warp * R + row0) * kD + d_lo] = f[0] + c0;
                red_o[(warp * R + row0) * kD + d_hi] = f[2] + c0;
            }
            if (row1 < n_rows) {
                red_o[(warp * R + row1) * kD + d_lo] = f[1] + c1;
                red_o[(warp * R + row1) * kD + d_hi] = f[3] + c1;
            }
        }
    }
    named_barrier_sync(1, 32 * kConsumers);
    const int d = threadIdx.x;
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
cudaError_t launch_r(const DecodeArgs& a, const void* k_ss, const void* v_ss, cudaStream_t stream, int* occ) {
    const size_t ring = NS * kStageBytes;
    const size_t red = (kConsumers * R * kD + 2 * kConsumers * R) * sizeof(float);
    const size_t smem = (ring > red ? ring : red) + 1024;
    auto kern = a.counters != nullptr ? decode_fp8_kernel<R, true> : decode_fp8_kernel<R, false>;
    if (occ != nullptr) return ctas_per_sm(kern, kThreads, smem, occ);
    CUtensorMap k_map, v_map, kw_map, vw_map;
    const uint64_t rows = static_cast<uint64_t>(a.num_pages) * a.page_size;
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(a.Hkv), rows};
        const uint64_t strides[2] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(a.Hkv) * a.D};
        const uint32_t box[3] = {kD, 1, kTileTok};
        if (!encode_tiled_map(&k_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.k_cache, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tiled_map(&v_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.v_cache, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(a.Hkv), rows};
        const uint64_t strides[1] = {static_cast<uint64_t>(a.Hkv) * 4};
        const uint32_t box[2] = {4, kTileTok};
        if (!encode_tiled_map(&kw_map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, k_ss, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_tiled_map(&vw_map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, v_ss, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
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
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    dim3 grid(a.n_split, a.Hkv * p.n_rg, a.B);
    kern<<<grid, kThreads, smem, stream>>>(k_map, v_map, kw_map, vw_map, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_fp8(const DecodeArgs& a, const void* k_scale_shift, const void* v_scale_shift,
                              cudaStream_t stream, int* occ) {
    if (decode_fp8_g32_supported(a)) return launch_decode_fp8_g32(a, k_scale_shift, v_scale_shift, stream, occ);
    switch (rows_per_cta(a)) {
        case 1: return launch_r<1>(a, k_scale_shift, v_scale_shift, stream, occ);
        case 2: return launch_r<2>(a, k_scale_shift, v_scale_shift, stream, occ);
        case 4: return launch_r<4>(a, k_scale_shift, v_scale_shift, stream, occ);
        case 8: return launch_r<8>(a, k_scale_shift, v_scale_shift, stream, occ);
        case 16: return launch_r<16>(a, k_scale_shift, v_scale_shift, stream, occ);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300
