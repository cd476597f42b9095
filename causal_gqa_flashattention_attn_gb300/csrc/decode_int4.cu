// decode_int4.cu - split-K paged decode over an int4 group-quantised KV cache.
//
// Row format ("splitk_kernels.py", docstring of _fwd_kernel_splitK,
// cast_uint32_to_half2, dequantize): per (token, kv head) a row of int32
// words, first n_groups coefficient words (fp16 scale in the low half, fp16
// offset in the high half), then D/8 code words group by group; nibble j of
// code word w of a group is element 8w+j of that group; value = scale*code +
// offset.
//
// The dequantisation is fused into the tensor-core operands instead of being
// materialised.  Scores use bf16 "code space": a code c becomes the exact
// bf16 value 128 + c by OR-ing the nibble (shifted to bits 0-3) into 0x4300.
// Values use fp16 code space: a code in bits 0-3 of a 16-bit half becomes the
// exact fp16 1024 + c by OR-ing it into 0x6400, a code in bits 4-7 the exact
// 1024 + 16 c (both within the 10 mantissa bits), and codes in the upper byte
// are first moved down by one byte permute, so no shifts.  With sigma_d = 16
// for the codes taken from bits 4-7 and 1 otherwise, the affine map is
// applied where it is cheap:
//   s[h,t]   = sum_g scale_g(t) * (sum_{d in g} q_hd c_td)  +  sum_g offset_g(t) * Qsum_g[h]
//              (computed as scale * (sum q (128 + c)) + (offset - 128 scale) * Qsum)
//   O[h,d]   = (sum_t w_ht (1024 + sigma_d c_td) - 1024 SP_g[h]) / sigma_d + OFF_g[h],
//              w = fp16(p_ht scale_g(t)),  SP_g = sum_t w_ht,  OFF_g = sum_t p_ht offset_g(t)
// where dividing by sigma_d is exact; the per-group affine terms cost a few
// FMAs per (token, head).
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

struct Params {
    const __nv_bfloat16* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    int max_pages, B, Hq, Hkv, num_pages, page_size, split_tokens, max_kv_len, n_split;
    int row_words;   // n_groups + D/8
    int G, nq, rpg, n_rg;   // heads per kv head, queries per sequence, rows per CTA, row groups
    float scale_log2;
    float* o_part;
    float* lse_part;
    int32_t* status;
    FusedOut fused;       // fused merge (counters NULL: partials only)
    int n_arrivals;       // CTAs per (sequence, KV head): splits x row groups
};

__device__ __forceinline__ float lo_half(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu))); }
__device__ __forceinline__ float hi_half(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))); }

// bf16x2 (128 + nibble q of the low half, 128 + nibble q of the high half)
__device__ __forceinline__ uint32_t nib_pair(uint32_t x, int q) {
    return ((x >> (4 * q)) & 0x000F000Fu) | 0x43004300u;
}

// fp16x2 (1024 + c, 1024 + c) of the codes in bits 0-3 of each 16-bit half of x
__device__ __forceinline__ uint32_t nib_lo(uint32_t x) { return (x & 0x000F000Fu) | 0x64006400u; }
// fp16x2 (1024 + 16 c, 1024 + 16 c) of the codes in bits 4-7 of each half
__device__ __forceinline__ uint32_t nib_hi(uint32_t x) { return (x & 0x00F000F0u) | 0x64006400u; }
// the upper byte of each 16-bit half moved to its lower byte (codes 2 and 3 of the half)
__device__ __forceinline__ uint32_t upper_bytes(uint32_t x) { return __byte_perm(x, 0u, 0x4341u); }

// Coordinates of the K-side operand of group-local k-step `ks` for lane
// quad index t: the code word (within the group) and the first nibble pair.
template <int NG>
__device__ __forceinline__ void k_word_of(int t, int ks, int& word, int& j0) {
    constexpr int E = kD / NG;        // elements per group
    if constexpr (E == 16) {          // half a word per thread
        word = t >> 1;
        j0 = 2 * (t & 1);
    } else {
        constexpr int WPT = E / 32;   // words per thread per group
        word = t * WPT + (ks >> 1);
        j0 = 2 * (ks & 1);
    }
}

// Row r of a CTA is the (query i, head h) pair rg * rpg + r = i * G + h; with
// one query per sequence the rows are the G heads of the KV group.
template <int R, int NG, int NS, bool kFused>
__global__ void __launch_bounds__(kThreads, (R > 8) ? 1 : 3) decode_int4_kernel(const __grid_constant__ CUtensorMap k_map,
                                                               const __grid_constant__ CUtensorMap v_map,
                                                               const Params p) {
    constexpr bool kTwoRows = (R > 8);
    constexpr int E = kD / NG;                 // elements per group
    constexpr int KS = E / 16;                 // k-steps per group
    constexpr int EPT = E / 8;                 // V elements per lane column per group
    constexpr int BW = (NG <= 4) ? 20 : 24;    // words per smem row (box width)
    constexpr int kTileBytes = kTileTok * BW * 4;
    constexpr int kStageBytes = 2 * kTileBytes;
    constexpr int kCfV = 2 * NG * 16 + 16;     // V half of a coefficient table (16 floats of bank padding)
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
    const int x0 = (kvh * p.row_words) & ~3;      // 16-byte aligned box start
    const int woff = kvh * p.row_words - x0;      // this head's row inside the box

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
                tma_load_2d(st, &k_map, &full_bar[slot], x0, row);
                tma_load_2d(st + kTileBytes, &v_map, &full_bar[slot], x0, row);
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t4 = lane & 3;
    // Q fragments in the nibble order of the K operand, and per-group sums of q
    // (the four lanes of a quad hold every element of a group once between
    // them, so a group's sum is a quad reduction of the fragment values).
    uint32_t qa[NG][KS][4];
    float qsum[NG][2];
    int lim[2];   // each row's last visible token (bottom-right causal: len - q_len + i)
    {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int row = g + 8 * rr;
            const bool real = (rr == 0 || kTwoRows) && row < n_rows;
            const __nv_bfloat16* qrow = p.q + out_row(real ? row : 0) * kD;
            lim[rr] = real ? len - p.nq + (first_row + row) / p.G : -1;
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) {
                float qs = 0.f;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    int word, j0;
                    k_word_of<NG>(t4, ks, word, j0);
                    const int e0 = gr * E + 8 * word + j0;  // element of nibble j0 (even)
                    uint32_t lo_pair = 0u, hi_pair = 0u;
                    if (real) {
                        const uint32_t x0 = *reinterpret_cast<const uint32_t*>(qrow + e0);      // e0, e0+1
                        const uint32_t x4 = *reinterpret_cast<const uint32_t*>(qrow + e0 + 4);  // e0+4, e0+5
                        lo_pair = __byte_perm(x0, x4, 0x5410);   // (e0, e0+4)
                        hi_pair = __byte_perm(x0, x4, 0x7632);   // (e0+1, e0+5)
                        const float2 fl = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&lo_pair));
                        const float2 fh = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi_pair));
                        qs += (fl.x + fl.y) + (fh.x + fh.y);
                    }
                    qa[gr][ks][rr] = lo_pair;        // a0 (row g) / a1 (row g+8): k = 2t, 2t+1
                    qa[gr][ks][rr + 2] = hi_pair;    // a2 / a3: k = 2t+8, 2t+9
                }
                qs += __shfl_xor_sync(0xffffffffu, qs, 1);
                qs += __shfl_xor_sync(0xffffffffu, qs, 2);
                qsum[gr][rr] = qs;
            }
        }
    }
    // smallest causal limit over this CTA's rows (rows are ordered by query)
    const int lim_min = len - p.nq + first_row / p.G;
    constexpr int kRows = kTwoRows ? 2 : 1;
    constexpr int MT = E / 16;                 // 16-row m-tiles of O^T per group
    // O^T accumulators: [head tile of 8][m-tile of 16 head-dim rows][fragment]
    float o_acc[kRows][8][4];
#pragma unroll
    for (int h = 0; h < kRows; ++h)
#pragma unroll
        for (int i = 0; i < 8; ++i) o_acc[h][i][0] = o_acc[h][i][1] = o_acc[h][i][2] = o_acc[h][i][3] = 0.f;
    // running sums of bf16(p * scale_g) and of p * offset_g, per group and row
    float2 sp2[NG][kRows], off2[NG][kRows];
#pragma unroll
    for (int gr = 0; gr < NG; ++gr)
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) sp2[gr][rr] = off2[gr][rr] = make_float2(0.f, 0.f);
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_part[2] = {0.f, 0.f};
    const float sl2 = p.scale_log2;
    // this warp's fp32 coefficient table for its 16 tokens of the current tile,
    // [group][token] blocks: K scale, K offset - 128 * K scale (both times
    // log2 e * softmax scale), then at kCfV: V scale, V offset
    float* cf = reinterpret_cast<float*>(smem + NS * kStageBytes) + warp * (2 * kCfV);

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
            const uint32_t* kt = reinterpret_cast<const uint32_t*>(smem + slot * kStageBytes) + woff;
            const uint32_t* vt = reinterpret_cast<const uint32_t*>(smem + slot * kStageBytes + kTileBytes) + woff;
            // ---- coefficient words -> fp32, once per (token, group); rows past the
            // end of the sequence may hold any bits and get weight 0
            if constexpr (NG % 4 == 0) {
                // rows of n_groups + 16 words start on 16 bytes (the box starts at
                // this head's row): one lane per (K or V, token) takes its row's
                // coefficient words four at a time
                const int kv = lane >> 4, tok = lane & 15;
                const bool ok = tok < n_valid;
                const uint32_t* crow = (kv == 0 ? kt : vt) + (warp * 16 + tok) * BW;
                float* dst = cf + kv * kCfV + tok;
#pragma unroll
                for (int q4 = 0; q4 < NG / 4; ++q4) {
                    const uint4 c4 = *reinterpret_cast<const uint4*>(crow + 4 * q4);
                    const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int gr = 4 * q4 + u;
                        const float sc = ok ? lo_half(cw[u]) : 0.f, of = ok ? hi_half(cw[u]) : 0.f;
                        dst[gr * 16] = kv == 0 ? sc * sl2 : sc;
                        dst[(NG + gr) * 16] = kv == 0 ? fmaf(-128.f, sc, of) * sl2 : of;
                    }
                }
            } else {
#pragma unroll
                for (int i = lane; i < 2 * 16 * NG; i += 32) {
                    const int kv = i / (16 * NG), rem = i % (16 * NG);
                    const int tok = rem / NG, gr = rem % NG;
                    const uint32_t cw = (kv == 0 ? kt : vt)[(warp * 16 + tok) * BW + gr];
                    const bool ok = tok < n_valid;
                    const float sc = ok ? lo_half(cw) : 0.f, of = ok ? hi_half(cw) : 0.f;
                    cf[kv * kCfV + gr * 16 + tok] = kv == 0 ? sc * sl2 : sc;
                    cf[kv * kCfV + (NG + gr) * 16 + tok] = kv == 0 ? fmaf(-128.f, sc, of) * sl2 : of;
                }
            }
            __syncwarp();
            // ---- scores in bf16 code space: per group T_g = sum_d q (128 + c), then
            //      s += scale_g * T_g + (offset_g - 128 scale_g) * Qsum_g
            float2 s2[2][kRows];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int rr = 0; rr < kRows; ++rr) s2[nt][rr] = make_float2(0.f, 0.f);
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    const uint32_t* krow = kt + (warp * 16 + nt * 8 + g) * BW + NG + gr * (E / 8);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        int word, j0;
                        k_word_of<NG>(t4, ks, word, j0);
                        const uint32_t w = krow[word];
                        mma_bf16_16816(acc, qa[gr][ks][0], qa[gr][ks][1], qa[gr][ks][2], qa[gr][ks][3],
                                       nib_pair(w, j0), nib_pair(w, j0 + 1));
                    }
                    const float2 scp = *reinterpret_cast<const float2*>(cf + (0 * NG + gr) * 16 + nt * 8 + 2 * t4);
                    const float2 c2p = *reinterpret_cast<const float2*>(cf + (1 * NG + gr) * 16 + nt * 8 + 2 * t4);
#pragma unroll
                    for (int rr = 0; rr < kRows; ++rr) {
                        s2[nt][rr] = __ffma2_rn(scp, make_float2(acc[2 * rr], acc[2 * rr + 1]), s2[nt][rr]);
                        s2[nt][rr] = __ffma2_rn(c2p, make_float2(qsum[gr][rr], qsum[gr][rr]), s2[nt][rr]);
                    }
                }
            }
            // scores are already in the exp2 domain (the table carries log2(e) * scale)
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                s[nt][0] = s2[nt][0].x;
                s[nt][1] = s2[nt][0].y;
                s[nt][2] = kTwoRows ? s2[nt][kRows - 1].x : 0.f;
                s[nt][3] = kTwoRows ? s2[nt][kRows - 1].y : 0.f;
            }
            // mask only sub-tiles that reach past the split end or some row's causal limit
            if (n_valid < 16 || tok0 + 15 > lim_min) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int tok = nt * 8 + 2 * t4 + (e & 1);
                        if (!(tok < n_valid && tok0 + tok <= lim[e >> 1])) s[nt][e] = -INFINITY;
                    }
            }
            // ---- online softmax (same as the bf16 path)
            float pv[2][4];   // [row][token slot: 2t, 2t+1, 2t+8, 2t+9]
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
            }
            if (__any_sync(0xffffffffu, need_rescale)) {
                // O^T columns are heads 8h + 2t and 8h + 2t + 1; their alphas live
                // in the lanes that hold those heads' score rows
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
#pragma unroll
                for (int gr = 0; gr < NG; ++gr)
#pragma unroll
                    for (int rr = 0; rr < kRows; ++rr) {
                        const float2 a2 = make_float2(alpha[rr], alpha[rr]);
                        sp2[gr][rr] = __fmul2_rn(sp2[gr][rr], a2);
                        off2[gr][rr] = __fmul2_rn(off2[gr][rr], a2);
                    }
            }
            // ---- O^T += (1024 + sigma codes)^T (P * scale_g)^T, group by group: M = 16
            //      head-dim rows, N = 8 heads, K = 16 tokens
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) {
                const float2 scA = *reinterpret_cast<const float2*>(cf + kCfV + gr * 16 + 2 * t4);
                const float2 scC = *reinterpret_cast<const float2*>(cf + kCfV + gr * 16 + 8 + 2 * t4);
                const float2 ofA = *reinterpret_cast<const float2*>(cf + kCfV + (NG + gr) * 16 + 2 * t4);
                const float2 ofC = *reinterpret_cast<const float2*>(cf + kCfV + (NG + gr) * 16 + 8 + 2 * t4);
                uint32_t pa[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int rr = 0; rr < kRows; ++rr) {
                    const float2 pA = make_float2(pv[rr][0], pv[rr][1]), pC = make_float2(pv[rr][2], pv[rr][3]);
                    const __half2 lo2 = __float22half2_rn(__fmul2_rn(pA, scA));
                    const __half2 hi2 = __float22half2_rn(__fmul2_rn(pC, scC));
                    pa[rr] = *reinterpret_cast<const uint32_t*>(&lo2);
                    pa[rr + 2] = *reinterpret_cast<const uint32_t*>(&hi2);
                    sp2[gr][rr] = __fadd2_rn(sp2[gr][rr], __fadd2_rn(__half22float2(lo2), __half22float2(hi2)));
                    off2[gr][rr] = __ffma2_rn(pC, ofC, __ffma2_rn(pA, ofA, off2[gr][rr]));
                }
                // A operand (codes): lane row g supplies elements g*EPT + q of the
                // group, q = 2*mt (m-tile row g) and 2*mt + 1 (m-tile row g + 8)
                const uint32_t* v_a = vt + (warp * 16 + 2 * t4) * BW + NG + gr * (E / 8);      // token 2t
                const uint32_t* v_c = vt + (warp * 16 + 8 + 2 * t4) * BW + NG + gr * (E / 8);  // token 2t+8
#pragma unroll
                for (int j = 0; j < EPT; j += 4) {
                    // nibbles [g*EPT + j, +4) (or +2 when EPT == 2) lie in one 16-bit half
                    const int nib = g * EPT + j;
                    const int word = nib >> 3;
                    const uint32_t sel = (nib & 4) ? 0x7632u : 0x5410u;
                    const uint32_t xa = __byte_perm(v_a[word], v_a[word + BW], sel);  // tokens 2t, 2t+1
                    const uint32_t xc = __byte_perm(v_c[word], v_c[word + BW], sel);  // tokens 2t+8, 2t+9
                    const int q0 = nib & 3;
#pragma unroll
                    for (int jj = 0; jj < (EPT < 4 ? EPT : 4); jj += 2) {
                        const int mt = gr * MT + (j + jj) / 2;
                        // codes q0 + jj (m-tile row g) and q0 + jj + 1 (row g + 8, times 16)
                        const bool upper = (q0 + jj) != 0;
                        const uint32_t ya = upper ? upper_bytes(xa) : xa, yc = upper ? upper_bytes(xc) : xc;
                        const uint32_t a0 = nib_lo(ya), a1 = nib_hi(ya), a2 = nib_lo(yc), a3 = nib_hi(yc);
#pragma unroll
                        for (int h = 0; h < kRows; ++h)
                            mma_f16_16816(o_acc[h][mt], a0, a1, a2, a3, pa[h], pa[h + 2]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }

    // ------------------------------------------- corrections and warp merge
    // OFF_g - 1024 SP_g (codes with sigma 1) and OFF_g - 64 SP_g (sigma 16, the
    // accumulator then divided by 16), summed over the four lanes of a row
    float corr_lo[NG][2], corr_hi[NG][2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        l_part[rr] += __shfl_xor_sync(0xffffffffu, l_part[rr], 1);
        l_part[rr] += __shfl_xor_sync(0xffffffffu, l_part[rr], 2);
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) {
            float off = 0.f, sp = 0.f;
            if (rr < kRows) {
                const float2 sp_v = sp2[gr][rr < kRows ? rr : 0], of_v = off2[gr][rr < kRows ? rr : 0];
                off = of_v.x + of_v.y;
                sp = sp_v.x + sp_v.y;
            }
            off += __shfl_xor_sync(0xffffffffu, off, 1);
            off += __shfl_xor_sync(0xffffffffu, off, 2);
            sp += __shfl_xor_sync(0xffffffffu, sp, 1);
            sp += __shfl_xor_sync(0xffffffffu, sp, 2);
            corr_lo[gr][rr] = fmaf(-1024.f, sp, off);
            corr_hi[gr][rr] = fmaf(-64.f, sp, off);
        }
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
    // O^T fragments: rows are head-dim elements, columns heads 8h + 2t, 8h + 2t + 1
#pragma unroll
    for (int h = 0; h < kRows; ++h) {
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) {
            const float c0 = __shfl_sync(0xffffffffu, corr_lo[gr][h], 8 * t4);
            const float c1 = __shfl_sync(0xffffffffu, corr_lo[gr][h], 8 * t4 + 4);
            const float c0h = __shfl_sync(0xffffffffu, corr_hi[gr][h], 8 * t4);
            const float c1h = __shfl_sync(0xffffffffu, corr_hi[gr][h], 8 * t4 + 4);
            const int head0 = 8 * h + 2 * t4, head1 = head0 + 1;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const float* f = o_acc[h][gr * MT + mt];
                // m-tile rows g (sigma 1) and g + 8 (sigma 16)
                const int d_lo = gr * E + g * EPT + 2 * mt, d_hi = d_lo + 1;
                if (head0 < n_rows) {
                    red_o[(warp * R + head0) * kD + d_lo] = f[0] + c0;
                    red_o[(warp * R + head0) * kD + d_hi] = fmaf(f[2], 0.0625f, c0h);
                }
                if (head1 < n_rows) {
                    red_o[(warp * R + head1) * kD + d_lo] = f[1] + c1;
                    red_o[(warp * R + head1) * kD + d_hi] = fmaf(f[3], 0.0625f, c1h);
                }
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

template <int R, int NG>
cudaError_t launch_g_ng(const DecodeArgs& a, cudaStream_t stream, int* occ) {
    constexpr int NS = 6;
    constexpr int BW = (NG <= 4) ? 20 : 24;
    constexpr int kStageBytes = 2 * kTileTok * BW * 4;
    const int row_words = a.n_groups + a.D / 8;
    const size_t ring = NS * kStageBytes + kConsumers * (4 * NG * 16 + 32) * sizeof(float);
    const size_t red = (kConsumers * R * kD + 2 * kConsumers * R) * sizeof(float);
    const size_t smem = (ring > red ? ring : red) + 1024;
    auto kern = a.counters != nullptr ? decode_int4_kernel<R, NG, NS, true> : decode_int4_kernel<R, NG, NS, false>;
    if (occ != nullptr) return ctas_per_sm(kern, kThreads, smem, occ);
    CUtensorMap k_map, v_map;
    const uint64_t dims[2] = {static_cast<uint64_t>(a.Hkv) * row_words,
                              static_cast<uint64_t>(a.num_pages) * a.page_size};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.Hkv) * row_words * 4};
    const uint32_t box[2] = {BW, kTileTok};
    if (!encode_tiled_map(&k_map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, a.k_cache, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tiled_map(&v_map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, a.v_cache, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
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
    p.row_words = row_words;
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
    // the merge scratch (4 warps x R rows x D floats) reuses the stage ring
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // two CTAs per SM: ask for the largest shared-memory carveout
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    dim3 grid(a.n_split, a.Hkv * p.n_rg, a.B);
    kern<<<grid, kThreads, smem, stream>>>(k_map, v_map, p);
    return cudaGetLastError();
}

template <int R>
cudaError_t launch_g(const DecodeArgs& a, cudaStream_t stream, int* occ) {
    switch (a.n_groups) {
        case 1: return launch_g_ng<R, 1>(a, stream, occ);
        case 2: return launch_g_ng<R, 2>(a, stream, occ);
        case 4: return launch_g_ng<R, 4>(a, stream, occ);
        case 8: return launch_g_ng<R, 8>(a, stream, occ);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode_int4(const DecodeArgs& a, cudaStream_t stream, int* occ) {
    if (decode_int4_g32_supported(a)) return launch_decode_int4_g32(a, stream, occ);
    switch (rows_per_cta(a)) {
        case 1: return launch_g<1>(a, stream, occ);
        case 2: return launch_g<2>(a, stream, occ);
        case 4: return launch_g<4>(a, stream, occ);
        case 8: return launch_g<8>(a, stream, occ);
        case 16: return launch_g<16>(a, stream, occ);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300
