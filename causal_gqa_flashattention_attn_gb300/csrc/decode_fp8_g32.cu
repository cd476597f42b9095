// decode_fp8_g32.cu - split-K paged decode over an fp8 (e4m3) row-wise
// quantised KV cache, for KV head counts that are multiples of 8 and at most 8
// (query, head) rows per KV head: persistent, eight KV heads per CTA.
//
// Format ("splitk_kernels.py", _fwd_kernel_splitK with FP8_QUANTIZED, the
// K/V_fp8_scale_shift tensors, cast_uint32_to_half2, dequantize): per
// (token, kv head) a row of D e4m3 bytes, and in a separate tensor one int32
// word per row holding the fp16 scale (low half) and fp16 shift (high half);
// value = fp8 * scale + shift.  The arithmetic is that of decode_fp8.cu: the
// e4m3 bytes become exact fp16 MMA operands by cvt.rn.f16x2.e4m3x2, Q is taken
// in fp16, and the row's affine map is applied outside the MMA in fp32:
//   s[t,r] = scale(t) (q_r . x_t) + shift(t) Qsum_r
//   O[r]   = sum_t fp16(p_rt scale(t)) x_t + sum_t p_rt shift(t)
//
// Work layout (persistent), as in decode_int4_g32.cu: one CTA per SM walks
// work units (sequence, split, group of 8 KV heads); a producer warp streams
// 32-token stages and copies each unit's queries ahead; eight consumer warps
// each own one KV head and every token of the unit (no cross-warp merge), and
// take a stage's 32 tokens as two 16-token sub-tiles.  A stage holds, per
// head, the 32 token rows of K codes and of V codes as one TMA box each
// ({128 bytes, 1 head, 32 tokens}, 128-byte swizzle: a head's rows are
// contiguous, so rows 0-7 sit on eight different swizzle phases and the
// consumers' 16-byte reads are free of bank conflicts) plus the 32 tokens'
// coefficient words of the 8 heads.  HBM is read in full 128-byte lines.
//
//   scores (S^T = K Q^T, M = 16 tokens, N = 8 rows, K = 16 head-dim elements):
//     lane (g, t4) of k-step ks takes bytes 4ks .. 4ks + 3 of its 32-byte slice
//     (elements 32 t4 ..) of token rows g and g + 8: one cvt per half gives the
//     A pairs (k = 2t4, 2t4+1) and (2t4+8, 2t4+9); Q's B fragments use the same
//     element order, so the k order inside an MMA is a permutation of D.
//   values (O^T = V^T W, M = 16 head-dim elements, N = 8 rows, K = 16 tokens):
//     lane (g, t4) reads the 16-byte chunk g (elements 16g ..) of tokens 2t4,
//     2t4+1, 2t4+8, 2t4+9; byte permutes pair two tokens' bytes of one element,
//     so m-tile mt's rows g and g + 8 are elements 16g + 2mt and 16g + 2mt + 1.
//     W = fp16(p scale) is made in the score layout and turned into the B
//     operand (tokens in k) by movmatrix transposes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "split_merge.cuh"

namespace gb300 {
namespace {

constexpr int kD = 128;
constexpr int kHeads = 8;                        // KV heads per CTA: one consumer warp each
constexpr int kTileTok = 32;                     // tokens per stage
constexpr int kHeadTile = kTileTok * kD;         // 4 KB: one head's 32 code rows
constexpr int kCodeTile = kHeads * kHeadTile;    // 32 KB of K (or V) codes
constexpr int kCoefTile = kTileTok * kHeads * 4; // 1 KB of K (or V) coefficient words, [token][head]
constexpr int kOffV = kCodeTile;
constexpr int kOffKw = 2 * kCodeTile;
constexpr int kOffVw = 2 * kCodeTile + kCoefTile;
constexpr int kStageBytes = 2 * kCodeTile + 2 * kCoefTile;
constexpr int kStages = 3;
constexpr int kConsumers = kHeads;
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kMaxRows = 8;                      // (query, head) rows per KV head: the MMA N
constexpr int kQBytes = kHeads * kMaxRows * kD * 2;
static_assert(kStageBytes % 1024 == 0 && kHeadTile % 1024 == 0, "tiles keep the 1024-byte swizzle phase");

struct Params {
    const __nv_bfloat16* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    int max_pages, B, Hq, Hkv, num_pages, page_size, split_tokens, max_kv_len, n_split;
    int G, nq, n_units;      // heads per kv head, queries per sequence, work units
    float scale_log2;
    float* o_part;
    float* lse_part;
    int32_t* status;
    FusedOut fused;          // fused merge (counters NULL: partials only)
};

// m16n8k16 fp16 MMA, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit elements held in fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Global -> shared bulk copy (16-byte aligned, a multiple of 16 bytes),
// completing on an mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// two e4m3 bytes (the low or the high 16-bit half of a word) -> f16x2
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

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float lo_half(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
__device__ __forceinline__ float hi_half(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
__device__ __forceinline__ int volatile_load(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

// Byte offset of 16-byte chunk c of token row r in a head's code tile (TMA,
// 128-byte swizzle: the chunk index is XOR-ed with the row index mod 8).
__device__ __forceinline__ uint32_t code_off(int r, int c) {
    return static_cast<uint32_t>(r * 128 + (((c ^ r) & 7) << 4));
}

// Per-warp state of the online softmax and the O^T accumulators.
struct WarpState {
    float o_acc[8][4];   // O^T m-tiles: elements 16g + 2mt (rows c0, c1) and + 1 (c2, c3), columns 2t4, 2t4 + 1
    float off_acc[2];    // this lane's share of sum_t p shift(t), columns 2t4, 2t4 + 1
    float m_run[2];      // running max of columns 2t4, 2t4 + 1 (exp2 domain)
    float m_thr[2];      // m_run + 8: a score above it triggers the rescale
    float m_use[2];      // m_run, or 0 while it is -inf
    float l_run[2];      // this lane's share of the running sums
};

__device__ __forceinline__ void reset(WarpState& st) {
#pragma unroll
    for (int i = 0; i < 8; ++i) st.o_acc[i][0] = st.o_acc[i][1] = st.o_acc[i][2] = st.o_acc[i][3] = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        st.off_acc[j] = 0.f;
        st.m_run[j] = st.m_thr[j] = -INFINITY;
        st.m_use[j] = 0.f;
        st.l_run[j] = 0.f;
    }
}

// This lane's offsets inside its head's code tile (first sub-tile; the second
// is 16 rows = 2048 bytes on, rows g + 8 are 1024 bytes on).
struct LaneOffsets {
    uint32_t k[2];   // K: chunks 2t4 and 2t4 + 1 of row g
    uint32_t v[2];   // V: chunk g of rows 2t4 and 2t4 + 1
};

// One warp's 32 tokens of a stage as two 16-token sub-tiles.  kPartial: some
// token is past the split end or past a row's causal limit, so scores are
// masked and the V codes and coefficient words of tokens past the end (which
// may hold any bits) are replaced by zeros.
template <bool kPartial>
__device__ __forceinline__ void subtiles(WarpState& st, const uint8_t* kt, const uint8_t* vt, const uint32_t* kw,
                                         const uint32_t* vw, const LaneOffsets& lo, const uint32_t (&qb)[8][2],
                                         const float (&qs)[2], float sl2, int lane, const int (&n_valid)[2],
                                         const int (&tok0)[2], const int (&lim)[2]) {
    const int g = lane >> 2, t4 = lane & 3;
    // ---- scores: sub-tile sb, tokens g (e = 0, 1) and g + 8 (e = 2, 3) by columns 2t4, 2t4 + 1
    float s[2][4];
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
        const uint32_t sbo = sb * 2048;
        const uint4 c0 = *reinterpret_cast<const uint4*>(kt + sbo + lo.k[0]);
        const uint4 c1 = *reinterpret_cast<const uint4*>(kt + sbo + lo.k[1]);
        const uint4 c2 = *reinterpret_cast<const uint4*>(kt + sbo + 1024 + lo.k[0]);
        const uint4 c3 = *reinterpret_cast<const uint4*>(kt + sbo + 1024 + lo.k[1]);
        const uint32_t wg[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const uint32_t wg8[8] = {c2.x, c2.y, c2.z, c2.w, c3.x, c3.y, c3.z, c3.w};
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma16816(acc, e4m3x2_lo(wg[ks]), e4m3x2_lo(wg8[ks]), e4m3x2_hi(wg[ks]), e4m3x2_hi(wg8[ks]), qb[ks][0],
                     qb[ks][1]);
        const uint32_t cw0 = kw[(16 * sb + g) * kHeads], cw1 = kw[(16 * sb + g + 8) * kHeads];
        const float sc0 = lo_half(cw0), sh0 = hi_half(cw0), sc1 = lo_half(cw1), sh1 = hi_half(cw1);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            s[sb][j] = (sc0 * acc[j] + sh0 * qs[j]) * sl2;
            s[sb][2 + j] = (sc1 * acc[2 + j] + sh1 * qs[j]) * sl2;
        }
        if constexpr (kPartial) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = g + 8 * (e >> 1);
                if (!(tok < n_valid[sb] && tok0[sb] + tok <= lim[e & 1])) s[sb][e] = -INFINITY;
            }
        }
    }
    // ---- the value side's shared-memory loads, issued before the softmax
    uint4 xv[2][4];   // chunk g of tokens 2t4, 2t4 + 1, 2t4 + 8, 2t4 + 9
    uint32_t vcw[2][2];
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
        const uint32_t sbo = sb * 2048;
        xv[sb][0] = *reinterpret_cast<const uint4*>(vt + sbo + lo.v[0]);
        xv[sb][1] = *reinterpret_cast<const uint4*>(vt + sbo + lo.v[1]);
        xv[sb][2] = *reinterpret_cast<const uint4*>(vt + sbo + 1024 + lo.v[0]);
        xv[sb][3] = *reinterpret_cast<const uint4*>(vt + sbo + 1024 + lo.v[1]);
        vcw[sb][0] = vw[(16 * sb + g) * kHeads];
        vcw[sb][1] = vw[(16 * sb + g + 8) * kHeads];
        if constexpr (kPartial) {
            // P is 0 past the end, but 0 * (NaN or Inf bits) is not: zero codes and coefficients
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tok = 2 * t4 + (i & 1) + 8 * (i >> 1);
                if (tok >= n_valid[sb]) xv[sb][i] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (g >= n_valid[sb]) vcw[sb][0] = 0u;
            if (g + 8 >= n_valid[sb]) vcw[sb][1] = 0u;
        }
    }
    // ---- online softmax per column; the max is reduced across the warp only
    // when some score passes the column's threshold (lazy rescale by 2^8)
    bool over = false;
#pragma unroll
    for (int sb = 0; sb < 2; ++sb)
        over |= (s[sb][0] > st.m_thr[0]) | (s[sb][2] > st.m_thr[0]) | (s[sb][1] > st.m_thr[1]) |
                (s[sb][3] > st.m_thr[1]);
    if (__any_sync(0xffffffffu, over)) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(fmaxf(s[0][j], s[0][2 + j]), fmaxf(s[1][j], s[1][2 + j]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            if (mx > st.m_thr[j]) {
                const float alpha = ex2(st.m_run[j] - mx);
                st.m_run[j] = mx;
                st.m_thr[j] = mx + 8.f;
                st.m_use[j] = mx;
                st.l_run[j] *= alpha;
                st.off_acc[j] *= alpha;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    st.o_acc[i][j] *= alpha;
                    st.o_acc[i][2 + j] *= alpha;
                }
            }
        }
    }
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
        float pr[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            pr[j] = ex2(s[sb][j] - st.m_use[j]);
            pr[2 + j] = ex2(s[sb][2 + j] - st.m_use[j]);
            st.l_run[j] += pr[j] + pr[2 + j];
        }
        const float sv0 = lo_half(vcw[sb][0]), sh0 = hi_half(vcw[sb][0]);
        const float sv1 = lo_half(vcw[sb][1]), sh1 = hi_half(vcw[sb][1]);
#pragma unroll
        for (int j = 0; j < 2; ++j) st.off_acc[j] += pr[j] * sh0 + pr[2 + j] * sh1;
        // W^T fragments (tokens 2t4, 2t4 + 1 / 2t4 + 8, 2t4 + 9 of column g): the B operand
        const uint32_t pt0 = movmatrix_trans(pack_f16x2(pr[0] * sv0, pr[1] * sv0));
        const uint32_t pt1 = movmatrix_trans(pack_f16x2(pr[2] * sv1, pr[3] * sv1));
        const uint32_t* xa = &xv[sb][0].x;
        const uint32_t* xb = &xv[sb][1].x;
        const uint32_t* xc = &xv[sb][2].x;
        const uint32_t* xd = &xv[sb][3].x;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int wi = mt >> 1;
            // bytes 2, 3 (odd mt) or 0, 1 of word wi, the two tokens interleaved
            const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
            const uint32_t xab = __byte_perm(xa[wi], xb[wi], sel);   // tokens 2t4, 2t4 + 1
            const uint32_t xcd = __byte_perm(xc[wi], xd[wi], sel);   // tokens 2t4 + 8, 2t4 + 9
            mma16816(st.o_acc[mt], e4m3x2_lo(xab), e4m3x2_hi(xab), e4m3x2_lo(xcd), e4m3x2_hi(xcd), pt0, pt1);
        }
    }
}

// Work unit u: KV head group u / (B * n_split), then sequence (u mod B) and
// split; `len` is the sequence length (clamped, and flagged when asked, if it
// is past the block table or max_kv_len).
struct Unit {
    int b, split, hg, len, lo, hi, n_tiles;
};

__device__ __forceinline__ Unit unit_of(const Params& p, int u, bool flag) {
    Unit w;
    const int per_group = p.B * p.n_split;
    w.hg = u / per_group;
    const int rem = u % per_group;
    w.b = rem % p.B;
    w.split = rem / p.B;
    int len = p.seq_lens[w.b];
    const int cap = min(p.max_kv_len, p.max_pages * p.page_size);
    if (len < 0 || len > cap) {
        if (flag) flag_status(p.status, ATTN_DEV_SEQ_TOO_LONG);
        len = len < 0 ? 0 : cap;
    }
    w.len = len;
    w.lo = w.split * p.split_tokens;
    w.hi = min(w.lo + p.split_tokens, len);
    w.n_tiles = w.lo < w.hi ? (w.hi - w.lo + kTileTok - 1) / kTileTok : 0;
    return w;
}

// kMode 0: partials only; 1: fused, the split that arrives last merges its
// (sequence, head group); 2: fused, cooperative launch, the whole grid merges
// every row once all CTAs have passed a grid barrier.
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fp8_g32_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                          const __grid_constant__ CUtensorMap kw_map, const __grid_constant__ CUtensorMap vw_map,
                          const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    uint8_t* qbuf = smem + kStages * kStageBytes;
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t q_full;
    __shared__ __align__(8) uint64_t q_empty;
    __shared__ int s_abort;
    __shared__ int s_skip[kStages];   // the stage was not loaded: its page id was out of range
    __shared__ __align__(8) uint64_t unit_bar;   // fused mode: the consumer warps have written a unit
    __shared__ __align__(8) uint64_t last_bar;   // fused modes: thread 0 has counted the CTA in (1) or met the grid (2)
    __shared__ int s_last;                       // mode 1: the CTA's split arrived last; 2: the grid barrier passed
    __shared__ __align__(8) uint64_t exit_bar;   // cooperative mode: the consumer warps are done

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rows = p.G * p.nq;    // <= 8 (query, head) rows per KV head
    const uint32_t q_bytes = kHeads * n_rows * kD * 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kConsumers);
        }
        mbar_init(&q_full, 1);
        mbar_init(&q_empty, kConsumers);
        mbar_init(&unit_bar, kConsumers);
        mbar_init(&last_bar, 1);
        mbar_init(&exit_bar, kConsumers);
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumers) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&k_map);
            tma_prefetch_desc(&v_map);
            tma_prefetch_desc(&kw_map);
            tma_prefetch_desc(&vw_map);
            const uint64_t pol = l2_policy_evict_first();   // every KV byte is read once
            int slot = 0;
            uint32_t phase = 0;   // parity of the stage ring's current round
            int t_all = 0;        // stages issued so far
            int n_q = 0;          // query copies issued so far
            for (int u = blockIdx.x; u < p.n_units && !volatile_load(&s_abort); u += gridDim.x) {
                const Unit w = unit_of(p, u, true);
                if (w.n_tiles == 0) continue;
                // the unit's queries: the rows of its 8 KV heads, G * q_len each, contiguous
                if (n_q > 0 && !mbar_wait(&q_empty, (n_q - 1) & 1)) {
                    flag_status(p.status, ATTN_DEV_WAIT_TIMEOUT);
                    atomicExch(&s_abort, 1);
                    break;
                }
                mbar_arrive_expect_tx(&q_full, q_bytes);
                bulk_load(qbuf, p.q + (static_cast<size_t>(w.b) * p.Hq + w.hg * kHeads * p.G) * p.nq * kD, q_bytes,
                          &q_full);
                ++n_q;
                const int32_t* table = p.block_table + static_cast<size_t>(w.b) * p.max_pages;
                for (int t = 0; t < w.n_tiles; ++t) {
                    if (t_all >= kStages && !mbar_wait(&empty_bar[slot], phase ^ 1u)) {
                        flag_status(p.status, ATTN_DEV_WAIT_TIMEOUT);
                        atomicExch(&s_abort, 1);
                        break;
                    }
                    const int tok = w.lo + t * kTileTok;
                    const int page = table[tok / p.page_size];
                    uint8_t* st = smem + slot * kStageBytes;
                    if (page < 0 || page >= p.num_pages) {
                        flag_status(p.status, ATTN_DEV_PAGE_OUT_OF_RANGE);
                        s_skip[slot] = 1;               // the consumers leave the page's tokens out
                        mbar_arrive(&full_bar[slot]);   // release the consumers; nothing is loaded
                    } else {
                        const int row = page * p.page_size + tok % p.page_size;
                        const int h0 = w.hg * kHeads;
                        s_skip[slot] = 0;
                        mbar_arrive_expect_tx(&full_bar[slot], kStageBytes);
                        for (int h = 0; h < kHeads; ++h) {
                            tma_load_3d_hint(st + h * kHeadTile, &k_map, &full_bar[slot], 0, h0 + h, row, pol);
                            tma_load_3d_hint(st + kOffV + h * kHeadTile, &v_map, &full_bar[slot], 0, h0 + h, row, pol);
                        }
                        tma_load_2d(st + kOffKw, &kw_map, &full_bar[slot], h0, row);
                        tma_load_2d(st + kOffVw, &vw_map, &full_bar[slot], h0, row);
                    }
                    ++t_all;
                    if (++slot == kStages) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t4 = lane & 3;
    LaneOffsets lo;
    lo.k[0] = code_off(g, 2 * t4);
    lo.k[1] = code_off(g, 2 * t4 + 1);
    lo.v[0] = code_off(2 * t4, g);
    lo.v[1] = code_off(2 * t4 + 1, g);
    const float sl2 = p.scale_log2;

    int slot = 0;
    uint32_t phase = 0;
    int n_q = 0;
    WarpState st;
    for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
        const Unit w = unit_of(p, u, false);
        const int kvh = w.hg * kHeads + warp;
        auto out_row = [&](int r) -> size_t {
            const int i = r / p.G, h = r % p.G;
            return (static_cast<size_t>(w.b) * p.Hq + kvh * p.G + h) * p.nq + i;
        };
        // fused mode: unit_fused_tail after every unit (an empty split included),
        // so its barriers' phase is the parity of the units this CTA took before
        auto fused_tail = [&]() -> bool {
            if constexpr (kMode != 1) return true;
            const uint32_t ph =
                static_cast<uint32_t>((u - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x)) & 1u;
            int32_t* cnt = p.fused.counters + static_cast<size_t>(w.b) * p.Hkv + w.hg * kHeads;
            return unit_fused_tail(p.fused, p.o_part, p.lse_part, p.n_split, p.status, cnt, out_row(0), n_rows, ph,
                                   &unit_bar, &last_bar, &s_last, &s_abort, warp, lane);
        };
        if (w.n_tiles == 0) {   // empty split: O = 0, LSE = -inf
            for (int i = lane; i < n_rows * kD; i += 32)
                p.o_part[(out_row(i / kD) * p.n_split + w.split) * kD + (i % kD)] = 0.f;
            if (lane < n_rows) p.lse_part[out_row(lane) * p.n_split + w.split] = -INFINITY;
            if (!fused_tail()) {
                flag_status(p.status, ATTN_DEV_WAIT_TIMEOUT);
                atomicExch(&s_abort, 1);
                break;
            }
            continue;
        }
        // ---- the unit's queries in fp16, as B fragments: column g is CTA row g
        // (zero past the rows); k-step ks, k pairs (2t4, 2t4+1) and (2t4+8,
        // 2t4+9) are elements 32t4 + 4ks + {0, 1} and {2, 3}
        if (!mbar_wait(&q_full, n_q & 1, &s_abort)) {
            flag_status(p.status, ATTN_DEV_WAIT_TIMEOUT);
            atomicExch(&s_abort, 1);
            break;
        }
        ++n_q;
        uint32_t qb[8][2];
        float qs[2];    // Q's row sums of columns 2t4, 2t4 + 1
        int lim[2];     // last visible token of columns 2t4, 2t4 + 1 (bottom-right causal: len - q_len + i)
        {
            const bool real = g < n_rows;
            // CTA row r = i * G + h is query row (warp * G + h) * q_len + i of the copied block
            const int qr = real ? (warp * p.G + g % p.G) * p.nq + g / p.G : 0;
            const __nv_bfloat16* qrow = reinterpret_cast<const __nv_bfloat16*>(qbuf) + qr * kD + 32 * t4;
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {   // elements 32t4 + 8c .. + 7: k-steps 2c and 2c + 1
                uint4 raw = make_uint4(0u, 0u, 0u, 0u);
                if (real) raw = *reinterpret_cast<const uint4*>(qrow + 8 * c);
                const uint32_t wq[4] = {raw.x, raw.y, raw.z, raw.w};
                float x[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wq[i]));
                    x[2 * i] = f.x;
                    x[2 * i + 1] = f.y;
                }
                qb[2 * c][0] = pack_f16x2(x[0], x[1]);
                qb[2 * c][1] = pack_f16x2(x[2], x[3]);
                qb[2 * c + 1][0] = pack_f16x2(x[4], x[5]);
                qb[2 * c + 1][1] = pack_f16x2(x[6], x[7]);
                sum += ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);   // row g's sum, in the quad's four lanes
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int col = 2 * t4 + j;
                qs[j] = __shfl_sync(0xffffffffu, sum, 4 * col);
                lim[j] = col < n_rows ? w.len - p.nq + col / p.G : -1;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_empty);   // the buffer may take the next unit's queries
        reset(st);
        // ---- the unit's stages
        const int lim_min = w.len - p.nq;   // the first row's limit, the smallest (rows are ordered by query)
        for (int t = 0; t < w.n_tiles; ++t) {
            if (!mbar_wait(&full_bar[slot], phase, &s_abort)) {
                flag_status(p.status, ATTN_DEV_WAIT_TIMEOUT);
                atomicExch(&s_abort, 1);
                break;
            }
            int tok0[2], n_valid[2];
#pragma unroll
            for (int sb = 0; sb < 2; ++sb) {
                tok0[sb] = w.lo + t * kTileTok + 16 * sb;
                n_valid[sb] = min(max(w.hi - tok0[sb], 0), 16);
            }
            if (!s_skip[slot]) {
                const uint8_t* sbase = smem + slot * kStageBytes;
                const uint8_t* kt = sbase + warp * kHeadTile;
                const uint8_t* vt = sbase + kOffV + warp * kHeadTile;
                const uint32_t* kw = reinterpret_cast<const uint32_t*>(sbase + kOffKw) + warp;
                const uint32_t* vw = reinterpret_cast<const uint32_t*>(sbase + kOffVw) + warp;
                if (n_valid[1] == 16 && tok0[0] + 31 <= lim_min)
                    subtiles<false>(st, kt, vt, kw, vw, lo, qb, qs, sl2, lane, n_valid, tok0, lim);
                else
                    subtiles<true>(st, kt, vt, kw, vw, lo, qb, qs, sl2, lane, n_valid, tok0, lim);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[slot]);
            if (++slot == kStages) {
                slot = 0;
                phase ^= 1u;
            }
        }
        if (volatile_load(&s_abort)) break;
        // ---- the unit's partial O and LSE for this KV head
        float l_tot[2], off_tot[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float l = st.l_run[j], o = st.off_acc[j];
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                l += __shfl_xor_sync(0xffffffffu, l, x);
                o += __shfl_xor_sync(0xffffffffu, o, x);
            }
            l_tot[j] = l;
            off_tot[j] = o;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int col = 2 * t4 + j;
            if (col >= n_rows) continue;
            const bool alive = l_tot[j] > 0.f;
            const float inv = alive ? 1.f / l_tot[j] : 0.f;
            const float off = off_tot[j];
            // this lane's 16 elements 16g .. 16g + 15: m-tile mt holds 16g + 2mt (rows j) and + 1 (rows 2 + j)
            float* orow = p.o_part + (out_row(col) * p.n_split + w.split) * kD + 16 * g;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4*>(orow + 4 * i) =
                    make_float4((st.o_acc[2 * i][j] + off) * inv, (st.o_acc[2 * i][2 + j] + off) * inv,
                                (st.o_acc[2 * i + 1][j] + off) * inv, (st.o_acc[2 * i + 1][2 + j] + off) * inv);
            if (g == 0)
                p.lse_part[out_row(col) * p.n_split + w.split] = alive ? st.m_run[j] * kLn2 + logf(l_tot[j])
                                                                         : -INFINITY;
        }
        if (!fused_tail()) {
            flag_status(p.status, ATTN_DEV_WAIT_TIMEOUT);
            atomicExch(&s_abort, 1);
            break;
        }
    }
    if constexpr (kMode == 2) {
        // every consumer warp of the CTA is done (bounded meeting); one thread
        // meets the grid, then every warp merges its share of the rows
        __syncwarp();
        if (lane == 0) mbar_arrive(&exit_bar);
        if (threadIdx.x == 0)
            s_last = mbar_wait(&exit_bar, 0, &s_abort) && volatile_load(&s_abort) == 0 &&
                     grid_barrier_once(p.fused.counters + p.B * p.Hkv, p.status);
        if (threadIdx.x == 0) mbar_arrive(&last_bar);
        if (mbar_wait(&last_bar, 0, &s_abort) && volatile_load(&s_last))
            grid_merge(p.o_part, p.lse_part, p.n_split, p.B * p.Hq * p.nq, p.fused, warp, kConsumers, lane);
    }
}

}  // namespace

bool decode_fp8_g32_shape_ok(const DecodeArgs& a) {
    return a.D == kD && a.Hkv % kHeads == 0 && (a.Hq / a.Hkv) * a.q_len <= kMaxRows;
}

bool decode_fp8_g32_supported(const DecodeArgs& a) {
    return decode_fp8_g32_shape_ok(a) && a.page_size % kTileTok == 0 && a.split_tokens % kTileTok == 0;
}

// With `occ` set nothing is launched: the kernel is persistent with one CTA
// per SM serving 8 KV heads at a time, reported as 8 (KV head, split) slots per SM.
cudaError_t launch_decode_fp8_g32(const DecodeArgs& a, const void* k_scale_shift, const void* v_scale_shift,
                                  cudaStream_t stream, int* occ) {
    const size_t smem = kStages * kStageBytes + kQBytes + 1024;
    auto kern = a.counters != nullptr ? decode_fp8_g32_kernel<1> : decode_fp8_g32_kernel<0>;
    if (occ != nullptr) {
        int ctas = 0;
        const cudaError_t e = ctas_per_sm(kern, kThreads, smem, &ctas);
        *occ = ctas * kHeads;
        return e;
    }
    CUtensorMap k_map, v_map, kw_map, vw_map;
    const uint64_t rows = static_cast<uint64_t>(a.num_pages) * a.page_size;
    {
        // codes [rows, Hkv, D] bytes: one box per head, {D bytes, 1 head, 32 tokens}
        const uint64_t dims[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(a.Hkv), rows};
        const uint64_t strides[2] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(a.Hkv) * kD};
        const uint32_t box[3] = {kD, 1, kTileTok};
        if (!encode_tiled_map(&k_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.k_cache, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tiled_map(&v_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.v_cache, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    {
        // coefficient words [rows, Hkv]: the 8 heads' words of 32 tokens (x starts at 32-byte multiples)
        const uint64_t dims[2] = {static_cast<uint64_t>(a.Hkv), rows};
        const uint64_t strides[1] = {static_cast<uint64_t>(a.Hkv) * 4};
        const uint32_t box[2] = {kHeads, kTileTok};
        if (!encode_tiled_map(&kw_map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, k_scale_shift, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_tiled_map(&vw_map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, v_scale_shift, dims, strides, box,
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
    p.n_units = a.B * a.n_split * (a.Hkv / kHeads);
    p.scale_log2 = a.scale * kLog2e;
    p.o_part = a.o_part;
    p.lse_part = a.lse_part;
    p.status = a.dev_status;
    p.fused.counters = a.counters;
    p.fused.o = static_cast<__nv_bfloat16*>(a.o_final);
    p.fused.lse = a.lse_final;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = p.n_units < sms ? p.n_units : sms;
    cudaError_t e;
    if (a.counters != nullptr && cooperative_launch_enabled()) {
        // fused: a cooperative launch (every CTA resident at once) lets the whole
        // grid merge after one grid barrier
        e = cudaFuncSetAttribute(decode_fp8_g32_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, decode_fp8_g32_kernel<2>, k_map, v_map, kw_map, vw_map, p);
        if (e == cudaSuccess) return e;
        // refused (too large to be resident at once, or a sharing mode without
        // cooperative launches): clear the launch error and merge by last arrival;
        // an error that is not the launch's own comes back from that launch too
        (void)cudaGetLastError();
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>(k_map, v_map, kw_map, vw_map, p);
    return cudaGetLastError();
}

}  // namespace gb300
