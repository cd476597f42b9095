// decode_int4_g32.cu - split-K paged decode over an int4 cache whose rows have
// four quantisation groups of 32 elements (N_GROUPS = 4 at D = 128), for KV
// head counts that are multiples of 8.
//
// Row format ("splitk_kernels.py", docstring of _fwd_kernel_splitK,
// cast_uint32_to_half2, dequantize): per (token, kv head) 20 int32 words, the
// four coefficient words (fp16 scale low, fp16 offset high) then 16 code
// words, four per group; nibble j of a group's word w is element 8w + j of the
// group; value = scale * code + offset.  With 20 words (80 bytes) per row every
// group's code words form one aligned 16-byte chunk.
//
// Work layout (persistent): one CTA per SM walks work units (sequence, split,
// group of 8 KV heads).  A producer warp streams 32-token stages of whole
// token rows (the 640 bytes of 8 heads' rows, contiguous in the pool) with
// TMA: a 3D box of 128-byte pieces with 128-byte swizzle, so HBM is read in
// full lines and the consumers' shared-memory reads are free of bank
// conflicts.  Eight consumer warps each own one KV head and every token of the
// unit, so no cross-warp merge is needed; each warp takes a stage's 32 tokens
// as two 16-token sub-tiles whose instruction streams interleave.  The
// producer runs ahead across unit boundaries (it also copies the next unit's
// queries), so the pipeline never drains between units.
//
// Codes enter the tensor cores as exact fp16 subnormals.  A code c in bits 0-3
// of a 16-bit half is the fp16 value c * 2^-24 and one in bits 4-7 the value
// 16c * 2^-24 (sigma = 16), so one AND per half pair makes an MMA operand; codes
// in a half's upper byte are first moved down by one byte permute.  The
// partner operand carries 1/sigma (Q) or the result is divided by sigma (O),
// both exact powers of two.
//
//   scores (S^T = K Q^T, M = 16 tokens, N = 8 rows, K = 16 elements):
//     T_g[t,r] = sum_{d in g} (sigma_d c_td 2^-24) (q_rd / sigma_d)   one accumulator per group
//     s[t,r]   = log2(e) scale_sm * (2^24 sum_g scale_g(t) T_g[t,r] + sum_g offset_g(t) Qsum_g[r])
//     the offset term is one more MMA with the offsets as A and the group sums of q as B.
//   values (O^T = V^T W, M = 16 head-dim elements, N = 8 rows, K = 16 tokens):
//     O[r,d]   = 2^24 / sigma_d sum_t (sigma_d c_td 2^-24) W_g(d)[t,r] + OFF_g(d)[r]
//     W_g[t,r] = fp16(p[t,r] * scale_g(t))       (the dequantised values' rounding on the pages)
//     OFF_g[r] = sum_t offset_g(t) p[t,r]        one more MMA with the offsets as A and P as B
//   The score fragment (tokens in rows) is turned into the B operand of the
//   value MMA (tokens in k) by movmatrix transposes.  K code fragments come
//   from ldmatrix, V code fragments from ldmatrix.trans (which pairs the two
//   tokens of a k pair in one register), straight from the TMA tile.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "split_merge.cuh"

namespace gb300 {
namespace {

constexpr int kD = 128;
constexpr int kGroups = 4;
constexpr int kRowWords = kGroups + kD / 8;     // 20 words per (token, head) row
constexpr int kRowBytes = 4 * kRowWords;        // 80
constexpr int kHeads = 8;                       // KV heads per CTA: one consumer warp each
constexpr int kTokBytes = kHeads * kRowBytes;   // 640: one token's rows of the 8 heads
constexpr int kPieces = kTokBytes / 128;        // 5 swizzled 128-byte pieces per token
constexpr int kTileTok = 32;                    // tokens per stage
constexpr int kTileBytes = kTileTok * kTokBytes;
constexpr int kStageBytes = 2 * kTileBytes;     // K then V
constexpr int kStages = 5;
constexpr int kConsumers = kHeads;
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kMaxRows = 8;                     // (query, head) rows per KV head: the MMA N
constexpr int kQBytes = kHeads * kMaxRows * kD * 2;
constexpr float kTwo24 = 16777216.0f;
constexpr uint32_t kRow8 = 8 * kTokBytes;       // 5120: eight token rows
static_assert(kTileBytes % 1024 == 0 && kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle phase");

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

// m16n8k16 fp16 MMA, fp32 accumulators (registers only, so the compiler may
// schedule it freely).
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

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t x) { return *reinterpret_cast<__half2*>(&x); }
__device__ __forceinline__ float lo_float(uint32_t w) { return __low2float(bits_h2(w)); }
__device__ __forceinline__ int volatile_load(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

// Codes of a 16-bit-half pair as fp16 subnormal operands: bits 0-3 of each
// half (sigma 1) and bits 4-7 (sigma 16), and the upper byte moved down.
__device__ __forceinline__ uint32_t nib0(uint32_t x) { return x & 0x000F000Fu; }
__device__ __forceinline__ uint32_t nib1(uint32_t x) { return x & 0x00F000F0u; }
__device__ __forceinline__ uint32_t upper(uint32_t x) { return __byte_perm(x, 0u, 0x4341u); }

// Byte offset of byte `o` of token row `r` inside a tile written by TMA with
// 128-byte swizzle: the 16-byte chunk index inside each 128-byte piece is
// XOR-ed with the piece's index mod 8.  Rows 8 apart have the same pattern (a
// token row is 5 pieces), so row r + 8k sits at offset(r) + 5120k.
__device__ __forceinline__ uint32_t swz(int r, int o) {
    const uint32_t lin = static_cast<uint32_t>(r * kTokBytes + o);
    return lin ^ (((lin >> 7) & 7u) << 4);
}

// Per-warp state of the online softmax and the O^T accumulators.
struct WarpState {
    float o_acc[2 * kGroups][4];   // O^T m-tiles: group c, element sets {4g, 4g+1} and {4g+2, 4g+3}
    float off_acc[4];              // OFF^T: rows = groups, columns = CTA rows
    float m_run[2];                // running max of columns 2t4, 2t4 + 1 (exp2 domain)
    float m_thr[2];                // m_run + 8: a score above it triggers the rescale
    float m_use[2];                // m_run, or 0 while it is -inf
    float l_run[2];                // this lane's share of the running sums
};

// This lane's (swizzled) shared-memory offsets inside a K or V tile.
struct LaneOffsets {
    uint32_t ldm[2];   // ldmatrix row address of groups {0,1} / {2,3}, first sub-tile
    uint32_t kc;       // coefficient words of token g
    uint32_t vc[2];    // coefficient words of tokens 2t4 and 2t4 + 1
};

__device__ __forceinline__ void reset(WarpState& st) {
#pragma unroll
    for (int i = 0; i < 2 * kGroups; ++i) st.o_acc[i][0] = st.o_acc[i][1] = st.o_acc[i][2] = st.o_acc[i][3] = 0.f;
    st.off_acc[0] = st.off_acc[1] = st.off_acc[2] = st.off_acc[3] = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        st.m_run[j] = st.m_thr[j] = -INFINITY;
        st.m_use[j] = 0.f;
        st.l_run[j] = 0.f;
    }
}

// One warp's 32 tokens of a stage, as two 16-token sub-tiles whose
// instruction streams interleave (the second hides the first's latencies).
// kPartial: some token is past the split end or past a row's causal limit, so
// scores are masked and the coefficient words of tokens past the end (which
// may hold any bits) are replaced by zeros.
template <bool kPartial>
__device__ __forceinline__ void subtiles(WarpState& st, const uint8_t* kt, const uint8_t* vt, const LaneOffsets& lo,
                                         const uint32_t (&qb)[kGroups][2][2], uint32_t qsb, float c24, int lane,
                                         const int (&n_valid)[2], const int (&tok0)[2], const int (&lim)[2]) {
    const int g = lane >> 2, t4 = lane & 3;
    const uint32_t kt_s = smem_u32(kt), vt_s = smem_u32(vt);
    // ---- scores: per sub-tile and group T_c (tokens g, g + 8 x columns 2t4, 2t4 + 1)
    float s[2][4];
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
        const uint32_t sbo = sb * 2 * kRow8;
        float tacc[kGroups][4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t r[4];   // (group 2h, token g), (2h, g + 8), (2h + 1, g), (2h + 1, g + 8)
            ldmatrix_x4(r[0], r[1], r[2], r[3], kt_s + lo.ldm[half] + sbo);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int c = 2 * half + u;
                const uint32_t x0 = r[2 * u], x1 = r[2 * u + 1];
                const uint32_t y0 = upper(x0), y1 = upper(x1);
                tacc[c][0] = tacc[c][1] = tacc[c][2] = tacc[c][3] = 0.f;
                mma16816(tacc[c], nib0(x0), nib0(x1), nib1(x0), nib1(x1), qb[c][0][0], qb[c][0][1]);
                mma16816(tacc[c], nib0(y0), nib0(y1), nib1(y0), nib1(y1), qb[c][1][0], qb[c][1][1]);
            }
        }
        // scale words of tokens g and g + 8; offset term: A = offsets (token rows;
        // groups 2t4, 2t4 + 1 in k, lanes t4 >= 2 repeat groups 0-3 against a zero B),
        // B = scaled group sums of q
        const uint8_t* kc = kt + lo.kc + sbo;
        const uint4 kc0 = *reinterpret_cast<const uint4*>(kc);
        const uint4 kc1 = *reinterpret_cast<const uint4*>(kc + kRow8);
        float r4[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int wo = 8 * (t4 & 1);
            const uint2 o0 = *reinterpret_cast<const uint2*>(kc + wo);
            const uint2 o1 = *reinterpret_cast<const uint2*>(kc + kRow8 + wo);
            mma16816(r4, __byte_perm(o0.x, o0.y, 0x7632u), __byte_perm(o1.x, o1.y, 0x7632u), 0u, 0u, qsb, 0u);
        }
        const uint32_t w0[4] = {kc0.x, kc0.y, kc0.z, kc0.w};
        const uint32_t w1[4] = {kc1.x, kc1.y, kc1.z, kc1.w};
        float2 u0 = make_float2(0.f, 0.f), u1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kGroups; ++c) {
            const float a = lo_float(w0[c]), a8 = lo_float(w1[c]);
            u0 = __ffma2_rn(make_float2(a, a), make_float2(tacc[c][0], tacc[c][1]), u0);
            u1 = __ffma2_rn(make_float2(a8, a8), make_float2(tacc[c][2], tacc[c][3]), u1);
        }
        const float2 c2 = make_float2(c24, c24);
        const float2 s0 = __ffma2_rn(c2, u0, make_float2(r4[0], r4[1]));
        const float2 s1 = __ffma2_rn(c2, u1, make_float2(r4[2], r4[3]));
        s[sb][0] = s0.x;
        s[sb][1] = s0.y;
        s[sb][2] = s1.x;
        s[sb][3] = s1.y;
        if constexpr (kPartial) {
            // mask tokens past the split end or a row's causal limit
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = g + 8 * (e >> 1);
                if (!(tok < n_valid[sb] && tok0[sb] + tok <= lim[e & 1])) s[sb][e] = -INFINITY;
            }
        }
    }
    // ---- the value side's shared-memory loads, issued before the softmax so
    // their latency hides behind it (none depends on P)
    uint4 vc_all[2][4];
    uint32_t woff[2][4];
    uint32_t rv[2][2][4];
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
        const uint32_t sbo = sb * 2 * kRow8;
        const uint8_t* va = vt + lo.vc[0] + sbo;
        const uint8_t* vb = vt + lo.vc[1] + sbo;
        const uint8_t* vrow[4] = {va, vb, va + kRow8, vb + kRow8};
        const int wo = 4 * (g & 3);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            vc_all[sb][i] = *reinterpret_cast<const uint4*>(vrow[i]);
            woff[sb][i] = *reinterpret_cast<const uint32_t*>(vrow[i] + wo);
        }
#pragma unroll
        for (int half = 0; half < 2; ++half)
            ldmatrix_x4_trans(rv[sb][half][0], rv[sb][half][1], rv[sb][half][2], rv[sb][half][3],
                              vt_s + lo.ldm[half] + sbo);
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
#pragma unroll
                for (int i = 0; i < 2 * kGroups; ++i) {
                    st.o_acc[i][j] *= alpha;
                    st.o_acc[i][2 + j] *= alpha;
                }
                st.off_acc[j] *= alpha;
                st.off_acc[2 + j] *= alpha;
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
        // P^T fragments (tokens 2t4, 2t4 + 1 / 2t4 + 8, 2t4 + 9 of column g): the B operand
        const uint32_t pt0 = movmatrix_trans(h2_bits(__floats2half2_rn(pr[0], pr[1])));
        const uint32_t pt1 = movmatrix_trans(h2_bits(__floats2half2_rn(pr[2], pr[3])));
        // V coefficient words of tokens 2t4, 2t4 + 1, 2t4 + 8, 2t4 + 9
        uint4 vc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            vc[i] = vc_all[sb][i];
            if constexpr (kPartial) {
                const int tok = 2 * t4 + (i & 1) + 8 * (i >> 1);
                if (tok >= n_valid[sb]) vc[i] = make_uint4(0u, 0u, 0u, 0u);   // P is 0 there; keep 0 * x finite
            }
        }
        // offset term of O: A = offsets of group g (rows 0-3 are read; rows 4-7 repeat
        // groups 0-3 and are discarded) by tokens, B = P^T
        {
            uint32_t w_a = woff[sb][0], w_b = woff[sb][1], w_c = woff[sb][2], w_d = woff[sb][3];
            if constexpr (kPartial) {
                w_a = 2 * t4 < n_valid[sb] ? w_a : 0u;
                w_b = 2 * t4 + 1 < n_valid[sb] ? w_b : 0u;
                w_c = 2 * t4 + 8 < n_valid[sb] ? w_c : 0u;
                w_d = 2 * t4 + 9 < n_valid[sb] ? w_d : 0u;
            }
            mma16816(st.off_acc, __byte_perm(w_a, w_b, 0x7632u), 0u, __byte_perm(w_c, w_d, 0x7632u), 0u, pt0, pt1);
        }
        // ---- O^T += codes^T W_c, two m-tiles per group
        const uint32_t vcw[4][4] = {{vc[0].x, vc[0].y, vc[0].z, vc[0].w}, {vc[1].x, vc[1].y, vc[1].z, vc[1].w},
                                    {vc[2].x, vc[2].y, vc[2].z, vc[2].w}, {vc[3].x, vc[3].y, vc[3].z, vc[3].w}};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint32_t* r = rv[sb][half];   // (group 2h, tokens 2t4..), (2h, 2t4+8..), (2h+1, 2t4..), (2h+1, 2t4+8..)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int c = 2 * half + u;
                const uint32_t wb0 =
                    h2_bits(__hmul2(bits_h2(pt0), bits_h2(__byte_perm(vcw[0][c], vcw[1][c], 0x5410u))));
                const uint32_t wb1 =
                    h2_bits(__hmul2(bits_h2(pt1), bits_h2(__byte_perm(vcw[2][c], vcw[3][c], 0x5410u))));
                const uint32_t x0 = r[2 * u], x1 = r[2 * u + 1];
                const uint32_t y0 = upper(x0), y1 = upper(x1);
                mma16816(st.o_acc[2 * c], nib0(x0), nib1(x0), nib0(x1), nib1(x1), wb0, wb1);
                mma16816(st.o_acc[2 * c + 1], nib0(y0), nib1(y0), nib0(y1), nib1(y1), wb0, wb1);
            }
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
__global__ void __launch_bounds__(kThreads, 1) decode_int4_g32_kernel(const __grid_constant__ CUtensorMap k_map,
                                                                      const __grid_constant__ CUtensorMap v_map,
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
                        s_skip[slot] = 0;
                        mbar_arrive_expect_tx(&full_bar[slot], kStageBytes);
                        tma_load_3d_hint(st, &k_map, &full_bar[slot], 0, w.hg * kPieces, row, pol);
                        tma_load_3d_hint(st + kTileBytes, &v_map, &full_bar[slot], 0, w.hg * kPieces, row, pol);
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
    const int head_off = warp * kRowBytes;   // this warp's KV head inside a token row
    LaneOffsets lo;
#pragma unroll
    for (int half = 0; half < 2; ++half)
        lo.ldm[half] = swz((lane & 7) + 8 * ((lane >> 3) & 1), head_off + 16 + 16 * (2 * half + (lane >> 4)));
    lo.kc = swz(g, head_off);
    lo.vc[0] = swz(2 * t4, head_off);
    lo.vc[1] = swz(2 * t4 + 1, head_off);
    const float c24 = kTwo24 * p.scale_log2;

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
        // ---- the unit's queries.  B operand of the score MMA: column g is CTA row g
        // (zero past the rows).  Group c, k-step 0 pairs elements (8t4, 8t4+4) and
        // (8t4+1, 8t4+5)/16, k-step 1 pairs (8t4+2, 8t4+6) and (8t4+3, 8t4+7)/16.
        if (!mbar_wait(&q_full, n_q & 1, &s_abort)) {
            flag_status(p.status, ATTN_DEV_WAIT_TIMEOUT);
            atomicExch(&s_abort, 1);
            break;
        }
        ++n_q;
        uint32_t qb[kGroups][2][2];
        uint32_t qsb;   // B operand of the offset MMA: (Qsum_{2t4}, Qsum_{2t4+1}) of row g, times log2 e * scale
        int lim[2];     // last visible token of columns 2t4, 2t4+1 (bottom-right causal: len - q_len + i)
        {
            const bool real = g < n_rows;
            // CTA row r = i * G + h is query row (warp * G + h) * q_len + i of the copied block
            const int qr = real ? (warp * p.G + g % p.G) * p.nq + g / p.G : 0;
            const __nv_bfloat16* qrow = reinterpret_cast<const __nv_bfloat16*>(qbuf) + qr * kD;
            float qs[kGroups];
#pragma unroll
            for (int c = 0; c < kGroups; ++c) {
                float x[8];
                if (real) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(qrow + 32 * c + 8 * t4);
                    const uint32_t wq[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wq[i]));
                        x[2 * i] = f.x;
                        x[2 * i + 1] = f.y;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] = 0.f;
                }
                qb[c][0][0] = h2_bits(__floats2half2_rn(x[0], x[4]));
                qb[c][0][1] = h2_bits(__floats2half2_rn(x[1] * 0.0625f, x[5] * 0.0625f));
                qb[c][1][0] = h2_bits(__floats2half2_rn(x[2], x[6]));
                qb[c][1][1] = h2_bits(__floats2half2_rn(x[3] * 0.0625f, x[7] * 0.0625f));
                float sq = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
                sq += __shfl_xor_sync(0xffffffffu, sq, 1);
                sq += __shfl_xor_sync(0xffffffffu, sq, 2);
                qs[c] = sq * p.scale_log2;
            }
            qsb = t4 == 0 ? h2_bits(__floats2half2_rn(qs[0], qs[1]))
                          : (t4 == 1 ? h2_bits(__floats2half2_rn(qs[2], qs[3])) : 0u);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int col = 2 * t4 + j;
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
                const uint8_t* kt = smem + slot * kStageBytes;
                if (n_valid[1] == 16 && tok0[0] + 31 <= lim_min)
                    subtiles<false>(st, kt, kt + kTileBytes, lo, qb, qsb, c24, lane, n_valid, tok0, lim);
                else
                    subtiles<true>(st, kt, kt + kTileBytes, lo, qb, qsb, c24, lane, n_valid, tok0, lim);
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
        float l_tot[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float l = st.l_run[j];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            l_tot[j] = l;
        }
        // OFF_c of columns 2t4, 2t4 + 1 lives in lane (c, t4)
        float offv[kGroups][2];
#pragma unroll
        for (int c = 0; c < kGroups; ++c) {
            offv[c][0] = __shfl_sync(0xffffffffu, st.off_acc[0], 4 * c + t4);
            offv[c][1] = __shfl_sync(0xffffffffu, st.off_acc[1], 4 * c + t4);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int col = 2 * t4 + j;
            if (col >= n_rows) continue;
            const bool alive = l_tot[j] > 0.f;
            const float inv = alive ? 1.f / l_tot[j] : 0.f;
            float* orow = p.o_part + (out_row(col) * p.n_split + w.split) * kD;
#pragma unroll
            for (int c = 0; c < kGroups; ++c) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float* f = st.o_acc[2 * c + hh];
                    const int d_lo = 32 * c + 4 * g + 2 * hh;   // sigma 1; d_lo + 1 has sigma 16
                    orow[d_lo] = fmaf(f[j], kTwo24, offv[c][j]) * inv;
                    orow[d_lo + 1] = fmaf(f[2 + j], kTwo24 * 0.0625f, offv[c][j]) * inv;
                }
            }
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

bool decode_int4_g32_shape_ok(const DecodeArgs& a) {
    return a.n_groups == kGroups && a.D == kD && a.Hkv % kHeads == 0 && (a.Hq / a.Hkv) * a.q_len <= kMaxRows;
}

bool decode_int4_g32_supported(const DecodeArgs& a) {
    return decode_int4_g32_shape_ok(a) && a.page_size % kTileTok == 0 && a.split_tokens % kTileTok == 0;
}

// With `occ` set nothing is launched: the kernel is persistent with one CTA
// per SM serving 8 KV heads at a time, reported as 8 (KV head, split) slots per SM.
cudaError_t launch_decode_int4_g32(const DecodeArgs& a, cudaStream_t stream, int* occ) {
    const size_t smem = kStages * kStageBytes + kQBytes + 1024;
    auto kern = a.counters != nullptr ? decode_int4_g32_kernel<1> : decode_int4_g32_kernel<0>;
    if (occ != nullptr) {
        int ctas = 0;
        const cudaError_t e = ctas_per_sm(kern, kThreads, smem, &ctas);
        *occ = ctas * kHeads;
        return e;
    }
    CUtensorMap k_map, v_map;
    // the pool [rows, Hkv * 20 words] as 128-byte pieces: {32 words, Hkv * 20 / 32 pieces, rows}
    const uint64_t dims[3] = {32, static_cast<uint64_t>(a.Hkv) * kRowWords / 32,
                              static_cast<uint64_t>(a.num_pages) * a.page_size};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(a.Hkv) * kRowBytes};
    const uint32_t box[3] = {32, kPieces, kTileTok};
    if (!encode_tiled_map(&k_map, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, a.k_cache, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled_map(&v_map, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, a.v_cache, dims, strides, box,
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
        e = cudaFuncSetAttribute(decode_int4_g32_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
        e = cudaLaunchKernelEx(&cfg, decode_int4_g32_kernel<2>, k_map, v_map, p);
        if (e == cudaSuccess) return e;
        // refused (too large to be resident at once, or a sharing mode without
        // cooperative launches): clear the launch error and merge by last arrival;
        // an error that is not the launch's own comes back from that launch too
        (void)cudaGetLastError();
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>(k_map, v_map, p);
    return cudaGetLastError();
}

}  // namespace gb300
