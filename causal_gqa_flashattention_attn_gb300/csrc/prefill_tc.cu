// prefill_tc.cu - causal GQA prefill on the 5th-generation tensor cores.
//
// What it computes follows "causal_forward_kernel.py" (flash-attention-scratch),
// _flash_attention_forward_gqa_kernel: Q tiles against streamed K/V tiles,
// S = Q K^T times the softmax scale and log2(e), so that the exponentials are powers of 2,
// an online softmax (running max m, running sum l, rescale by exp2(m_old -
// m_new)), P rounded to bf16 before O += P V, skipping of tiles above the
// causal diagonal and masking of the diagonal tiles only, then O = acc / l
// and a per-row LSE.  Causal alignment is bottom-right as in
// "gpt-o3 / triton6fd1ef", _gqa_prefill_kernel (query i sees the first
// i + 1 + delta keys, at most kv_len of them); the LSE is the natural log with no epsilon; the
// fully-masked-row guard is that of "splitk_kernels.py", _fwd_kernel_splitK.
//
// GB300 design:
//   * GQA packing: a 128-row Q tile holds P = floor(128/G) consecutive query
//     positions for each of the G query heads that share one KV head, so every
//     K/V tile brought on chip serves the whole group (when G does not divide
//     128, the last 128 - P G rows are never loaded and never stored);
//   * a CTA owns two such tiles (2P positions) and one KV head: the two
//     softmax warpgroups ping-pong so the tensor core always has work;
//   * warp roles: warps 0-3 softmax of tile 0, warps 4-7 softmax of tile 1,
//     warp 8 TMA producer, warp 9 MMA issuer (one elected lane), warps 10-11
//     idle; registers move from the control warpgroup to the softmax ones;
//   * one elected lane of the MMA warp issues every tcgen05.mma with
//     prebuilt descriptor words, a handful of instructions per MMA, so the
//     tensor core is not left waiting on the issuing thread;
//   * TMA (128-byte swizzle) stages Q once per work item and K/V through a
//     two-stage ring whose K and V stages are freed separately (K once both
//     S MMAs have read it, V after both P.V); tcgen05.mma accumulates S
//     (2 x 128 columns) and O (2 x 128 columns) in the 512 TMEM columns; P is
//     written back over S in TMEM as bf16 and fed to the P.V MMA from TMEM;
//   * the max is rescaled lazily (only when it grows by more than 2^8), so
//     the O accumulator in TMEM is rarely touched by the softmax warps;
//   * O leaves TMEM in one round trip and is released to the next item's P.V
//     before it is written; the dense layout writes it through a 16 KB
//     shared-memory stage per softmax warpgroup with TMA stores;
//   * a persistent grid walks whole work items longest-first in a snake
//     order, in sections of (batch, KV head) pairs whose K/V stays in L2;
//   * with caller scratch, shapes with too few items to fill the GPU take
//     a split schedule: the (item, KV tile) steps are cut into equal ranges
//     per CTA and a cut item is merged by the piece that finishes last.
//
// Ragged mode (kVarlen, "gpt-o3 / triton6fd1ef", run): a batch of sequences
// with CSR extents over a paged KV cache in one launch.  Work items are
// (sequence, query block, KV head), sorted longest-first in every CTA.  K/V
// tiles come either from the pool, gathered row by row with cp.async by the
// producer warp, or by TMA from a contiguous copy of the listed pages made
// beforehand by gather_pages_kernel.
#include <cuda_bf16.h>

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;          // rows per Q tile
constexpr int kBN = 128;          // keys per KV tile
constexpr int kThreads = 384;     // 12 warps = 3 warpgroups
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kNoRow = 0xffffffffu;
// Registers: launched at 168 per thread (384 x 168 = 64512); the
// producer/MMA warpgroup drops to 72 and each softmax warpgroup rises to
// 216 (2 x 128 x 216 + 128 x 72 = 64512, the launch total).
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsControl = 72;
constexpr int kHalf = 128 * 128;  // bytes of one 64-column half of a 128-row tile
constexpr int kTile = 2 * kHalf;  // 32 KB: 128 rows x 128 bf16
constexpr int kStages = 2;
// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffQ = 0;                        // 2 tiles
constexpr int kOffK = kOffQ + 2 * kTile;        // kStages tiles
constexpr int kOffV = kOffK + kStages * kTile;  // kStages tiles
constexpr int kSmemBytes = kOffV + kStages * kTile;
// dense layout only: a 64-column half of each softmax warpgroup's O tile,
// staged for a TMA store (the ragged mode's static tables leave no room)
constexpr int kOffStage = kSmemBytes;
constexpr int kSmemDense = kOffStage + 2 * kHalf;
// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // + 128 * tile
constexpr uint32_t kColO = 256;  // + 128 * tile

struct Params {
    __nv_bfloat16* o;
    float* lse;
    int32_t* status;
    int B, Hq, Hkv, q_len, kv_len, G, P, n_qb, n_items;
    int halves;   // 64-column halves of a head's row, D / 64 (dense: 1 or 2; ragged: 2)
    int sec_bh;   // whole items: (batch, KV head) pairs per section of the order (their K/V fits in L2)
    float scale_log2;
    // ragged batch over a paged cache (varlen mode only)
    const int32_t* qo_indptr;   // [B+1]
    const int32_t* kv_indptr;   // [B+1], in pages
    const int32_t* kv_indices;  // pool page of each listed page
    const int32_t* kv_last;     // [B] tokens in the last page (NULL: full pages)
    const __nv_bfloat16* k_pool;   // [pool_rows, Hkv, D]
    const __nv_bfloat16* v_pool;
    int page_size, pool_rows;
    int gathered;   // K/V come by TMA from a contiguous copy in page-list order
    // split schedule (dense only): the (item, KV tile) steps in item order
    // (batch, KV head, query block), cut into gridDim.x equal ranges
    long long sk_total;   // KV tile steps of all items
    long long sk_per_bh;  // KV tile steps of one (batch, KV head)
    int sk_zero_qb;       // leading query blocks that see no key
    int32_t* sk_count;    // [n_items][2 tiles][arrived, stored], zero between launches
    float* sk_o;          // [2 * gridDim.x slots][2 tiles][32 column quads][128 rows][4]
    float* sk_ml;         // [2 * gridDim.x slots][2 tiles][m, l][128 rows]
};

struct Item {
    int b, kvh, p0, n_kv;
    int q_start, q_len, delta, kv_len, kv_base;   // per-sequence extent (varlen: ragged)
    int j0, j1;           // KV tiles [j0, j1) of this piece of the item
};

constexpr int kMaxVarlenSeqs = 2048;   // sequences per ragged batch (prefix table in shared memory)
// Ragged batches of up to kMaxOrder (sequence, query block) pairs are walked
// longest-first through a sorted list in shared memory; larger ones in
// sequence order.  Pair word: sequence << kPairQbBits | query block.
constexpr int kMaxOrder = 4096;
constexpr int kOrderBuckets = 512;      // sort keys: KV tiles, 511 and more share the top bucket
constexpr int kPairQbBits = 21;

// KV tiles that query block qb (2P positions) of the dense layout sees.
__host__ __device__ __forceinline__ int dense_qb_tiles(int q_len, int kv_len, int P, int qb) {
    const int p_last = min(qb * 2 * P + 2 * P, q_len) - 1;
    const int kv_end = min(kv_len, p_last + kv_len - q_len + 1);
    return kv_end > 0 ? (kv_end + kBN - 1) / kBN : 0;
}

// The whole item of (batch * Hkv + KV head) bh and query block qb.
__device__ __forceinline__ Item dense_item(const Params& p, int bh, int qb) {
    Item it;
    it.b = bh / p.Hkv;
    it.kvh = bh % p.Hkv;
    it.p0 = qb * 2 * p.P;
    it.q_start = 0;
    it.q_len = p.q_len;
    it.kv_len = p.kv_len;
    it.kv_base = 0;
    it.delta = p.kv_len - p.q_len;
    it.n_kv = dense_qb_tiles(p.q_len, p.kv_len, p.P, qb);
    it.j0 = 0;
    it.j1 = it.n_kv;
    return it;
}

// Work item `idx` of the whole-item order: sections of sec_bh (batch, KV
// head) pairs, whose K/V stays in L2 while the section runs; within a
// section longest first (query blocks from the last), pairs inner.
__host__ __device__ __forceinline__ void whole_item(int idx, int bh_count, int n_qb, int sec_bh, int& bh, int& qb) {
    const int per_sec = sec_bh * n_qb;
    const int sec = idx / per_sec, local = idx - sec * per_sec;
    const int in_sec = min(sec_bh, bh_count - sec * sec_bh);   // the last section may be short
    qb = n_qb - 1 - local / in_sec;
    bh = sec * sec_bh + local % in_sec;
}
__device__ __forceinline__ Item item_of(const Params& p, int idx) {
    int bh, qb;
    whole_item(idx, p.B * p.Hkv, p.n_qb, p.sec_bh, bh, qb);
    return dense_item(p, bh, qb);
}

// Split schedule: the CTA whose range [L0, L1) holds step L, where CTA c
// owns [c * total / grid, (c + 1) * total / grid).
__device__ __forceinline__ int split_cta_of(const Params& p, long long L) {
    return static_cast<int>(((L + 1) * gridDim.x - 1) / p.sk_total);
}

// Position of a CTA's walk through the split schedule: step L of the
// current item (bh, qb), which starts at step `start`; the range ends at L1.
// After split_next it still describes the item of the piece it returned.
struct SplitWalk {
    long long L, L1, start;
    int bh, qb;
};

// Next piece of this CTA's range: the steps of one item that fall in it.
// Items that see no key are skipped (the softmax warps write them apart).
__device__ __forceinline__ bool split_next(const Params& p, SplitWalk& w, Item& it) {
    while (w.L < w.L1) {
        const int n = dense_qb_tiles(p.q_len, p.kv_len, p.P, w.qb);
        const long long end = w.start + n;
        if (w.L >= end) {
            w.start = end;
            if (++w.qb == p.n_qb) {
                w.qb = 0;
                ++w.bh;
            }
            continue;
        }
        it = dense_item(p, w.bh, w.qb);
        it.j0 = static_cast<int>(w.L - w.start);
        const long long stop = end < w.L1 ? end : w.L1;
        it.j1 = static_cast<int>(stop - w.start);
        w.L = stop;
        return true;
    }
    return false;
}

// Split schedule (one warp): the item holding this CTA's first step.
// Lanes take 32 query blocks at a time and scan their tile counts.
__device__ void split_find_start(const Params& p, long long L0, SplitWalk& w, int lane) {
    const int bh = static_cast<int>(L0 / p.sk_per_bh);
    const long long r = L0 - bh * p.sk_per_bh;
    long long acc = 0;
    w.bh = bh;
    w.qb = 0;
    w.start = static_cast<long long>(bh) * p.sk_per_bh;
    for (int q0 = 0; q0 < p.n_qb; q0 += 32) {
        const int q = q0 + lane;
        const long long n = q < p.n_qb ? dense_qb_tiles(p.q_len, p.kv_len, p.P, q) : 0;
        long long cum = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, cum, off);
            if (lane >= off) cum += v;
        }
        const long long total = __shfl_sync(0xffffffffu, cum, 31);
        if (acc + total > r) {
            const int first = __ffs(__ballot_sync(0xffffffffu, acc + cum > r)) - 1;
            const long long cum_f = __shfl_sync(0xffffffffu, cum, first);
            const long long n_f = __shfl_sync(0xffffffffu, n, first);
            w.qb = q0 + first;
            w.start += acc + cum_f - n_f;
            return;
        }
        acc += total;
    }
}

// Ragged batch: the item of sequence b, query block qb (2P positions) and KV
// head kvh.
__device__ __forceinline__ Item varlen_item(const Params& p, int b, int qb, int kvh) {
    Item it;
    it.b = b;
    it.q_start = p.qo_indptr[b];
    it.q_len = p.qo_indptr[b + 1] - it.q_start;
    it.kv_base = p.kv_indptr[b];
    const int n_pages = p.kv_indptr[b + 1] - it.kv_base;
    const int last = (p.kv_last != nullptr) ? p.kv_last[b] : p.page_size;
    it.kv_len = n_pages > 0 ? (n_pages - 1) * p.page_size + last : 0;
    it.delta = it.kv_len - it.q_len;
    it.kvh = kvh;
    it.p0 = qb * 2 * p.P;
    const int p_last = min(it.p0 + 2 * p.P, it.q_len) - 1;
    const int kv_end = min(it.kv_len, p_last + it.delta + 1);
    it.n_kv = kv_end > 0 ? (kv_end + kBN - 1) / kBN : 0;
    it.j0 = 0;
    it.j1 = it.n_kv;
    return it;
}

// Ragged batch, unsorted order: the pair word of item `idx` in
// sequence-major order, within a sequence the furthest query block (longest
// KV range) first.  `prefix[b]` counts the items of sequences before b.
__device__ __forceinline__ uint32_t pair_of_varlen(const Params& p, const int* prefix, int idx) {
    int lo = 0, hi = p.B;   // last b with prefix[b] <= idx
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= idx) lo = mid; else hi = mid;
    }
    const int q_len = p.qo_indptr[lo + 1] - p.qo_indptr[lo];
    const int n_qb = (q_len + 2 * p.P - 1) / (2 * p.P);
    const int qb = n_qb - 1 - (idx - prefix[lo]) / p.Hkv;
    return (static_cast<uint32_t>(lo) << kPairQbBits) | static_cast<uint32_t>(qb);
}

// Ragged batch: KV tiles of sequence b's query block qb, clamped to the
// counting-sort range.
__device__ __forceinline__ int varlen_pair_key(const Params& p, int q_len, int kv_len, int qb) {
    const int p_last = min(qb * 2 * p.P + 2 * p.P, q_len) - 1;
    const int kv_end = min(kv_len, p_last + kv_len - q_len + 1);
    const int n_kv = kv_end > 0 ? (kv_end + kBN - 1) / kBN : 0;
    return min(n_kv, kOrderBuckets - 1);
}

// Ragged batch: new-token and KV lengths of sequence b.
__device__ __forceinline__ void varlen_lens(const Params& p, int b, int& q_len, int& kv_len) {
    q_len = p.qo_indptr[b + 1] - p.qo_indptr[b];
    const int n_pages = p.kv_indptr[b + 1] - p.kv_indptr[b];
    const int last = (p.kv_last != nullptr) ? p.kv_last[b] : p.page_size;
    kv_len = n_pages > 0 ? (n_pages - 1) * p.page_size + last : 0;
}

// Ragged batch (one warp): prefix[b] = work items of the sequences before b,
// prefix[B] = all items.  One lane per sequence, 32 sequences per round.
__device__ void varlen_prefix(const Params& p, int* prefix, int lane) {
    int carry = 0;
#pragma unroll 4
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int items = 0;
        if (b < p.B) {
            const int ql = p.qo_indptr[b + 1] - p.qo_indptr[b];
            items = ((ql + 2 * p.P - 1) / (2 * p.P)) * p.Hkv;
        }
        int incl = items;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (b < p.B) prefix[b] = carry + incl - items;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[p.B] = carry;
}

// Ragged batch, sorted order (one warp, identical in every CTA): the
// (sequence, query block) pairs by decreasing KV tile count.  A counting
// sort: histogram of the keys, exclusive scan from the largest key down,
// then a scatter in a fixed order (rounds of 32 sequences, one lane each;
// within a round the furthest query blocks first, ties by lane) so that
// every CTA writes the same list.
__device__ void varlen_sort_pairs(const Params& p, uint32_t* order, int* bucket, int lane) {
    for (int k = lane; k < kOrderBuckets; k += 32) bucket[k] = 0;
    __syncwarp();
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int q_len = 0, kv_len = 0;
        if (b < p.B) varlen_lens(p, b, q_len, kv_len);
        const int n_qb = (q_len + 2 * p.P - 1) / (2 * p.P);
        for (int qb = 0; qb < n_qb; ++qb) atomicAdd(&bucket[varlen_pair_key(p, q_len, kv_len, qb)], 1);
    }
    __syncwarp();
    constexpr int per = kOrderBuckets / 32;   // lane 0 owns the largest keys
    int sum = 0;
#pragma unroll
    for (int e = 0; e < per; ++e) sum += bucket[kOrderBuckets - 1 - (per * lane + e)];
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int e = 0; e < per; ++e) {
        const int k = kOrderBuckets - 1 - (per * lane + e);
        const int c = bucket[k];
        bucket[k] = run;
        run += c;
    }
    __syncwarp();
    const uint32_t below = (1u << lane) - 1u;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int q_len = 0, kv_len = 0;
        if (b < p.B) varlen_lens(p, b, q_len, kv_len);
        const int n_qb = (q_len + 2 * p.P - 1) / (2 * p.P);
        const int rounds = __reduce_max_sync(0xffffffffu, n_qb);
        for (int k = 0; k < rounds; ++k) {
            const bool valid = k < n_qb;
            const int qb = n_qb - 1 - k;
            const uint32_t act = __ballot_sync(0xffffffffu, valid);
            int key = 0, pos = 0;
            uint32_t grp = 0;
            if (valid) {
                key = varlen_pair_key(p, q_len, kv_len, qb);
                grp = __match_any_sync(act, key);
                pos = bucket[key] + __popc(grp & below);
            }
            __syncwarp();
            if (valid) {
                order[pos] = (static_cast<uint32_t>(b) << kPairQbBits) | static_cast<uint32_t>(qb);
                if (lane == __ffs(grp) - 1) bucket[key] += __popc(grp);
            }
            __syncwarp();
        }
    }
}

// i-th item of this CTA: rounds of gridDim.x items, every other round reversed.
__device__ __forceinline__ int cta_item(int i) {
    const int round = i;
    const int pos = (round & 1) ? (gridDim.x - 1 - blockIdx.x) : blockIdx.x;
    return round * gridDim.x + pos;
}

// kVarlen: Q is ragged [total_q, Hq, D] (tile rows ordered position-major,
// r = pos * G + head) and K/V rows are gathered from a paged pool through the
// page list by the producer warp with 16-byte cp.async copies into the
// 128-byte-swizzled tile layout (TMA tile loads need contiguous rows).
// kSplit (dense only): the split schedule, where an item whose KV tiles are
// cut between CTAs is finished by the piece that ends last (see the epilogue).
// kD64 (dense, D = 64): the tiles hold only their first 64-column half, so
// S = Q K^T takes that half's 4 K steps and P.V runs at N = 64 (an
// instantiation of its own: the D = 128 kernels' MMA-issuing loop is left as
// it is, which the tensor core's rate is sensitive to).
template <bool kVarlen, bool kSplit, bool kD64 = false>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                      const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap o_map,
                      const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    __shared__ int prefix[kVarlen ? kMaxVarlenSeqs + 1 : 1];
    __shared__ uint32_t order[kVarlen ? kMaxOrder : 1];  // sorted (sequence, query block) pairs
    __shared__ int bucket[kVarlen ? kOrderBuckets : 1];
    __shared__ __align__(8) uint64_t q_full, q_empty;
    __shared__ __align__(8) uint64_t k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages];
    __shared__ __align__(8) uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    __shared__ SplitWalk walk_sh[kThreads / 32];          // split schedule: each warp's position
    __shared__ __align__(8) uint64_t sk_bar[2];           // split epilogue: a tile's 128 threads meet
    __shared__ __align__(8) uint64_t epi_bar[2];          // O staging: a tile's 128 threads meet
    __shared__ int sk_word[2];                            // split epilogue: arrival order / go flag

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&q_full, 1);
        mbar_init(&q_empty, 1);
        for (int s = 0; s < kStages; ++s) {
            // ragged, gathered in the kernel: one cp.async arrival per lane of the gather warp
            const uint32_t n_arrive = (kVarlen && !p.gathered) ? 32 : 1;
            mbar_init(&k_full[s], n_arrive);
            mbar_init(&v_full[s], n_arrive);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 128);
            mbar_init(&o_full[t], 1);
            mbar_init(&o_empty[t], 128);
            mbar_init(&sk_bar[t], 128);
            mbar_init(&epi_bar[t], 128);
        }
        abort_sh = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    if (!kVarlen && p.halves == 1) {
        // D = 64: the tiles' second 64-column halves are never loaded, and the
        // kD64 kernel's MMAs never read them; they are zeroed all the same
        static_assert(kStages == 2, "six tiles: two Q, two K, two V");
        constexpr int kVecs = kHalf / 16;
        for (int i = threadIdx.x; i < 6 * kVecs; i += kThreads) {
            const int tile = i / kVecs;   // Q0, Q1, K0, K1, V0, V1: consecutive 32 KB tiles from kOffQ
            *reinterpret_cast<uint4*>(smem + kOffQ + tile * kTile + kHalf + (i % kVecs) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();   // generic-proxy writes -> the tensor core's reads
    }
    int n_items = p.n_items;
    if constexpr (kVarlen) {
        if (warp == 0) {
            varlen_prefix(p, prefix, lane);
            __syncwarp();
            if (prefix[p.B] / p.Hkv <= kMaxOrder) varlen_sort_pairs(p, order, bucket, lane);
        }
    }
    if constexpr (kSplit) {
        if (warp == 0) {
            const long long L0 = static_cast<long long>(blockIdx.x) * p.sk_total / gridDim.x;
            SplitWalk w;
            split_find_start(p, L0, w, lane);
            if (lane == 0) {
                w.L = L0;
                w.L1 = static_cast<long long>(blockIdx.x + 1) * p.sk_total / gridDim.x;
                for (int k = 0; k < kThreads / 32; ++k) walk_sh[k] = w;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    if constexpr (kVarlen) n_items = prefix[p.B];
    const bool sorted = kVarlen && n_items / p.Hkv <= kMaxOrder;
    auto get_item = [&](int idx) -> Item {
        if constexpr (kVarlen) {
            const uint32_t pair = sorted ? order[idx / p.Hkv] : pair_of_varlen(p, prefix, idx);
            return varlen_item(p, static_cast<int>(pair >> kPairQbBits),
                               static_cast<int>(pair & ((1u << kPairQbBits) - 1u)), idx % p.Hkv);
        } else {
            return item_of(p, idx);
        }
    };
    // every role walks the same sequence of items (or, split, of item
    // pieces); the split position lives in shared memory, one per warp, so
    // that it holds no registers across the KV loops
    struct Walker {
        int i;
    };
    auto walk_begin = [&]() -> Walker { return Walker{0}; };
    auto walk_next = [&](Walker& k, Item& it) -> bool {
        if constexpr (kSplit) {
            const unsigned act = __activemask();
            SplitWalk w = walk_sh[warp];
            const bool got = split_next(p, w, it);
            __syncwarp(act);
            if (lane == __ffs(act) - 1) walk_sh[warp] = w;
            __syncwarp(act);
            return got;
        } else {
            const int idx = cta_item(k.i++);
            if (idx >= n_items) return false;
            it = get_item(idx);
            return true;
        }
    };

    auto fail = [&]() {
        flag_status(p.status, ATTN_DEV_WAIT_TIMEOUT);
        atomicExch(&abort_sh, 1);
    };
    // bounded wait that also gives up once any role has given up
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_wait(bar, parity, &abort_sh)) return true;
        fail();
        return false;
    };

    if (warp < 8) {
        regs_inc<kRegsSoftmax>();
        // ---------------------------------------------------------- softmax warpgroups
        const int t = warp >> 2;                       // which Q tile
        const int r = threadIdx.x & 127;               // row of the tile == TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_addr = tmem + lane_addr + kColS + 128 * t;
        const uint32_t o_addr = tmem + lane_addr + kColO + 128 * t;
        const float sl2 = p.scale_log2;
        uint32_t kv_iter = 0, item_iter = 0;
        bool ok = true;
        // this thread's row of item `it`: query position, head, output row
        // rows past P G are padding when G does not divide 128: never stored
        const bool row_used = r < p.P * p.G;
        auto row_of = [&](const Item& it, int& pos, size_t& row_id) {
            // head-major rows for the dense layout, position-major rows for
            // the ragged [total_q, Hq, D] layout
            const int head = it.kvh * p.G + (kVarlen ? r % p.G : r / p.P);
            pos = it.p0 + t * p.P + (kVarlen ? r / p.G : r % p.P);
            row_id = kVarlen ? (static_cast<size_t>(it.q_start) + pos) * p.Hq + head
                             : (static_cast<size_t>(it.b) * p.Hq + head) * p.q_len + pos;
        };
        // a row that sees no key: O = 0, LSE = -inf
        const int d_out = 64 * p.halves;   // D: the row stride of O
        auto write_empty = [&](size_t row_id) {
            uint4* orow = reinterpret_cast<uint4*>(p.o + row_id * d_out);
            for (int c = 0; c < d_out / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
            if (p.lse != nullptr) p.lse[row_id] = -INFINITY;
        };
        if constexpr (kSplit) {
            // the split walk skips the leading query blocks that see no key
            const int zq = p.sk_zero_qb;
            for (int k = blockIdx.x; k < p.B * p.Hkv * zq; k += gridDim.x) {
                int pos;
                size_t row_id;
                row_of(dense_item(p, k / zq, k % zq), pos, row_id);
                if (row_used && pos < p.q_len) write_empty(row_id);
            }
        }
        Walker wk = walk_begin();
        for (Item it; ok && walk_next(wk, it);) {
            const int delta = it.delta;
            int pos;
            size_t row_id;
            row_of(it, pos, row_id);
            const bool row_real = row_used && pos < it.q_len;
            if (it.n_kv == 0) {
                if (row_real) write_empty(row_id);
                continue;
            }
            const int pos_min = it.p0 + t * p.P;     // smallest position of this tile
            const int lim_row = pos + delta;         // last visible key of this row
            float m = -INFINITY, l = 0.f;
            bool o_live = false;   // O_t holds this piece's accumulation (after its first P.V)
            for (int j = it.j0; j < it.j1; ++j, ++kv_iter) {
                if (!(ok = wait(&s_full[t], kv_iter & 1))) break;
                tc_fence_after();
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + 32 * c, sr[c]);
                tmem_ld_wait();
                const int kv0 = j * kBN;
                // causal mask only on tiles that cross this tile's diagonal
                if (kv0 + kBN - 1 > pos_min + delta) {
                    const int lim = lim_row - kv0;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (32 * c + e > lim) sr[c][e] = __float_as_uint(-INFINITY);
                }
                // row max: four independent chains of 3-input max
                float mc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < 32; e += 2)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        mc[c] = max3f(mc[c], __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
                float mx = max3f(mc[0], mc[1], fmaxf(mc[2], mc[3])) * sl2;
                float alpha = 1.f;
                const bool grow = mx > m + 8.f;
                if (grow) {
                    alpha = ex2(m - mx);   // 0 when m = -inf
                    m = mx;
                    l *= alpha;
                }
                if (o_live && __any_sync(0xffffffffu, grow)) {
                    // O_t is idle here: the commit that announced S_t also covers
                    // the P.V of the previous tile
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t orr[32];
                        tmem_ld32(o_addr + 32 * c, orr);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                        tmem_st32(o_addr + 32 * c, orr);
                    }
                }
                const float neg_m = (m == -INFINITY) ? 0.f : -m;
                // p = 2^(s * scale * log2 e - m): packed pair FMAs, MUFU ex2,
                // four independent pair-sum chains, bf16x2 packing into TMEM
                const float2 scl2 = make_float2(sl2, sl2), nm2 = make_float2(neg_m, neg_m);
                float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int c = 2 * hh + (e >> 4), col = 2 * (e & 15);
                        const float2 y = __ffma2_rn(
                            make_float2(__uint_as_float(sr[c][col]), __uint_as_float(sr[c][col + 1])), scl2, nm2);
                        const float2 pp = make_float2(ex2(y.x), ex2(y.y));
                        ls[e & 3] = __fadd2_rn(ls[e & 3], pp);
                        pk[e] = pack_bf16x2(pp.x, pp.y);
                    }
                    tmem_st32(s_addr + 32 * hh, pk);
                }
                const float2 l01 = __fadd2_rn(ls[0], ls[1]), l23 = __fadd2_rn(ls[2], ls[3]);
                l += (l01.x + l01.y) + (l23.x + l23.y);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&p_full[t]);
                o_live = true;
            }
            if (!ok) break;
            // -------------------------------------------------------------- epilogue
            // Split schedule, an item cut between CTAs: each piece takes an
            // arrival ticket (while its last P.V still runs).  Every piece but
            // the last stores its unnormalised O, m and l (fp32) in its CTA's
            // slot; the last waits until they are stored, merges them with its
            // own by LSE weighting, writes O and LSE and zeroes the counters.
            // Pieces that arrived never wait, so the wait always ends.
            int np = 1, c0 = 0, arrival = 0;
            int32_t* ctr = nullptr;
            // the tile's 128 threads meet (bounded wait); every cut piece meets
            // twice, so the barrier's phases go 0, 1, 0, 1, ...
            auto wg_sync = [&](uint32_t phase) -> bool {
                mbar_arrive(&sk_bar[t]);
                return wait(&sk_bar[t], phase);
            };
            if constexpr (kSplit) {
                const SplitWalk w = walk_sh[warp];   // still the item of this piece
                const long long item_end = w.start + dense_qb_tiles(p.q_len, p.kv_len, p.P, w.qb);
                c0 = split_cta_of(p, w.start);
                np = split_cta_of(p, item_end - 1) - c0 + 1;
                if (np > 1) {
                    ctr = p.sk_count + ((static_cast<size_t>(w.bh) * p.n_qb + w.qb) * 2 + t) * 2;
                    if (r == 0) {
                        const int a = atomicAdd(ctr, 1);
                        // a ticket past the piece count: the counters did not start at zero
                        if (a >= np) flag_status(p.status, ATTN_DEV_WORKSPACE_STATE);
                        sk_word[t] = a;
                    }
                    if (!(ok = wg_sync(0))) break;
                    arrival = sk_word[t];
                }
            }
            if (!(ok = wait(&o_full[t], item_iter & 1))) break;
            tc_fence_after();
            row_of(it, pos, row_id);   // recomputed: not held in registers across the KV loop
            if (np == 1 || arrival < np - 1) {
                // O leaves TMEM in one round trip, and the next item's P.V may
                // overwrite it while this one is written out
                uint32_t ov[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(o_addr + 32 * c, ov[c]);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&o_empty[t]);
                ++item_iter;
                if (np == 1) {
                    const bool alive = l > 0.f;
                    const float inv_l = alive ? 1.f / l : 0.f;
                    auto pack8 = [&](int c, int e) {   // columns 32 c + e .. + 7 of this row, as bf16
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(ov[c][e]) * inv_l, __uint_as_float(ov[c][e + 1]) * inv_l);
                        v.y = pack_bf16x2(__uint_as_float(ov[c][e + 2]) * inv_l, __uint_as_float(ov[c][e + 3]) * inv_l);
                        v.z = pack_bf16x2(__uint_as_float(ov[c][e + 4]) * inv_l, __uint_as_float(ov[c][e + 5]) * inv_l);
                        v.w = pack_bf16x2(__uint_as_float(ov[c][e + 6]) * inv_l, __uint_as_float(ov[c][e + 7]) * inv_l);
                        return v;
                    };
                    if constexpr (!kVarlen) {
                        // Each 64-column half of the tile goes through this warpgroup's
                        // 16 KB stage (128-byte swizzle, row r at r * 128) and leaves
                        // by one TMA store of the box {64, P, G} its Q came in by, so
                        // the rows reach memory as whole lines; rows past q_len are
                        // clipped by the store.  Four meetings per item: phases 0 1 0 1.
                        uint8_t* stage = smem + kOffStage + t * kHalf;
                        const bool tile_real = it.p0 + t * p.P < p.q_len;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (h >= p.halves) break;
                            if (r == 0) bulk_wait_read_all();   // the stage's last store has read it
                            mbar_arrive(&epi_bar[t]);
                            if (!(ok = wait(&epi_bar[t], 0))) break;
#pragma unroll
                            for (int cc = 0; cc < 8; ++cc)
                                *reinterpret_cast<uint4*>(stage + r * 128 + ((cc ^ (r & 7)) << 4)) =
                                    pack8(2 * h + (cc >> 2), 8 * (cc & 3));
                            fence_proxy_async_smem();   // generic-proxy writes -> the TMA's reads
                            mbar_arrive(&epi_bar[t]);
                            if (!(ok = wait(&epi_bar[t], 1))) break;
                            if (r == 0 && tile_real) {
                                tma_store_3d(&o_map, stage, h * 64, it.p0 + t * p.P, it.b * p.Hq + it.kvh * p.G);
                                bulk_commit();
                            }
                        }
                        if (!ok) break;
                    } else if (row_real) {
                        uint4* orow = reinterpret_cast<uint4*>(p.o + row_id * kD);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int e = 0; e < 32; e += 8) orow[(32 * c + e) / 8] = pack8(c, e);
                    }
                    if (row_real && p.lse != nullptr) p.lse[row_id] = alive ? (m * kLn2 + logf(l)) : -INFINITY;
                } else {
                    // the item's first piece (on CTA c0) has slot 2 c0 + 1, the others 2 c
                    const int slot = 2 * static_cast<int>(blockIdx.x) + (c0 == static_cast<int>(blockIdx.x) ? 1 : 0);
                    float4* dst = reinterpret_cast<float4*>(p.sk_o) + (static_cast<size_t>(slot) * 2 + t) * 32 * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[(c * 8 + q) * 128 + r] =
                                make_float4(__uint_as_float(ov[c][4 * q]), __uint_as_float(ov[c][4 * q + 1]),
                                            __uint_as_float(ov[c][4 * q + 2]), __uint_as_float(ov[c][4 * q + 3]));
                    float* ml = p.sk_ml + (static_cast<size_t>(slot) * 2 + t) * 256;
                    ml[r] = m;
                    ml[128 + r] = l;
                    __threadfence();
                    if (!(ok = wg_sync(1))) break;   // sk_word[t] is read by every thread by now
                    if (r == 0) atomicAdd(ctr + 1, 1);
                }
                continue;
            }
            if constexpr (kSplit) {
                // the last piece to arrive: wait until the others are stored
                if (r == 0) {
                    bool stored = false;
                    const uint64_t t0 = global_ns();
                    for (uint32_t spin = 0;; ++spin) {
                        const int done = ld_acquire_gpu(ctr + 1);
                        if (done >= np - 1) {
                            if (done > np - 1) flag_status(p.status, ATTN_DEV_WORKSPACE_STATE);
                            stored = true;
                            break;
                        }
                        if ((spin & 63u) == 63u &&
                            (global_ns() - t0 > kWaitLimitNs || *reinterpret_cast<volatile int*>(&abort_sh)))
                            break;
                    }
                    if (stored) {
                        ctr[0] = 0;
                        ctr[1] = 0;
                    } else {
                        fail();
                    }
                    sk_word[t] = stored ? 1 : 0;
                }
                if (!(ok = wg_sync(1))) break;
                if (!(ok = sk_word[t] != 0)) break;
                // Pieces in CTA order, this CTA's own from TMEM, the others
                // from their slots (the first piece, on CTA c0, in slot
                // 2 c0 + 1, a later one in 2 c): the same sums whichever
                // piece merges, so the result does not depend on timing.
                const int self = static_cast<int>(blockIdx.x);
                auto slot_of = [&](int c) { return static_cast<size_t>((2 * c + (c == c0 ? 1 : 0)) * 2 + t); };
                float mm = m;
                for (int c = c0; c < c0 + np; ++c)
                    if (c != self) mm = fmaxf(mm, __ldcg(p.sk_ml + slot_of(c) * 256 + r));
                const bool none = mm == -INFINITY;
                float lsum = 0.f;
                for (int c = c0; c < c0 + np; ++c) {
                    const float mc = c == self ? m : __ldcg(p.sk_ml + slot_of(c) * 256 + r);
                    const float lc = c == self ? l : __ldcg(p.sk_ml + slot_of(c) * 256 + 128 + r);
                    lsum += none ? 0.f : lc * ex2(mc - mm);
                }
                const bool alive = lsum > 0.f;
                const float inv = alive ? 1.f / lsum : 0.f;
                uint4* orow = reinterpret_cast<uint4*>(p.o + row_id * d_out);
#pragma unroll 1
                for (int c = 0; c < 2 * p.halves; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(o_addr + 32 * c, orr);
                    tmem_ld_wait();
                    float acc[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
                    for (int cc = c0; cc < c0 + np && !none; ++cc) {
                        if (cc == self) {
                            const float w = ex2(m - mm);
#pragma unroll
                            for (int e = 0; e < 32; ++e) acc[e] = fmaf(w, __uint_as_float(orr[e]), acc[e]);
                            continue;
                        }
                        const size_t so = slot_of(cc);
                        const float w = ex2(__ldcg(p.sk_ml + so * 256 + r) - mm);
                        const float4* src = reinterpret_cast<const float4*>(p.sk_o) + so * 32 * 128;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 v = __ldcg(src + (c * 8 + q) * 128 + r);
                            acc[4 * q] = fmaf(w, v.x, acc[4 * q]);
                            acc[4 * q + 1] = fmaf(w, v.y, acc[4 * q + 1]);
                            acc[4 * q + 2] = fmaf(w, v.z, acc[4 * q + 2]);
                            acc[4 * q + 3] = fmaf(w, v.w, acc[4 * q + 3]);
                        }
                    }
                    if (row_real) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            uint4 v;
                            v.x = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
                            v.y = pack_bf16x2(acc[e + 2] * inv, acc[e + 3] * inv);
                            v.z = pack_bf16x2(acc[e + 4] * inv, acc[e + 5] * inv);
                            v.w = pack_bf16x2(acc[e + 6] * inv, acc[e + 7] * inv);
                            orow[(32 * c + e) / 8] = v;
                        }
                    }
                }
                if (row_real && p.lse != nullptr) p.lse[row_id] = alive ? (mm * kLn2 + logf(lsum)) : -INFINITY;
                tc_fence_before();
                mbar_arrive(&o_empty[t]);
                ++item_iter;
            }
        }
        if (!kVarlen && r == 0) bulk_wait_all();   // O's TMA stores done before the CTA exits
    } else {
        regs_dec<kRegsControl>();
        if (warp == kProducerWarp && kVarlen && p.gathered) {
            // ------------------------- producer, ragged batch from the contiguous copy
            // Token t of sequence b is row kv_indptr[b] * page_size + t of the copy
            // [rows, Hkv, D]; the tile halves are 2D TMA boxes {64, 128}.  Rows past a sequence's end belong to the next sequence, or
            // are zero: the causal limit masks them.
            if (lane == 0) {
                tma_prefetch_desc(&q_map);
                tma_prefetch_desc(&k_map);
                tma_prefetch_desc(&v_map);
                uint32_t kv_iter = 0, item_iter = 0;
                bool ok = true;
                Walker wk = walk_begin();
                for (Item it; ok && walk_next(wk, it);) {
                    if (it.n_kv == 0) continue;
                    if (item_iter > 0 && !(ok = wait(&q_empty, (item_iter - 1) & 1))) break;
                    mbar_arrive_expect_tx(&q_full, 2 * p.P * p.G * 256);
                    for (int t = 0; t < 2; ++t)
                        for (int h = 0; h < 2; ++h)
                            tma_load_3d(smem + kOffQ + t * kTile + h * kHalf, &q_map, &q_full, h * 64,
                                        it.kvh * p.G, it.q_start + it.p0 + t * p.P);
                    const int row0 = it.kv_base * p.page_size;
                    for (int j = 0; j < it.n_kv; ++j, ++kv_iter) {
                        const int s = kv_iter % kStages;
                        const uint32_t par = ((kv_iter / kStages) - 1) & 1;
                        const int row = row0 + j * kBN;
                        const int x = it.kvh * kD;
                        if (kv_iter >= kStages && !(ok = wait(&k_empty[s], par))) break;
                        mbar_arrive_expect_tx(&k_full[s], kTile);
                        tma_load_2d(smem + kOffK + s * kTile, &k_map, &k_full[s], x, row);
                        tma_load_2d(smem + kOffK + s * kTile + kHalf, &k_map, &k_full[s], x + 64, row);
                        if (kv_iter >= kStages && !(ok = wait(&v_empty[s], par))) break;
                        mbar_arrive_expect_tx(&v_full[s], kTile);
                        tma_load_2d(smem + kOffV + s * kTile, &v_map, &v_full[s], x, row);
                        tma_load_2d(smem + kOffV + s * kTile + kHalf, &v_map, &v_full[s], x + 64, row);
                    }
                    ++item_iter;
                }
            }
        } else if (warp == kProducerWarp && kVarlen) {
            // ------------------------------------------ producer, ragged batch over a paged pool
            // Q tiles by TMA; K/V rows gathered by the whole warp with 16-byte
            // cp.async copies: lane i copies token rows i, i+32, i+64, i+96 of
            // each 128-token tile, 16 chunks per row.  Rows 32 apart share their
            // swizzle phase, so one instruction's 32 chunks fill every bank
            // four times over (the minimum for 512 bytes).  The pool rows of the
            // next tile are looked up while this tile's copies are issued; K
            // arrives on its own barrier before the V copies start; tokens past
            // the sequence are zero-filled.  (A second gather warp was slower:
            // its issue slots come out of the softmax warps of its SM quarter.)
            if (lane == 0) tma_prefetch_desc(&q_map);
            const size_t row_elems = static_cast<size_t>(p.Hkv) * kD;
            const uint32_t swz = static_cast<uint32_t>(lane & 7);
            uint32_t kv_iter = 0, item_iter = 0;
            bool ok = true;
            Walker wk = walk_begin();
            for (Item it; ok && walk_next(wk, it);) {
                if (it.n_kv == 0) continue;
                if (lane == 0) {
                    if (item_iter > 0) ok = wait(&q_empty, (item_iter - 1) & 1);
                    if (ok) {
                        mbar_arrive_expect_tx(&q_full, 2 * p.P * p.G * 256);
                        for (int t = 0; t < 2; ++t)
                            for (int h = 0; h < 2; ++h)
                                tma_load_3d(smem + kOffQ + t * kTile + h * kHalf, &q_map, &q_full, h * 64,
                                            it.kvh * p.G, it.q_start + it.p0 + t * p.P);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                // pool rows of tokens i + 32e of tile j (kNoRow past the sequence)
                auto resolve = [&](int j, uint32_t (&r4)[4]) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int tok = j * kBN + 32 * e + lane;
                        r4[e] = kNoRow;
                        if (tok < it.kv_len) {
                            const int page = p.kv_indices[it.kv_base + tok / p.page_size];
                            if (page >= 0 && static_cast<long long>(page) * p.page_size < p.pool_rows)
                                r4[e] = static_cast<uint32_t>(page) * p.page_size + tok % p.page_size;
                            else
                                flag_status(p.status, ATTN_DEV_PAGE_OUT_OF_RANGE);
                        }
                    }
                };
                uint32_t nxt[4];
                resolve(0, nxt);
                for (int j = 0; j < it.n_kv; ++j, ++kv_iter) {
                    const int s = kv_iter % kStages;
                    const uint32_t par = ((kv_iter / kStages) - 1) & 1;
                    uint32_t cur[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) cur[e] = nxt[e];
                    if (j + 1 < it.n_kv) resolve(j + 1, nxt);   // index loads overlap this tile's copies
#pragma unroll 1
                    for (int kv = 0; kv < 2 && ok; ++kv) {
                        // K's stage frees once both S MMAs have read it, V's after both P.V
                        if (lane == 0 && kv_iter >= kStages) ok = wait(kv == 0 ? &k_empty[s] : &v_empty[s], par);
                        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                        if (!ok) break;
                        const __nv_bfloat16* base = (kv == 0 ? p.k_pool : p.v_pool) + it.kvh * kD;
                        uint8_t* dst = smem + (kv == 0 ? kOffK : kOffV) + s * kTile + lane * 128;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const bool real = cur[e] != kNoRow;
                            const __nv_bfloat16* src = base + (real ? static_cast<size_t>(cur[e]) * row_elems : 0);
                            const uint32_t nb = real ? 16u : 0u;
#pragma unroll
                            for (int c = 0; c < 16; ++c)
                                cp_async16(dst + e * 32 * 128 + (c >> 3) * kHalf + (((c & 7) ^ swz) << 4),
                                           src + 8 * c, nb);
                        }
                        cp_async_mbar_arrive(kv == 0 ? &k_full[s] : &v_full[s]);
                    }
                    if (!ok) break;
                }
                ++item_iter;
            }
            cp_async_wait_all();   // no copy may land after an early exit has released the CTA
        } else if (warp == kProducerWarp) {
            // ------------------------------------------------------------ TMA producer
            if (lane == 0) {
                tma_prefetch_desc(&q_map);
                tma_prefetch_desc(&k_map);
                tma_prefetch_desc(&v_map);
                uint32_t kv_iter = 0, item_iter = 0;
                bool ok = true;
                Walker wk = walk_begin();
                for (Item it; ok && walk_next(wk, it);) {
                    if (it.n_kv == 0) continue;
                    if (item_iter > 0 && !(ok = wait(&q_empty, (item_iter - 1) & 1))) break;
                    mbar_arrive_expect_tx(&q_full, 2 * p.P * p.G * 128 * p.halves);
                    const int head0 = it.b * p.Hq + it.kvh * p.G;
                    for (int t = 0; t < 2; ++t)
                        for (int h = 0; h < p.halves; ++h)
                            tma_load_3d(smem + kOffQ + t * kTile + h * kHalf, &q_map, &q_full, h * 64, it.p0 + t * p.P,
                                        head0);
                    const int kvrow = it.b * p.Hkv + it.kvh;
                    for (int j = it.j0; j < it.j1; ++j, ++kv_iter) {
                        const int s = kv_iter % kStages;
                        const uint32_t par = ((kv_iter / kStages) - 1) & 1;
                        if (kv_iter >= kStages && !(ok = wait(&k_empty[s], par))) break;
                        mbar_arrive_expect_tx(&k_full[s], kHalf * p.halves);
                        tma_load_3d(smem + kOffK + s * kTile, &k_map, &k_full[s], 0, j * kBN, kvrow);
                        if (p.halves == 2)
                            tma_load_3d(smem + kOffK + s * kTile + kHalf, &k_map, &k_full[s], 64, j * kBN, kvrow);
                        if (kv_iter >= kStages && !(ok = wait(&v_empty[s], par))) break;
                        mbar_arrive_expect_tx(&v_full[s], kHalf * p.halves);
                        tma_load_3d(smem + kOffV + s * kTile, &v_map, &v_full[s], 0, j * kBN, kvrow);
                        if (p.halves == 2)
                            tma_load_3d(smem + kOffV + s * kTile + kHalf, &v_map, &v_full[s], 64, j * kBN, kvrow);
                    }
                    ++item_iter;
                }
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------- MMA issuer
            if (lane == 0) {
                // tiles written by cp.async (the generic proxy) need a proxy fence
                // before the tensor core reads them; TMA-written tiles do not
                const bool cp_async_tiles = kVarlen && !p.gathered;
                constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, false);
                constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, kD64 ? 64 : kD, true);
                // This one thread issues every MMA of the CTA, so its instruction
                // count per MMA bounds the tensor core: the descriptors' low words
                // are built once and an MMA only adds a constant start-address
                // offset (>> 4); the high word is an immediate in the instruction.
                // (Full 64-bit descriptors rebuilt per MMA left the tensor core idle
                // about a third of the time.)
                const uint32_t d_base = sw128_desc_lo(smem_u32(smem), 16);   // low word of a descriptor at smem
                auto issue_s = [&](int t, int stage) {  // S_t = Q_t K^T
                    const uint32_t dq = d_base + ((kOffQ + t * kTile) >> 4), dk = d_base + ((kOffK + stage * kTile) >> 4);
                    const uint32_t d = tmem + kColS + 128 * t;
                    umma_ss_lo<0>(d, dq, dk, idesc_qk);
    #pragma unroll
                    for (int kk = 1; kk < (kD64 ? 4 : kD / 16); ++kk) {
                        const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                        umma_ss_lo<1>(d, dq + off, dk + off, idesc_qk);
                    }
                };
                auto issue_pv = [&](int t, int stage, bool acc) {  // O_t (+)= P_t V
                    // V: leading offset kHalf (the two 64-column halves) in bits 16-29
                    const uint32_t dv = d_base + ((kOffV + stage * kTile) >> 4) + (((kHalf - 16) >> 4) << 16);
                    const uint32_t d = tmem + kColO + 128 * t, a = tmem + kColS + 128 * t;
                    umma_ts_lo(d, a, dv, idesc_pv, acc ? 1u : 0u);
    #pragma unroll
                    for (int kk = 1; kk < kBN / 16; ++kk) umma_ts_lo(d, a + kk * 8, dv + ((kk * 16 * 128) >> 4), idesc_pv, 1u);
                };
                uint32_t kv_iter = 0, item_iter = 0;
                bool ok = true;
                Walker wk = walk_begin();
                for (Item it; ok && walk_next(wk, it);) {
                    if (it.n_kv == 0) continue;
                    if (!(ok = wait(&q_full, item_iter & 1))) break;
                    if (!(ok = wait(&k_full[kv_iter % kStages], (kv_iter / kStages) & 1))) break;
                    if (cp_async_tiles) fence_proxy_async_smem();   // cp.async writes -> tensor-core reads
                    tc_fence_after();
                    issue_s(0, kv_iter % kStages);
                    umma_commit(&s_full[0]);
                    issue_s(1, kv_iter % kStages);
                    umma_commit(&s_full[1]);
                    umma_commit(&k_empty[kv_iter % kStages]);   // K_j no longer read
                    if (it.j1 - it.j0 == 1) umma_commit(&q_empty);  // Q no longer read: the producer may refill it
                    for (int j = it.j0; j < it.j1 && ok; ++j, ++kv_iter) {
                        const int s = kv_iter % kStages;
                        const bool last = (j + 1 == it.j1);
                        const uint32_t nxt = kv_iter + 1;
                        if (!(ok = wait(&v_full[s], (kv_iter / kStages) & 1))) break;
                        if (cp_async_tiles) fence_proxy_async_smem();
                        for (int t = 0; t < 2; ++t) {
                            if (!(ok = wait(&p_full[t], kv_iter & 1))) break;
                            if (j == it.j0 && item_iter > 0 && !(ok = wait(&o_empty[t], (item_iter - 1) & 1))) break;
                            tc_fence_after();
                            issue_pv(t, s, j > it.j0);                   // O_t (+)= P_t V_j
                            if (t == 1) umma_commit(&v_empty[s]);     // V_j no longer read
                            if (!last) {
                                if (t == 0) {
                                    if (!(ok = wait(&k_full[nxt % kStages], (nxt / kStages) & 1))) break;
                                    if (cp_async_tiles) fence_proxy_async_smem();
                                    tc_fence_after();
                                }
                                issue_s(t, nxt % kStages);            // S_t = Q_t K_{j+1}^T (after P_t is read)
                                umma_commit(&s_full[t]);
                                if (t == 1) umma_commit(&k_empty[nxt % kStages]);   // K_{j+1} no longer read
                                if (t == 1 && j + 2 == it.j1) umma_commit(&q_empty);  // last S read Q
                            } else {
                                umma_commit(&o_full[t]);
                            }
                        }
                    }
                    if (!ok) break;
                    ++item_iter;
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Copies the K and V rows of every listed page into contiguous buffers in
// page-list order (row r = list entry r / page_size, offset r % page_size),
// one warp per row, 16-byte vectors; the 128 rows after the last one are
// zeroed so that the last tile of the last sequence reads zeros.  A page id
// outside the pool gives zero rows and ATTN_DEV_PAGE_OUT_OF_RANGE; a list
// longer than the copy sets ATTN_DEV_SEQ_TOO_LONG and is cut.
__global__ void __launch_bounds__(256) gather_pages_kernel(const uint4* __restrict__ k_pool,
                                                           const uint4* __restrict__ v_pool,
                                                           const int32_t* __restrict__ kv_indptr,
                                                           const int32_t* __restrict__ kv_indices, int B,
                                                           int page_size, int num_pages, int row_vecs,
                                                           uint4* __restrict__ k_ws, uint4* __restrict__ v_ws,
                                                           int max_rows, int32_t* status) {
    const long long listed = static_cast<long long>(kv_indptr[B]) * page_size;
    if (listed > max_rows && blockIdx.x == 0 && threadIdx.x == 0) flag_status(status, ATTN_DEV_SEQ_TOO_LONG);
    const long long rows = listed < max_rows ? listed : max_rows;
    const long long zero_end = (rows + kBN < max_rows) ? rows + kBN : max_rows;
    const int lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (long long r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < zero_end; r += warps) {
        bool real = false;
        size_t src = 0;
        if (r < rows) {
            const int page = kv_indices[r / page_size];
            real = page >= 0 && page < num_pages;
            if (!real && lane == 0) flag_status(status, ATTN_DEV_PAGE_OUT_OF_RANGE);
            src = (static_cast<size_t>(real ? page : 0) * page_size + r % page_size) * row_vecs;
        }
        const size_t dst = static_cast<size_t>(r) * row_vecs;
        for (int v = lane; v < row_vecs; v += 32) {
            const uint4 kx = real ? k_pool[src + v] : zero;
            const uint4 vx = real ? v_pool[src + v] : zero;
            k_ws[dst + v] = kx;
            v_ws[dst + v] = vx;
        }
    }
}

}  // namespace

namespace {

// Cost model of the two schedules, in KV tile steps of one CTA (a step is
// about 1.8 us on GB300): a piece costs its steps plus kPieceCost (Q load,
// pipeline fill, epilogue: measured at about 2 steps), a piece of a cut item
// kMergeCost more (its fp32 partial stored, or the others merged).  The
// split schedule is taken only when it is expected to be kSplitGain faster.
constexpr double kPieceCost = 2.0;
constexpr double kMergeCost = 1.5;
constexpr double kSplitGain = 0.9;

struct SplitPlan {
    bool split;
    long long total, per_bh;
    int zero_qb, grid;
};

// Chooses between whole items, longest first in snake order, and the split
// schedule; the split one only when it is expected to finish sooner.  Few
// items (the tail of whole items is then large) is where splitting pays.
SplitPlan plan_schedule(int B, int Hkv, int q_len, int kv_len, int P, int n_qb, int sec_bh, int sms,
                        bool have_ws) {
    SplitPlan pl{false, 0, 0, 0, 0};
    const long long bh = static_cast<long long>(B) * Hkv;
    if (!have_ws || bh * n_qb >= 8LL * sms) return pl;
    std::vector<int> tiles(n_qb);
    for (int qb = 0; qb < n_qb; ++qb) {
        tiles[qb] = dense_qb_tiles(q_len, kv_len, P, qb);
        pl.per_bh += tiles[qb];
        if (tiles[qb] == 0) pl.zero_qb = qb + 1;
    }
    pl.total = bh * pl.per_bh;
    if (pl.total == 0) return pl;
    // whole items: the kernel's snake order over the longest-first list
    const long long n_items = bh * n_qb;
    const int grid_w = static_cast<int>(n_items < sms ? n_items : sms);
    std::vector<double> load(grid_w, 0.0);
    for (long long idx = 0; idx < n_items; ++idx) {
        const long long round = idx / grid_w, k = idx % grid_w;
        const int cta = static_cast<int>((round & 1) ? grid_w - 1 - k : k);
        int b_h, qb;
        whole_item(static_cast<int>(idx), static_cast<int>(bh), n_qb, sec_bh, b_h, qb);
        const int n = tiles[qb];
        if (n > 0) load[cta] += n + kPieceCost;
    }
    const double whole = *std::max_element(load.begin(), load.end());
    // split: equal ranges of the (item, KV tile) order
    const int grid_s = static_cast<int>(pl.total < sms ? pl.total : sms);
    std::vector<double> sload(grid_s, 0.0);
    long long start = 0;
    for (long long i = 0; i < n_items; ++i) {
        const int n = tiles[i % n_qb];
        if (n == 0) continue;
        const long long end = start + n;
        const int c0 = static_cast<int>(((start + 1) * grid_s - 1) / pl.total);
        const int c1 = static_cast<int>((end * grid_s - 1) / pl.total);
        for (int c = c0; c <= c1; ++c) {
            const long long lo = std::max(start, static_cast<long long>(c) * pl.total / grid_s);
            const long long hi = std::min(end, static_cast<long long>(c + 1) * pl.total / grid_s);
            sload[c] += static_cast<double>(hi - lo) + kPieceCost + (c1 > c0 ? kMergeCost : 0.0);
        }
        start = end;
    }
    const double split = *std::max_element(sload.begin(), sload.end());
    if (split < kSplitGain * whole) {
        pl.split = true;
        pl.grid = grid_s;
    }
    return pl;
}

size_t round16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

// (batch, KV head) pairs per section of the whole-item order.  A section's
// K/V must fit in kSectionBytes (half of the 126 MB L2, the rest for the
// streaming Q and O), and its items must fill whole rounds of `grid` CTAs:
// the longest-first snake balances the CTAs only while item sizes fall from
// round to round, and a round shared by two sections would mix the shortest
// items of one with the longest of the next.  Without such a size, a single
// section (all pairs, the plain longest-first order).
constexpr double kSectionBytes = 64.0 * (1 << 20);
int section_pairs(const PrefillArgs& a, int n_qb, int grid) {
    const double kv_pair = 2.0 * a.kv_len * a.D * 2;   // K and V of one pair, bf16
    const int bh = a.B * a.Hkv;
    const int most = static_cast<int>(kSectionBytes / kv_pair);
    if (most >= bh) return bh;
    for (int s = most; s >= 1; --s)
        if ((static_cast<long long>(s) * n_qb) % grid == 0) return s;
    return bh;
}

}  // namespace

size_t prefill_tc_workspace_bytes(const PrefillArgs& a, int sms) {
    const int G = a.Hq / a.Hkv;
    const int P = kBM / G;
    const long long n_items = static_cast<long long>(a.B) * a.Hkv * ((a.q_len + 2 * P - 1) / (2 * P));
    const size_t counters = round16(static_cast<size_t>(n_items) * 2 * 2 * sizeof(int32_t));
    const size_t o_part = static_cast<size_t>(2) * sms * 2 * kD * kBM * sizeof(float);
    const size_t ml_part = static_cast<size_t>(2) * sms * 2 * 2 * kBM * sizeof(float);
    return counters + o_part + ml_part;
}

size_t prefill_tc_counter_bytes(const PrefillArgs& a) {
    const int G = a.Hq / a.Hkv;
    const int P = kBM / G;
    const long long n_items = static_cast<long long>(a.B) * a.Hkv * ((a.q_len + 2 * P - 1) / (2 * P));
    return round16(static_cast<size_t>(n_items) * 2 * 2 * sizeof(int32_t));
}

int prefill_tc_plan(const PrefillArgs& a, int sms, int* grid) {
    const int G = a.Hq / a.Hkv;
    const int P = kBM / G;
    const int n_qb = (a.q_len + 2 * P - 1) / (2 * P);
    const long long n_items = static_cast<long long>(a.B) * a.Hkv * n_qb;
    const int grid_w = static_cast<int>(n_items < sms ? n_items : sms);
    const SplitPlan pl =
        plan_schedule(a.B, a.Hkv, a.q_len, a.kv_len, P, n_qb, section_pairs(a, n_qb, grid_w), sms, true);
    if (grid != nullptr) *grid = pl.split ? pl.grid : grid_w;
    return pl.split ? 1 : 0;
}

bool prefill_tc_supported(const PrefillArgs& a) {
    if (a.dtype != ATTN_BF16 || (a.D != kD && a.D != 64)) return false;
    const int G = a.Hq / a.Hkv;
    if (G < 1 || G > 128) return false;
    return true;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream) {
    const int G = a.Hq / a.Hkv;
    const int P = kBM / G;
    const uint64_t D = static_cast<uint64_t>(a.D);   // 128, or 64 (loaded into the first half of each tile)
    CUtensorMap q_map, k_map, v_map;
    {
        const uint64_t dims[3] = {D, static_cast<uint64_t>(a.q_len), static_cast<uint64_t>(a.B) * a.Hq};
        const uint64_t strides[2] = {D * 2, static_cast<uint64_t>(a.q_len) * D * 2};
        const uint32_t box[3] = {64, static_cast<uint32_t>(P), static_cast<uint32_t>(G)};
        if (!encode_tiled_map(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {D, static_cast<uint64_t>(a.kv_len), static_cast<uint64_t>(a.B) * a.Hkv};
        const uint64_t strides[2] = {D * 2, static_cast<uint64_t>(a.kv_len) * D * 2};
        const uint32_t box[3] = {64, kBN, 1};
        if (!encode_tiled_map(&k_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.k, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tiled_map(&v_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.v, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    CUtensorMap o_map;   // O [B * Hq, q_len, D]: the Q map's geometry over the output
    {
        const uint64_t dims[3] = {D, static_cast<uint64_t>(a.q_len), static_cast<uint64_t>(a.B) * a.Hq};
        const uint64_t strides[2] = {D * 2, static_cast<uint64_t>(a.q_len) * D * 2};
        const uint32_t box[3] = {64, static_cast<uint32_t>(P), static_cast<uint32_t>(G)};
        if (!encode_tiled_map(&o_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.o, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    Params p;
    p.o = static_cast<__nv_bfloat16*>(a.o);
    p.lse = a.lse;
    p.status = a.dev_status;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.q_len = a.q_len;
    p.kv_len = a.kv_len;
    p.G = G;
    p.P = P;
    p.n_qb = (a.q_len + 2 * P - 1) / (2 * P);
    p.n_items = a.B * a.Hkv * p.n_qb;
    p.halves = a.D / 64;
    p.scale_log2 = a.scale * kLog2e;
    p.qo_indptr = p.kv_indptr = p.kv_indices = p.kv_last = nullptr;
    p.k_pool = p.v_pool = nullptr;
    p.page_size = p.pool_rows = 0;
    p.gathered = 0;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    p.sec_bh = section_pairs(a, p.n_qb, p.n_items < sms ? p.n_items : sms);
    const SplitPlan pl = plan_schedule(a.B, a.Hkv, a.q_len, a.kv_len, P, p.n_qb, p.sec_bh, sms,
                                       a.ws != nullptr && a.ws_bytes >= prefill_tc_workspace_bytes(a, sms));
    p.sk_total = pl.total;
    p.sk_per_bh = pl.per_bh;
    p.sk_zero_qb = pl.zero_qb;
    p.sk_count = nullptr;
    p.sk_o = p.sk_ml = nullptr;
    const size_t smem = kSmemDense + 1024;
    if (pl.split) {
        uint8_t* w = static_cast<uint8_t*>(a.ws);
        p.sk_count = reinterpret_cast<int32_t*>(w);
        p.sk_o = reinterpret_cast<float*>(w + prefill_tc_counter_bytes(a));
        p.sk_ml = p.sk_o + static_cast<size_t>(2) * sms * 2 * kD * kBM;
        auto kern = p.halves == 1 ? prefill_tc_kernel<false, true, true> : prefill_tc_kernel<false, true>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        kern<<<pl.grid, kThreads, smem, stream>>>(q_map, k_map, v_map, o_map, p);
        return cudaGetLastError();
    }
    const int grid = p.n_items < sms ? p.n_items : sms;
    auto kern = p.halves == 1 ? prefill_tc_kernel<false, false, true> : prefill_tc_kernel<false, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>(q_map, k_map, v_map, o_map, p);
    return cudaGetLastError();
}

int varlen_max_seqs() { return kMaxVarlenSeqs; }

cudaError_t launch_prefill_varlen_tc(const VarlenArgs& a, cudaStream_t stream) {
    const int G = a.Hq / a.Hkv;
    const int P = kBM / G;
    CUtensorMap q_map, k_map, v_map;   // K/V maps only over the contiguous copy
    {
        // ragged Q [total_q, Hq, D]: box {64 dims, G heads, P positions} -> rows pos * G + head
        const uint64_t dims[3] = {kD, static_cast<uint64_t>(a.Hq), static_cast<uint64_t>(a.total_q)};
        const uint64_t strides[2] = {kD * 2, static_cast<uint64_t>(a.Hq) * kD * 2};
        const uint32_t box[3] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(P)};
        if (!encode_tiled_map(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    Params p;
    p.o = static_cast<__nv_bfloat16*>(a.o);
    p.lse = a.lse;
    p.status = a.dev_status;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.q_len = p.kv_len = 0;
    p.G = G;
    p.P = P;
    p.n_qb = 0;
    p.n_items = 0;   // counted on the device from qo_indptr
    p.halves = 2;
    p.sec_bh = 1;
    p.scale_log2 = a.scale * kLog2e;
    p.qo_indptr = a.qo_indptr;
    p.kv_indptr = a.kv_indptr;
    p.kv_indices = a.kv_indices;
    p.kv_last = a.kv_last_page_len;
    p.page_size = a.page_size;
    p.pool_rows = a.num_pages * a.page_size;
    p.k_pool = static_cast<const __nv_bfloat16*>(a.k_cache);
    p.v_pool = static_cast<const __nv_bfloat16*>(a.v_cache);
    p.gathered = a.kv_ws != nullptr;
    p.sk_total = p.sk_per_bh = 0;
    p.sk_zero_qb = 0;
    p.sk_count = nullptr;
    p.sk_o = p.sk_ml = nullptr;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    k_map = v_map = q_map;
    if (p.gathered) {
        // K copy [max_kv_rows, Hkv, D] then V copy, each viewed as the 2D
        // [Hkv * D, rows]: a tile half is the box {64, 128} at x = kvh * D + 64 h
        const size_t row_bytes = static_cast<size_t>(a.Hkv) * kD * 2;
        uint8_t* k_ws = static_cast<uint8_t*>(a.kv_ws);
        uint8_t* v_ws = k_ws + row_bytes * static_cast<size_t>(a.max_kv_rows);
        const uint64_t dims[2] = {static_cast<uint64_t>(a.Hkv) * kD, static_cast<uint64_t>(a.max_kv_rows)};
        const uint64_t strides[1] = {row_bytes};
        const uint32_t box[2] = {64, kBN};
        if (!encode_tiled_map(&k_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k_ws, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tiled_map(&v_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, v_ws, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        const int row_vecs = static_cast<int>(row_bytes / 16);
        gather_pages_kernel<<<sms * 8, 256, 0, stream>>>(
            static_cast<const uint4*>(a.k_cache), static_cast<const uint4*>(a.v_cache), a.kv_indptr, a.kv_indices,
            a.B, a.page_size, a.num_pages, row_vecs, reinterpret_cast<uint4*>(k_ws), reinterpret_cast<uint4*>(v_ws),
            a.max_kv_rows, a.dev_status);
        const cudaError_t ge = cudaGetLastError();
        if (ge != cudaSuccess) return ge;
    }
    const size_t smem = kSmemBytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<true, false><<<sms, kThreads, smem, stream>>>(q_map, k_map, v_map, q_map, p);
    return cudaGetLastError();
}

}  // namespace gb300
