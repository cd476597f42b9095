// attn_api.cu - the C ABI declared in include/attn.h: argument validation,
// workspace accounting, TMA descriptor encoding and kernel dispatch.
//
// The errors the pages' Python wrappers raise become status codes: the
// Hq % Hkv assertion of "causal_forward_kernel.py" flash_attention_forward,
// the shape checks of "gpt-o3 / triton6fd1ef" run, and the static_asserts of
// "splitk_kernels.py" _fwd_kernel_splitK (N_GROUPS in {1, 2, 4, 8}).
#include <atomic>
#include <cudaTypedefs.h>

#include <cmath>
#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace gb300 {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
}  // namespace

bool encode_tiled_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle) {
    std::call_once(g_encode_once, load_encode);
    if (g_encode == nullptr) return false;
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    cuuint64_t d[5], s[4];
    cuuint32_t bx[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) s[i] = strides_bytes[i];
    const CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s, bx,
                                elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

std::atomic<int> g_cooperative{1};

bool cooperative_launch_enabled() { return g_cooperative.load(std::memory_order_relaxed) != 0; }

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices && g_sm_count[dev] > 0) return g_sm_count[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev] = n;
    return n;
}

}  // namespace gb300

using namespace gb300;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

attn_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

int split_count(int max_kv_len, int split_tokens) {
    const long long s = (static_cast<long long>(max_kv_len) + split_tokens - 1) / split_tokens;
    return s < 1 ? 1 : static_cast<int>(s);
}

size_t round16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

// Sizes, group and dtype checks of the dense prefill (pointers aside).
attn_status_t prefill_shape_check(attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len, int kv_len, int D,
                                  float scale) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || q_len <= 0 || kv_len <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * Hq * q_len >= (1LL << 31) || static_cast<long long>(B) * Hkv * kv_len >= (1LL << 31))
        return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

}  // namespace

namespace {

// Shared by the single- and multi-query decode entry points.
attn_status_t decode_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                          int max_pages_per_seq, const int32_t* seq_lens, attn_dtype_t kv_dtype, int n_groups, int B,
                          int Hq, int Hkv, int q_len, int D, int num_pages, int page_size, int split_tokens,
                          int max_kv_len, float scale, void* workspace, size_t workspace_bytes, void* o, float* lse,
                          int32_t* dev_status, void* stream, const void* k_scale_shift = nullptr,
                          const void* v_scale_shift = nullptr, bool fused = false) {
    if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr || seq_lens == nullptr)
        return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || num_pages <= 0 || page_size <= 0 || split_tokens <= 0 ||
        max_kv_len < 0 || max_pages_per_seq <= 0 || q_len <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || (o != nullptr && !aligned16(o)))
        return ATTN_ERR_INVALID_ARG;
    if (D != 128) return ATTN_ERR_UNSUPPORTED;
    const int G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return ATTN_ERR_UNSUPPORTED;
    if (q_len > 16) return ATTN_ERR_UNSUPPORTED;
    // the persistent int4 and fp8 kernels (int4 with N_GROUPS 4; Hkv a multiple
    // of 8, at most 8 rows per KV head) take splits in 32-token steps, the
    // others in 64-token steps
    const bool tile32 = ((kv_dtype == ATTN_INT4_PACKED && n_groups == 4) || kv_dtype == ATTN_FP8_E4M3) && D == 128 &&
                        Hkv % 8 == 0 && G * q_len <= 8;
    if (page_size % 64 != 0 || split_tokens % (tile32 ? 32 : 64) != 0) return ATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(num_pages) * page_size >= (1LL << 31)) return ATTN_ERR_UNSUPPORTED;
    int fmt = 0;
    if (kv_dtype == ATTN_BF16) {
        fmt = 0;
    } else if (kv_dtype == ATTN_INT4_PACKED) {
        fmt = 1;
        if (n_groups != 1 && n_groups != 2 && n_groups != 4 && n_groups != 8) return ATTN_ERR_UNSUPPORTED;
        if ((static_cast<long long>(Hkv) * (n_groups + D / 8)) % 4 != 0) return ATTN_ERR_UNSUPPORTED;
    } else if (kv_dtype == ATTN_FP8_E4M3) {
        fmt = 2;
        if (k_scale_shift == nullptr || v_scale_shift == nullptr) return ATTN_ERR_INVALID_ARG;
        if (!aligned16(k_scale_shift) || !aligned16(v_scale_shift)) return ATTN_ERR_INVALID_ARG;
        if (Hkv % 4 != 0) return ATTN_ERR_UNSUPPORTED;
    } else {
        return ATTN_ERR_UNSUPPORTED;
    }
    const int rows_q = Hq * q_len;   // output rows per sequence
    const size_t partial_bytes = attn_decode_workspace_bytes(B, rows_q, max_kv_len, split_tokens, D);
    const size_t need = fused ? attn_decode_fused_workspace_bytes(B, Hq, Hkv, q_len, max_kv_len, split_tokens, D)
                              : partial_bytes;
    if (need == 0) return ATTN_ERR_INVALID_ARG;
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
    if (fused && o == nullptr) return ATTN_ERR_INVALID_ARG;
    const int S = split_count(max_kv_len, split_tokens);
    const size_t rows = static_cast<size_t>(B) * rows_q;
    float* o_part = static_cast<float*>(workspace);
    float* lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + round16(rows * S * D * sizeof(float)));
    DecodeArgs a{q,         k_cache,   v_cache,      block_table, max_pages_per_seq, seq_lens, fmt, n_groups,
                 B,         Hq,        Hkv,          D,           num_pages,         page_size, split_tokens,
                 max_kv_len, S,        scale,        q_len,       o_part,            lse_part,  dev_status};
    if (fused) {
        a.counters = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + partial_bytes);
        a.o_final = o;
        a.lse_final = lse;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = (fmt == 2) ? launch_decode_fp8(a, k_scale_shift, v_scale_shift, s) : launch_decode(a, s);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    if (o != nullptr && !fused) e = launch_merge(o_part, lse_part, static_cast<int>(rows), S, D, o, lse, ATTN_BF16, s);
    return from_cuda(e);
}

}  // namespace

namespace {

attn_status_t varlen_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* qo_indptr,
                          const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* kv_last_page_len,
                          void* o, float* lse, int B, int Hq, int Hkv, int D, int total_q, int num_pages,
                          int page_size, float scale, int32_t* dev_status, void* stream, void* kv_ws,
                          int max_kv_rows) {
    if (q == nullptr || k_cache == nullptr || v_cache == nullptr || qo_indptr == nullptr || kv_indptr == nullptr ||
        kv_indices == nullptr || o == nullptr)
        return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || total_q < 0 || num_pages <= 0 || page_size <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    if (D != 128) return ATTN_ERR_UNSUPPORTED;
    const int G = Hq / Hkv;
    if (G > 128) return ATTN_ERR_UNSUPPORTED;
    if (B > varlen_max_seqs()) return ATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(num_pages) * page_size >= (1LL << 31) - 1) return ATTN_ERR_UNSUPPORTED;
    // work items (query blocks x KV heads) are counted in int and a query
    // block index is packed in 21 bits
    if (total_q >= (1 << 22) || (static_cast<long long>(total_q) + B) * Hkv >= (1LL << 31))
        return ATTN_ERR_UNSUPPORTED;
    if (total_q == 0) return ATTN_OK;
    VarlenArgs a{q,  k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, o,      lse,
                 B,  Hq,      Hkv,     D,         total_q,   num_pages,  page_size,        scale,  dev_status,
                 kv_ws, max_kv_rows};
    return from_cuda(launch_prefill_varlen_tc(a, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

const char* attn_status_string(attn_status_t status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_DEVICE_FAULT: return "device-side fault";
        default: return "unknown status";
    }
}

int attn_abi_version(void) { return 112; }

int attn_decode_cooperative(int enable) {
    if (enable < 0) return g_cooperative.load();
    return g_cooperative.exchange(enable != 0 ? 1 : 0);
}

attn_status_t attn_selftest_wait_timeout(int32_t* dev_status, unsigned int limit_us, void* stream) {
    if (dev_status == nullptr || limit_us == 0 || limit_us > 1000000u) return ATTN_ERR_INVALID_ARG;
    return from_cuda(launch_wait_timeout_selftest(dev_status, static_cast<uint64_t>(limit_us) * 1000u,
                                                  static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_prefill_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                               attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len, int kv_len, int D,
                               float scale, int32_t* dev_status, void* stream) {
    return attn_prefill_fwd_ws(q, k, v, o, lse, dtype, B, Hq, Hkv, q_len, kv_len, D, scale, nullptr, 0, dev_status,
                               stream);
}

size_t attn_prefill_workspace_bytes(attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len, int kv_len, int D) {
    if (prefill_shape_check(dtype, B, Hq, Hkv, q_len, kv_len, D, 1.f) != ATTN_OK) return 0;
    PrefillArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, static_cast<int>(dtype), B, Hq, Hkv, q_len, kv_len,
                  D, 1.f, nullptr, nullptr, 0};
    if (dtype != ATTN_BF16 || !prefill_tc_supported(a)) return 0;
    const int sms = device_sm_count();
    return sms > 0 ? prefill_tc_workspace_bytes(a, sms) : 0;
}

int attn_prefill_plan_sms(attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len, int kv_len, int D, int sms,
                          int* grid) {
    if (grid != nullptr) *grid = 0;
    if (sms <= 0 || prefill_shape_check(dtype, B, Hq, Hkv, q_len, kv_len, D, 1.f) != ATTN_OK) return -1;
    PrefillArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, static_cast<int>(dtype), B, Hq, Hkv, q_len, kv_len,
                  D, 1.f, nullptr, nullptr, 0};
    if (dtype != ATTN_BF16 || !prefill_tc_supported(a)) return 0;
    return prefill_tc_plan(a, sms, grid);
}

int attn_prefill_plan(attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len, int kv_len, int D, int* grid) {
    if (grid != nullptr) *grid = 0;
    if (prefill_shape_check(dtype, B, Hq, Hkv, q_len, kv_len, D, 1.f) != ATTN_OK) return -1;
    PrefillArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, static_cast<int>(dtype), B, Hq, Hkv, q_len, kv_len,
                  D, 1.f, nullptr, nullptr, 0};
    if (dtype != ATTN_BF16 || !prefill_tc_supported(a)) return 0;
    return attn_prefill_plan_sms(dtype, B, Hq, Hkv, q_len, kv_len, D, device_sm_count(), grid);
}

attn_status_t attn_prefill_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse,
                                  attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len, int kv_len, int D,
                                  float scale, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                  void* stream) {
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    const attn_status_t shape_ok = prefill_shape_check(dtype, B, Hq, Hkv, q_len, kv_len, D, scale);
    if (shape_ok != ATTN_OK) return shape_ok;
    if (workspace != nullptr) {
        if (!aligned16(workspace) ||
            workspace_bytes < attn_prefill_workspace_bytes(dtype, B, Hq, Hkv, q_len, kv_len, D))
            return ATTN_ERR_WORKSPACE;
    }
    PrefillArgs a{q, k, v, o, lse, static_cast<int>(dtype), B, Hq, Hkv, q_len, kv_len, D, scale, dev_status,
                  workspace, workspace_bytes};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == ATTN_BF16 && prefill_tc_supported(a)) return from_cuda(launch_prefill_tc(a, s));
    return from_cuda(launch_prefill_simt(a, s));
}

size_t attn_prefill_host_workspace_bytes(attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len, int kv_len,
                                         int D) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || q_len <= 0 || kv_len <= 0 || D <= 0) return 0;
    if (dtype != ATTN_F32 && dtype != ATTN_BF16) return 0;
    const size_t elem = dtype == ATTN_F32 ? 4 : 2;
    const size_t qb = static_cast<size_t>(B) * Hq * q_len * D * elem;
    const size_t kvb = static_cast<size_t>(B) * Hkv * kv_len * D * elem;
    const size_t lb = static_cast<size_t>(B) * Hq * q_len * sizeof(float);
    // Q, O, K, V, LSE, then the split-schedule scratch
    return 2 * round16(qb) + 2 * round16(kvb) + round16(lb) +
           attn_prefill_workspace_bytes(dtype, B, Hq, Hkv, q_len, kv_len, D);
}

attn_status_t attn_prefill_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                                    float* lse_host, attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len,
                                    int kv_len, int D, float scale, void* workspace, size_t workspace_bytes,
                                    int32_t* dev_status, void* stream) {
    if (q_host == nullptr || k_host == nullptr || v_host == nullptr || o_host == nullptr) return ATTN_ERR_INVALID_ARG;
    const attn_status_t shape_ok = prefill_shape_check(dtype, B, Hq, Hkv, q_len, kv_len, D, scale);
    if (shape_ok != ATTN_OK) return shape_ok;   // before anything is enqueued
    const size_t need = attn_prefill_host_workspace_bytes(dtype, B, Hq, Hkv, q_len, kv_len, D);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
    const size_t elem = dtype == ATTN_F32 ? 4 : 2;
    const size_t qb = static_cast<size_t>(B) * Hq * q_len * D * elem;
    const size_t kvb = static_cast<size_t>(B) * Hkv * kv_len * D * elem;
    const size_t lb = static_cast<size_t>(B) * Hq * q_len * sizeof(float);
    char* w = static_cast<char*>(workspace);
    void* dq = w;
    void* dout = w + round16(qb);
    void* dk = w + 2 * round16(qb);
    void* dv = w + 2 * round16(qb) + round16(kvb);
    float* dl = reinterpret_cast<float*>(w + 2 * round16(qb) + 2 * round16(kvb));
    char* split_ws = w + 2 * round16(qb) + 2 * round16(kvb) + round16(lb);
    const size_t split_bytes = attn_prefill_workspace_bytes(dtype, B, Hq, Hkv, q_len, kv_len, D);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // one copy per tensor, in, then the prefill, then one copy per result, out
    if (cudaMemcpyAsync(dq, q_host, qb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(dk, k_host, kvb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(dv, v_host, kvb, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (split_bytes > 0) {
        // this workspace is the caller's scratch: the split counters start at zero here
        PrefillArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, static_cast<int>(dtype), B, Hq, Hkv, q_len,
                      kv_len, D, scale, nullptr, nullptr, 0};
        if (cudaMemsetAsync(split_ws, 0, prefill_tc_counter_bytes(a), s) != cudaSuccess) return ATTN_ERR_CUDA;
    }
    const attn_status_t st = attn_prefill_fwd_ws(dq, dk, dv, dout, lse_host != nullptr ? dl : nullptr, dtype, B, Hq,
                                                 Hkv, q_len, kv_len, D, scale, split_bytes > 0 ? split_ws : nullptr,
                                                 split_bytes, dev_status, stream);
    if (st != ATTN_OK) return st;
    if (cudaMemcpyAsync(o_host, dout, qb, cudaMemcpyDeviceToHost, s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (lse_host != nullptr && cudaMemcpyAsync(lse_host, dl, lb, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

int attn_decode_split_tokens_for(int sms, int ctas_per_sm, int B, int Hq, int Hkv, int q_len, int max_kv_len) {
    if (sms <= 0 || ctas_per_sm <= 0 || B <= 0 || Hq <= 0 || Hkv <= 0 || q_len <= 0 || q_len > 16 || max_kv_len <= 0)
        return 0;
    if (Hq % Hkv != 0) return 0;
    const int G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return 0;
    // rows per CTA: the (query, head) pairs of a KV head, a power of two up to 16
    int R = 1;
    while (R < G * q_len && R < 16) R *= 2;
    const double slots = static_cast<double>(sms) * ctas_per_sm;
    const double units = static_cast<double>(B) * Hkv * ((G * q_len + R - 1) / R);
    // fewest splits whose CTAs fill at least one wave, the last one 90 % full
    const int tiles = (max_kv_len + 63) / 64;
    int best = 64 * tiles;
    double best_eff = -1.0;
    for (int n = 1; n <= tiles; ++n) {
        const int split = 64 * ((tiles + n - 1) / n);
        if ((max_kv_len + split - 1) / split != n) continue;   // this split gives fewer pieces
        const double waves = units * n / slots;
        const double eff = waves / std::ceil(waves);
        if (waves >= 1.0 && eff >= 0.9) return split;
        if (eff > best_eff) {
            best_eff = eff;
            best = split;
        }
    }
    return best;
}

int attn_decode_split_tokens_balanced_for(int sms, int B, int head_groups, int max_kv_len, int tile) {
    if (sms <= 0 || B <= 0 || head_groups <= 0 || max_kv_len <= 0 || (tile != 32 && tile != 64)) return 0;
    constexpr long long kUnitCost = 64;   // a unit's fixed cost, in tokens
    const int tiles = (max_kv_len + tile - 1) / tile;
    int best = 0;
    long long best_cost = -1;
    std::vector<long long> load;
    for (int split = tile * tiles; split >= tile; split -= tile) {
        const int S = (max_kv_len + split - 1) / split;
        const long long per_group = static_cast<long long>(B) * S;
        const long long units = per_group * head_groups;
        const int grid = units < sms ? static_cast<int>(units) : sms;
        // every CTA c takes units c, c + grid, ...: all of `split` tokens but the
        // last chunk of each sequence, which is max_kv_len - (S - 1) * split long
        load.assign(grid, 0);
        for (int c = 0; c < grid; ++c) load[c] = ((units - c + grid - 1) / grid) * (split + kUnitCost);
        const long long short_by = split - (max_kv_len - static_cast<long long>(S - 1) * split);
        if (short_by > 0)
            for (long long hg = 0; hg < head_groups; ++hg)
                for (long long b = 0; b < B; ++b) load[(hg * per_group + (S - 1) * static_cast<long long>(B) + b) % grid] -= short_by;
        const long long cost = *std::max_element(load.begin(), load.end());
        if (best_cost < 0 || cost < best_cost) {   // ties keep the larger split, found first
            best_cost = cost;
            best = split;
        }
    }
    return best;
}

int attn_decode_split_tokens(attn_dtype_t kv_dtype, int n_groups, int B, int Hq, int Hkv, int q_len, int max_kv_len,
                             int D) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || q_len <= 0 || q_len > 16 || max_kv_len <= 0 || D != 128) return 0;
    if (Hq % Hkv != 0) return 0;
    const int G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return 0;
    int fmt = 0;
    if (kv_dtype == ATTN_INT4_PACKED) {
        if (n_groups != 1 && n_groups != 2 && n_groups != 4 && n_groups != 8) return 0;
        fmt = 1;
    } else if (kv_dtype == ATTN_FP8_E4M3) {
        fmt = 2;
    } else if (kv_dtype != ATTN_BF16) {
        return 0;
    }
    DecodeArgs a{};
    a.kv_format = fmt;
    a.n_groups = n_groups;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.q_len = q_len;
    if ((fmt == 1 && decode_int4_g32_shape_ok(a)) || (fmt == 2 && decode_fp8_g32_shape_ok(a)))
        return attn_decode_split_tokens_balanced_for(device_sm_count(), B, Hkv / 8, max_kv_len, 32);
    int occ = 0;
    const cudaError_t e = (fmt == 2) ? launch_decode_fp8(a, nullptr, nullptr, nullptr, &occ)
                                     : launch_decode(a, nullptr, &occ);
    if (e != cudaSuccess) return 0;
    return attn_decode_split_tokens_for(device_sm_count(), occ, B, Hq, Hkv, q_len, max_kv_len);
}

size_t attn_decode_workspace_bytes(int B, int Hq, int max_kv_len, int split_tokens, int D) {
    if (B <= 0 || Hq <= 0 || max_kv_len < 0 || split_tokens <= 0 || D <= 0) return 0;
    const size_t S = static_cast<size_t>(split_count(max_kv_len, split_tokens));
    const size_t rows = static_cast<size_t>(B) * Hq;
    return round16(rows * S * D * sizeof(float)) + round16(rows * S * sizeof(float));
}

attn_status_t attn_decode_paged_splitk(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, int max_pages_per_seq,
                                       const int32_t* seq_lens, attn_dtype_t kv_dtype, int n_groups, int B,
                                       int Hq, int Hkv, int D, int num_pages, int page_size, int split_tokens,
                                       int max_kv_len, float scale, void* workspace, size_t workspace_bytes,
                                       void* o, float* lse, int32_t* dev_status, void* stream) {
    return decode_impl(q, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens, kv_dtype, n_groups, B, Hq,
                       Hkv, 1, D, num_pages, page_size, split_tokens, max_kv_len, scale, workspace, workspace_bytes,
                       o, lse, dev_status, stream);
}

attn_status_t attn_decode_paged_splitk_mq(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_table, int max_pages_per_seq,
                                          const int32_t* seq_lens, attn_dtype_t kv_dtype, int n_groups, int B,
                                          int Hq, int Hkv, int q_len, int D, int num_pages, int page_size,
                                          int split_tokens, int max_kv_len, float scale, void* workspace,
                                          size_t workspace_bytes, void* o, float* lse, int32_t* dev_status,
                                          void* stream) {
    return decode_impl(q, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens, kv_dtype, n_groups, B, Hq,
                       Hkv, q_len, D, num_pages, page_size, split_tokens, max_kv_len, scale, workspace,
                       workspace_bytes, o, lse, dev_status, stream);
}

attn_status_t attn_decode_paged_splitk_fp8(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* k_scale_shift, const int32_t* v_scale_shift,
                                           const int32_t* block_table, int max_pages_per_seq,
                                           const int32_t* seq_lens, int B, int Hq, int Hkv, int q_len, int D,
                                           int num_pages, int page_size, int split_tokens, int max_kv_len,
                                           float scale, void* workspace, size_t workspace_bytes, void* o,
                                           float* lse, int32_t* dev_status, void* stream) {
    return decode_impl(q, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens, ATTN_FP8_E4M3, 1, B, Hq, Hkv,
                       q_len, D, num_pages, page_size, split_tokens, max_kv_len, scale, workspace, workspace_bytes,
                       o, lse, dev_status, stream, k_scale_shift, v_scale_shift);
}

size_t attn_decode_fused_workspace_bytes(int B, int Hq, int Hkv, int q_len, int max_kv_len, int split_tokens,
                                         int D) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || q_len <= 0 || Hq % Hkv != 0) return 0;
    const size_t partials = attn_decode_workspace_bytes(B, Hq * q_len, max_kv_len, split_tokens, D);
    if (partials == 0) return 0;
    // the arrival counters, then the three words of the cooperative kernels' grid barrier
    return partials + round16((static_cast<size_t>(B) * Hkv + 3) * sizeof(int32_t));
}

attn_status_t attn_decode_paged_fused(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* k_scale_shift, const int32_t* v_scale_shift,
                                      const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                                      attn_dtype_t kv_dtype, int n_groups, int B, int Hq, int Hkv, int q_len, int D,
                                      int num_pages, int page_size, int split_tokens, int max_kv_len, float scale,
                                      void* workspace, size_t workspace_bytes, void* o, float* lse,
                                      int32_t* dev_status, void* stream) {
    return decode_impl(q, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens, kv_dtype, n_groups, B, Hq, Hkv,
                       q_len, D, num_pages, page_size, split_tokens, max_kv_len, scale, workspace, workspace_bytes, o,
                       lse, dev_status, stream, k_scale_shift, v_scale_shift, true);
}

attn_status_t attn_prefill_paged_varlen(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* qo_indptr, const int32_t* kv_indptr,
                                        const int32_t* kv_indices, const int32_t* kv_last_page_len, void* o,
                                        float* lse, int B, int Hq, int Hkv, int D, int total_q, int num_pages,
                                        int page_size, float scale, int32_t* dev_status, void* stream) {
    return varlen_impl(q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, o, lse, B, Hq, Hkv,
                       D, total_q, num_pages, page_size, scale, dev_status, stream, nullptr, 0);
}

size_t attn_prefill_varlen_workspace_bytes(int max_kv_rows, int Hkv, int D) {
    if (max_kv_rows <= 0 || Hkv <= 0 || D <= 0) return 0;
    return 2 * static_cast<size_t>(max_kv_rows) * Hkv * D * 2;
}

attn_status_t attn_prefill_paged_varlen_ws(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* qo_indptr, const int32_t* kv_indptr,
                                           const int32_t* kv_indices, const int32_t* kv_last_page_len, void* o,
                                           float* lse, int B, int Hq, int Hkv, int D, int total_q, int num_pages,
                                           int page_size, int max_kv_rows, float scale, void* workspace,
                                           size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (max_kv_rows <= 0) return ATTN_ERR_INVALID_ARG;
    if (Hkv > 0 && D > 0 && static_cast<long long>(max_kv_rows) * Hkv * D >= (1LL << 40)) return ATTN_ERR_UNSUPPORTED;
    const size_t need = attn_prefill_varlen_workspace_bytes(max_kv_rows, Hkv, D);
    if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    return varlen_impl(q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, o, lse, B, Hq, Hkv,
                       D, total_q, num_pages, page_size, scale, dev_status, stream, workspace, max_kv_rows);
}

attn_status_t attn_lse_merge(const float* o_part, const float* lse_part, int N, int S, int D, void* o, float* lse,
                             attn_dtype_t o_dtype, void* stream) {
    if (o_part == nullptr || lse_part == nullptr || o == nullptr) return ATTN_ERR_INVALID_ARG;
    if (N < 0 || S < 1 || D < 4 || D % 4 != 0) return ATTN_ERR_INVALID_ARG;
    if (D > 1024) return ATTN_ERR_UNSUPPORTED;
    if (o_dtype != ATTN_F32 && o_dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(o_part) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    return from_cuda(launch_merge(o_part, lse_part, N, S, D, o, lse, o_dtype, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_lse_merge_bwd(const float* o_part, const float* lse_part, const float* d_o, const float* d_lse,
                                 int N, int S, int D, float* d_o_part, float* d_lse_part, void* stream) {
    if (o_part == nullptr || lse_part == nullptr || d_o == nullptr || d_o_part == nullptr || d_lse_part == nullptr)
        return ATTN_ERR_INVALID_ARG;
    if (N < 0 || S < 1 || D < 4 || D % 4 != 0) return ATTN_ERR_INVALID_ARG;
    if (D > 1024) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(o_part) || !aligned16(d_o) || !aligned16(d_o_part)) return ATTN_ERR_INVALID_ARG;
    return from_cuda(launch_merge_bwd(o_part, lse_part, d_o, d_lse, N, S, D, d_o_part, d_lse_part,
                                      static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
