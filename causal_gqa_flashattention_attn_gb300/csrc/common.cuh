// common.cuh - host/device declarations shared by the kernels and the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/attn.h"

namespace gb300 {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Records a device-side error bit (never traps).
__device__ __forceinline__ void flag_status(int32_t* status, int32_t bit) {
    if (status != nullptr) atomicOr(status, bit);
}

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- host side

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).  Returns false on failure.
bool encode_tiled_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle);

int device_sm_count();
// Whether the fused decodes may use cooperative launches (attn_decode_cooperative).
bool cooperative_launch_enabled();

// Launchers (return a cudaError_t from the launch).
struct DecodeArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_table;
    int max_pages;
    const int32_t* seq_lens;
    int kv_format;   // 0 bf16, 1 int4
    int n_groups;
    int B, Hq, Hkv, D, num_pages, page_size, split_tokens, max_kv_len, n_split;
    float scale;
    int q_len;   // queries per sequence (causal multi-query decode when > 1)
    float* o_part;
    float* lse_part;
    int32_t* dev_status;
    // fused mode (counters not NULL): the last split of each (sequence, KV head)
    // merges its partials into o_final / lse_final inside the launch
    int32_t* counters;   // [B * Hkv], zero when the launch starts
    void* o_final;       // bf16 [B, Hq, q_len, D]
    float* lse_final;    // [B, Hq, q_len] or NULL
};
// With `occ` set, a decode launcher launches nothing: it writes how many CTAs
// of the kernel it would launch fit on one SM at once.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream, int* occ = nullptr);
cudaError_t launch_decode_int4(const DecodeArgs& a, cudaStream_t stream, int* occ = nullptr);
// int4 rows of four 32-element groups and at most 8 (query, head) rows per KV
// head: the fp16-subnormal code-space kernel of decode_int4_g32.cu.
bool decode_int4_g32_shape_ok(const DecodeArgs& a);   // shape only (no page or split size)
bool decode_int4_g32_supported(const DecodeArgs& a);
cudaError_t launch_decode_int4_g32(const DecodeArgs& a, cudaStream_t stream, int* occ = nullptr);
// fp8 rows, KV head counts that are multiples of 8 and at most 8 (query, head)
// rows per KV head: the persistent kernel of decode_fp8_g32.cu.
bool decode_fp8_g32_shape_ok(const DecodeArgs& a);   // shape only (no page or split size)
bool decode_fp8_g32_supported(const DecodeArgs& a);
cudaError_t launch_decode_fp8_g32(const DecodeArgs& a, const void* k_scale_shift, const void* v_scale_shift,
                                  cudaStream_t stream, int* occ = nullptr);
cudaError_t launch_decode_fp8(const DecodeArgs& a, const void* k_scale_shift, const void* v_scale_shift,
                              cudaStream_t stream, int* occ = nullptr);
int rows_per_cta(const DecodeArgs& a);

// CTAs of `kern` (with its shared-memory attributes set as for a launch)
// resident on one SM at once.
template <typename K>
cudaError_t ctas_per_sm(K kern, int threads, size_t smem, int* occ) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    return e == cudaSuccess ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, kern, threads, smem) : e;
}

cudaError_t launch_wait_timeout_selftest(int32_t* status, uint64_t limit_ns, cudaStream_t stream);

cudaError_t launch_merge(const float* o_part, const float* lse_part, int N, int S, int D, void* o,
                         float* lse, int o_dtype, cudaStream_t stream);
cudaError_t launch_merge_bwd(const float* o_part, const float* lse_part, const float* d_o, const float* d_lse, int N,
                             int S, int D, float* d_o_part, float* d_lse_part, cudaStream_t stream);

struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    int dtype;  // ATTN_F32 / ATTN_BF16
    int B, Hq, Hkv, q_len, kv_len, D;
    float scale;
    int32_t* dev_status;
    void* ws;          // split-schedule scratch (NULL: whole items only)
    size_t ws_bytes;
};
cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream);
bool prefill_tc_supported(const PrefillArgs& a);
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream);
// Scratch of the split schedule on a device with `sms` SMs, and the leading
// part of it (the counters) that must be zero when a launch starts.
size_t prefill_tc_workspace_bytes(const PrefillArgs& a, int sms);
size_t prefill_tc_counter_bytes(const PrefillArgs& a);
// 1 if a launch with a workspace takes the split schedule, else 0; *grid = its CTAs.
int prefill_tc_plan(const PrefillArgs& a, int sms, int* grid);

struct VarlenArgs {
    const void* q;          // [total_q, Hq, D] bf16
    const void* k_cache;    // [num_pages, page_size, Hkv, D] bf16
    const void* v_cache;
    const int32_t* qo_indptr;
    const int32_t* kv_indptr;
    const int32_t* kv_indices;
    const int32_t* kv_last_page_len;   // may be NULL
    void* o;                // [total_q, Hq, D] bf16
    float* lse;             // [total_q, Hq]
    int B, Hq, Hkv, D, total_q, num_pages, page_size;
    float scale;
    int32_t* dev_status;
    void* kv_ws;            // NULL: gather rows inside the kernel; else contiguous K then V copy
    int max_kv_rows;        // rows the copy holds (>= kv_indptr[B] * page_size)
};
int varlen_max_seqs();
cudaError_t launch_prefill_varlen_tc(const VarlenArgs& a, cudaStream_t stream);

}  // namespace gb300
