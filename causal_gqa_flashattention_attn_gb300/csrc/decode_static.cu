// decode_static.cu - attn_decode_paged_splitk_static: the paged split-K decode
// for callers that cannot allocate device memory.
//
// Some callers of a decode step have no way to obtain scratch memory on the
// call path: plugin or callback interfaces that hand over only the input and
// output buffers, and serving loops that forbid cudaMalloc once they are
// running (an allocation can synchronise the device, and it can fail under
// memory pressure in the middle of a request).  This entry point needs no
// workspace from them: the split partials live in one fixed array of device
// memory that is part of the library image, reserved on every GPU that loads
// the library until the process exits.
//
// Host code cannot pass the array's name to a kernel (in host code it names a
// host-side stand-in, not device memory), so the device address is looked up
// with cudaGetSymbolAddress once per device, with that device current, on the
// first call made on that device.  That first call should therefore come
// before any stream capture.  The address is kept per device ordinal for the
// life of the process; a cudaDeviceReset (or a non-primary context) would
// leave it stale, and the entry point does not support either.  Nothing in the array has to start at zero: the
// decode kernel writes every partial (O_s and LSE_s, including empty splits)
// before the merge reads it.  Every call shares the one array and it keeps
// the last call's contents, so calls whose work overlaps on the GPU (on
// different streams, or from different host threads) race with each other.
#include <mutex>

#include "common.cuh"

// Largest split-partial area this entry point serves (32 MiB).
static constexpr size_t kStaticScratchBytes = ATTN_DECODE_STATIC_SCRATCH_BYTES;

// The split partials of attn_decode_paged_splitk_static (file scope, one per device).
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (nullptr on failure).
void* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

attn_status_t attn_decode_paged_splitk_static(const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* block_table, int max_pages_per_seq,
                                              const int32_t* seq_lens, attn_dtype_t kv_dtype, int n_groups, int B,
                                              int Hq, int Hkv, int D, int num_pages, int page_size,
                                              int split_tokens, int max_kv_len, float scale, void* o, float* lse,
                                              int32_t* dev_status, void* stream) {
    if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr || seq_lens == nullptr)
        return ATTN_ERR_INVALID_ARG;
    if (o == nullptr) return ATTN_ERR_INVALID_ARG;  // the partials stay private here, so O is required
    const size_t need = attn_decode_workspace_bytes(B, Hq, max_kv_len, split_tokens, D);
    if (need == 0) return ATTN_ERR_INVALID_ARG;
    if (need > kStaticScratchBytes) return ATTN_ERR_WORKSPACE;  // beyond the fixed maximum
    // The remaining checks are the ones of attn_decode_paged_splitk, which is
    // called with the fixed array as its workspace; it allocates nothing.
    void* scratch = scratch_on_current_device();
    if (scratch == nullptr) return ATTN_ERR_CUDA;
    return attn_decode_paged_splitk(q, k_cache, v_cache, block_table, max_pages_per_seq, seq_lens, kv_dtype,
                                    n_groups, B, Hq, Hkv, D, num_pages, page_size, split_tokens, max_kv_len, scale,
                                    scratch, kStaticScratchBytes, o, lse, dev_status, stream);
}

}  // extern "C"
