/*
 * attn.h - C ABI of the GB300 (sm_103a) causal grouped-query attention library.
 *
 * What the library computes (the pages it follows are named per entry point):
 *   O = softmax(scale * Q K^T + causal mask) V, plus the per-row natural-log
 *   log-sum-exp LSE = log(sum_j exp(scale * q_i . k_j)) over the visible keys.
 * Query head h reads key/value head h / (Hq / Hkv) (grouped-query attention).
 * Causal alignment is bottom-right: with delta = kv_len - q_len, key j is
 * visible to query i iff j <= i + delta.  A query row with no visible key gets
 * O = 0 and LSE = -inf.
 *
 * Conventions shared by every entry point:
 *   - All tensor arguments are DEVICE pointers to dense, contiguous,
 *     row-major buffers that the CALLER allocates and owns; the library never
 *     allocates, frees or synchronises.  Pointers must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL means the legacy default stream).  A returned ATTN_OK means the
 *     work was validated and enqueued, not that it has finished.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and returned as ATTN_ERR_INVALID_ARG / ATTN_ERR_UNSUPPORTED /
 *     ATTN_ERR_WORKSPACE; a failed launch returns ATTN_ERR_CUDA.
 *   - Errors only the device can see (a block-table entry outside the page
 *     pool, a sequence longer than its block table, a bounded wait that ran
 *     out) are OR-ed as ATTN_DEV_* bits into the optional int32 device word
 *     `dev_status` (may be NULL).  The kernel skips the offending access and
 *     never traps; the caller reads the word after synchronising.
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = -1,   /* null pointer, non-positive size, Hq % Hkv != 0, ... */
    ATTN_ERR_UNSUPPORTED = -2,   /* valid but not implemented (head dim, dtype, group count) */
    ATTN_ERR_WORKSPACE = -3,     /* workspace missing or smaller than attn_decode_workspace_bytes */
    ATTN_ERR_CUDA = -4,          /* a CUDA runtime/driver call or a launch failed */
    ATTN_ERR_DEVICE_FAULT = -5   /* reserved for callers that translate dev_status */
} attn_status_t;

typedef enum {
    ATTN_F32 = 0,
    ATTN_BF16 = 1,
    ATTN_F16 = 2,
    ATTN_INT4_PACKED = 3,        /* int32 words, see attn_decode_paged_splitk */
    ATTN_FP8_E4M3 = 4            /* e4m3 bytes + a scale/shift word per row, see attn_decode_paged_splitk_fp8 */
} attn_dtype_t;

/* Bits OR-ed into *dev_status by a kernel. */
#define ATTN_DEV_PAGE_OUT_OF_RANGE 0x1  /* block_table entry < 0 or >= num_pages */
#define ATTN_DEV_SEQ_TOO_LONG      0x2  /* seq_lens[b] > max_kv_len or > max_pages_per_seq * page_size */
#define ATTN_DEV_WAIT_TIMEOUT      0x4  /* a bounded mbarrier wait gave up */
#define ATTN_DEV_WORKSPACE_STATE   0x8  /* attn_prefill_fwd_ws: the split counters were not zero */

/*
 * attn_prefill_fwd - causal GQA prefill.
 *
 * Follows "causal_forward_kernel.py" (flash-attention-scratch),
 * _flash_attention_forward_gqa_kernel and its wrapper flash_attention_forward
 * (tiled online-softmax forward, GQA head map, O in the input dtype, an LSE
 * row per query), with the bottom-right alignment of "gpt-o3 / triton6fd1ef",
 * _gqa_prefill_kernel: query i sees the first i + 1 + delta keys, at most
 * kv_len of them, delta = kv_len - q_len.
 *
 *   q    [B, Hq,  q_len,  D]  dtype            (read)
 *   k    [B, Hkv, kv_len, D]  dtype            (read)
 *   v    [B, Hkv, kv_len, D]  dtype            (read)
 *   o    [B, Hq,  q_len,  D]  dtype            (written)
 *   lse  [B, Hq,  q_len]      float32, natural log (written; may be NULL)
 *   dtype   ATTN_BF16 (tensor-core path for Hq/Hkv <= 128, larger groups use
 *           the CUDA-core path) or ATTN_F32 (exact fp32 CUDA-core path, no
 *           TF32).
 *   D       64 or 128.
 *   scale   softmax scale; pass 1/sqrt(D) for the usual attention.
 *   Requires Hq % Hkv == 0, all sizes > 0.
 */
attn_status_t attn_prefill_fwd(const void* q, const void* k, const void* v,
                               void* o, float* lse, attn_dtype_t dtype,
                               int B, int Hq, int Hkv, int q_len, int kv_len, int D,
                               float scale, int32_t* dev_status, void* stream);

/*
 * attn_prefill_fwd_ws - attn_prefill_fwd with scratch for a split schedule.
 *
 * Same operation, arguments and results as attn_prefill_fwd.  With a
 * workspace, the bf16 tensor-core path may cut the KV range of a query block
 * between CTAs when there are too few blocks to keep every SM busy to the
 * end (few heads, short prompts).  Each piece keeps its own unnormalised O,
 * running max m and sum l; the piece that finishes last combines them,
 * O = sum_i 2^(m_i - M) O_i / sum_i 2^(m_i - M) l_i with M = max_i m_i, the
 * LSE-weighted combination of "splitk_kernels.py", _splitK_reduce.  The host
 * picks the schedule from the sizes alone; results agree with
 * attn_prefill_fwd within rounding, not bit for bit.
 *
 *   workspace        device, 16-byte aligned, at least
 *                    attn_prefill_workspace_bytes() bytes, or NULL (the
 *                    whole-item schedule of attn_prefill_fwd).  Its first
 *                    bytes are counters that must be zero when a call starts:
 *                    zero the workspace once; every call that completes
 *                    without a device error leaves them zero again, so
 *                    consecutive calls on one stream can share it.  After a
 *                    device error (dev_status != 0) zero it again.  Calls
 *                    that may run at the same time need separate workspaces.
 *                    A counter found past its range sets
 *                    ATTN_DEV_WORKSPACE_STATE (the results are then not valid).
 *   workspace_bytes  its size.
 * Errors as attn_prefill_fwd; ATTN_ERR_WORKSPACE for a misaligned or short
 * workspace.
 */
size_t attn_prefill_workspace_bytes(attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len, int kv_len, int D);
/* The schedule attn_prefill_fwd_ws takes on the current device: 1 split,
 * 0 whole items (always 0 for the CUDA-core paths), -1 for invalid sizes or
 * no device.  If grid is not NULL, *grid = the CTAs of the tensor-core launch
 * (0 for the CUDA-core paths and on error). */
int attn_prefill_plan(attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len, int kv_len, int D, int* grid);
/* The same for a device with `sms` SMs (nothing is asked of the driver), for
 * planning ahead; -1 also for sms <= 0. */
int attn_prefill_plan_sms(attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len, int kv_len, int D, int sms,
                          int* grid);
attn_status_t attn_prefill_fwd_ws(const void* q, const void* k, const void* v,
                                  void* o, float* lse, attn_dtype_t dtype,
                                  int B, int Hq, int Hkv, int q_len, int kv_len, int D,
                                  float scale, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, void* stream);

/*
 * attn_prefill_fwd_host - attn_prefill_fwd on host buffers.
 *
 * Enqueues on `stream`: one host -> device copy each of q, k and v into
 * `workspace`, the prefill of attn_prefill_fwd, and one device -> host copy
 * each of O and (if lse_host is not NULL) LSE.  Returns once enqueued; the
 * results are in o_host / lse_host when the stream has reached this work, and
 * the host buffers must not be reused before then.  Page-locked host memory
 * (cudaHostAlloc / cudaHostRegister) lets the copies run asynchronously and
 * overlap work on other streams; with pageable memory they stall the host.
 *
 *   q_host, k_host, v_host, o_host, lse_host  host memory, shapes and dtype
 *                as the device buffers of attn_prefill_fwd
 *   workspace    device, 16-byte aligned, attn_prefill_host_workspace_bytes()
 *                bytes (the device copies of Q, O, K, V and LSE, then the
 *                scratch of attn_prefill_fwd_ws, whose counters this call
 *                zeroes on the stream first; overwritten)
 * Other arguments and errors as attn_prefill_fwd; ATTN_ERR_WORKSPACE for a
 * missing, misaligned or short workspace; ATTN_ERR_CUDA if a copy cannot be
 * enqueued.
 */
size_t attn_prefill_host_workspace_bytes(attn_dtype_t dtype, int B, int Hq, int Hkv, int q_len, int kv_len,
                                         int D);
attn_status_t attn_prefill_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                                    void* o_host, float* lse_host, attn_dtype_t dtype,
                                    int B, int Hq, int Hkv, int q_len, int kv_len, int D, float scale,
                                    void* workspace, size_t workspace_bytes,
                                    int32_t* dev_status, void* stream);

/*
 * attn_decode_workspace_bytes - bytes of scratch attn_decode_paged_splitk needs.
 *
 * The workspace holds the split partials of "splitk_kernels.py",
 * _fwd_kernel_splitK (Out_splitK / LSE_splitk), laid out as
 *   o_part   float32 [B, Hq, S, D]   at offset 0
 *   lse_part float32 [B, Hq, S]      right after o_part (16-byte aligned)
 * with S = ceil(max_kv_len / split_tokens) (at least 1).  Returns 0 for
 * invalid sizes.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int max_kv_len, int split_tokens, int D);

/*
 * attn_decode_split_tokens - a split size for the paged decode entries that
 * fills the current device.
 *
 * "splitk_kernels.py", _fwd_kernel_splitK cuts every sequence's keys into
 * chunks of split_tokens, one program each.  Here each (chunk, KV head,
 * sequence) is one CTA.  This returns the split_tokens (a multiple of 64) that
 * gives the fewest chunks per sequence while the CTAs, at the number of them
 * that fit on the device at once, come to at least one wave with the last
 * wave at least 90 % full (else the fullest last wave found).  It counts every
 * sequence at max_kv_len, so it suits batches of similar lengths.
 *
 *   kv_dtype   ATTN_BF16, ATTN_INT4_PACKED (with n_groups) or ATTN_FP8_E4M3
 * The int4 decode with N_GROUPS 4, Hkv a multiple of 8 and G * q_len <= 8
 * runs one persistent CTA per SM over work units (sequence, chunk, group of 8
 * KV heads); for it the choice is attn_decode_split_tokens_balanced_for with
 * 32-token steps (so the returned split may be a multiple of 32 only).
 * Returns 0 for sizes the decode entries do not take, or without a device.
 */
int attn_decode_split_tokens(attn_dtype_t kv_dtype, int n_groups, int B, int Hq, int Hkv, int q_len, int max_kv_len,
                             int D);
/* The same choice for `sms` SMs holding ctas_per_sm decode CTAs each
 * (nothing is asked of the driver); 0 for sizes the decode entries do not take
 * or a non-positive device description. */
int attn_decode_split_tokens_for(int sms, int ctas_per_sm, int B, int Hq, int Hkv, int q_len, int max_kv_len);
/* The split for a persistent decode whose `sms` CTAs walk the work units
 * (head group, chunk, sequence) round-robin, B sequences and head_groups groups
 * of KV heads, every sequence counted at max_kv_len: the multiple of `tile`
 * (32 or 64) that minimises the largest per-CTA sum of unit tokens, each unit
 * counted 64 tokens longer for its fixed cost; ties go to the larger split.
 * 0 for non-positive sizes or another tile. */
int attn_decode_split_tokens_balanced_for(int sms, int B, int head_groups, int max_kv_len, int tile);

/*
 * attn_prefill_paged_varlen - causal GQA prefill of a ragged batch over a
 * paged KV cache, in one launch.
 *
 * Follows "gpt-o3 / triton6fd1ef", run and _gqa_prefill_kernel: CSR
 * qo_indptr / kv_indptr / kv_indices, kv_head = q_head / (Hq / Hkv), and per
 * sequence bottom-right causal alignment (delta = kv_len - q_len).  The
 * sequences' extents are read on the device; nothing is synchronised.
 *
 *   q            [total_q, Hq, D] bfloat16; sequence b owns rows
 *                [qo_indptr[b], qo_indptr[b+1])                      (read)
 *   k_cache,
 *   v_cache      bfloat16 [num_pages, page_size, Hkv, D] (any page_size >= 1) (read)
 *   qo_indptr    int32 [B+1]; kv_indptr int32 [B+1], in pages;
 *   kv_indices   int32 [kv_indptr[B]], the pool page of each listed page;
 *   kv_last_page_len  int32 [B], tokens in each sequence's last page
 *                (NULL: every page full); kv_len_b = (pages_b - 1) *
 *                page_size + last_b                                  (read, device)
 *   o            [total_q, Hq, D] bfloat16; lse [total_q, Hq] fp32 (written; lse may be NULL)
 *   D = 128, Hq / Hkv <= 128, B <= 2048, total_q < 2^22 and
 *   (total_q + B) * Hkv < 2^31 (ATTN_ERR_UNSUPPORTED otherwise).
 * A page id outside [0, num_pages) sets ATTN_DEV_PAGE_OUT_OF_RANGE and is
 * read as zeros.
 */
attn_status_t attn_prefill_paged_varlen(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* qo_indptr, const int32_t* kv_indptr,
                                        const int32_t* kv_indices, const int32_t* kv_last_page_len,
                                        void* o, float* lse, int B, int Hq, int Hkv, int D, int total_q,
                                        int num_pages, int page_size, float scale,
                                        int32_t* dev_status, void* stream);

/*
 * attn_prefill_paged_varlen_ws - attn_prefill_paged_varlen with a workspace:
 * the K and V rows of every listed page are first copied into contiguous
 * buffers in page-list order (token t of sequence b is row
 * kv_indptr[b] * page_size + t), then read by TMA tiles as in the dense
 * prefill.  Same results; faster when pages are small (the in-kernel gather
 * of attn_prefill_paged_varlen cannot hide the latency of page-size-1 rows).
 *
 *   max_kv_rows  rows the workspace holds: at least kv_indptr[B] * page_size
 *                (a longer list sets ATTN_DEV_SEQ_TOO_LONG and is cut)
 *   workspace    device, 16-byte aligned, attn_prefill_varlen_workspace_bytes()
 *                bytes: the K copy [max_kv_rows, Hkv, D] bf16, then the V copy
 *                (scratch, overwritten)
 * Other arguments, limits and errors as attn_prefill_paged_varlen;
 * ATTN_ERR_WORKSPACE for a missing, misaligned or short workspace.
 */
size_t attn_prefill_varlen_workspace_bytes(int max_kv_rows, int Hkv, int D);
attn_status_t attn_prefill_paged_varlen_ws(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* qo_indptr, const int32_t* kv_indptr,
                                           const int32_t* kv_indices, const int32_t* kv_last_page_len,
                                           void* o, float* lse, int B, int Hq, int Hkv, int D, int total_q,
                                           int num_pages, int page_size, int max_kv_rows, float scale,
                                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                           void* stream);

/*
 * attn_decode_paged_splitk - single-query split-K decode over a paged KV cache.
 *
 * Follows "splitk_kernels.py" (xformers), _fwd_kernel_splitK (split chunks,
 * block-table indirection, per-split O already divided by its own l, natural
 * LSE, empty split -> O = 0 / LSE = -inf) and load_dequantize_k_v_group /
 * cast_uint32_to_half2 / dequantize (int4 rows); then _splitK_reduce merges.
 *
 *   q            [B, Hq, D] bfloat16 (one query per sequence)      (read)
 *   k_cache,
 *   v_cache      page pool, token-major inside a page:
 *                  ATTN_BF16:        bfloat16 [num_pages, page_size, Hkv, D]
 *                  ATTN_INT4_PACKED: int32    [num_pages, page_size, Hkv, n_groups + D/8]
 *                int4 row: n_groups coefficient words (fp16 scale in the low
 *                16 bits, fp16 offset in the high 16 bits), then D/8 code
 *                words group by group; nibble j (bits 4j..4j+3) of word w of
 *                a group is element 8w+j of that group; value =
 *                scale * code + offset.                            (read)
 *   block_table  int32 [B, max_pages_per_seq]; entry p of sequence b is the
 *                pool page holding its tokens [p*page_size, (p+1)*page_size).
 *                Entries past the sequence's last page are never read.  (read)
 *   seq_lens     int32 [B], 0 <= seq_lens[b] <= max_kv_len  (device)  (read)
 *   n_groups     1, 2, 4 or 8 for ATTN_INT4_PACKED; ignored for ATTN_BF16.
 *   D            128.  Hq / Hkv in {1, 2, 4, 8, 16}.
 *   page_size    a multiple of 64.  split_tokens: a multiple of 64, or of 32
 *                for an int4 cache with n_groups 4, Hkv a multiple of 8 and
 *                Hq / Hkv * q_len <= 8 (the persistent int4 kernel).
 *   workspace    >= attn_decode_workspace_bytes(B, Hq, max_kv_len, split_tokens, D)
 *                bytes of device memory owned by the caller; it receives the
 *                split partials in the layout documented above.
 *   o            [B, Hq, D] bfloat16 (written), lse [B, Hq] float32 (written,
 *                may be NULL).  If o is NULL only the partials are produced
 *                (for callers that merge across devices themselves).
 * Split s of sequence b covers tokens [s*split_tokens, min((s+1)*split_tokens, len_b)).
 * A block-table entry outside [0, num_pages) sets ATTN_DEV_PAGE_OUT_OF_RANGE;
 * that page is not read and its tokens are left out of their split (as if
 * masked), so the outputs stay defined: the decode of the sequence without
 * that page.  This holds for every decode entry (mq, fp8, static as well).
 */
attn_status_t attn_decode_paged_splitk(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, int max_pages_per_seq,
                                       const int32_t* seq_lens, attn_dtype_t kv_dtype, int n_groups,
                                       int B, int Hq, int Hkv, int D, int num_pages, int page_size,
                                       int split_tokens, int max_kv_len, float scale,
                                       void* workspace, size_t workspace_bytes,
                                       void* o, float* lse, int32_t* dev_status, void* stream);

/*
 * attn_decode_paged_splitk_mq - causal multi-query split-K decode.
 *
 * Follows "splitk_kernels.py", _fwd_kernel_splitK with IS_CAUSAL and
 * NUM_QUERIES_CAUSAL (the kernel's own explanation of its causal mask): the
 * q_len queries of a sequence are its last q_len
 * positions, so query i (0-based) sees cached tokens t <= len_b - q_len + i
 * (bottom-right alignment).  A split in which a query sees nothing yields
 * O_s = 0, LSE_s = -inf for that query.  Used for speculative decoding.
 *
 * Arguments as attn_decode_paged_splitk, except:
 *   q       [B, Hq, q_len, D] bfloat16;   1 <= q_len <= 16
 *   o       [B, Hq, q_len, D] bfloat16 (or NULL: partials only);  lse [B, Hq, q_len] fp32
 *   workspace >= attn_decode_workspace_bytes(B, Hq * q_len, max_kv_len, split_tokens, D);
 *           it receives o_part [B, Hq, q_len, S, D] and lse_part [B, Hq, q_len, S].
 * With q_len = 1 this is exactly attn_decode_paged_splitk.
 */
attn_status_t attn_decode_paged_splitk_mq(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_table, int max_pages_per_seq,
                                          const int32_t* seq_lens, attn_dtype_t kv_dtype, int n_groups,
                                          int B, int Hq, int Hkv, int q_len, int D, int num_pages,
                                          int page_size, int split_tokens, int max_kv_len, float scale,
                                          void* workspace, size_t workspace_bytes,
                                          void* o, float* lse, int32_t* dev_status, void* stream);

/*
 * attn_decode_paged_splitk_fp8 - split-K decode over an fp8 (e4m3) row-wise
 * quantised paged KV cache, single- or multi-query.
 *
 * Follows "splitk_kernels.py", _fwd_kernel_splitK with FP8_QUANTIZED (row-wise
 * only), the K_fp8_scale_shift / V_fp8_scale_shift tensors,
 * cast_uint32_to_half2 and dequantize: value = e4m3(byte) * scale + shift.
 *
 *   k_cache, v_cache          uint8 [num_pages, page_size, Hkv, D], e4m3 bytes
 *   k_scale_shift, v_scale_shift
 *                             int32 [num_pages, page_size, Hkv]: fp16 scale in
 *                             the low 16 bits, fp16 shift in the high 16 bits
 *   q                         [B, Hq, q_len, D] bfloat16, 1 <= q_len <= 16
 *                             (converted to fp16 on chip: |q| < 65504)
 *   Hkv                       a multiple of 4.
 * Every other argument, the workspace and the causal rule for q_len > 1 are
 * those of attn_decode_paged_splitk_mq; o [B, Hq, q_len, D] bfloat16.
 */
attn_status_t attn_decode_paged_splitk_fp8(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* k_scale_shift, const int32_t* v_scale_shift,
                                           const int32_t* block_table, int max_pages_per_seq,
                                           const int32_t* seq_lens, int B, int Hq, int Hkv, int q_len, int D,
                                           int num_pages, int page_size, int split_tokens, int max_kv_len,
                                           float scale, void* workspace, size_t workspace_bytes,
                                           void* o, float* lse, int32_t* dev_status, void* stream);

/*
 * attn_decode_paged_fused - the paged split-K decode with the LSE merge
 * inside the same launch.
 *
 * Computes what attn_decode_paged_splitk (q_len == 1), attn_decode_paged_splitk_mq
 * (q_len > 1) or attn_decode_paged_splitk_fp8 computes, and then merges: the
 * split of each (sequence, KV head) that finishes last reads that head's
 * partials and writes its O and LSE ("splitk_kernels.py", _splitK_reduce:
 * M = max_s LSE_s, w_s = exp(LSE_s - M), O = sum_s w_s O_s / sum_s w_s,
 * LSE = M + log sum_s w_s; O = 0 and LSE = -inf when every LSE_s is -inf).
 * No CTA waits for another: arrival is counted, and the last arrival merges.
 * The persistent int4 and fp8 kernels (KV head counts that are multiples of 8,
 * at most 8 rows per KV head) are launched cooperatively instead, every CTA
 * resident at once: after its last split each CTA meets the others at one
 * grid barrier (a bounded wait; ATTN_DEV_WAIT_TIMEOUT if it runs out), and then
 * every warp of the grid merges a share of the rows.  If the device refuses
 * the cooperative launch, they fall back to the last-arrival merge.
 *
 *   kv_dtype       ATTN_BF16, ATTN_INT4_PACKED (with n_groups) or
 *                  ATTN_FP8_E4M3 (with k_scale_shift / v_scale_shift, as for
 *                  attn_decode_paged_splitk_fp8; NULL otherwise)
 *   q              [B, Hq, q_len, D] bfloat16 (query i of a sequence sees
 *                  tokens t <= len - q_len + i)                       (read)
 *   workspace      >= attn_decode_fused_workspace_bytes(...) bytes: the split
 *                  partials (layout as for attn_decode_paged_splitk with
 *                  Hq * q_len rows per sequence), then one int32 arrival
 *                  counter per (sequence, KV head) and three int32 words of
 *                  the grid barrier.  The counters and words must be 0 when a
 *                  call starts: zero the workspace once; every call that
 *                  completes without a device error leaves them 0 again (so a
 *                  replayed CUDA graph needs no re-zeroing).  A
 *                  counter found past its range sets ATTN_DEV_WORKSPACE_STATE.
 *                  Calls that share a workspace must not overlap on the GPU.
 *   o              [B, Hq, q_len, D] bfloat16 (written, required); lse
 *                  [B, Hq, q_len] fp32 (written, may be NULL)
 * Other arguments, limits and errors as the entries named above.
 *
 * attn_decode_cooperative - whether attn_decode_paged_fused may use
 * cooperative launches (process-wide, default on).  enable = 1 allows them,
 * 0 makes every fused decode use the last-arrival merge (for callers whose
 * device or sharing mode refuses cooperative launches, or to compare the
 * two), -1 only reads the setting.  Returns the setting before the call.
 */
size_t attn_decode_fused_workspace_bytes(int B, int Hq, int Hkv, int q_len, int max_kv_len, int split_tokens,
                                         int D);
attn_status_t attn_decode_paged_fused(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* k_scale_shift, const int32_t* v_scale_shift,
                                      const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                                      attn_dtype_t kv_dtype, int n_groups, int B, int Hq, int Hkv, int q_len, int D,
                                      int num_pages, int page_size, int split_tokens, int max_kv_len, float scale,
                                      void* workspace, size_t workspace_bytes, void* o, float* lse,
                                      int32_t* dev_status, void* stream);
int attn_decode_cooperative(int enable);

/*
 * attn_decode_paged_splitk_static - attn_decode_paged_splitk without a workspace.
 *
 * The pages have no counterpart of this entry point.  It serves callers that
 * cannot allocate device memory on the call path: plugin or callback
 * interfaces that hand over only input and output buffers, and serving loops
 * that forbid cudaMalloc once running (an allocation can synchronise the
 * device and can fail under memory pressure mid-request).  It computes
 * exactly what attn_decode_paged_splitk computes, with the same arguments
 * minus the workspace, and allocates nothing: the split partials go to one
 * fixed array of ATTN_DECODE_STATIC_SCRATCH_BYTES bytes of device memory that
 * belongs to the library image and stays reserved on every GPU that loads the
 * library until the process exits.
 *
 *   - o is required (the partials are not visible to the caller); lse may be NULL.
 *   - Returns ATTN_ERR_WORKSPACE when
 *     attn_decode_workspace_bytes(B, Hq, max_kv_len, split_tokens, D) exceeds
 *     ATTN_DECODE_STATIC_SCRATCH_BYTES; all other checks and errors are those
 *     of attn_decode_paged_splitk.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  ATTN_ERR_CUDA if the lookup fails.  The
 *     address is kept per device ordinal for the life of the process, so the
 *     entry point is not for use across a cudaDeviceReset (or with a context
 *     other than the device's primary context current): the kept address
 *     would then be stale.
 *   - All calls share the one array, which keeps the last call's contents
 *     (nothing in it needs to start at zero: every partial is written before
 *     it is read).  Calls whose work overlaps on the GPU (different streams or
 *     host threads) race with each other and must be serialised by the caller.
 */
#define ATTN_DECODE_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

attn_status_t attn_decode_paged_splitk_static(const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* block_table, int max_pages_per_seq,
                                              const int32_t* seq_lens, attn_dtype_t kv_dtype, int n_groups,
                                              int B, int Hq, int Hkv, int D, int num_pages, int page_size,
                                              int split_tokens, int max_kv_len, float scale,
                                              void* o, float* lse, int32_t* dev_status, void* stream);

/*
 * attn_lse_merge - LSE-weighted merge of split partials.
 *
 * Follows "splitk_kernels.py", _splitK_reduce: per row n,
 *   M = max_s lse_part[n, s];  w_s = exp(lse_part[n, s] - M);
 *   o[n] = sum_s w_s o_part[n, s] / sum_s w_s;  lse[n] = M + log(sum_s w_s);
 *   a row whose partial LSEs are all -inf gets o = 0, lse = -inf; the o_part
 *   entries of a split whose LSE is -inf add nothing, whatever they hold.
 *
 *   o_part   float32 [N, S, D]  (read)      lse_part float32 [N, S] (read)
 *   o        [N, D] in o_dtype (ATTN_F32 or ATTN_BF16) (written)
 *   lse      float32 [N] (written; may be NULL)
 *   D <= 1024 and a multiple of 4;  S >= 1.
 */
attn_status_t attn_lse_merge(const float* o_part, const float* lse_part, int N, int S, int D,
                             void* o, float* lse, attn_dtype_t o_dtype, void* stream);

/*
 * attn_lse_merge_bwd - gradient of attn_lse_merge.
 *
 * Follows "splitk_kernels.py", _splitK_reduce_varargs_backward: with the
 * merged O and LSE of each row and w_s = exp(lse_part[n, s] - LSE[n]),
 *   d_o_part[n, s]   = w_s * d_o[n]
 *   d_lse_part[n, s] = w_s * d_lse[n] + sum_d (o_part[n, s, d] - O[n, d]) * w_s * d_o[n, d].
 * O and LSE are recomputed from the partials in fp32.  Splits with LSE -inf,
 * and every split of a row whose partials are all -inf, get zero gradients.
 *
 *   o_part float32 [N, S, D], lse_part float32 [N, S]            (read)
 *   d_o    float32 [N, D], d_lse float32 [N] (may be NULL = 0)   (read)
 *   d_o_part float32 [N, S, D], d_lse_part float32 [N, S]        (written)
 *   D <= 1024 and a multiple of 4;  S >= 1.
 */
attn_status_t attn_lse_merge_bwd(const float* o_part, const float* lse_part, const float* d_o,
                                 const float* d_lse, int N, int S, int D,
                                 float* d_o_part, float* d_lse_part, void* stream);

/*
 * attn_selftest_wait_timeout - check that a pipeline wait which is never
 * satisfied ends with a status, not a hang.
 *
 * Launches one thread that waits, with the bounded mbarrier wait all the
 * kernels above use, on a barrier nothing arrives on.  After limit_us
 * microseconds of device time the wait gives up, ATTN_DEV_WAIT_TIMEOUT is
 * OR-ed into *dev_status and the kernel returns; the CUDA context stays
 * usable.  (The library's own kernels give up after 4 s.)
 *
 *   dev_status  int32 on the device (written; required)
 *   limit_us    1 .. 1000000
 * ATTN_ERR_INVALID_ARG for a NULL status word or a limit out of range.
 */
attn_status_t attn_selftest_wait_timeout(int32_t* dev_status, unsigned int limit_us, void* stream);

/* Static, human-readable name of a status code. */
const char* attn_status_string(attn_status_t status);

/* ABI version of this header (major * 100 + minor); 101 added attn_selftest_wait_timeout,
 * 102 attn_prefill_paged_varlen_ws, 103 attn_prefill_fwd_host,
 * 104 attn_prefill_fwd_ws, attn_prefill_workspace_bytes, attn_prefill_plan,
 * 105 attn_decode_split_tokens,
 * 106 attn_prefill_plan_sms, attn_decode_split_tokens_for.
 * 107 attn_decode_split_tokens_balanced_for; bad decode pages are left out.
 * 108 attn_decode_paged_fused, attn_decode_fused_workspace_bytes.
 * 109 32-token splits for the persistent int4 decode; the balanced split takes a tile.
 * 110 the tensor-core prefill takes any Hq / Hkv up to 128 (not only divisors of 128), and D = 64.
 * 111 the fused decode's workspace holds three more words (the cooperative grid merge).
 * 112 attn_decode_cooperative. */
int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_H */
