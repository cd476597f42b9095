"""GB300 (sm_103a) causal grouped-query attention: Python binding of libattn.so.

This module only marshals arguments: it takes torch tensors that already live
on the GPU, passes their device pointers and sizes to the C ABI declared in
``include/attn.h`` and raises on a non-OK status.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback of any
kind, and importing a function of this module fails loudly when the library
has not been built.

Entry points (names as in the C ABI):
  attn_prefill_fwd          causal GQA prefill -> (O, LSE)
  attn_prefill_fwd_ws       the same with scratch for the split schedule
  attn_prefill_paged_varlen ragged causal GQA prefill over a paged KV cache
  attn_decode_workspace_bytes
  attn_decode_paged_splitk  single-query split-K decode over a paged cache
  attn_decode_paged_splitk_mq      causal multi-query decode (q_len <= 16 per sequence)
  attn_decode_paged_splitk_fp8     the same over an fp8 e4m3 row-wise cache
  attn_decode_paged_splitk_static  the same decode with no workspace argument
  attn_decode_paged_fused   the decode with the LSE merge inside the same launch
  attn_lse_merge            LSE-weighted merge of split partials
  attn_lse_merge_bwd        its gradient
  attn_status_string
"""

import ctypes
import math
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libattn.so")

# status and dtype codes of include/attn.h
ATTN_OK = 0
ATTN_F32, ATTN_BF16, ATTN_F16, ATTN_INT4_PACKED, ATTN_FP8_E4M3 = 0, 1, 2, 3, 4
ATTN_DEV_PAGE_OUT_OF_RANGE = 0x1
ATTN_DEV_SEQ_TOO_LONG = 0x2
ATTN_DEV_WAIT_TIMEOUT = 0x4
ATTN_DEV_WORKSPACE_STATE = 0x8

EXPORTED = ("attn_prefill_fwd", "attn_prefill_workspace_bytes", "attn_prefill_plan", "attn_prefill_plan_sms", "attn_prefill_fwd_ws", "attn_prefill_host_workspace_bytes", "attn_prefill_fwd_host", "attn_prefill_paged_varlen", "attn_prefill_varlen_workspace_bytes",
            "attn_prefill_paged_varlen_ws", "attn_decode_workspace_bytes", "attn_decode_split_tokens", "attn_decode_split_tokens_for", "attn_decode_split_tokens_balanced_for", "attn_decode_paged_splitk", "attn_decode_paged_splitk_mq",
            "attn_decode_paged_splitk_fp8", "attn_decode_paged_fused", "attn_decode_fused_workspace_bytes", "attn_decode_cooperative",
            "attn_decode_paged_splitk_static", "attn_lse_merge", "attn_lse_merge_bwd", "attn_selftest_wait_timeout",
            "attn_status_string", "attn_abi_version")
ATTN_DECODE_STATIC_SCRATCH_BYTES = 32 << 20

_lib = None


class AttnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {attn_status_string(status)} ({status})")


def lib():
    """The loaded library (ctypes), with argument and result types declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(or python causal_gqa_flashattention_attn_gb300/_build.py)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_prefill_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp, vp]
    L.attn_prefill_fwd.restype = i32
    L.attn_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    L.attn_prefill_workspace_bytes.restype = sz
    L.attn_prefill_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int)]
    L.attn_prefill_plan.restype = i32
    L.attn_prefill_plan_sms.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int)]
    L.attn_prefill_plan_sms.restype = i32
    L.attn_decode_split_tokens_for.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    L.attn_decode_split_tokens_for.restype = i32
    L.attn_decode_split_tokens_balanced_for.argtypes = [i32, i32, i32, i32, i32]
    L.attn_decode_split_tokens_balanced_for.restype = i32
    L.attn_prefill_fwd_ws.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp, sz, vp, vp]
    L.attn_prefill_fwd_ws.restype = i32
    L.attn_prefill_host_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    L.attn_prefill_host_workspace_bytes.restype = sz
    L.attn_prefill_fwd_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp, sz, vp, vp]
    L.attn_prefill_fwd_host.restype = i32
    L.attn_prefill_paged_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                            f32, vp, vp]
    L.attn_prefill_paged_varlen.restype = i32
    L.attn_prefill_varlen_workspace_bytes.argtypes = [i32, i32, i32]
    L.attn_prefill_varlen_workspace_bytes.restype = sz
    L.attn_prefill_paged_varlen_ws.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                               i32, f32, vp, sz, vp, vp]
    L.attn_prefill_paged_varlen_ws.restype = i32
    L.attn_decode_split_tokens.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
    L.attn_decode_split_tokens.restype = i32
    L.attn_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.attn_decode_workspace_bytes.restype = sz
    L.attn_decode_paged_splitk.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                           i32, f32, vp, sz, vp, vp, vp, vp]
    L.attn_decode_paged_splitk.restype = i32
    L.attn_decode_paged_splitk_mq.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                              i32, i32, f32, vp, sz, vp, vp, vp, vp]
    L.attn_decode_paged_splitk_mq.restype = i32
    L.attn_decode_paged_splitk_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32,
                                               i32, i32, f32, vp, sz, vp, vp, vp, vp]
    L.attn_decode_paged_splitk_fp8.restype = i32
    L.attn_decode_fused_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    L.attn_decode_fused_workspace_bytes.restype = sz
    L.attn_decode_paged_fused.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                          i32, i32, i32, f32, vp, sz, vp, vp, vp, vp]
    L.attn_decode_paged_fused.restype = i32
    L.attn_decode_paged_splitk_static.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32,
                                                  i32, i32, i32, f32, vp, vp, vp, vp]
    L.attn_decode_paged_splitk_static.restype = i32
    L.attn_lse_merge.argtypes = [vp, vp, i32, i32, i32, vp, vp, i32, vp]
    L.attn_lse_merge.restype = i32
    L.attn_lse_merge_bwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp, vp]
    L.attn_lse_merge_bwd.restype = i32
    L.attn_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint, vp]
    L.attn_selftest_wait_timeout.restype = i32
    L.attn_status_string.argtypes = [i32]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_abi_version.argtypes = []
    L.attn_abi_version.restype = i32
    L.attn_decode_cooperative.argtypes = [i32]
    L.attn_decode_cooperative.restype = i32
    _lib = L
    return L


def attn_decode_cooperative(enable=None):
    """Allow (True) or forbid (False) cooperative launches in the fused
    decodes, process-wide; None only reads the setting.  Returns the setting
    before the call."""
    return bool(lib().attn_decode_cooperative(-1 if enable is None else int(bool(enable))))


def attn_status_string(status):
    return lib().attn_status_string(int(status)).decode()


def attn_selftest_wait_timeout(dev_status, limit_us=20000, stream=None):
    """Run one bounded wait that nothing satisfies; ``ATTN_DEV_WAIT_TIMEOUT``
    is OR-ed into ``dev_status`` (int32 CUDA tensor) after ``limit_us``."""
    _need_cuda(dev_status)
    if dev_status.dtype != torch.int32:
        raise ValueError("dev_status must be int32")
    _check("attn_selftest_wait_timeout",
           lib().attn_selftest_wait_timeout(_ptr(dev_status), int(limit_us), _stream_ptr(stream)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, status):
    if status != ATTN_OK:
        raise AttnError(fn, status)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


_DT = {torch.float32: ATTN_F32, torch.bfloat16: ATTN_BF16, torch.float16: ATTN_F16}


def attn_prefill_fwd(q, k, v, o=None, lse=None, scale=None, dev_status=None, stream=None, want_lse=True):
    """Causal GQA prefill (bottom-right alignment).

    ``q [B, Hq, q_len, D]``, ``k, v [B, Hkv, kv_len, D]`` (bf16 or fp32).
    Returns ``(o, lse)`` with ``o`` like ``q`` and ``lse [B, Hq, q_len]``
    float32 (natural log), allocating them when not given.
    """
    _need_cuda(q, k, v, o, lse, dev_status)
    bsz, hq, q_len, d = q.shape
    hkv, kv_len = k.shape[1], k.shape[2]
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(bsz, hq, q_len, dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib().attn_prefill_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _DT.get(q.dtype, -1), bsz, hq,
                                hkv, q_len, kv_len, d, float(scale), _ptr(dev_status), _stream_ptr(stream))
    _check("attn_prefill_fwd", st)
    return o, lse


def attn_prefill_workspace_bytes(dtype, B, Hq, Hkv, q_len, kv_len, D):
    """Bytes of split-schedule scratch attn_prefill_fwd_ws takes (0: none used)."""
    return int(lib().attn_prefill_workspace_bytes(_DT.get(dtype, -1), B, Hq, Hkv, q_len, kv_len, D))


def attn_prefill_plan(dtype, B, Hq, Hkv, q_len, kv_len, D):
    """(schedule, grid) of attn_prefill_fwd_ws on the current device:
    schedule 1 = split, 0 = whole items, -1 = invalid sizes or no device."""
    grid = ctypes.c_int(0)
    sched = lib().attn_prefill_plan(_DT.get(dtype, -1), B, Hq, Hkv, q_len, kv_len, D, ctypes.byref(grid))
    return int(sched), int(grid.value)


def attn_prefill_plan_sms(dtype, B, Hq, Hkv, q_len, kv_len, D, sms):
    """(schedule, grid) of attn_prefill_fwd_ws on a device with ``sms`` SMs."""
    grid = ctypes.c_int(0)
    sched = lib().attn_prefill_plan_sms(_DT.get(dtype, -1), B, Hq, Hkv, q_len, kv_len, D, sms, ctypes.byref(grid))
    return int(sched), int(grid.value)


def attn_decode_split_tokens_balanced_for(sms, B, head_groups, max_kv_len, tile=32):
    """The split of the persistent int4 decode for a described device (no driver call)."""
    return int(lib().attn_decode_split_tokens_balanced_for(sms, B, head_groups, max_kv_len, tile))


def attn_decode_split_tokens_for(sms, ctas_per_sm, B, Hq, Hkv, max_kv_len, q_len=1):
    """attn_decode_split_tokens for ``sms`` SMs holding ``ctas_per_sm`` decode CTAs each."""
    return int(lib().attn_decode_split_tokens_for(sms, ctas_per_sm, B, Hq, Hkv, q_len, max_kv_len))


def attn_prefill_fwd_ws(q, k, v, workspace=None, o=None, lse=None, scale=None, dev_status=None, stream=None,
                        want_lse=True):
    """attn_prefill_fwd with scratch for the split schedule.

    ``workspace`` is a uint8 CUDA tensor of at least
    attn_prefill_workspace_bytes() bytes whose leading counters are zero (a
    zeroed tensor stays reusable: every completed call leaves them zero);
    None allocates a zeroed one for this call.  Returns ``(o, lse)``.
    """
    _need_cuda(q, k, v, o, lse, dev_status, workspace)
    bsz, hq, q_len, d = q.shape
    hkv, kv_len = k.shape[1], k.shape[2]
    need = attn_prefill_workspace_bytes(q.dtype, bsz, hq, hkv, q_len, kv_len, d)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(bsz, hq, q_len, dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().attn_prefill_fwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _DT.get(q.dtype, -1), bsz, hq,
                                   hkv, q_len, kv_len, d, float(scale), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                   _stream_ptr(stream))
    _check("attn_prefill_fwd_ws", st)
    return o, lse


def attn_prefill_host_workspace_bytes(dtype, B, Hq, Hkv, q_len, kv_len, D):
    return int(lib().attn_prefill_host_workspace_bytes(_DT.get(dtype, -1), B, Hq, Hkv, q_len, kv_len, D))


def attn_prefill_fwd_host(q, k, v, o, lse=None, workspace=None, scale=None, dev_status=None, stream=None):
    """:func:`attn_prefill_fwd` on CPU tensors (pinned for asynchronous
    copies): ``q, k, v`` are copied in, ``o`` (and ``lse``) copied out, all
    enqueued on ``stream``; synchronise the stream before reading ``o``."""
    for t in (q, k, v, o, lse):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("q, k, v, o, lse must be contiguous host tensors")
    _need_cuda(workspace, dev_status)
    bsz, hq, q_len, d = q.shape
    hkv, kv_len = k.shape[1], k.shape[2]
    if workspace is None:
        need = attn_prefill_host_workspace_bytes(q.dtype, bsz, hq, hkv, q_len, kv_len, d)
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib().attn_prefill_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _DT.get(q.dtype, -1), bsz, hq,
                                     hkv, q_len, kv_len, d, float(scale), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                     _stream_ptr(stream))
    _check("attn_prefill_fwd_host", st)
    return o, lse


def attn_prefill_paged_varlen(q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, kv_last_page_len=None,
                              o=None, lse=None, scale=None, dev_status=None, stream=None):
    """Ragged causal GQA prefill over a paged cache: ``q [total_q, Hq, D]``,
    caches ``[num_pages, page_size, Hkv, D]`` (bf16), CSR ``qo_indptr``,
    ``kv_indptr`` (pages), ``kv_indices`` and optional ``kv_last_page_len``
    (int32, on the device).  Returns ``(o [total_q, Hq, D], lse [total_q, Hq])``."""
    _need_cuda(q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, o, lse, dev_status)
    total_q, hq, d = q.shape
    num_pages, page_size, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    bsz = qo_indptr.numel() - 1
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(total_q, hq, dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib().attn_prefill_paged_varlen(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(qo_indptr), _ptr(kv_indptr),
                                         _ptr(kv_indices), _ptr(kv_last_page_len), _ptr(o), _ptr(lse), bsz, hq, hkv,
                                         d, total_q, num_pages, page_size, float(scale), _ptr(dev_status),
                                         _stream_ptr(stream))
    _check("attn_prefill_paged_varlen", st)
    return o, lse


def attn_prefill_varlen_workspace_bytes(max_kv_rows, Hkv, D):
    return int(lib().attn_prefill_varlen_workspace_bytes(int(max_kv_rows), int(Hkv), int(D)))


def attn_prefill_paged_varlen_ws(q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, kv_last_page_len=None,
                                 max_kv_rows=None, workspace=None, o=None, lse=None, scale=None, dev_status=None,
                                 stream=None):
    """As :func:`attn_prefill_paged_varlen`, with the pages first copied into a
    contiguous workspace (``max_kv_rows`` rows of K and of V, at least
    ``kv_indptr[B] * page_size``; by default the pool's row count)."""
    _need_cuda(q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, o, lse, dev_status,
               workspace)
    total_q, hq, d = q.shape
    num_pages, page_size, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    bsz = qo_indptr.numel() - 1
    if max_kv_rows is None:
        max_kv_rows = num_pages * page_size
    need = attn_prefill_varlen_workspace_bytes(max_kv_rows, hkv, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(total_q, hq, dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib().attn_prefill_paged_varlen_ws(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(qo_indptr),
                                            _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len), _ptr(o),
                                            _ptr(lse), bsz, hq, hkv, d, total_q, num_pages, page_size,
                                            int(max_kv_rows), float(scale), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                            _stream_ptr(stream))
    _check("attn_prefill_paged_varlen_ws", st)
    return o, lse


def attn_decode_workspace_bytes(B, Hq, max_kv_len, split_tokens, D):
    return int(lib().attn_decode_workspace_bytes(B, Hq, max_kv_len, split_tokens, D))


def attn_decode_split_tokens(kv_dtype, B, Hq, Hkv, max_kv_len, q_len=1, n_groups=4, D=128):
    """Split size that fills the current GPU with the decode's CTAs (0: unsupported).
    ``kv_dtype``: "bf16", "int4" or "fp8"."""
    code = {"bf16": ATTN_BF16, "int4": ATTN_INT4_PACKED, "fp8": ATTN_FP8_E4M3}[kv_dtype]
    return int(lib().attn_decode_split_tokens(code, n_groups, B, Hq, Hkv, q_len, max_kv_len, D))


def attn_decode_paged_splitk(q, k_cache, v_cache, block_table, seq_lens, split_tokens, max_kv_len, scale=None,
                             n_groups=1, workspace=None, o=None, lse=None, dev_status=None, stream=None,
                             write_output=True):
    """Single-query split-K decode over a paged KV cache.

    ``q [B, Hq, D]`` bf16; caches ``[num_pages, page_size, Hkv, D]`` bf16 or
    ``[num_pages, page_size, Hkv, n_groups + D/8]`` int32 (int4 rows);
    ``block_table [B, max_pages]`` and ``seq_lens [B]`` int32.  Returns
    ``(o, lse, workspace)``; with ``write_output=False`` only the split
    partials are produced in ``workspace`` (``o`` and ``lse`` are None).
    """
    _need_cuda(q, k_cache, v_cache, block_table, seq_lens, workspace, o, lse, dev_status)
    bsz, hq, d = q.shape
    num_pages, page_size, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    kv_dtype = ATTN_INT4_PACKED if k_cache.dtype == torch.int32 else _DT.get(k_cache.dtype, -1)
    need = attn_decode_workspace_bytes(bsz, hq, max_kv_len, split_tokens, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if write_output:
        if o is None:
            o = torch.empty(bsz, hq, d, dtype=q.dtype, device=q.device)
        if lse is None:
            lse = torch.empty(bsz, hq, dtype=torch.float32, device=q.device)
    else:
        o = lse = None
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib().attn_decode_paged_splitk(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), kv_dtype,
        n_groups, bsz, hq, hkv, d, num_pages, page_size, split_tokens, max_kv_len, float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(o), _ptr(lse), _ptr(dev_status), _stream_ptr(stream))
    _check("attn_decode_paged_splitk", st)
    return o, lse, workspace


def attn_decode_paged_splitk_mq(q, k_cache, v_cache, block_table, seq_lens, split_tokens, max_kv_len, scale=None,
                                n_groups=1, workspace=None, o=None, lse=None, dev_status=None, stream=None,
                                write_output=True):
    """Causal multi-query decode: ``q [B, Hq, q_len, D]``; query i of sequence
    b sees tokens ``t <= len_b - q_len + i``.  Returns ``(o [B, Hq, q_len, D],
    lse [B, Hq, q_len], workspace)``."""
    _need_cuda(q, k_cache, v_cache, block_table, seq_lens, workspace, o, lse, dev_status)
    bsz, hq, nq, d = q.shape
    num_pages, page_size, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    kv_dtype = ATTN_INT4_PACKED if k_cache.dtype == torch.int32 else _DT.get(k_cache.dtype, -1)
    need = attn_decode_workspace_bytes(bsz, hq * nq, max_kv_len, split_tokens, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if write_output:
        if o is None:
            o = torch.empty(bsz, hq, nq, d, dtype=q.dtype, device=q.device)
        if lse is None:
            lse = torch.empty(bsz, hq, nq, dtype=torch.float32, device=q.device)
    else:
        o = lse = None
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib().attn_decode_paged_splitk_mq(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), kv_dtype,
        n_groups, bsz, hq, hkv, nq, d, num_pages, page_size, split_tokens, max_kv_len, float(scale),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(o), _ptr(lse), _ptr(dev_status),
        _stream_ptr(stream))
    _check("attn_decode_paged_splitk_mq", st)
    return o, lse, workspace


def attn_decode_paged_splitk_fp8(q, k_cache, v_cache, k_scale_shift, v_scale_shift, block_table, seq_lens,
                                 split_tokens, max_kv_len, scale=None, workspace=None, o=None, lse=None,
                                 dev_status=None, stream=None, write_output=True):
    """Decode over an fp8 e4m3 cache: ``k/v_cache`` uint8 ``[num_pages,
    page_size, Hkv, D]``, ``k/v_scale_shift`` int32 ``[num_pages, page_size,
    Hkv]``; ``q [B, Hq, D]`` (single query) or ``[B, Hq, q_len, D]``."""
    _need_cuda(q, k_cache, v_cache, k_scale_shift, v_scale_shift, block_table, seq_lens, workspace, o, lse,
               dev_status)
    single = q.dim() == 3
    q4 = q[:, :, None, :] if single else q
    bsz, hq, nq, d = q4.shape
    num_pages, page_size, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    need = attn_decode_workspace_bytes(bsz, hq * nq, max_kv_len, split_tokens, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if write_output:
        if o is None:
            o = torch.empty(q.shape, dtype=q.dtype, device=q.device)
        if lse is None:
            lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    else:
        o = lse = None
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib().attn_decode_paged_splitk_fp8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale_shift), _ptr(v_scale_shift), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), bsz, hq, hkv, nq, d, num_pages, page_size, split_tokens, max_kv_len,
        float(scale), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(o), _ptr(lse),
        _ptr(dev_status), _stream_ptr(stream))
    _check("attn_decode_paged_splitk_fp8", st)
    return o, lse, workspace


def attn_decode_fused_workspace_bytes(B, Hq, Hkv, max_kv_len, split_tokens, D=128, q_len=1):
    return int(lib().attn_decode_fused_workspace_bytes(B, Hq, Hkv, q_len, max_kv_len, split_tokens, D))


def attn_decode_paged_fused(q, k_cache, v_cache, block_table, seq_lens, split_tokens, max_kv_len, scale=None,
                            n_groups=1, k_scale_shift=None, v_scale_shift=None, workspace=None, o=None, lse=None,
                            dev_status=None, stream=None):
    """The paged split-K decode with the merge inside the same launch.

    ``q [B, Hq, D]`` (one query per sequence) or ``[B, Hq, q_len, D]`` bf16;
    the cache is bf16, int4 words (int32, with ``n_groups``) or fp8 e4m3 bytes
    (uint8, with ``k/v_scale_shift``).  ``workspace`` holds the partials and the
    arrival counters, which must be zero when a call starts (a new workspace is
    allocated zeroed here; every completed call leaves the counters zero).
    Returns ``(o, lse, workspace)``."""
    _need_cuda(q, k_cache, v_cache, k_scale_shift, v_scale_shift, block_table, seq_lens, workspace, o, lse,
               dev_status)
    single = q.dim() == 3
    q4 = q[:, :, None, :] if single else q
    bsz, hq, nq, d = q4.shape
    num_pages, page_size, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    if k_cache.dtype == torch.int32:
        kv_dtype = ATTN_INT4_PACKED
    elif k_cache.dtype == torch.uint8:
        kv_dtype = ATTN_FP8_E4M3
    else:
        kv_dtype = _DT.get(k_cache.dtype, -1)
    need = attn_decode_fused_workspace_bytes(bsz, hq, hkv, max_kv_len, split_tokens, d, q_len=nq)
    if workspace is None:
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib().attn_decode_paged_fused(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale_shift), _ptr(v_scale_shift), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), kv_dtype, n_groups, bsz, hq, hkv, nq, d, num_pages, page_size,
        split_tokens, max_kv_len, float(scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(o), _ptr(lse), _ptr(dev_status), _stream_ptr(stream))
    _check("attn_decode_paged_fused", st)
    return o, lse, workspace


def attn_decode_paged_splitk_static(q, k_cache, v_cache, block_table, seq_lens, split_tokens, max_kv_len,
                                    scale=None, n_groups=1, o=None, lse=None, dev_status=None, stream=None):
    """The same decode for callers that cannot allocate device memory: no
    workspace argument, the split partials go to a fixed array inside the
    library (at most ATTN_DECODE_STATIC_SCRATCH_BYTES).  Calls share that
    array, so calls that overlap on the GPU race; the first call on a device
    looks up the array's address and should come before any stream capture.
    Returns ``(o, lse)``; ``o`` and ``lse`` are allocated here (by torch, on
    the Python side) only when not given."""
    _need_cuda(q, k_cache, v_cache, block_table, seq_lens, o, lse, dev_status)
    bsz, hq, d = q.shape
    num_pages, page_size, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    kv_dtype = ATTN_INT4_PACKED if k_cache.dtype == torch.int32 else _DT.get(k_cache.dtype, -1)
    if o is None:
        o = torch.empty(bsz, hq, d, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(bsz, hq, dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib().attn_decode_paged_splitk_static(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), kv_dtype,
        n_groups, bsz, hq, hkv, d, num_pages, page_size, split_tokens, max_kv_len, float(scale), _ptr(o), _ptr(lse),
        _ptr(dev_status), _stream_ptr(stream))
    _check("attn_decode_paged_splitk_static", st)
    return o, lse


def decode_partials_view(workspace, B, Hq, max_kv_len, split_tokens, D):
    """Views ``(o_part [B, Hq, S, D], lse_part [B, Hq, S])`` of a decode
    workspace, in the layout documented for attn_decode_workspace_bytes."""
    S = max(1, -(-max_kv_len // split_tokens))
    n_o = B * Hq * S * D
    off = ((n_o * 4 + 15) // 16) * 16
    f = workspace.view(torch.uint8)
    o_part = f[:n_o * 4].view(torch.float32).view(B, Hq, S, D)
    lse_part = f[off:off + B * Hq * S * 4].view(torch.float32).view(B, Hq, S)
    return o_part, lse_part


def attn_lse_merge(o_part, lse_part, o=None, lse=None, o_dtype=torch.float32, stream=None):
    """Merge ``o_part [N, S, D]`` / ``lse_part [N, S]`` (float32) by LSE weight.
    Returns ``(o [N, D], lse [N])``."""
    _need_cuda(o_part, lse_part, o, lse)
    n, s, d = o_part.shape
    if o is None:
        o = torch.empty(n, d, dtype=o_dtype, device=o_part.device)
    if lse is None:
        lse = torch.empty(n, dtype=torch.float32, device=o_part.device)
    st = lib().attn_lse_merge(_ptr(o_part), _ptr(lse_part), n, s, d, _ptr(o), _ptr(lse), _DT.get(o.dtype, -1),
                              _stream_ptr(stream))
    _check("attn_lse_merge", st)
    return o, lse


def attn_lse_merge_bwd(o_part, lse_part, d_o, d_lse=None, d_o_part=None, d_lse_part=None, stream=None):
    """Gradient of the merge: ``(d_o_part [N, S, D], d_lse_part [N, S])`` from
    the partials and the gradients ``d_o [N, D]``, ``d_lse [N]`` (float32)."""
    _need_cuda(o_part, lse_part, d_o, d_lse, d_o_part, d_lse_part)
    n, s, d = o_part.shape
    if d_o_part is None:
        d_o_part = torch.empty_like(o_part)
    if d_lse_part is None:
        d_lse_part = torch.empty_like(lse_part)
    st = lib().attn_lse_merge_bwd(_ptr(o_part), _ptr(lse_part), _ptr(d_o), _ptr(d_lse), n, s, d, _ptr(d_o_part),
                                  _ptr(d_lse_part), _stream_ptr(stream))
    _check("attn_lse_merge_bwd", st)
    return d_o_part, d_lse_part
