"""The C-ABI library loads, exports every entry point include/attn.h declares,
and rejects bad arguments on the host before touching a GPU (none here)."""

import ctypes
import os
import re

import pytest
import torch

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    import causal_gqa_flashattention_attn_gb300 as attn
    return attn.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("attn_prefill_fwd", "attn_decode_paged_splitk", "attn_lse_merge", "attn_decode_workspace_bytes",
              "attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    import causal_gqa_flashattention_attn_gb300 as attn
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in attn.EXPORTED
    assert L.attn_abi_version() == 112


def test_status_strings(L):
    import causal_gqa_flashattention_attn_gb300 as attn
    assert attn.attn_status_string(0) == "ok"
    assert "invalid" in attn.attn_status_string(-1)
    assert "unsupported" in attn.attn_status_string(-2)
    assert "workspace" in attn.attn_status_string(-3)


FAKE = ctypes.c_void_p(0x10000)   # aligned, never dereferenced: validation fails first


def _prefill(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, dtype=1, B=1, Hq=4, Hkv=2, q_len=8, kv_len=8, D=128,
             scale=0.1, status=None, stream=None)
    a.update(kw)
    return L.attn_prefill_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dtype"], a["B"], a["Hq"], a["Hkv"],
                              a["q_len"], a["kv_len"], a["D"], a["scale"], a["status"], a["stream"])


def test_prefill_host_validation(L):
    assert _prefill(L, q=None) == -1
    assert _prefill(L, Hq=6, Hkv=4) == -1                # Hq % Hkv != 0
    assert _prefill(L, B=0) == -1
    assert _prefill(L, kv_len=-3) == -1
    assert _prefill(L, scale=float("nan")) == -1
    assert _prefill(L, o=ctypes.c_void_p(0x10004)) == -1  # misaligned
    assert _prefill(L, D=96) == -2                       # unsupported head dim
    assert _prefill(L, dtype=2) == -2                    # fp16 not implemented
    assert _prefill(L, dtype=3) == -2


def test_prefill_host_buffers_validation(L):
    import causal_gqa_flashattention_attn_gb300 as attn
    # Q and O [1, 4, 8, 128] bf16, K and V [1, 2, 8, 128] bf16, LSE [1, 4, 8] fp32
    need = 2 * 1 * 4 * 8 * 128 * 2 + 2 * 1 * 2 * 8 * 128 * 2 + 1 * 4 * 8 * 4
    assert attn.attn_prefill_host_workspace_bytes(torch.bfloat16, 1, 4, 2, 8, 8, 128) == need
    assert attn.attn_prefill_host_workspace_bytes(torch.float16, 1, 4, 2, 8, 8, 128) == 0

    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, dtype=1, B=1, Hq=4, Hkv=2, q_len=8, kv_len=8, D=128,
                 scale=0.1, ws=FAKE, ws_bytes=need, status=None, stream=None)
        a.update(kw)
        return L.attn_prefill_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dtype"], a["B"], a["Hq"],
                                       a["Hkv"], a["q_len"], a["kv_len"], a["D"], a["scale"], a["ws"],
                                       a["ws_bytes"], a["status"], a["stream"])
    assert call(q=None) == -1
    assert call(B=0) == -1
    assert call(dtype=2) == -2
    assert call(ws=None) == -3
    assert call(ws_bytes=need - 1) == -3
    assert call(ws=ctypes.c_void_p(0x10008)) == -3
    assert call(Hq=6, Hkv=4, ws_bytes=1 << 20) == -1     # Hq % Hkv != 0, before any copy is enqueued
    assert call(D=96, ws_bytes=1 << 20) == -2


def test_prefill_ws_validation(L):
    import causal_gqa_flashattention_attn_gb300 as attn

    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, dtype=1, B=1, Hq=4, Hkv=2, q_len=8, kv_len=8, D=128,
                 scale=0.1, ws=FAKE, ws_bytes=1 << 30, status=None, stream=None)
        a.update(kw)
        return L.attn_prefill_fwd_ws(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dtype"], a["B"], a["Hq"],
                                     a["Hkv"], a["q_len"], a["kv_len"], a["D"], a["scale"], a["ws"], a["ws_bytes"],
                                     a["status"], a["stream"])
    assert call(q=None) == -1
    assert call(o=ctypes.c_void_p(0x10004)) == -1
    assert call(B=0) == -1
    assert call(Hq=6, Hkv=4) == -1
    assert call(scale=float("nan")) == -1
    assert call(dtype=2) == -2
    assert call(D=96) == -2
    assert call(ws=ctypes.c_void_p(0x10008)) == -3        # misaligned workspace
    # sizes of the split scratch and the schedule need a device; invalid sizes never do
    assert attn.attn_prefill_plan(torch.bfloat16, 1, 4, 3, 8, 8, 128) == (-1, 0)
    assert attn.attn_prefill_plan(torch.float32, 1, 4, 2, 8, 8, 64) == (0, 0)   # CUDA-core path: no split
    assert attn.attn_prefill_workspace_bytes(torch.float32, 1, 4, 2, 8, 8, 64) == 0
    assert attn.attn_prefill_workspace_bytes(torch.bfloat16, 0, 4, 2, 8, 8, 128) == 0


def test_decode_split_tokens_validation(L):
    import causal_gqa_flashattention_attn_gb300 as attn
    # sizes the decode entries do not take give 0; so does a machine without a GPU
    assert attn.attn_decode_split_tokens("int4", 16, 32, 8, 16384, n_groups=3) == 0
    assert attn.attn_decode_split_tokens("bf16", 16, 32, 8, 16384, q_len=17) == 0
    assert attn.attn_decode_split_tokens("bf16", 16, 32, 8, 16384, D=64) == 0
    assert attn.attn_decode_split_tokens("bf16", 16, 24, 8, 16384) == 0        # G = 3
    assert attn.attn_decode_split_tokens("bf16", 0, 32, 8, 16384) == 0
    assert L.attn_decode_split_tokens(0, 1, 16, 32, 8, 1, 16384, 128) == 0     # fp32 cache: no decode kernel
    if not torch.cuda.is_available():
        assert attn.attn_decode_split_tokens("bf16", 16, 32, 8, 16384) == 0


def _decode(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, table=FAKE, max_pages=4, lens=FAKE, kv_dtype=1, ng=1, B=2, Hq=32, Hkv=8,
             D=128, num_pages=8, page_size=256, split=2048, max_len=1024, scale=0.1, ws=FAKE, ws_bytes=1 << 30,
             o=FAKE, lse=None, status=None, stream=None)
    a.update(kw)
    return L.attn_decode_paged_splitk(a["q"], a["k"], a["v"], a["table"], a["max_pages"], a["lens"], a["kv_dtype"],
                                      a["ng"], a["B"], a["Hq"], a["Hkv"], a["D"], a["num_pages"], a["page_size"],
                                      a["split"], a["max_len"], a["scale"], a["ws"], a["ws_bytes"], a["o"],
                                      a["lse"], a["status"], a["stream"])


def test_decode_host_validation(L):
    assert _decode(L, table=None) == -1
    assert _decode(L, Hq=12, Hkv=8) == -1
    assert _decode(L, num_pages=0) == -1
    assert _decode(L, D=64) == -2
    assert _decode(L, Hq=24, Hkv=8) == -2               # group of 3
    assert _decode(L, page_size=100) == -2
    assert _decode(L, split=1000) == -2
    assert _decode(L, kv_dtype=0) == -2                 # fp32 cache not implemented
    assert _decode(L, kv_dtype=3, ng=3) == -2           # N_GROUPS must be 1, 2, 4 or 8
    assert _decode(L, ws=None) == -3
    assert _decode(L, ws_bytes=16) == -3


def _varlen(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, qo=FAKE, kvp=FAKE, kvi=FAKE, last=None, o=FAKE, lse=None, B=2, Hq=32, Hkv=4,
             D=128, total_q=100, num_pages=64, page_size=1, scale=0.1, status=None, stream=None)
    a.update(kw)
    return L.attn_prefill_paged_varlen(a["q"], a["k"], a["v"], a["qo"], a["kvp"], a["kvi"], a["last"], a["o"],
                                       a["lse"], a["B"], a["Hq"], a["Hkv"], a["D"], a["total_q"], a["num_pages"],
                                       a["page_size"], a["scale"], a["status"], a["stream"])


def test_varlen_host_validation(L):
    assert _varlen(L, qo=None) == -1
    assert _varlen(L, kvi=None) == -1
    assert _varlen(L, B=0) == -1
    assert _varlen(L, total_q=-1) == -1
    assert _varlen(L, page_size=0) == -1
    assert _varlen(L, Hq=30, Hkv=4) == -1                 # Hq % Hkv != 0
    assert _varlen(L, scale=float("inf")) == -1
    assert _varlen(L, o=ctypes.c_void_p(0x10008)) == -1   # misaligned
    assert _varlen(L, D=64) == -2
    assert _varlen(L, Hq=129, Hkv=1) == -2                # a group of more than 128 heads
    assert _varlen(L, B=2049) == -2                       # prefix table holds 2048 sequences
    assert _varlen(L, total_q=1 << 22) == -2              # query block index packed in 21 bits
    assert _varlen(L, Hq=1024, Hkv=1024, total_q=(1 << 21) + 1) == -2   # item count overflows int
    assert _varlen(L, num_pages=1 << 30, page_size=4) == -2
    assert _varlen(L, total_q=0) == 0                     # nothing to do, nothing launched


def _varlen_ws(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, qo=FAKE, kvp=FAKE, kvi=FAKE, last=None, o=FAKE, lse=None, B=2, Hq=32, Hkv=4,
             D=128, total_q=100, num_pages=64, page_size=1, rows=64, scale=0.1, ws=FAKE, ws_bytes=1 << 30,
             status=None, stream=None)
    a.update(kw)
    return L.attn_prefill_paged_varlen_ws(a["q"], a["k"], a["v"], a["qo"], a["kvp"], a["kvi"], a["last"], a["o"],
                                          a["lse"], a["B"], a["Hq"], a["Hkv"], a["D"], a["total_q"],
                                          a["num_pages"], a["page_size"], a["rows"], a["scale"], a["ws"],
                                          a["ws_bytes"], a["status"], a["stream"])


def test_varlen_ws_host_validation(L):
    import causal_gqa_flashattention_attn_gb300 as attn
    need = 2 * 64 * 4 * 128 * 2   # K and V copies of 64 rows x 4 heads x 128 dims, bf16
    assert attn.attn_prefill_varlen_workspace_bytes(64, 4, 128) == need
    assert attn.attn_prefill_varlen_workspace_bytes(0, 4, 128) == 0
    assert _varlen_ws(L, rows=0) == -1
    assert _varlen_ws(L, ws=None) == -3
    assert _varlen_ws(L, ws_bytes=need - 1) == -3
    assert _varlen_ws(L, ws=ctypes.c_void_p(0x10008)) == -3   # misaligned
    assert _varlen_ws(L, qo=None) == -1                       # the shared checks still apply
    assert _varlen_ws(L, D=64) == -2
    assert _varlen_ws(L, total_q=0, ws_bytes=need) == 0


def _decode_mq(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, table=FAKE, max_pages=4, lens=FAKE, kv_dtype=1, ng=1, B=2, Hq=32, Hkv=8,
             q_len=4, D=128, num_pages=8, page_size=256, split=2048, max_len=1024, scale=0.1, ws=FAKE,
             ws_bytes=1 << 30, o=FAKE, lse=None, status=None, stream=None)
    a.update(kw)
    return L.attn_decode_paged_splitk_mq(a["q"], a["k"], a["v"], a["table"], a["max_pages"], a["lens"],
                                         a["kv_dtype"], a["ng"], a["B"], a["Hq"], a["Hkv"], a["q_len"], a["D"],
                                         a["num_pages"], a["page_size"], a["split"], a["max_len"], a["scale"],
                                         a["ws"], a["ws_bytes"], a["o"], a["lse"], a["status"], a["stream"])


def test_decode_mq_host_validation(L):
    assert _decode_mq(L, q_len=0) == -1
    assert _decode_mq(L, q_len=17) == -2                 # at most 16 query rows per sequence
    assert _decode_mq(L, Hq=12, Hkv=8) == -1
    assert _decode_mq(L, kv_dtype=4) == -1               # fp8 needs its scale/shift tensors
    # workspace rows scale with q_len: [B, Hq * q_len, S, D] + [B, Hq * q_len, S]
    import causal_gqa_flashattention_attn_gb300 as attn
    need = attn.attn_decode_workspace_bytes(2, 32 * 4, 1024, 2048, 128)
    assert _decode_mq(L, ws_bytes=need - 16) == -3


def _decode_fp8(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, ks=FAKE, vs=FAKE, table=FAKE, max_pages=4, lens=FAKE, B=2, Hq=32, Hkv=8,
             q_len=1, D=128, num_pages=8, page_size=256, split=2048, max_len=1024, scale=0.1, ws=FAKE,
             ws_bytes=1 << 30, o=FAKE, lse=None, status=None, stream=None)
    a.update(kw)
    return L.attn_decode_paged_splitk_fp8(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["table"], a["max_pages"],
                                          a["lens"], a["B"], a["Hq"], a["Hkv"], a["q_len"], a["D"],
                                          a["num_pages"], a["page_size"], a["split"], a["max_len"], a["scale"],
                                          a["ws"], a["ws_bytes"], a["o"], a["lse"], a["status"], a["stream"])


def test_decode_fp8_host_validation(L):
    assert _decode_fp8(L, ks=None) == -1
    assert _decode_fp8(L, vs=ctypes.c_void_p(0x10004)) == -1   # misaligned scale/shift
    assert _decode_fp8(L, Hq=8, Hkv=2) == -2                   # coefficient box needs Hkv % 4 == 0
    assert _decode_fp8(L, page_size=32) == -2
    assert _decode_fp8(L, ws=None) == -3


def _decode_fused(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, ks=None, vs=None, table=FAKE, max_pages=4, lens=FAKE, kv_dtype=1, ng=1, B=2,
             Hq=32, Hkv=8, nq=1, D=128, num_pages=8, page_size=256, split=512, max_len=1024, scale=0.1, ws=FAKE,
             ws_bytes=1 << 30, o=FAKE, lse=None, status=None, stream=None)
    a.update(kw)
    return L.attn_decode_paged_fused(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["table"], a["max_pages"], a["lens"],
                                     a["kv_dtype"], a["ng"], a["B"], a["Hq"], a["Hkv"], a["nq"], a["D"],
                                     a["num_pages"], a["page_size"], a["split"], a["max_len"], a["scale"], a["ws"],
                                     a["ws_bytes"], a["o"], a["lse"], a["status"], a["stream"])


def test_decode_fused_host_validation(L):
    """The fused entry: O is required (the partials stay in the workspace), the
    workspace must hold the partials and the counters, and the format checks
    are those of the separate entries."""
    import causal_gqa_flashattention_attn_gb300 as attn
    assert _decode_fused(L, o=None) == -1
    assert _decode_fused(L, table=None) == -1
    assert _decode_fused(L, kv_dtype=4) == -1                    # fp8 without scale/shift words
    assert _decode_fused(L, kv_dtype=3, ng=3) == -2
    assert _decode_fused(L, nq=17) == -2
    assert _decode_fused(L, ws=None) == -3
    partial = attn.attn_decode_workspace_bytes(2, 32, 1024, 512, 128)
    fused = attn.attn_decode_fused_workspace_bytes(2, 32, 8, 1024, 512, 128)
    assert fused == partial + 80          # 2 x 8 int32 counters and 3 grid-barrier words, rounded to 16 bytes
    assert attn.attn_decode_fused_workspace_bytes(2, 32, 8, 1024, 512, 128, q_len=4) == \
        attn.attn_decode_workspace_bytes(2, 128, 1024, 512, 128) + 80
    assert _decode_fused(L, ws_bytes=partial) == -3               # room for the partials only
    assert attn.attn_decode_fused_workspace_bytes(2, 12, 8, 1024, 512, 128) == 0


def test_workspace_bytes(L):
    import causal_gqa_flashattention_attn_gb300 as attn
    # [B, Hq, S, D] + [B, Hq, S] floats, each rounded to 16 bytes; S = ceil(32768 / 2048) = 16
    assert attn.attn_decode_workspace_bytes(64, 32, 32768, 2048, 128) == 64 * 32 * 16 * 128 * 4 + 64 * 32 * 16 * 4
    assert attn.attn_decode_workspace_bytes(1, 1, 0, 64, 128) == 128 * 4 + 16   # at least one split
    assert attn.attn_decode_workspace_bytes(0, 1, 10, 64, 128) == 0


def test_merge_host_validation(L):
    assert L.attn_lse_merge(None, FAKE, 4, 2, 128, FAKE, None, 0, None) == -1
    assert L.attn_lse_merge(FAKE, FAKE, 4, 0, 128, FAKE, None, 0, None) == -1
    assert L.attn_lse_merge(FAKE, FAKE, 4, 2, 130, FAKE, None, 0, None) == -1
    assert L.attn_lse_merge(FAKE, FAKE, 4, 2, 2048, FAKE, None, 0, None) == -2
    assert L.attn_lse_merge(FAKE, FAKE, 4, 2, 128, FAKE, None, 2, None) == -2


def test_selftest_host_validation(L):
    assert L.attn_selftest_wait_timeout(None, 1000, None) == -1
    assert L.attn_selftest_wait_timeout(FAKE, 0, None) == -1
    assert L.attn_selftest_wait_timeout(FAKE, 1000001, None) == -1


def test_merge_bwd_host_validation(L):
    assert L.attn_lse_merge_bwd(None, FAKE, FAKE, None, 4, 2, 128, FAKE, FAKE, None) == -1
    assert L.attn_lse_merge_bwd(FAKE, FAKE, FAKE, None, 4, 0, 128, FAKE, FAKE, None) == -1
    assert L.attn_lse_merge_bwd(FAKE, FAKE, FAKE, None, 4, 2, 2048, FAKE, FAKE, None) == -2


def test_product_path_has_no_cpu_fallback():
    """The binding must not import the oracle or reach a CPU implementation."""
    pkg = os.path.join(ROOT, "causal_gqa_flashattention_attn_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            src = open(os.path.join(pkg, f)).read()
            assert "import oracle" not in src and "from oracle" not in src
