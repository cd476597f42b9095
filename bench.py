"""Benchmark of the causal GQA attention hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input,
inputs resident in HBM:
  1. causal GQA prefill, Llama-style workload: B=1, Hq=32, Hkv=4, q_len=2048,
     kv_len=4096 (bottom-right, delta=2048), D=128, bf16;
  2. paged split-K decode, bf16 cache: B=64, Hq=32, Hkv=8, D=128, lengths
     U[512, 32768], 256-token pages, split 2048, then the LSE merge;
  3. paged split-K decode, int4 cache (N_GROUPS=4): B=16, length 16384, then
     the LSE merge.
Each kernel is timed with CUDA events on the stream it runs on; before each
kernel a 256 MiB buffer is written and another 256 MiB buffer read, which
flushes the 129 MB L2 and leaves no dirty lines of the flush to be written back
during the kernel (the flush is outside the kernel timings).  The headline
value is prefill TFLOP/s with causal-halved FLOPs = 2*B*Hq*D*(visible
pairs)*2; decode is reported in GB/s of algorithmic bytes.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun every rank runs its own replica of the step (independent
problems, no collective on the data path); rank 0 prints one JSON line.
"""

import argparse
from dataclasses import replace
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal GQA prefill TFLOP/s and paged decode KV GB/s, % of GB300 roofline"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- accounting

def visible_pairs(q_len, kv_len):
    """Number of (query, key) pairs with key <= query + (kv_len - q_len)."""
    delta = kv_len - q_len
    return sum(max(0, min(kv_len, i + delta + 1)) for i in range(q_len))


def prefill_flops(shape):
    return 2 * shape.B * shape.Hq * shape.D * visible_pairs(shape.q_len, shape.kv_len) * 2


def kv_row_bytes(shape):
    """Bytes of one cached (token, KV head) row of K (or of V)."""
    if shape.kv_format == "dense":
        return shape.D * 2
    if shape.kv_format == "fp8":
        return shape.D + 4       # e4m3 bytes + the row's scale/shift word
    return (shape.n_groups + shape.D // 8) * 4


def decode_bytes(shape, lens):
    """Algorithmic bytes of one decode: every cached K and V row once, Q, the
    block-table entries and lengths read; O and LSE written.  The split
    partials (kernel-to-kernel scratch) are not counted."""
    row = kv_row_bytes(shape)
    kv = sum(lens) * shape.Hkv * row * 2
    pages = sum(-(-n // shape.page_size) for n in lens)
    q = shape.B * shape.Hq * shape.D * 2
    o = shape.B * shape.Hq * shape.D * 2 + shape.B * shape.Hq * 4
    return {"kv": kv, "q": q, "o": o, "table": pages * 4 + shape.B * 4,
            "kernel": kv + q + pages * 4 + shape.B * 4, "path": kv + q + o + pages * 4 + shape.B * 4}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def filled_split(shape):
    """The int4 and fp8 decode workloads fix no split size: take the library's
    choice (attn_decode_split_tokens: for the persistent int4 and fp8 kernels
    the split that balances their CTAs, 864 tokens here).  The bf16 workload
    keeps its stated 2048."""
    import causal_gqa_flashattention_attn_gb300 as attn
    if shape.kv_format not in ("int4", "fp8"):
        return shape
    s = attn.attn_decode_split_tokens(shape.kv_format, shape.B, shape.Hq, shape.Hkv, shape.len_hi,
                                      n_groups=shape.n_groups, D=shape.D)
    return replace(shape, split_tokens=s) if s > 0 else shape


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, keyed by kernel,
    kept only while the kernel's source is unchanged since the capture."""
    out = {}
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return out
    for line in open(path):
        parts = line.split()
        if len(parts) != 4 or line.startswith("#"):
            continue
        name, nbytes, src, digest = parts
        srcp = os.path.join(ROOT, "causal_gqa_flashattention_attn_gb300", "csrc", src)
        if os.path.exists(srcp) and hashlib.sha256(open(srcp, "rb").read()).hexdigest()[:16] == digest:
            out[name] = float(nbytes)
    return out


def max_over_ranks(values, dist, device=None):
    """Whole-job timing: element-wise maximum of `values` (a list of floats,
    one per timed quantity) over all ranks of the process group `dist`
    (torch.distributed, any backend); `values` unchanged when dist is None."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(values, dtype=torch.float64)
    if device is not None:
        t = t.to(device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


def job_throughput(work_per_rank, world, ms):
    """Units processed by all ranks divided by the slowest rank's time (per second)."""
    return world * work_per_rank / (ms * 1e-3)


# ------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(gpu_id)], stdout=subprocess.PIPE,
                                         stderr=subprocess.PIPE, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, err = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, err = self.proc.communicate()
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"error": (err or out or "no samples").strip()[:200]}
        sms.sort()
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sms)}


def gpu_id_for_smi(torch, dev):
    try:
        uuid = torch.cuda.get_device_properties(dev).uuid
        s = str(uuid)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x for x in vis.split(",") if x.strip()]
        return ids[dev.index or 0] if ids else str(dev.index or 0)


class L2Flush:
    """Evicts the L2 before a timed kernel: writes a buffer larger than L2, then
    reads another one, so the timed kernel starts with none of its inputs in
    L2 and with no dirty lines of the flush left to write back inside its own
    time.  Both passes run outside the timed region."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.fill_(1.0)
        self.torch.sum(self.r, dim=0, out=self.out)


# ------------------------------------------------------------- CPU baseline

def oracle_prefill_sample(seconds, shape):
    """The oracle as it stands on the host cores: whole heads of the prefill
    workload (every query row of head h of batch 0) until `seconds` pass."""
    import oracle
    import synth
    q, k, v = synth.prefill_inputs(shape, seed=0)
    qn = q[:1].double().numpy()
    kn, vn = k[:1].double().numpy(), v[:1].double().numpy()
    per_head = 2 * shape.D * visible_pairs(shape.q_len, shape.kv_len) * 2
    rows = list(range(shape.q_len))
    heads, t0 = 0, time.perf_counter()
    while True:
        oracle.prefill_rows(qn, kn, vn, 0, heads % shape.Hq, rows)
        heads += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return per_head * heads / el / 1e12, heads, el


def oracle_decode_sample(seconds, shape, inp):
    """The oracle as it stands on the host cores: whole sequences of a decode
    workload (every head, every split, merged), in order, until `seconds`
    pass.  Each sequence's pages are first gathered into a compact pool with a
    matching block table (outside the timed region); the oracle then walks
    that table token by token itself.  Returns KV GB/s of algorithmic bytes."""
    import numpy as np

    import oracle
    ps = shape.page_size
    qn = inp["q"].double().numpy()
    table = inp["block_table"].numpy()
    done_bytes, done, el = 0, 0, 0.0
    row = kv_row_bytes(shape)
    for b, n in enumerate(inp["lens"]):
        pages = table[b, :-(-n // ps)]
        kc, vc = inp["k_cache"][pages], inp["v_cache"][pages]
        if shape.kv_format == "dense":
            kc, vc = kc.float().numpy(), vc.float().numpy()
        else:
            kc, vc = kc.numpy(), vc.numpy()
        extra = {}
        if shape.kv_format == "fp8":
            extra = dict(k_scale_shift=inp["k_scale_shift"][pages].numpy(),
                         v_scale_shift=inp["v_scale_shift"][pages].numpy())
        t_b = np.arange(len(pages))[None, :]
        t0 = time.perf_counter()
        oracle.decode(qn[b:b + 1], kc, vc, t_b, [n], ps, shape.split_tokens, kv_format=shape.kv_format,
                      n_groups=shape.n_groups, **extra)
        el += time.perf_counter() - t0
        done_bytes += n * shape.Hkv * row * 2
        done += 1
        if el >= seconds:
            break
    return done_bytes / el / 1e9, done, el


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# --------------------------------------------------------------- the bench

def run_ours(args, rank, world, dist):
    import torch

    import causal_gqa_flashattention_attn_gb300 as attn
    import synth

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    attn.lib()
    stream = torch.cuda.current_stream(dev)

    pf = synth.LLAMA_GQA_PREFILL
    d16 = synth.PAGED_DECODE_BF16
    d4 = filled_split(synth.PAGED_DECODE_INT4)
    seed = 1000 * rank
    q, k, v = (t.to(dev) for t in synth.prefill_inputs(pf, seed=seed))
    o = torch.empty_like(q)
    lse = torch.empty(pf.B, pf.Hq, pf.q_len, dtype=torch.float32, device=dev)
    pb = synth.BATCHED_SQUARE_PREFILL
    qb, kb, vb = (t.to(dev) for t in synth.prefill_inputs(pb, seed=seed))
    ob = torch.empty_like(qb)
    lseb = torch.empty(pb.B, pb.Hq, pb.q_len, dtype=torch.float32, device=dev)
    dec = {}
    for name, shape in (("decode_bf16", d16), ("decode_int4", d4)):
        inp = synth.decode_inputs(shape, seed=seed)
        t = {kk: vv.to(dev) for kk, vv in inp.items() if torch.is_tensor(vv)}
        max_len = shape.len_hi
        ws = torch.empty(attn.attn_decode_workspace_bytes(shape.B, shape.Hq, max_len, shape.split_tokens, shape.D),
                         dtype=torch.uint8, device=dev)
        o_part, lse_part = attn.decode_partials_view(ws, shape.B, shape.Hq, max_len, shape.split_tokens, shape.D)
        dec[name] = dict(shape=shape, t=t, lens=inp["lens"], max_len=max_len, ws=ws,
                         o_part=o_part.view(shape.B * shape.Hq, -1, shape.D),
                         lse_part=lse_part.view(shape.B * shape.Hq, -1),
                         o=torch.empty(shape.B * shape.Hq, shape.D, dtype=torch.bfloat16, device=dev),
                         lse=torch.empty(shape.B * shape.Hq, dtype=torch.float32, device=dev),
                         bytes=decode_bytes(shape, inp["lens"]))
        if rank == 0 and not args.no_cpu_baseline:
            dec[name]["cpu_inp"] = inp     # the oracle's decode baseline reads the same draws
        del inp
    # the int4 decode again at the 2048-token split the workload description
    # gives for the bf16 cache (the leg above takes the split that fills the GPU)
    d4s = synth.PAGED_DECODE_INT4
    ws4s = torch.empty(attn.attn_decode_workspace_bytes(d4s.B, d4s.Hq, d4s.len_hi, d4s.split_tokens, d4s.D),
                       dtype=torch.uint8, device=dev)
    # the same two decodes through attn_decode_paged_fused (the merge inside the
    # launch): workspaces with the arrival counters, zeroed once
    fused = {}
    for name in ("decode_bf16", "decode_int4"):
        d = dec[name]
        sh = d["shape"]
        fused[name] = dict(ws=torch.zeros(attn.attn_decode_fused_workspace_bytes(sh.B, sh.Hq, sh.Hkv, d["max_len"],
                                                                                 sh.split_tokens, sh.D),
                                          dtype=torch.uint8, device=dev),
                           o=torch.empty(sh.B, sh.Hq, sh.D, dtype=torch.bfloat16, device=dev),
                           lse=torch.empty(sh.B, sh.Hq, dtype=torch.float32, device=dev))
    flush = L2Flush(torch, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # split-schedule scratch of the two prefills (zeroed once; each call leaves it zeroed)
    pws = torch.zeros(attn.attn_prefill_workspace_bytes(torch.bfloat16, pf.B, pf.Hq, pf.Hkv, pf.q_len, pf.kv_len,
                                                        pf.D), dtype=torch.uint8, device=dev)
    pwsb = torch.zeros(attn.attn_prefill_workspace_bytes(torch.bfloat16, pb.B, pb.Hq, pb.Hkv, pb.q_len, pb.kv_len,
                                                         pb.D), dtype=torch.uint8, device=dev)

    kernels = ["prefill", "prefill_batched", "decode_bf16", "merge_bf16", "decode_int4", "merge_int4",
               "decode_int4_split2048", "decode_bf16_fused", "decode_int4_fused", "merge_bwd", "decode_mq",
               "decode_fp8", "prefill_varlen", "prefill_varlen_ws"]
    # the method's own steps (dense prefill, paged split-K decode, merge); the
    # other legs are the widened rows (merge backward, multi-query, fp8, ragged)
    hot = ["prefill", "prefill_batched", "decode_bf16", "merge_bf16", "decode_int4", "merge_int4"]
    # ragged prefill over a page-size-1 cache (8 sequences)
    vl = synth.VARLEN_PAGED_PREFILL
    inpv = synth.varlen_inputs(vl, seed=seed)
    tv = {kk: vv.to(dev) for kk, vv in inpv.items() if torch.is_tensor(vv)}
    vl_flops = sum(2 * vl.Hq * vl.D * visible_pairs(ql, kl) * 2 for ql, kl in zip(inpv["q_lens"], inpv["kv_lens"]))
    vo = torch.empty_like(tv["q"])
    vlse = torch.empty(tv["q"].shape[0], vl.Hq, dtype=torch.float32, device=dev)
    v_rows = inpv["k_cache"].shape[0] * vl.page_size
    vws = torch.empty(attn.attn_prefill_varlen_workspace_bytes(v_rows, vl.Hkv, vl.D), dtype=torch.uint8, device=dev)
    # fp8 e4m3 row-wise cache on the int4 workload's shape
    d8 = filled_split(synth.PAGED_DECODE_FP8)
    inp8 = synth.decode_inputs(d8, seed=seed)
    t8 = {kk: vv.to(dev) for kk, vv in inp8.items() if torch.is_tensor(vv)}
    ws8 = torch.empty(attn.attn_decode_workspace_bytes(d8.B, d8.Hq, d8.len_hi, d8.split_tokens, d8.D),
                      dtype=torch.uint8, device=dev)
    lens8 = inp8["lens"]
    del inp8
    # causal multi-query decode (4 draft queries per sequence) over the bf16 paged cache
    mq_n = 4
    gmq = torch.Generator().manual_seed(seed + 11)
    mq_q = torch.randn(d16.B, d16.Hq, mq_n, d16.D, generator=gmq).to(torch.bfloat16).to(dev)
    mq_ws = torch.empty(attn.attn_decode_workspace_bytes(d16.B, d16.Hq * mq_n, d16.len_hi, d16.split_tokens, d16.D),
                        dtype=torch.uint8, device=dev)
    # merge backward on the bf16 decode's split partials, with seeded upstream gradients
    mbw = dec["decode_bf16"]
    gmb = torch.Generator().manual_seed(seed + 7)
    mb_do = torch.randn(mbw["o"].shape, generator=gmb).to(dev)
    mb_dlse = torch.randn(mbw["lse"].shape, generator=gmb).to(dev)
    mb_go = torch.empty_like(mbw["o_part"])
    mb_gl = torch.empty_like(mbw["lse_part"])
    launches_per_step = len(kernels) + 1   # the copied-pages ragged prefill launches two kernels

    def dec_call(name, fused_out=False):
        d = dec[name]
        sh, t = d["shape"], d["t"]
        if fused_out:
            f = fused[name]
            return lambda: attn.attn_decode_paged_fused(
                t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"], sh.split_tokens, d["max_len"],
                n_groups=sh.n_groups, workspace=f["ws"], o=f["o"], lse=f["lse"], dev_status=status, stream=stream)
        return lambda: attn.attn_decode_paged_splitk(
            t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"], sh.split_tokens, d["max_len"],
            n_groups=sh.n_groups, workspace=d["ws"], dev_status=status, stream=stream, write_output=False)

    def merge_call(name):
        d = dec[name]
        return lambda: attn.attn_lse_merge(d["o_part"], d["lse_part"], o=d["o"], lse=d["lse"], stream=stream)

    t4 = dec["decode_int4"]["t"]
    t16 = dec["decode_bf16"]["t"]
    # one launch (two for the copied-pages ragged prefill) per leg, in step order
    calls = {
        "prefill": lambda: attn.attn_prefill_fwd_ws(q, k, v, workspace=pws, o=o, lse=lse, dev_status=status,
                                                    stream=stream),
        "prefill_batched": lambda: attn.attn_prefill_fwd_ws(qb, kb, vb, workspace=pwsb, o=ob, lse=lseb,
                                                            dev_status=status, stream=stream),
        "decode_bf16": dec_call("decode_bf16"),
        "merge_bf16": merge_call("decode_bf16"),
        "decode_int4": dec_call("decode_int4"),
        "merge_int4": merge_call("decode_int4"),
        "decode_bf16_fused": dec_call("decode_bf16", fused_out=True),
        "decode_int4_fused": dec_call("decode_int4", fused_out=True),
        "decode_int4_split2048": lambda: attn.attn_decode_paged_splitk(
            t4["q"], t4["k_cache"], t4["v_cache"], t4["block_table"], t4["seq_lens"], d4s.split_tokens, d4s.len_hi,
            n_groups=d4s.n_groups, workspace=ws4s, dev_status=status, stream=stream, write_output=False),
        "merge_bwd": lambda: attn.attn_lse_merge_bwd(mbw["o_part"], mbw["lse_part"], mb_do, mb_dlse,
                                                     d_o_part=mb_go, d_lse_part=mb_gl, stream=stream),
        "decode_mq": lambda: attn.attn_decode_paged_splitk_mq(
            mq_q, t16["k_cache"], t16["v_cache"], t16["block_table"], t16["seq_lens"], d16.split_tokens,
            d16.len_hi, workspace=mq_ws, dev_status=status, stream=stream, write_output=False),
        "decode_fp8": lambda: attn.attn_decode_paged_splitk_fp8(
            t8["q"], t8["k_cache"], t8["v_cache"], t8["k_scale_shift"], t8["v_scale_shift"], t8["block_table"],
            t8["seq_lens"], d8.split_tokens, d8.len_hi, workspace=ws8, dev_status=status, stream=stream,
            write_output=False),
        "prefill_varlen": lambda: attn.attn_prefill_paged_varlen(
            tv["q"], tv["k_cache"], tv["v_cache"], tv["qo_indptr"], tv["kv_indptr"], tv["kv_indices"],
            tv["kv_last_page_len"], o=vo, lse=vlse, dev_status=status, stream=stream),
        "prefill_varlen_ws": lambda: attn.attn_prefill_paged_varlen_ws(
            tv["q"], tv["k_cache"], tv["v_cache"], tv["qo_indptr"], tv["kv_indptr"], tv["kv_indices"],
            tv["kv_last_page_len"], max_kv_rows=v_rows, workspace=vws, o=vo, lse=vlse, dev_status=status,
            stream=stream),
    }
    assert set(calls) == set(kernels)
    # a merge runs right after its decode, on the partials the decode left in L2
    after_decode = {"merge_bf16", "merge_int4"}

    def step(ev):
        for kn in calls:
            if kn not in after_decode:
                flush()
            ev[kn][0].record(stream)
            calls[kn]()
            ev[kn][1].record(stream)

    # Legs whose inputs are larger than L2 (the paged caches, 0.34-4.1 GB, and
    # the batched prefill's Q/K/V, 0.4 GB) are also timed args.steps launches
    # back to back between one pair of events, with no flush or event between
    # launches: what a launch costs in a stream kept busy, as a serving loop
    # keeps it.  The decode paths run decode + merge per step, each merge on
    # the partials its decode has just written.
    b2b_legs = {kn: [calls[kn]] for kn in ("prefill_batched", "decode_bf16", "decode_int4",
                                           "decode_int4_split2048", "decode_bf16_fused", "decode_int4_fused",
                                           "decode_mq", "decode_fp8")}
    b2b_legs["decode_bf16_path"] = [calls["decode_bf16"], calls["merge_bf16"]]
    b2b_legs["decode_int4_path"] = [calls["decode_int4"], calls["merge_int4"]]

    def back_to_back():
        out = {}
        for kn, fns in b2b_legs.items():
            for f in fns:   # the leg's own warm-up
                f()
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                for f in fns:
                    f()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            out[kn] = e0.elapsed_time(e1) / args.steps
        return out

    def new_events():
        return {kn: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for kn in kernels}

    for _ in range(args.warmup):
        step(new_events())
    torch.cuda.synchronize(dev)
    # nvidia-smi samples every 200 ms, far longer than K steps take: the
    # sampler covers a loaded window of untimed steps (about args.clock_window
    # seconds) that ends with the timed region itself
    sampler = ClockSampler(gpu_id_for_smi(torch, dev)) if rank == 0 else None
    t_end = time.perf_counter() + args.clock_window
    while time.perf_counter() < t_end:
        for _ in range(8):
            step(new_events())
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    evs = [new_events() for _ in range(args.steps)]
    region0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    region1.record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    b2b = back_to_back()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler is not None else None
    assert status.item() == 0, f"device status {status.item()}"

    ms = {kn: sum(e[kn][0].elapsed_time(e[kn][1]) for e in evs) / args.steps for kn in kernels}
    region_ms = region0.elapsed_time(region1) / args.steps
    if dist is not None:
        vals = max_over_ranks([ms[kn] for kn in kernels] + [region_ms], dist,
                              device=dev if dist.get_backend() == "nccl" else None)
        ms = dict(zip(kernels, vals[:-1]))
        region_ms = vals[-1]
        b2b = dict(zip(b2b, max_over_ranks(list(b2b.values()), dist,
                                           device=dev if dist.get_backend() == "nccl" else None)))
    # the roofline of a leg timed back to back takes that time; the others
    # (the Llama prefill, whose inputs fit in L2, the merges, merge backward
    # and the ragged prefills) their flushed per-launch time
    ms_flushed = dict(ms)
    ms = {kn: b2b.get(kn, ms_flushed[kn]) for kn in kernels}

    # ---------------------------------------------------------------- e2e
    # the same prefill through the public host-buffer call: every step copies
    # Q, K, V in from pinned host memory and O, LSE back out (all enqueued by
    # attn_prefill_fwd_host).  Steps rotate over three streams, each with its
    # own workspace and host outputs, so that a step's inbound copies, the
    # previous step's kernel and the one before's outbound copies overlap, as
    # a serving loop would (the host link, about 205 GB/s in and 190 GB/s out,
    # bounds it; a fourth stream measured no faster).
    n_e2e = 3
    hq_, hk_, hv_ = (t.cpu().pin_memory() for t in (q, k, v))
    e2e_streams = [stream] + [torch.cuda.Stream(dev) for _ in range(n_e2e - 1)]
    need_h = attn.attn_prefill_host_workspace_bytes(q.dtype, pf.B, pf.Hq, pf.Hkv, pf.q_len, pf.kv_len, pf.D)
    e2e_ws = [torch.empty(need_h, dtype=torch.uint8, device=dev) for _ in range(n_e2e)]
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(n_e2e)]
    hl = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(n_e2e)]

    def e2e_step(i):
        j = i % n_e2e
        attn.attn_prefill_fwd_host(hq_, hk_, hv_, ho[j], hl[j], workspace=e2e_ws[j], stream=e2e_streams[j])

    def join(e_from, e_to):
        ev = torch.cuda.Event()
        ev.record(e_from)
        e_to.wait_event(ev)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s_ in e2e_streams[1:]:
        join(stream, s_)
    for i in range(args.steps):
        e2e_step(i)
    for s_ in e2e_streams[1:]:
        join(s_, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / args.steps
    if dist is not None:
        e2e_ms = max_over_ranks([e2e_ms], dist, device=dev if dist.get_backend() == "nccl" else None)[0]
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()

    if rank != 0:
        return None

    # ------------------------------------------------------------ report
    peaks, peak_src = load_peaks()
    traffic = load_traffic()
    flops = prefill_flops(pf)
    tflops = job_throughput(flops, world, ms["prefill"]) / 1e12
    rep = {}
    rep["prefill"] = dict(bound="tensor", achieved=flops / (ms["prefill"] * 1e-3) / 1e12,
                          peak=peaks["bf16_tflops"], unit="TFLOP/s", work=flops, src="prefill_tc.cu",
                          kernel="prefill_tc_kernel")
    flops_b = prefill_flops(pb)
    rep["prefill_batched"] = dict(bound="tensor", achieved=flops_b / (ms["prefill_batched"] * 1e-3) / 1e12,
                                  peak=peaks["bf16_tflops"], unit="TFLOP/s", work=flops_b, src="prefill_tc.cu",
                                  kernel="prefill_tc_kernel")
    for name in ("decode_bf16", "decode_int4"):
        d = dec[name]
        kb = d["bytes"]["kernel"]
        rep[name] = dict(bound="hbm", achieved=kb / (ms[name] * 1e-3) / 1e9, peak=peaks["hbm_gbs"], unit="GB/s",
                         work=kb, src="decode.cu" if name == "decode_bf16" else "decode_int4_g32.cu",
                         kernel="decode_bf16_kernel" if name == "decode_bf16" else "decode_int4_g32_kernel")
        mname = name.replace("decode", "merge")
        n_rows = d["shape"].B * d["shape"].Hq
        s_max = d["o_part"].shape[1]
        mb = n_rows * s_max * (d["shape"].D + 1) * 4 + n_rows * (d["shape"].D * 2 + 4)
        rep[mname] = dict(bound="hbm", achieved=mb / (ms[mname] * 1e-3) / 1e9, peak=peaks["hbm_gbs"], unit="GB/s",
                          work=mb, src="merge.cu", kernel="lse_merge_kernel")
    kb4 = dec["decode_int4"]["bytes"]["kernel"]
    rep["decode_int4_split2048"] = dict(bound="hbm", achieved=kb4 / (ms["decode_int4_split2048"] * 1e-3) / 1e9,
                                        peak=peaks["hbm_gbs"], unit="GB/s", work=kb4, src="decode_int4_g32.cu",
                                        kernel="decode_int4_g32_kernel (split 2048)")
    for name in ("decode_bf16", "decode_int4"):
        pb_ = dec[name]["bytes"]["path"]
        rep[name + "_fused"] = dict(bound="hbm", achieved=pb_ / (ms[name + "_fused"] * 1e-3) / 1e9,
                                    peak=peaks["hbm_gbs"], unit="GB/s", work=pb_,
                                    src="decode.cu" if name == "decode_bf16" else "decode_int4_g32.cu",
                                    kernel=("decode_bf16_kernel" if name == "decode_bf16" else "decode_int4_g32_kernel")
                                    + " (merge inside the launch)")
    n_rows, s_max, dd = mbw["o_part"].shape
    # algorithmic bytes: partials read once, gradients in, gradient partials out
    mbb = n_rows * s_max * (dd + 1) * 4 * 2 + n_rows * (dd + 1) * 4
    rep["merge_bwd"] = dict(bound="hbm", achieved=mbb / (ms["merge_bwd"] * 1e-3) / 1e9, peak=peaks["hbm_gbs"],
                            unit="GB/s", work=mbb, src="merge.cu", kernel="lse_merge_bwd_short_kernel")
    mqb = dec["decode_bf16"]["bytes"]["kernel"] + mq_q.numel() * 2 - d16.B * d16.Hq * d16.D * 2
    rep["decode_mq"] = dict(bound="hbm", achieved=mqb / (ms["decode_mq"] * 1e-3) / 1e9, peak=peaks["hbm_gbs"],
                            unit="GB/s", work=mqb, src="decode.cu", kernel="decode_bf16_kernel (q_len 4)")
    fp8b = decode_bytes(d8, lens8)["kernel"]
    rep["decode_fp8"] = dict(bound="hbm", achieved=fp8b / (ms["decode_fp8"] * 1e-3) / 1e9, peak=peaks["hbm_gbs"],
                             unit="GB/s", work=fp8b, src="decode_fp8_g32.cu", kernel="decode_fp8_g32_kernel")
    rep["prefill_varlen"] = dict(bound="tensor", achieved=vl_flops / (ms["prefill_varlen"] * 1e-3) / 1e12,
                                 peak=peaks["bf16_tflops"], unit="TFLOP/s", work=vl_flops, src="prefill_tc.cu",
                                 kernel="prefill_tc_kernel (ragged, paged)")
    rep["prefill_varlen_ws"] = dict(bound="tensor", achieved=vl_flops / (ms["prefill_varlen_ws"] * 1e-3) / 1e12,
                                    peak=peaks["bf16_tflops"], unit="TFLOP/s", work=vl_flops, src="prefill_tc.cu",
                                    kernel="gather_pages_kernel + prefill_tc_kernel (ragged, pages copied first)")
    kernels_out = []
    for kn in kernels:
        r = rep[kn]
        kernels_out.append({"name": kn, "kernel": r["kernel"], "ms": round(ms[kn], 5), "bound": r["bound"],
                            "achieved": round(r["achieved"], 2), "peak": r["peak"], "unit": r["unit"],
                            "frac": round(r["achieved"] / r["peak"], 4),
                            "timing": "back to back" if kn in b2b else
                            ("right after its decode" if kn in after_decode else "L2 flushed"),
                            "ms_flushed": round(ms_flushed[kn], 5),
                            "traffic": traffic.get(kn),
                            "row": "hot path" if kn in hot else
                            ("hot path, split 2048 (not in ms_per_step)" if kn == "decode_int4_split2048"
                             else "hot path, decode and merge in one launch (not in ms_per_step)"
                             if kn.endswith("_fused") else "widened")})
    dominant = max(hot, key=lambda kn: ms[kn])
    dom = rep[dominant]
    path = {}
    for name in ("decode_bf16", "decode_int4"):
        d = dec[name]
        t_ms = b2b[name + "_path"]
        t_fl = ms_flushed[name] + ms_flushed[name.replace("decode", "merge")]
        path[name] = {"value": round(world * d["bytes"]["path"] / (t_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                      "ms": round(t_ms, 5), "kv_bytes": d["bytes"]["kv"], "algorithmic_bytes": d["bytes"]["path"],
                      "frac_of_hbm": round(d["bytes"]["path"] / (t_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                      "timing": "decode + merge per step, back to back",
                      "ms_flushed": round(t_fl, 5)}

    cpu = None
    if not args.no_cpu_baseline:
        val, heads, el = oracle_prefill_sample(args.cpu_seconds, pf)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"{heads} whole heads (all {pf.q_len} query rows x {pf.kv_len} keys) of the prefill "
                         f"workload, {el:.1f} s of numpy float64 on the host"}
        for name in ("decode_bf16", "decode_int4"):
            d = dec[name]
            gbs, n_seq, el_d = oracle_decode_sample(args.cpu_seconds / 2, d["shape"], d.pop("cpu_inp"))
            cpu[name] = {"value": gbs, "unit": "GB/s", "kind": "oracle", "cores": host_cores(),
                         "sample": f"{n_seq} whole sequences (every head and split, merged) of the {name} "
                                   f"workload, {el_d:.1f} s of numpy float64 on the host; KV bytes read"}
    line = {
        "metric": METRIC,
        "value": round(tflops, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(sum(ms_flushed[kn] for kn in hot), 5),
        "ms_per_step_back_to_back": round(ms_flushed["prefill"] + b2b["prefill_batched"]
                                          + b2b["decode_bf16_path"] + b2b["decode_int4_path"], 5),
        "ms_widened_rows_per_step": round(sum(ms_flushed[kn] for kn in kernels if kn not in hot), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": "prefill B1 Hq32 Hkv4 q2048 kv4096 D128 bf16 (bottom-right causal; the headline value) "
                        "+ batched prefill B8 Hq32 Hkv8 q=kv=4096 D128 + paged split-K decode bf16 B64 Hq32 Hkv8 "
                        "D128 len U[512,32768] page256 split2048 + int4 (N_GROUPS=4) paged decode B16 len16384",
            "prefill": {"B": pf.B, "Hq": pf.Hq, "Hkv": pf.Hkv, "q_len": pf.q_len, "kv_len": pf.kv_len, "D": pf.D,
                        "flops": flops},
            "decode_bf16": {"B": d16.B, "Hq": d16.Hq, "Hkv": d16.Hkv, "D": d16.D, "tokens": sum(dec["decode_bf16"]["lens"]),
                            "page": d16.page_size, "split": d16.split_tokens},
            "decode_int4": {"B": d4.B, "Hq": d4.Hq, "Hkv": d4.Hkv, "D": d4.D, "tokens": sum(dec["decode_int4"]["lens"]),
                            "n_groups": d4.n_groups, "page": d4.page_size, "split": d4.split_tokens},
            "global_batch": world,
            "parallelism": f"replicas x{world}",
            "l2": "per step, before each kernel a 256 MiB buffer is written, then another 256 MiB buffer is read "
                  "(the kernel's inputs leave L2 and no dirty flush lines are written back inside its time; "
                  "flush excluded from kernel times; a merge follows its decode unflushed); the legs whose inputs "
                  "are larger than L2 (paged caches 0.34-4.1 GB, batched prefill Q/K/V 0.4 GB) are also timed "
                  "steps launches back to back between one event pair, and their roofline uses that time "
                  "(kernels[].timing; ms_flushed beside it); ms_per_step sums the flushed hot-path legs",
            "peaks": peak_src,
        },
        "decode": path,
        "roofline": {"kernel": dominant, "bound": dom["bound"], "achieved": round(dom["achieved"], 2),
                     "peak": dom["peak"], "unit": dom["unit"], "frac": round(dom["achieved"] / dom["peak"], 4),
                     "traffic": traffic.get(dominant), "peak_source": f"{peak_src} (MEASURED_PEAKS.json)"
                     if peak_src == "measured" else "fallback"},
        "prefill_batched": {"value": round(job_throughput(flops_b, world, ms["prefill_batched"]) / 1e12, 3),
                            "unit": "TFLOP/s", "ms": round(ms["prefill_batched"], 5), "flops": flops_b,
                            "frac": round(rep["prefill_batched"]["achieved"] / peaks["bf16_tflops"], 4),
                            "workload": "B8 Hq32 Hkv8 q=kv=4096 D128 bf16, K x2"},
        "prefill_roofline": {"bound": "tensor", "achieved": round(rep["prefill"]["achieved"], 2),
                             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": round(rep["prefill"]["achieved"] / peaks["bf16_tflops"], 4),
                             "traffic": traffic.get("prefill")},
        "kernels": kernels_out,
        "region_ms_per_step_incl_flush": round(region_ms, 5),
        "cpu_baseline": cpu,
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms": round(e2e_ms, 5),
                "what": "prefill through the C-ABI host-buffer call attn_prefill_fwd_host: pinned host Q/K/V "
                        "copied in and O/LSE copied out every step, steps rotating over three streams"},
        "gpu_launches": launches_per_step * args.steps + sum(len(f) for f in b2b_legs.values()) * args.steps,
        "clocks": clocks,
    }
    return line


def run_reference(args, rank):
    """The oracle arm: the CPU oracle as it stands, timed on the host cores on
    bounded samples of the same workloads.  Each step runs one whole head of
    the Llama-style prefill (the headline TFLOP/s), one whole sequence of the
    bf16 paged decode and one of the int4 paged decode (KV GB/s, every head
    and split of the sequence, merged)."""
    import synth
    if rank != 0:
        return None
    import numpy as np

    import oracle
    pf = synth.LLAMA_GQA_PREFILL
    per_head = 2 * pf.D * visible_pairs(pf.q_len, pf.kv_len) * 2
    q, k, v = synth.prefill_inputs(pf, seed=0)
    qn, kn, vn = q[:1].double().numpy(), k[:1].double().numpy(), v[:1].double().numpy()
    rows = list(range(pf.q_len))
    dec = {}
    for name, shape in (("decode_bf16", synth.PAGED_DECODE_BF16), ("decode_int4", synth.PAGED_DECODE_INT4)):
        inp = synth.decode_inputs(shape, seed=0)
        ps = shape.page_size
        seqs = []
        for i in range(args.warmup + args.steps):   # the pages of each sampled sequence, in a compact pool
            b = i % shape.B
            n = inp["lens"][b]
            pages = inp["block_table"][b, :-(-n // ps)].numpy()
            kc, vc = inp["k_cache"][pages], inp["v_cache"][pages]
            conv = (lambda x: x.float().numpy()) if shape.kv_format == "dense" else (lambda x: x.numpy())
            seqs.append((inp["q"][b:b + 1].double().numpy(), conv(kc), conv(vc), np.arange(len(pages))[None, :], n))
        dec[name] = dict(shape=shape, seqs=seqs, row=kv_row_bytes(shape))
        del inp

    def decode_one(name, i):
        d = dec[name]
        sh = d["shape"]
        qb, kc, vc, table, n = d["seqs"][i]
        oracle.decode(qb, kc, vc, table, [n], sh.page_size, sh.split_tokens, kv_format=sh.kv_format,
                      n_groups=sh.n_groups)
        return n * sh.Hkv * d["row"] * 2

    for i in range(args.warmup):
        oracle.prefill_rows(qn, kn, vn, 0, i % pf.Hq, rows)
        decode_one("decode_bf16", i)
        decode_one("decode_int4", i)
    t_pf = 0.0
    t_dec = {"decode_bf16": 0.0, "decode_int4": 0.0}
    kv_bytes = {"decode_bf16": 0, "decode_int4": 0}
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle.prefill_rows(qn, kn, vn, 0, i % pf.Hq, rows)
        t_pf += time.perf_counter() - t0
        for name in ("decode_bf16", "decode_int4"):
            t0 = time.perf_counter()
            kv_bytes[name] += decode_one(name, args.warmup + i)
            t_dec[name] += time.perf_counter() - t0
    val = per_head * args.steps / t_pf / 1e12
    cores = host_cores()
    sample = f"one whole head (all {pf.q_len} query rows x {pf.kv_len} keys) of the prefill workload per step"
    decode = {name: {"value": kv_bytes[name] / t_dec[name] / 1e9, "unit": "GB/s", "kind": "oracle", "cores": cores,
                     "sample": f"one whole sequence of the {name} workload per step (every head and split, "
                               f"merged); KV bytes read"}
              for name in t_dec}
    total = t_pf + sum(t_dec.values())
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "prefill B1 Hq32 Hkv4 q2048 kv4096 D128 (bottom-right causal) + paged split-K "
                                   "decode bf16 B64 len U[512,32768] + int4 decode B16 len16384, CPU oracle"},
            "decode": decode,
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample, **decode},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_profile(args):
    """One kernel on its workload, `args.warmup + args.steps` launches, for an
    ncu capture of that kernel (`-k` and `-s/-c` pick the launches)."""

    import torch

    import causal_gqa_flashattention_attn_gb300 as attn
    import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    attn.lib()
    n = args.warmup + args.steps
    if args.profile.startswith("prefill_varlen"):
        vl = synth.VARLEN_PAGED_PREFILL
        t = {kk: vv.to(dev) for kk, vv in synth.varlen_inputs(vl, seed=0).items() if torch.is_tensor(vv)}
        rows = t["k_cache"].shape[0] * vl.page_size
        for _ in range(n):
            if args.profile == "prefill_varlen_ws":
                attn.attn_prefill_paged_varlen_ws(t["q"], t["k_cache"], t["v_cache"], t["qo_indptr"],
                                                  t["kv_indptr"], t["kv_indices"], t["kv_last_page_len"],
                                                  max_kv_rows=rows)
            else:
                attn.attn_prefill_paged_varlen(t["q"], t["k_cache"], t["v_cache"], t["qo_indptr"], t["kv_indptr"],
                                               t["kv_indices"], t["kv_last_page_len"])
    elif args.profile == "merge_bwd":
        # partials of the bf16 decode's shape (rows = B * Hq, its split count, D), synthetic values
        shape = synth.PAGED_DECODE_BF16
        n_split = -(-shape.len_hi // shape.split_tokens)
        o_part, lse_part = synth.merge_inputs(shape.B * shape.Hq, n_split, shape.D, seed=0)
        g = torch.Generator().manual_seed(1)
        d_o = torch.randn(shape.B * shape.Hq, shape.D, generator=g).to(dev)
        d_lse = torch.randn(shape.B * shape.Hq, generator=g).to(dev)
        op, lp = o_part.to(dev), lse_part.to(dev)
        go, gl = torch.empty_like(op), torch.empty_like(lp)
        for _ in range(n):
            attn.attn_lse_merge_bwd(op, lp, d_o, d_lse, d_o_part=go, d_lse_part=gl)
    elif args.profile.startswith("prefill"):
        shape = synth.LLAMA_GQA_PREFILL if args.profile == "prefill" else synth.BATCHED_SQUARE_PREFILL
        q, k, v = (t.to(dev) for t in synth.prefill_inputs(shape, seed=0))
        ws = torch.zeros(attn.attn_prefill_workspace_bytes(q.dtype, *q.shape[:2], k.shape[1], q.shape[2], k.shape[2],
                                                           q.shape[3]), dtype=torch.uint8, device=dev)
        for _ in range(n):
            attn.attn_prefill_fwd_ws(q, k, v, workspace=ws)
    else:
        shape = {"decode_bf16": synth.PAGED_DECODE_BF16, "decode_int4": synth.PAGED_DECODE_INT4,
                 "decode_fp8": synth.PAGED_DECODE_FP8}[args.profile]
        if args.decode_batch:
            shape = replace(shape, B=args.decode_batch)
        shape = filled_split(shape)
        inp = synth.decode_inputs(shape, seed=0)
        t = {kk: vv.to(dev) for kk, vv in inp.items() if torch.is_tensor(vv)}
        ws = torch.empty(attn.attn_decode_workspace_bytes(shape.B, shape.Hq, shape.len_hi, shape.split_tokens,
                                                          shape.D), dtype=torch.uint8, device=dev)
        for _ in range(n):
            if shape.kv_format == "fp8":
                attn.attn_decode_paged_splitk_fp8(t["q"], t["k_cache"], t["v_cache"], t["k_scale_shift"],
                                                  t["v_scale_shift"], t["block_table"], t["seq_lens"],
                                                  shape.split_tokens, shape.len_hi, workspace=ws, write_output=False)
            else:
                attn.attn_decode_paged_splitk(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                                              shape.split_tokens, shape.len_hi, n_groups=shape.n_groups,
                                              workspace=ws, write_output=False)
    torch.cuda.synchronize(dev)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-window", type=float, default=2.0,
                    help="seconds of loaded, untimed steps sampled by nvidia-smi before the timed region")
    ap.add_argument("--profile", choices=["prefill", "prefill_batched", "prefill_varlen", "prefill_varlen_ws", "decode_bf16", "decode_int4",
                                          "decode_fp8", "merge_bwd"],
                    help="run only one kernel on its workload (for ncu captures); prints no JSON line")
    ap.add_argument("--decode-batch", type=int, default=0, help="with --profile: shrink the decode batch")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.profile:
        run_profile(args)
        return
    if args.impl == "reference":
        line = run_reference(args, rank)
    else:
        if world > 1:
            import torch
            import torch.distributed as tdist
            tdist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
            dist = tdist
        line = run_ours(args, rank, world, dist)
        if dist is not None:
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
