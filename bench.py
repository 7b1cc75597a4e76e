"""Benchmark of the attention hot path on one GB300 (or N independent ranks).

A step is one paged-decode step of the Llama-3-8B-shaped workload (64
requests, one new token each, 32 query / 8 KV heads, head size 128, bf16,
contexts U[512, 4096], block size 16, 40960-block pool): write the 64 new
tokens' K/V through slot_mapping, then attention over the paged cache
(split-KV kernel + combine).  `value` is algorithmic HBM bytes per step over
the device time per step (GB/s).

The same line carries every other workload, each timed on its own with CUDA
events and its own clock record, with its roofline:
  prefill       chunked varlen causal prefill (16 requests, new U[1k, 8k] on
                cached U[0, 4k], bs 64), TFLOP/s, with the fp64 oracle timed
                on a seeded sample of its rows (cpu_baseline)
  tiny          4 packed requests {6, 4, 17, 33} then one decode step (us)
  longctx-bs*   long-context split-KV decode, block sizes 16 / 64 / 256
  cascade       decode over a shared 4096-token prefix (prefix + suffix +
                merge, one CUDA graph)
  swa           sliding-window decode with sinks
  verify        multi-token verification (2-8 query tokens per request)
  fp8decode     the decode shape over an e4m3 cache
  fp8prefill    the chunked prefill shape over an e4m3 cache
  fp8mixed      128 decode requests + 4 prefill chunks in one call, e4m3 cache

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline] [--decode-only]

--workload NAME prints the line of that one workload alone.
--impl reference times the fp64 CPU oracle on the same decode workload
(host cores; every step is a bounded sample of the decode batch), the
deliberately slow reference arm.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from varlen_flashattention_causal_gb300 import workloads as W  # noqa: E402

METRIC = "paged-decode KV GB/s + varlen-prefill TFLOP/s, % of 1×GB300 roofline"
# the workload both arms of the default line measure (they are paired by it)
DECODE_WORKLOAD = ("paged decode, Llama-3-8B shaped: B=64, Hq=32, Hkv=8, D=128, bf16, "
                   "ctx U[512,4096], block_size 16, 40960-block pool")
L2_BYTES = 129 * 1024 * 1024


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the decode split kernel on this workload, from one ncu capture of those
# metrics (its summary under profiles/ gives the command).  It is reported only while
# the kernel's sources hash to the value recorded with the capture.
DECODE_TRAFFIC = {
    "bytes": 593428480 + 5424640,        # dram__bytes_read.sum + dram__bytes_write.sum, 4 segments
    "sources": ["varlen_flashattention_causal_gb300/csrc/attn_mma.cu",
                "varlen_flashattention_causal_gb300/csrc/common.cuh",
                "varlen_flashattention_causal_gb300/csrc/internal.h"],
    "sha256": "2c561e466aaf2a6cde3139e63656fdbd1a24f82f66cb9348ffeeb833a01e602e",
}


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def decode_traffic():
    t = DECODE_TRAFFIC
    if t["bytes"] is None or source_hash(t["sources"]) != t["sha256"]:
        return None
    return t["bytes"]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, ws, device=None):
    """The slowest rank's value (every rank times the same K steps of its own
    replica); the value itself when there is one rank."""
    if ws <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def decode_bytes(b, elem=2):
    """Algorithmic bytes of one decode attention call: every cached K and V
    row once per KV head, q and out once, the block-table entries and
    lengths read."""
    kv = sum(b.kv_lens) * b.Hkv * b.D * 2 * elem
    qo = 2 * b.T * b.Hq * b.D * 2
    tables = sum((L + b.bs - 1) // b.bs for L in b.kv_lens) * 4 + b.B * 4
    return kv + qo + tables


def kv_write_bytes(T, Hkv, D, elem=2):
    return T * Hkv * D * 2 * (2 + elem) + T * 8


def visible_pairs(q_len, kv_len):
    """Unmasked (query, key) pairs of one causal, bottom-right-aligned request."""
    ctx = kv_len - q_len
    return q_len * ctx + q_len * (q_len + 1) // 2


def prefill_flops(b):
    """4 * D * Hq * (unmasked query-key pairs): QK^T and PV, 2 flops per MAC."""
    pairs = sum(visible_pairs(q, kv) for q, kv in zip(b.q_lens, b.kv_lens))
    return 4 * b.D * b.Hq * pairs


def roofline(bound, work, ms, peak, unit):
    """achieved = algorithmic work per launch / launch time; frac of the peak."""
    scale = 1e9 if unit == "GB/s" else 1e12
    ach = work / (ms * 1e-3) / scale
    return {"bound": bound, "achieved": round(ach, 1), "peak": peak, "unit": unit, "frac": round(ach / peak, 4)}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, which):
        setattr(self, which, time.time())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = getattr(self, "start", 0.0), getattr(self, "stop", float("inf"))
        for ts, r in self.rows:
            if not (lo - 0.1 <= ts <= hi + 0.3):
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for n, v in zip(names, r[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
            except Exception:
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _time(fn, steps, warmup, flush=None, min_s=0.5):
    """CUDA-event times of fn over `steps` calls after `warmup` calls (and at
    least 1 s of running, so the clock sampler is up): (median ms, mean ms,
    clocks seen during the timed calls).  flush, if given, runs before every
    timed call, outside the events (an L2 flush).  The timed loop repeats
    until it has covered at least min_s seconds, so every leg has a clock
    sample of its own."""
    with ClockSampler(torch.cuda.current_device()) as clk:
        t_w = time.time()
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        while time.time() - t_w < 1.0:
            fn()
            torch.cuda.synchronize()
        clk.mark("start")
        t = []
        t_start = time.time()
        while not t or (time.time() - t_start < min_s and len(t) < 100 * steps):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for a, c in evs:
                if flush is not None:
                    flush()
                a.record()
                fn()
                c.record()
            torch.cuda.synchronize()
            t += [a.elapsed_time(c) for a, c in evs]
        clk.mark("stop")
    return statistics.median(t), statistics.mean(t), dict(clk.summary(), timed_calls=len(t))


def _e4m3_scale(x):
    """Per-tensor scale: the largest magnitude maps to e4m3's 448."""
    return float(x.float().abs().max()) / 448.0


def _device_cache(b, dev, kv_dtype=torch.bfloat16, seed=0):
    """A paged cache on the device for every cached token of b: N(0, 1)
    K/V drawn on the device and written through kv_cache_write at the
    engine's slots (bf16), or quantised to e4m3 with per-tensor scales
    amax/448 (untimed set-up).  Returns (k_cache, v_cache, k_scale, v_scale)."""
    import varlen_flashattention_causal_gb300 as va
    g = torch.Generator(device=dev)
    g.manual_seed(W.SEED0 + 500 + seed)
    shape = (b.num_blocks, b.bs, b.Hkv, b.D)
    if kv_dtype != torch.float8_e4m3fn:
        return (torch.randn(shape, generator=g, device=dev).to(kv_dtype),
                torch.randn(shape, generator=g, device=dev).to(kv_dtype), 1.0, 1.0)
    n = sum(b.kv_lens)
    k = torch.randn((n, b.Hkv, b.D), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((n, b.Hkv, b.D), generator=g, device=dev).to(torch.bfloat16)
    ks, vs = _e4m3_scale(k), _e4m3_scale(v)
    sl = torch.cat([W.slots(b.block_table, r, range(L), b.bs) for r, L in enumerate(b.kv_lens)]).to(dev)
    kc = torch.zeros(shape, dtype=kv_dtype, device=dev)
    vc = torch.zeros_like(kc)
    va.kv_cache_write(k, v, kc, vc, sl, ks, vs)
    del k, v
    return kc, vc, ks, vs


def _steps(args):
    """Timed calls per workload leg of the default line."""
    return max(10, min(args.steps, 50))


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- workloads
# Each returns one dict: the workload, its metric and value, its roofline
# (bound, achieved, peak, frac of the measured peak) and the clocks seen.

def wl_prefill(va, dev, steps, warmup, pk):
    hbm, tc = pk
    b = W.chunked_prefill(gen_kv=False)
    kc, vc, _, _ = _device_cache(b, dev)
    q, out = b.q.to(dev), torch.empty(b.q.shape, dtype=torch.bfloat16, device=dev)
    cu, su, bt = b.cu_seqlens_q.to(dev), b.seqused_k.to(dev), b.block_table.to(dev)
    wsp = torch.empty(va.attn_workspace_size(b.T, b.Hq, b.D, 1), dtype=torch.uint8, device=dev)
    fn = lambda: va.attn_varlen_prefill(q, kc, vc, out, cu, su, bt, b.max_seqlen_q, b.max_seqlen_k,
                                        b.softmax_scale, causal=True, num_splits=1, workspace=wsp)
    med, mean, clk = _time(fn, max(3, min(steps, 20)), warmup)
    fl = prefill_flops(b)
    return {"workload": "chunked varlen causal prefill: B=16, new U[1k,8k] on cached U[0,4k], Hq=32, Hkv=8, "
                        "D=128, bf16, block_size 64",
            "metric": "varlen causal prefill TFLOP/s", "value": round(fl / (med * 1e-3) / 1e12, 1),
            "unit": "TFLOP/s", "ms": round(med, 4), "flops": fl, "kernel": "fwd_tc2_kernel (tcgen05 cta_group::2, pairs of SMs)",
            "roofline": roofline("tensor", fl, med, tc, "TFLOP/s"), "clocks": clk}


def wl_tiny(va, dev, steps, warmup, pk):
    """The pages' packed example grown to four requests, then one decode
    step: latency of the two attention calls (L2 flushed between calls)."""
    pre, dec = W.tiny()
    kc = torch.zeros((pre.num_blocks, pre.bs, pre.Hkv, pre.D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    for b in (pre, dec):
        va.kv_cache_write(b.k_tok.to(dev), b.v_tok.to(dev), kc, vc, b.slot_mapping.to(dev))
    l2buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    flush = lambda: l2buf.fill_(1)
    res = {"workload": "tiny: 4 packed requests {6,4,17,33}, Hq=8, Hkv=2, D=64, bf16, bs 16, 16-block pool, "
                       "then 1 decode step each", "metric": "latency us", "unit": "us",
           "l2": "flushed between timed calls"}
    for name, b in (("prefill", pre), ("decode", dec)):
        q, out = b.q.to(dev), torch.empty(b.q.shape, dtype=torch.bfloat16, device=dev)
        cu, su, bt = b.cu_seqlens_q.to(dev), b.seqused_k.to(dev), b.block_table.to(dev)
        fn = lambda: va.attn_varlen_prefill(q, kc, vc, out, cu, su, bt, b.max_seqlen_q, b.max_seqlen_k,
                                            b.softmax_scale, causal=True, num_splits=1)
        med, mean, clk = _time(fn, steps, warmup, flush)
        res[name + "_us"] = round(med * 1e3, 2)
        res["clocks"] = clk
    res["value"] = round(res["prefill_us"] + res["decode_us"], 2)
    res["roofline"] = {"bound": "latency", "note": "a few KB of K/V: launch latency, not bandwidth or flops"}
    return res


def wl_longctx(bs):
    def run(va, dev, steps, warmup, pk):
        hbm, tc = pk
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        b = W.decode_longctx(bs=bs, gen_kv=False)
        kc, vc, _, _ = _device_cache(b, dev)
        q, out = b.q.to(dev), torch.empty(b.q.shape, dtype=torch.bfloat16, device=dev)
        su, bt = b.seqused_k.to(dev), b.block_table.to(dev)
        ns = va.attn_num_splits(b.B, 1, b.max_seqlen_k, b.Hq, b.Hkv, sms)
        wsp = torch.empty(va.attn_workspace_size(b.B, b.Hq, b.D, ns), dtype=torch.uint8, device=dev)
        fn = lambda: va.attn_paged_decode(q, kc, vc, out, su, bt, b.max_seqlen_k, b.softmax_scale,
                                          num_splits=ns, workspace=wsp)
        med, mean, clk = _time(fn, steps, warmup)
        by = decode_bytes(b)
        return {"workload": "long-context split-KV decode: B=4, ctx {32k,64k,96k,128k}, Hq=64, Hkv=8, D=128, "
                            "bf16, block_size %d" % bs,
                "metric": "long-context paged decode GB/s", "value": round(by / (med * 1e-3) / 1e9, 1),
                "unit": "GB/s", "ms": round(med, 4), "bytes": by, "num_splits": ns,
                "roofline": roofline("hbm", by, med, hbm, "GB/s"), "clocks": clk}
    return run


def wl_cascade(va, dev, steps, warmup, pk):
    hbm, tc = pk
    b = W.cascade_decode()
    kc, vc, _, _ = _device_cache(b, dev)
    P = b.extra["prefix"]
    nblk = P // b.bs
    T, Hq, D = b.q.shape
    q = b.q.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    cu0 = torch.tensor([0, T], dtype=torch.int32, device=dev)
    su0 = torch.tensor([P], dtype=torch.int32, device=dev)
    bt = b.block_table.to(dev)
    cu, su = b.cu_seqlens_q.to(dev), (b.seqused_k - P).to(dev)
    # one attn_cascade call: the prefix half on a second stream, both halves'
    # segments merged by one combine; the library picks both split counts
    ns_pair = va.attn_cascade_splits(b.B, T, 1, P, b.max_seqlen_k - P, Hq, b.Hkv, D)
    wsp = torch.empty(va.attn_workspace_size(T, Hq, D, sum(ns_pair)), dtype=torch.uint8, device=dev)
    aux = torch.cuda.Stream()

    def step():
        va.attn_cascade(q, kc, vc, out, cu0, su0, bt[0], P, cu, su, bt[:, nblk:], 1, b.max_seqlen_k - P,
                        b.softmax_scale, lse_out=lse, workspace=wsp, aux_stream=aux)

    # the step as a serving loop runs it: captured once in a CUDA graph and
    # replayed (no host work between the launches)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    # the step touches ~185 MB, under twice the L2: write a 258 MB buffer
    # between timed steps so that no input stays resident
    l2buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    flush = lambda: l2buf.fill_(1)
    med, mean, clk = _time(g.replay, steps, warmup, flush)
    kvb = (P + sum(b.extra["suffix"])) * b.Hkv * b.D * 2 * 2
    by = kvb + 2 * T * Hq * D * 2
    return {"workload": "cascade decode: 64 requests share a 4096-token prefix, private suffix U[256,1024], "
                        "Hq=32, Hkv=8, D=128, bf16, block_size 64",
            "metric": "cascade decode GB/s (prefix read once)", "value": round(by / (med * 1e-3) / 1e9, 1),
            "unit": "GB/s", "ms": round(med, 4), "bytes": by, "splits": list(ns_pair),
            "timing": "cuda graph of one attn_cascade call (prefix half on a second stream, one combine)",
            "l2": "flushed between timed steps (%d MB write)" % (2 * L2_BYTES >> 20),
            "roofline": roofline("hbm", by, med, hbm, "GB/s"), "clocks": clk}


def wl_swa(va, dev, steps, warmup, pk):
    hbm, tc = pk
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    b = W.swa_decode(gen_kv=False)
    kc, vc, _, _ = _device_cache(b, dev)
    q, out = b.q.to(dev), torch.empty(b.q.shape, dtype=torch.bfloat16, device=dev)
    cu, su, bt = b.cu_seqlens_q.to(dev), b.seqused_k.to(dev), b.block_table.to(dev)
    win, sinks = b.extra["window"], b.extra["sinks"].to(dev)
    span = min(b.max_seqlen_k, win[0] + 1)
    ns = va.attn_num_splits(b.B, 1, span, b.Hq, b.Hkv, sms)
    wsp = torch.empty(va.attn_workspace_size(b.T, b.Hq, b.D, ns), dtype=torch.uint8, device=dev)
    fn = lambda: va.attn_varlen_prefill(q, kc, vc, out, cu, su, bt, 1, b.max_seqlen_k, b.softmax_scale,
                                        causal=True, window=win, sinks=sinks, num_splits=0, workspace=wsp)
    med, mean, clk = _time(fn, steps, warmup)
    # algorithmic bytes: the keys inside each query's window, K and V once per KV head
    by = sum(min(L, win[0] + 1) for L in b.kv_lens) * b.Hkv * b.D * 2 * 2 + 2 * b.T * b.Hq * b.D * 2
    return {"workload": "sliding-window decode with sinks: B=64, ctx U[4k,32k], window 4096, Hq=32, Hkv=8, "
                        "D=128, bf16, block_size 16",
            "metric": "sliding-window decode GB/s (window keys)", "value": round(by / (med * 1e-3) / 1e9, 1),
            "unit": "GB/s", "ms": round(med, 4), "bytes": by,
            "roofline": roofline("hbm", by, med, hbm, "GB/s"), "clocks": clk}


def wl_verify(va, dev, steps, warmup, pk):
    hbm, tc = pk
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    b = W.verify_decode(gen_kv=False)
    kc, vc, _, _ = _device_cache(b, dev)
    q, out = b.q.to(dev), torch.empty(b.q.shape, dtype=torch.bfloat16, device=dev)
    cu, su, bt = b.cu_seqlens_q.to(dev), b.seqused_k.to(dev), b.block_table.to(dev)
    ns = va.attn_num_splits(b.B, b.max_seqlen_q, b.max_seqlen_k, b.Hq, b.Hkv, sms)
    wsp = torch.empty(va.attn_workspace_size(b.T, b.Hq, b.D, ns), dtype=torch.uint8, device=dev)
    fn = lambda: va.attn_varlen_prefill(q, kc, vc, out, cu, su, bt, b.max_seqlen_q, b.max_seqlen_k,
                                        b.softmax_scale, causal=True, num_splits=0, workspace=wsp)
    med, mean, clk = _time(fn, steps, warmup)
    by = decode_bytes(b)
    return {"workload": "multi-token verify: B=64, q_len U[2,8] over ctx U[512,8192], Hq=32, Hkv=8, D=128, "
                        "bf16, block_size 16",
            "metric": "multi-token verify GB/s", "value": round(by / (med * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms": round(med, 4), "bytes": by, "roofline": roofline("hbm", by, med, hbm, "GB/s"), "clocks": clk}


def _q8(q):
    """e4m3 queries with a per-tensor scale (q_descale = amax / 448)."""
    qs = _e4m3_scale(q)
    return (q.float() / qs).to(torch.float8_e4m3fn), qs


def wl_fp8decode(va, dev, steps, warmup, pk):
    """The decode shape on an e4m3 cache, with bf16 queries and with e4m3
    queries (q_descale; Q K^T on e4m3 operands)."""
    hbm, tc = pk
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    b = W.decode_llama8b(gen_kv=False)
    kc, vc, ks, vs = _device_cache(b, dev, torch.float8_e4m3fn)
    su, bt, cu = b.seqused_k.to(dev), b.block_table.to(dev), b.cu_seqlens_q.to(dev)
    ns = va.attn_num_splits(b.B, 1, b.max_seqlen_k, b.Hq, b.Hkv, sms, b.D, va.ATTN_BF16, va.ATTN_FP8_E4M3)
    wsp = torch.empty(va.attn_workspace_size(b.B, b.Hq, b.D, ns), dtype=torch.uint8, device=dev)
    by = decode_bytes(b, elem=1)
    q8, qs = _q8(b.q)
    out = torch.empty(b.q.shape, dtype=torch.bfloat16, device=dev)
    lines, clocks = {}, None
    for name, q, qd in (("q_bf16", b.q.to(dev), 1.0), ("q_e4m3", q8.to(dev), qs)):
        fn = lambda: va.attn_varlen_prefill(q, kc, vc, out, cu, su, bt, 1, b.max_seqlen_k, b.softmax_scale,
                                            causal=True, q_descale=qd, k_descale=ks, v_descale=vs,
                                            num_splits=0, workspace=wsp)
        med, mean, clocks = _time(fn, steps, warmup)
        lines[name] = {"ms": round(med, 4), "gbs": round(by / (med * 1e-3) / 1e9, 1),
                       "frac": round(by / (med * 1e-3) / 1e9 / hbm, 4)}
    best = max(lines.values(), key=lambda x: x["gbs"])
    return {"workload": "paged decode, Llama-3-8B shaped, e4m3 cache (per-tensor amax/448 scales)",
            "metric": "fp8-KV decode GB/s", "value": best["gbs"], "unit": "GB/s", "ms": best["ms"],
            "kernel": "fwd_dec_kernel (S^T = K Q^T, O^T = V^T P^T, 8-row CTAs, TMA tile gather) + combine_light_kernel",
            "bytes": by, "variants": lines,
            "roofline": roofline("hbm", by, best["ms"], hbm, "GB/s"), "clocks": clocks}


def wl_fp8prefill(va, dev, steps, warmup, pk):
    """The chunked prefill shape on an e4m3 cache: bf16 queries (K, V and Q
    widened to fp16, f16 MMAs) and e4m3 queries (S = Q K^T on e4m3
    operands; P V on fp16 with V widened)."""
    hbm, tc = pk
    b = W.chunked_prefill(gen_kv=False)
    kc, vc, ks, vs = _device_cache(b, dev, torch.float8_e4m3fn)
    cu, su, bt = b.cu_seqlens_q.to(dev), b.seqused_k.to(dev), b.block_table.to(dev)
    q8, qs = _q8(b.q)
    out = torch.empty(b.q.shape, dtype=torch.bfloat16, device=dev)
    wsp = torch.empty(va.attn_workspace_size(b.T, b.Hq, b.D, 1), dtype=torch.uint8, device=dev)
    fl = prefill_flops(b)
    lines, clocks = {}, None
    for name, q, qd in (("q_bf16", b.q.to(dev), 1.0), ("q_e4m3", q8.to(dev), qs)):
        fn = lambda: va.attn_varlen_prefill(q, kc, vc, out, cu, su, bt, b.max_seqlen_q, b.max_seqlen_k,
                                            b.softmax_scale, causal=True, q_descale=qd, k_descale=ks,
                                            v_descale=vs, num_splits=1, workspace=wsp)
        med, mean, clocks = _time(fn, max(3, min(steps, 20)), warmup)
        tf = fl / (med * 1e-3) / 1e12
        lines[name] = {"ms": round(med, 4), "tflops": round(tf, 1), "frac_of_bf16_peak": round(tf / tc, 4)}
    best = max(lines.values(), key=lambda x: x["tflops"])
    r = roofline("tensor", fl, best["ms"], tc, "TFLOP/s")
    r["note"] = "P V runs on fp16 MMAs, so the bf16 GEMM peak is the denominator"
    return {"workload": "chunked varlen causal prefill shape, e4m3 cache (per-tensor amax/448 scales)",
            "metric": "fp8-KV chunked prefill TFLOP/s", "value": best["tflops"], "unit": "TFLOP/s",
            "ms": best["ms"], "flops": fl, "variants": lines, "roofline": r, "clocks": clocks}


def wl_fp8mixed(va, dev, steps, warmup, pk):
    hbm, tc = pk
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    b = W.fp8_mixed(gen_kv=False)
    kc, vc, ks, vs = _device_cache(b, dev, torch.float8_e4m3fn)
    q, out = b.q.to(dev), torch.empty(b.q.shape, dtype=torch.bfloat16, device=dev)
    cu, su, bt = b.cu_seqlens_q.to(dev), b.seqused_k.to(dev), b.block_table.to(dev)
    ns = va.attn_num_splits(b.B, b.max_seqlen_q, b.max_seqlen_k, b.Hq, b.Hkv, sms, b.D, va.ATTN_BF16,
                            va.ATTN_FP8_E4M3)
    wsp = torch.empty(va.attn_workspace_size(b.T, b.Hq, b.D, ns), dtype=torch.uint8, device=dev)
    fn = lambda: va.attn_varlen_prefill(q, kc, vc, out, cu, su, bt, b.max_seqlen_q, b.max_seqlen_k,
                                        b.softmax_scale, causal=True, k_descale=ks, v_descale=vs,
                                        num_splits=0, workspace=wsp)
    med, mean, clk = _time(fn, steps, warmup)
    n_dec = sum(1 for x in b.q_lens if x == 1)
    dec = sum(b.kv_lens[:n_dec]) * b.Hkv * b.D * 2
    fl = prefill_flops(b)
    t_star = max(dec / hbm / 1e6, fl / tc / 1e9)
    return {"workload": "fp8 mixed batch: 128 decode requests ctx log-uniform [128,16k] + 4 prefill chunks of "
                        "2048, e4m3 cache (per-tensor amax/448 scales), Hq=32, Hkv=8, D=128, block_size 32",
            "metric": "fp8-KV mixed batch ms", "value": round(med, 4), "unit": "ms", "ms": round(med, 4),
            "decode_bytes": dec, "prefill_flops": fl, "num_splits": ns,
            "roofline": {"bound": "mixed", "t_star_ms": round(t_star, 4),
                         "sum_bound_ms": round(dec / hbm / 1e6 + fl / tc / 1e9, 4),
                         "frac": round(t_star / med, 4),
                         "note": "t* = max(decode bytes / HBM peak, prefill flops / bf16 peak); frac = t* / time"},
            "clocks": clk}


WORKLOADS = {
    "prefill": wl_prefill, "tiny": wl_tiny,
    "longctx-bs16": wl_longctx(16), "longctx-bs64": wl_longctx(64), "longctx-bs256": wl_longctx(256),
    "cascade": wl_cascade, "swa": wl_swa, "verify": wl_verify,
    "fp8decode": wl_fp8decode, "fp8prefill": wl_fp8prefill, "fp8mixed": wl_fp8mixed,
}
# the default line's extra legs (prefill has its own key)
DEFAULT_LEGS = ["tiny", "longctx-bs16", "longctx-bs64", "longctx-bs256", "cascade", "swa", "verify",
                "fp8decode", "fp8prefill", "fp8mixed"]


# ---------------------------------------------------------------- the line

def run_ours(args):
    import varlen_flashattention_causal_gb300 as va
    from varlen_flashattention_causal_gb300 import build
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    build.build()
    hbm, tc, tc_sus, peak_kind = peaks()

    # ---------------- decode workload: history resident in the paged cache
    b = W.decode_llama8b(device="cpu")
    # the step's own new tokens are the last position of each request
    last = torch.tensor([sum(b.kv_lens[:r + 1]) - 1 for r in range(b.B)])
    g = torch.Generator(device=dev)
    g.manual_seed(W.SEED0 + 1)
    kc = torch.randn((b.num_blocks, b.bs, b.Hkv, b.D), generator=g, device=dev).to(torch.bfloat16)
    vc = torch.randn((b.num_blocks, b.bs, b.Hkv, b.D), generator=g, device=dev).to(torch.bfloat16)
    q = b.q.to(dev)
    k_new = b.k_tok[last].to(dev)
    v_new = b.v_tok[last].to(dev)
    slots = b.slot_mapping[last].to(dev)
    seq_lens = b.seqused_k.to(dev)
    bt = b.block_table.to(dev)
    out = torch.empty_like(q)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ns = va.attn_num_splits(b.B, 1, b.max_seqlen_k, b.Hq, b.Hkv, sms)
    wsp = torch.empty(va.attn_workspace_size(b.B, b.Hq, b.D, ns), dtype=torch.uint8, device=dev)

    def step(stream=None):
        va.kv_cache_write(k_new, v_new, kc, vc, slots)
        va.attn_paged_decode(q, kc, vc, out, seq_lens, bt, b.max_seqlen_k, b.softmax_scale,
                             num_splits=ns, workspace=wsp)

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with ClockSampler(dev.index) as clk:
        t_w = time.time()
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        while time.time() - t_w < 1.0:        # the sampler is up before timing starts
            step()
            torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        clk.mark("start")
        # the K timed steps, with nothing between the launches (an event
        # between two launches would cut their programmatic chaining)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(K):
            step()
        t1.record()
        torch.cuda.synchronize()
        # the attention call alone, for its roofline: events around each call
        for i in range(K):
            va.kv_cache_write(k_new, v_new, kc, vc, slots)
            ev[i][0].record()
            va.attn_paged_decode(q, kc, vc, out, seq_lens, bt, b.max_seqlen_k, b.softmax_scale,
                                 num_splits=ns, workspace=wsp)
            ev[i][1].record()
        torch.cuda.synchronize()
        clk.mark("stop")
    if ws > 1:
        dist.barrier()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), ws, dev)
    attn_ms = statistics.mean(a.elapsed_time(c) for a, c in ev)
    dbytes = decode_bytes(b)
    step_bytes = dbytes + kv_write_bytes(b.B, b.Hkv, b.D)
    ms_per_step = elapsed_ms / K
    value = step_bytes * ws / (ms_per_step * 1e-3) / 1e9
    achieved = dbytes / (attn_ms * 1e-3) / 1e9

    # ---------------- e2e: host inputs -> device -> result back, per step
    # The step's inputs (q, new K/V rows, slots, lengths, block table) sit
    # packed in one pinned host buffer and go up in one copy; the result
    # comes back in one copy.  As a serving loop runs it, both copies run on
    # a copy stream with two device buffer sets: step k+1's inputs upload
    # and step k's result downloads while the next step computes.
    ins = (q, k_new, v_new, slots, seq_lens, bt)
    offs, total = [], 0
    for t in ins:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for t, o in zip(ins, offs):
        n = t.numel() * t.element_size()
        h_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    d_in = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]

    def views(buf):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(ins, offs)]

    d_views = [views(d) for d in d_in]
    outs = [torch.empty_like(out) for _ in range(2)]
    h_outs = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    bi = sum(t.numel() * t.element_size() for t in ins)
    bo = out.numel() * out.element_size()
    cur, cp = torch.cuda.current_stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]       # the compute that used buffer set i finished
    out_free = [torch.cuda.Event() for _ in range(2)]   # the result in outs[i] has been copied back

    def upload(i):
        with torch.cuda.stream(cp):
            cp.wait_event(done[i])                       # the step two back has read d_in[i]
            d_in[i].copy_(h_in, non_blocking=True)
            in_ready[i].record(cp)

    def e2e_steps(n):
        upload(0)
        for k in range(n):
            i = k & 1
            if k + 1 < n:
                upload(1 - i)
            cur.wait_event(in_ready[i])
            cur.wait_event(out_free[i])
            dq, dk, dv, dslots, dlens, dbt = d_views[i]
            va.kv_cache_write(dk, dv, kc, vc, dslots)
            va.attn_paged_decode(dq, kc, vc, outs[i], dlens, dbt, b.max_seqlen_k, b.softmax_scale,
                                 num_splits=ns, workspace=wsp)
            done[i].record(cur)
            with torch.cuda.stream(cp):
                cp.wait_event(done[i])
                h_outs[i].copy_(outs[i], non_blocking=True)
                out_free[i].record(cp)
        cur.wait_stream(cp)

    e2e_steps(3)
    torch.cuda.synchronize()
    Ke = max(100, K)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    e2e_steps(Ke)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / Ke
    assert torch.equal(h_outs[(Ke - 1) & 1], out.cpu()), "e2e result differs from the device-timed step"
    e2e_value = step_bytes * ws / (e2e_ms * 1e-3) / 1e9
    del kc, vc, d_in, outs
    _free()

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD,
                   "step": "kv_cache_write of 64 new tokens + attn_paged_decode (split-KV + combine)",
                   "num_splits": ns, "bytes_per_step": step_bytes,
                   "l2": "inputs larger than L2: %.0f MB of K/V read per step vs %d MB L2"
                         % (sum(b.kv_lens) * b.Hkv * b.D * 4 / 1e6, L2_BYTES >> 20),
                   "parallelism": "replicas x%d (independent batches, no collective)" % ws},
        "roofline": {"kernel": "attn_paged_decode (fwd_mma_kernel + combine_light_kernel; time of the whole call)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_source": peak_kind, "traffic": decode_traffic(),
                     "traffic_kernel": "fwd_mma_kernel (ncu, one launch)",
                     "algorithmic_bytes_per_launch": dbytes, "avg_launch_ms": round(attn_ms, 5)},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "ms_per_step": round(e2e_ms, 5), "steps": Ke,
                "copies": "one packed pinned-host upload and one result download per step, on a copy "
                          "stream overlapping the neighbouring steps' compute (two buffer sets)"},
        "gpu_launches": 3 * K,
        "clocks": clk.summary(),
    }
    if not args.decode_only:
        pk = (hbm, tc)
        pf = wl_prefill(va, dev, _steps(args), args.warmup, pk)
        _free()
        if rank == 0 and not args.no_cpu_baseline:
            pf["cpu_baseline"] = cpu_baseline_prefill()
        res["prefill"] = pf
        legs = {}
        for name in DEFAULT_LEGS:
            legs[name] = WORKLOADS[name](va, dev, _steps(args), args.warmup, pk)
            _free()
        res["workloads"] = legs
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args)
    if rank == 0:
        print(json.dumps(res))
    if ws > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------ CPU baseline

def _oracle_decode_setup():
    import oracle
    b = W.decode_llama8b(device="cpu", pool=16384)
    kc = torch.zeros((b.num_blocks, b.bs, b.Hkv, b.D), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    oracle.kv_write(b.k_tok, b.v_tok, kc, vc, b.slot_mapping)
    return b, kc, vc


def _oracle_decode(b, kc, vc, rows, cores):
    import oracle
    oracle.attention(b.q, kc, vc, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                     causal=True, rows=rows, nthreads=cores)


def _sample_bytes(b, rows):
    kv = sum(b.kv_lens[r] for r in rows) * b.Hkv * b.D * 2 * 2
    return kv + 2 * len(rows) * b.Hq * b.D * 2 + sum((b.kv_lens[r] + b.bs - 1) // b.bs for r in rows) * 4


def cpu_baseline(args, budget_s=10.0):
    """The fp64 oracle on the full decode batch, on this host's cores,
    repeated until about budget_s seconds of CPU work."""
    b, kc, vc = _oracle_decode_setup()
    cores = os.cpu_count() or 1
    rows = list(range(b.B))
    n, t0 = 0, time.perf_counter()
    while n < 30 and (n == 0 or time.perf_counter() - t0 < budget_s):
        _oracle_decode(b, kc, vc, rows, cores)
        n += 1
    dt = (time.perf_counter() - t0) / n
    return {"value": round(decode_bytes(b) / dt / 1e9, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "full decode batch (64 requests x 32 heads, %d cached keys), fp64, %d pass(es), %.2f s/pass"
                      % (sum(b.kv_lens), n, dt)}


def prefill_sample_rows(b, per_request, seed):
    """Seeded query rows of a prefill batch: per request, per_request
    distinct rows in a random order (all of a shorter request's rows).
    Returns one list of packed token indices per request."""
    g = torch.Generator().manual_seed(W.SEED0 + 800 + seed)
    cu = b.cu_seqlens_q.tolist()
    return [[cu[r] + i for i in torch.randperm(cu[r + 1] - cu[r], generator=g)[:per_request].tolist()]
            for r in range(b.B)]


def rows_pairs(b, rows):
    """Unmasked (query, key) pairs of the given packed token rows (causal,
    bottom-right aligned)."""
    cu = b.cu_seqlens_q.tolist()
    pairs = 0
    for t in rows:
        r = max(i for i in range(b.B) if cu[i] <= t and cu[i + 1] > t)
        ql, kv = cu[r + 1] - cu[r], b.kv_lens[r]
        pairs += kv - ql + (t - cu[r]) + 1
    return pairs


def cpu_baseline_prefill(per_request=256, rounds_of=32, budget_s=25.0):
    """The fp64 oracle on the chunked prefill workload, on every host core:
    a seeded sample of up to per_request query rows per request (all heads),
    evaluated in rounds of rounds_of rows per request until the sample is
    done or about budget_s seconds of CPU work have run; the full batch's
    time is extrapolated by the unmasked (query, key) pairs covered."""
    import oracle
    b = W.chunked_prefill(device="cpu")
    kc = torch.zeros((b.num_blocks, b.bs, b.Hkv, b.D), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    oracle.kv_write(b.k_tok, b.v_tok, kc, vc, b.slot_mapping)
    per_req = prefill_sample_rows(b, per_request, seed=3)
    cores = os.cpu_count() or 1
    done, pairs, dt = 0, 0, 0.0
    for k in range(0, per_request, rounds_of):
        rows = sorted(t for rr in per_req for t in rr[k:k + rounds_of])
        if not rows:
            break
        t0 = time.perf_counter()
        oracle.attention(b.q, kc, vc, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                         causal=True, rows=rows, nthreads=cores)
        dt += time.perf_counter() - t0
        done += len(rows)
        pairs += rows_pairs(b, rows)
        if dt >= budget_s:
            break
    fl = 4 * b.D * b.Hq * pairs
    full = prefill_flops(b)
    return {"value": round(fl / dt / 1e12, 5), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": "%d seeded query rows (up to %d per request, all 32 heads) of the chunked prefill batch, "
                      "fp64, %.1f s" % (done, per_request, dt),
            "extrapolated_full_s": round(dt * full / fl, 1)}


def run_reference(args, budget_s=150.0):
    """Reference arm: the fp64 CPU oracle timed on the host cores.  Every
    step is a bounded sample of the decode batch (the first n requests, all
    heads), n chosen so that warm-up plus timed steps take about budget_s."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    b, kc, vc = _oracle_decode_setup()
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    _oracle_decode(b, kc, vc, list(range(b.B)), cores)          # calibration pass
    full = time.perf_counter() - t0
    per_step = budget_s / max(1, args.steps + args.warmup)
    n = max(1, min(b.B, int(b.B * per_step / max(full, 1e-6))))
    rows = list(range(n))
    for _ in range(args.warmup):
        _oracle_decode(b, kc, vc, rows, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_decode(b, kc, vc, rows, cores)
    dt = (time.perf_counter() - t0) / args.steps
    v = _sample_bytes(b, rows) / dt / 1e9
    sample = "first %d of 64 decode requests (all 32 heads) per step, fp64 oracle" % n
    res = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "GB/s", "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": DECODE_WORKLOAD},
           "cpu_baseline": {"value": round(v, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(v, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def run_workload(args):
    """One workload alone on one GPU (its attention calls only)."""
    import varlen_flashattention_causal_gb300 as va
    from varlen_flashattention_causal_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm, tc, _, peak_kind = peaks()
    res = WORKLOADS[args.workload](va, dev, args.steps, args.warmup, (hbm, tc))
    res.update(n_gpus=1, steps=args.steps, warmup=args.warmup, data="synthetic", peak_source=peak_kind,
               name=args.workload)
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-only", action="store_true", help="the decode line alone, without the other legs")
    ap.add_argument("--workload", default="decode", choices=["decode"] + sorted(WORKLOADS),
                    help="decode is the benchmark line (with every other workload as a leg); "
                         "the others print one workload alone")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from oracle.build import build_oracle
    if args.impl == "ours" and args.workload != "decode":
        run_workload(args)
        return
    if args.impl == "reference":
        build_oracle()
        run_reference(args)
    else:
        if not args.no_cpu_baseline:
            build_oracle()
        run_ours(args)


if __name__ == "__main__":
    main()
