#!/usr/bin/env python
"""Benchmark of the KVarN KV-cache hot path on GB300.

Step = one decode step of the ragged serving mix (Qwen3-32B layer: 64 query
heads, 8 KV heads, head_dim 128, fp16; 256 sequences with context lengths
U[128, 32768], never a multiple of 128): append one token per sequence to
the raw open tile (tiles that fill are quantised into their paged block on
the spot), then decode attention of one query per sequence and head over the
packed cache plus the open tile.  Every row of the hot path runs in every
step.  Inputs (the prefilled cache, every step's new tokens and queries) are
resident in HBM before the timed region; the packed cache (~3.5 GB) is far
larger than L2.

Also reported, as components: the 16K-context decode (32 x 16384 tokens) of
the packed kernel beside the in-repo 16-bit paged decode kernel on the same
shapes, and the write-path quantiser on 32 x 16384 x 8 heads of bf16.

With N > 1 GPUs the step is split by KV head (`--shard heads`, the
default): rank r of N owns KV heads [8r/N, 8(r+1)/N) of every sequence,
their query heads, pool, open tiles and output slice, as tensor-parallel
attention would place them; no data crosses ranks.  `--shard replicas` runs
N independent serving batches instead.

`--impl reference` times the CPU oracle (the plain fp64 restatement of the
method) on the host cores on a bounded sample of the same step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn tokens/s & packed-KV HBM GB/s (% of 8 TB/s); quantized tiles/s"
T = D = 128


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.lines, self.proc = gpu, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        time.sleep(0.25)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1])); mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# DRAM bytes actually moved by one decode call per algorithmic byte, from an
# ncu capture of the 16K decode call (32 x 16384 tokens, 64 q / 8 KV heads:
# 446 744 832 B of DRAM traffic for 437 796 992 algorithmic bytes).  The
# serving step's call is too large to capture, and its traffic grows with the
# records it reads.
DECODE_TRAFFIC_PER_BYTE = 446744832 / 437796992


# The quantiser's FP32 work per (tile, head) job: 8 normalisation iterations x
# 2 half-steps x 16384 elements x 3 lane operations (shifted product, sum,
# sum of squares) plus ~6 per element for the row range and the encode.
QUANT_LANE_OPS_PER_JOB = 8 * 2 * 16384 * 3 + 6 * 16384
FP32_LANES_PER_SM = 128          # FP32 lanes of one SM (4 sub-partitions x 32)


def fp32_lane_ops_peak(dev, sm_mhz=None):
    """FP32 lane operations per second of the device: its SM count (from the
    device properties) x 128 lanes x the SM clock (the median sampled under
    load when given, else the device's maximum clock)."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    mhz = sm_mhz
    if not mhz:
        try:
            mhz = float(subprocess.check_output(
                ["nvidia-smi", "-i", str(dev.index), "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits"],
                text=True).strip().splitlines()[0])
        except Exception:
            mhz = 2070.0
    return props.multi_processor_count * FP32_LANES_PER_SM * mhz * 1e6, props.multi_processor_count, mhz


def decode_bytes(lens, w, H=None, Hq=None):
    """Algorithmic bytes of one decode call over H KV heads and Hq query
    heads (default: all of the workload's): packed records of the closed
    tiles, raw open-tile tokens, queries, outputs, block ids and lengths."""
    H = w.num_kv_heads if H is None else H
    Hq = w.num_q_heads if Hq is None else Hq
    closed = sum(n // T for n in lens)
    tail = sum(n % T for n in lens)
    head_rec = 2 * 512 + T * D * (w.k_bits + w.v_bits) // 8   # K and V record of one (tile, head)
    return (closed * H * head_rec + tail * H * 2 * D * 2 + len(lens) * Hq * D * (2 + 4)
            + closed * 4 + len(lens) * 4)


# --------------------------------------------------------------------------- multi-rank host logic
def rank_seed(rank):
    """Seed of rank's own serving batch under `--shard replicas`: every rank
    draws its own sequences, so ranks share no (sequence, KV head) unit and
    exchange no data."""
    return 4 + 1000 * rank


def reduce_max_ms(ms, device=None):
    """The slowest rank's time (MAX all-reduce; a no-op without a process group)."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(batch, steps, world, ms, shard="replicas"):
    """Whole-job throughput in decoded tokens (one per sequence and step) per
    second of the slowest rank: with replicas every rank decodes its own
    batch; with KV-head sharding the ranks decode parts of the same tokens."""
    return batch * steps * (world if shard == "replicas" else 1) / (ms / 1e3)


# --------------------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world):
    import torch
    from bit_kv_cache_quantize_gb300 import build as B
    from bit_kv_cache_quantize_gb300 import inputs as I
    from bit_kv_cache_quantize_gb300 import kvarn as K
    from bit_kv_cache_quantize_gb300.cache import PagedCache

    B.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    from bit_kv_cache_quantize_gb300 import shard as S
    hbm_peak, _, peak_src = measured_peaks()
    steps, warm = args.steps, args.warmup
    n_dec = max(64, steps + warm)
    mode = args.shard if world > 1 else "single"
    w = I.ragged_32b(steps=n_dec, seed=rank_seed(rank) if mode == "replicas" else 4)
    h0, h1 = S.head_range(rank, world, w.num_kv_heads) if mode == "heads" else (0, w.num_kv_heads)
    c = PagedCache(w, dev, heads=(h0, h1))
    c.prefill()
    torch.cuda.synchronize()
    assert c.check_error() == 0, "device error during prefill"

    # every step's inputs, resident before timing (this rank's heads only)
    B_, H, Hq = w.batch, c.H, c.Hq
    qh0, qh1 = h0 * w.G, h1 * w.G
    dt = I.torch_dtype(w.dtype)
    base = torch.tensor(w.seq_lens, dtype=torch.int64)
    pos_all = (base[None, :] + torch.arange(n_dec)[:, None]).to(torch.int32)          # [S, B]
    kn = torch.empty(n_dec, B_, H, D, dtype=dt, device=dev)
    vn = torch.empty_like(kn)
    for b in range(B_):
        kn[:, b] = I.kv_values(w, "k", b, w.seq_lens[b], n_dec, dev, heads=range(h0, h1))
        vn[:, b] = I.kv_values(w, "v", b, w.seq_lens[b], n_dec, dev, heads=range(h0, h1))
    qs = torch.stack([I.queries(w, step=s + 1, device=dev)[:, qh0:qh1] for s in range(n_dec)]).contiguous()
    pos_d = pos_all.to(dev)
    lens_d = (pos_all + 1).to(dev)
    out = torch.empty(B_, Hq, D, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(s):
        c.append(kn[s], vn[s], pos_d[s], stream)
        c.decode(qs[s], out, lens=lens_d[s], stream=stream)

    for s in range(warm):
        step(s)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t0.record(stream)
        for i in range(steps):
            s = warm + i
            c.append(kn[s], vn[s], pos_d[s], stream)
            evs[i][0].record(stream)
            c.decode(qs[s], out, lens=lens_d[s], stream=stream)
            evs[i][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = t0.elapsed_time(t1)
    assert c.check_error() == 0, "device error during the timed steps"
    if world > 1:
        ms = reduce_max_ms(ms, dev)
    dec_ms = [a.elapsed_time(b) for a, b in evs]
    dec_avg_s = sum(dec_ms) / len(dec_ms) / 1e3
    dec_bytes = statistics.mean(decode_bytes([int(x) + 1 for x in pos_all[warm + i]], w, H, Hq)
                                for i in range(steps))
    achieved = dec_bytes / dec_avg_s / 1e9
    shard_mode = "replicas" if mode == "replicas" else "heads"
    tokens_per_s = job_tokens_per_s(B_, steps, world, ms, shard_mode)

    # e2e: the same steps through the public API with host buffers
    e2e = run_e2e(c, w, kn, vn, qs, pos_all, dev, warm, steps)
    if world > 1:
        e2e_ms = reduce_max_ms(e2e["ms_per_step"] * steps, dev)
        e2e["value"] = job_tokens_per_s(B_, steps, world, e2e_ms, shard_mode)
        e2e["ms_per_step"] = e2e_ms / steps
        e2e["h2d_bytes_per_step"] *= world      # every rank copies its own slices
        e2e["d2h_bytes_per_step"] *= world
    parallelism = {"single": "single GPU", "replicas": f"replicas x{world}",
                   "heads": f"KV heads split {world} ways ({H} KV / {Hq} q heads per rank), no collective"}[mode]

    res = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": ms / steps, "higher_is_better": True,
        "scaling": "strong" if mode == "heads" else "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": serving_config(B_, statistics.mean(w.seq_lens), n_dec, parallelism),
        "roofline": {"kernel": "kvarn_decode_attention (split-K decode + combine)", "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "peak_source": peak_src, "traffic": DECODE_TRAFFIC_PER_BYTE * dec_bytes,
                     "traffic_source": "ncu capture of the 16K decode call, scaled by algorithmic bytes",
                     "algorithmic_bytes_per_launch": dec_bytes,
                     "avg_launch_us": dec_avg_s * 1e6},
        "e2e": e2e,
        "gpu_launches": steps * 3,
        "bits_per_element": {"k": 4.25, "v": 2.25, "mean": 3.25, "vs_16bit": 16 / 3.25},
    }
    del c, kn, vn, qs
    torch.cuda.empty_cache()
    res["clocks"] = clk.summary()
    if not args.no_components and rank == 0:
        res["components"] = components(dev, hbm_peak, measured_peaks()[1], res["clocks"].get("sm_mhz"))
    return res


def run_e2e(c, w, kn, vn, qs, pos_all, dev, warm, steps):
    """Serving steps through the public API with host buffers: each step's new
    K/V tokens, queries and positions are copied from pinned host memory and
    its output read back, the copies on their own streams and double
    buffered so that they overlap the neighbouring steps' compute (step i's
    inputs land while step i-1 computes, its output drains while step i+1
    computes).  The timed region runs from the first upload to the last
    download."""
    import torch
    hk = kn.cpu().pin_memory(); hv = vn.cpu().pin_memory(); hq = qs.cpu().pin_memory()
    hp = pos_all.pin_memory(); hl = (pos_all + 1).pin_memory()
    Hq = qs.shape[2]                          # query heads of this rank
    hout = [torch.empty(w.batch, Hq, D, dtype=torch.float32).pin_memory() for _ in range(2)]
    bufs = []
    for _ in range(2):
        bufs.append(dict(k=torch.empty_like(kn[0]), v=torch.empty_like(vn[0]), q=torch.empty_like(qs[0]),
                         p=torch.empty(w.batch, dtype=torch.int32, device=dev),
                         l=torch.empty(w.batch, dtype=torch.int32, device=dev),
                         o=torch.empty(w.batch, Hq, D, dtype=torch.float32, device=dev)))
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    b0 = bufs[0]
    h2d = b0["k"].numel() * b0["k"].element_size() * 2 + b0["q"].numel() * b0["q"].element_size() + b0["p"].numel() * 8
    d2h = b0["o"].numel() * 4

    def run(first, n):
        for i in range(n):
            s, j = first + i, i & 1
            bj = bufs[j]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(in_free[j])
                bj["k"].copy_(hk[s], non_blocking=True); bj["v"].copy_(hv[s], non_blocking=True)
                bj["q"].copy_(hq[s], non_blocking=True); bj["p"].copy_(hp[s], non_blocking=True)
                bj["l"].copy_(hl[s], non_blocking=True)
                in_ready[j].record(up)
            comp.wait_event(in_ready[j])
            if i >= 2:
                comp.wait_event(out_free[j])
            c.append(bj["k"], bj["v"], bj["p"], comp)
            c.decode(bj["q"], bj["o"], lens=bj["l"], stream=comp)
            in_free[j].record(comp)
            out_ready[j].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(out_ready[j])
                hout[j].copy_(bj["o"], non_blocking=True)
                out_free[j].record(down)
        comp.wait_stream(down)

    # replay the same positions: the state a step writes is the state it reads
    run(0, warm)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    up.wait_stream(comp)
    run(warm, steps)
    b.record(comp)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    return {"value": w.batch * steps / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / steps,
            "copies": "own streams, double buffered, overlapping the neighbouring steps' compute"}


def flush_l2(buf):
    buf.zero_()


def components(dev, hbm_peak, bf16_peak, sm_mhz=None):
    """16K decode (packed vs 16-bit kernel) and the prefill quantiser."""
    import torch
    from bit_kv_cache_quantize_gb300 import inputs as I
    from bit_kv_cache_quantize_gb300 import kvarn as K
    from bit_kv_cache_quantize_gb300.cache import PagedCache

    out = {}
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # 2 x L2
    stream = torch.cuda.current_stream()

    def timed(fn, reps):
        ts = []
        for _ in range(3):
            fn()
        for _ in range(reps):
            flush_l2(scratch)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream); fn(); b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) / 1e3)
        return statistics.median(ts)

    # --- 16K decode: packed KVarN vs 16-bit paged kernel, same table and shapes
    w = I.qwen3_32b()
    c = PagedCache(w, dev, fp16_pool=True)
    c.prefill()
    q = I.queries(w, device=dev)
    o = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    t_pk = timed(lambda: c.decode(q, o), 50)
    t_16 = timed(lambda: c.decode_fp16(q, o), 20)
    b_pk = decode_bytes(w.seq_lens, w)
    b_16 = sum(w.seq_lens) * w.num_kv_heads * 2 * D * 2 + w.batch * w.num_q_heads * D * 6
    assert c.check_error() == 0
    # --- multi-query: the last 16 tokens of every sequence as causal queries
    #     (a prefill chunk / speculative verify), one call vs 16 decode calls
    Qn = 16
    qm = I.multi_queries(w, Qn, device=dev)
    om = torch.empty(w.batch, Qn, w.num_q_heads, D, dtype=torch.float32, device=dev)
    t_mq = timed(lambda: c.multiquery(qm, Qn, om), 20)
    lens_i = [c.lens - (Qn - 1 - i) for i in range(Qn)]
    qd = [qm[:, i].contiguous() for i in range(Qn)]
    od = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    t_dq = timed(lambda: [c.decode(qd[i], od, lens=lens_i[i]) for i in range(Qn)], 5)
    assert c.check_error() == 0
    L = w.seq_lens[0]
    flops = 4 * D * w.batch * w.num_q_heads * sum(L - Qn + i + 1 for i in range(Qn))
    out["multiquery_16k"] = {
        "workload": "qwen3_32b_decode_16k cache, last 16 tokens of each of the 32 sequences as causal queries "
                    "(16 x 8 GQA rows = one 128-row block per KV head)",
        "us": t_mq * 1e6, "query_tokens_per_s": w.batch * Qn / t_mq,
        "algorithmic_tflops": flops / t_mq / 1e12, "frac_bf16_peak": flops / t_mq / 1e12 / bf16_peak,
        "executed_over_algorithmic": 2.25, "bytes": b_pk, "GBps": b_pk / t_mq / 1e9,
        "sixteen_decode_calls_us": t_dq * 1e6, "speedup_vs_decode_calls": t_dq / t_mq,
    }
    out["decode_16k"] = {
        "workload": "qwen3_32b_decode_16k: 32 seqs x 16384 tokens, 64 q / 8 KV heads, fp16, permuted blocks",
        "kvarn_us": t_pk * 1e6, "kvarn_tokens_per_s": w.batch / t_pk, "kvarn_GBps": b_pk / t_pk / 1e9,
        "kvarn_frac_hbm": b_pk / t_pk / 1e9 / hbm_peak, "kvarn_bytes": b_pk,
        "fp16_us": t_16 * 1e6, "fp16_tokens_per_s": w.batch / t_16, "fp16_GBps": b_16 / t_16 / 1e9,
        "fp16_frac_hbm": b_16 / t_16 / 1e9 / hbm_peak, "fp16_bytes": b_16,
        "speedup_vs_fp16": t_16 / t_pk,
        "context_tokens_per_s": w.batch * w.seq_lens[0] / t_pk,
    }
    del c
    torch.cuda.empty_cache()

    # --- the same decode over 2-bit keys (K2/V2 records, 9216 B per tile and head)
    w.k_bits = 2
    c = PagedCache(w, dev)
    c.prefill()
    t_k2 = timed(lambda: c.decode(q, o), 50)
    b_k2 = decode_bytes(w.seq_lens, w)
    assert c.check_error() == 0
    out["decode_16k_k2v2"] = {
        "workload": "qwen3_32b_decode_16k with 2-bit keys and values (K2/V2 records)",
        "us": t_k2 * 1e6, "tokens_per_s": w.batch / t_k2, "GBps": b_k2 / t_k2 / 1e9,
        "frac_hbm": b_k2 / t_k2 / 1e9 / hbm_peak, "bytes": b_k2, "speedup_vs_fp16": t_16 / t_k2,
    }
    del c
    torch.cuda.empty_cache()

    # --- the same decode over 4-bit values (K4/V4 records, 17408 B per tile and head)
    w.k_bits, w.v_bits = 4, 4
    c = PagedCache(w, dev)
    c.prefill()
    t_v4 = timed(lambda: c.decode(q, o), 50)
    b_v4 = decode_bytes(w.seq_lens, w)
    assert c.check_error() == 0
    out["decode_16k_k4v4"] = {
        "workload": "qwen3_32b_decode_16k with 4-bit keys and values (K4/V4 records)",
        "us": t_v4 * 1e6, "tokens_per_s": w.batch / t_v4, "GBps": b_v4 / t_v4 / 1e9,
        "frac_hbm": b_v4 / t_v4 / 1e9 / hbm_peak, "bytes": b_v4, "speedup_vs_fp16": t_16 / t_v4,
    }
    del c, q, o
    torch.cuda.empty_cache()

    # --- one tile (latency of a quantise call and a decode call)
    w = I.single_tile()
    c = PagedCache(w, dev)
    k1 = I.kv_sequence(w, "k", 0, T, dev)
    v1 = I.kv_sequence(w, "v", 0, T, dev)
    q1 = I.queries(w, device=dev)
    o1 = torch.empty(1, 1, D, dtype=torch.float32, device=dev)
    t_q1 = timed(lambda: c.quantize_sequence(0, k1, v1), 50)
    t_d1 = timed(lambda: c.decode(q1, o1), 50)
    assert c.check_error() == 0
    out["single_tile"] = {"workload": "1 KV head, 1 query head, 128 tokens, fp16: latency of one call",
                          "quantize_us": t_q1 * 1e6, "decode_us": t_d1 * 1e6}
    del c

    # --- Qwen3-4B-shaped layer decode: 8 x 4096 tokens, 32 q / 8 KV heads, bf16 (27 MB packed: L2 flushed)
    w = I.qwen3_4b()
    c = PagedCache(w, dev)
    c.prefill()
    q4 = I.queries(w, device=dev)
    o4 = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    t_4b = timed(lambda: c.decode(q4, o4), 50)
    b_4b = decode_bytes(w.seq_lens, w)
    assert c.check_error() == 0
    out["decode_qwen3_4b"] = {"workload": "qwen3_4b_layer: 8 seqs x 4096 tokens, 32 q / 8 KV heads, bf16",
                              "us": t_4b * 1e6, "tokens_per_s": w.batch / t_4b, "GBps": b_4b / t_4b / 1e9,
                              "frac_hbm": b_4b / t_4b / 1e9 / hbm_peak, "bytes": b_4b}
    del c
    torch.cuda.empty_cache()

    # --- write path: quantise 32 x 16384 tokens x 8 heads of bf16 (65536 tile jobs)
    w = I.prefill_32b()
    c = PagedCache(w, dev)
    Bn, n = w.batch, w.seq_lens[0]
    k = torch.empty(Bn * n, w.num_kv_heads, D, dtype=I.torch_dtype(w.dtype), device=dev)
    v = torch.empty_like(k)
    for b in range(Bn):
        k[b * n:(b + 1) * n] = I.kv_sequence(w, "k", b, n, dev)
        v[b * n:(b + 1) * n] = I.kv_sequence(w, "v", b, n, dev)
    n_tiles = Bn * n // T
    first = torch.arange(n_tiles, dtype=torch.int64, device=dev) * T
    dst = c.table[:, : n // T].reshape(-1).contiguous()
    fn = lambda: K.kvarn_quantize_tiles(c.cfg, k, v, w.num_kv_heads * D, Bn * n, first, dst, n_tiles, c.pool,
                                        c.err)
    t_q = timed(fn, 10)
    assert c.check_error() == 0
    jobs = n_tiles * w.num_kv_heads * 2
    byt = jobs * (T * D * 2) + n_tiles * w.num_kv_heads * 13312 + n_tiles * 12
    alu_ops = jobs * QUANT_LANE_OPS_PER_JOB
    alu_peak, sms, mhz = fp32_lane_ops_peak(dev, sm_mhz)
    out["quantizer"] = {
        "workload": "prefill_32b_16k: 32 x 16384 tokens x 8 KV heads, bf16, K and V tiles (65536 tile jobs)",
        "us": t_q * 1e6, "tiles_per_s": jobs / t_q, "GBps": byt / t_q / 1e9, "frac_hbm": byt / t_q / 1e9 / hbm_peak,
        "bytes": byt,
        "alu": {"bound": "alu", "lane_ops_per_job": QUANT_LANE_OPS_PER_JOB, "achieved_tops": alu_ops / t_q / 1e12,
                "peak_tops": alu_peak / 1e12, "frac": alu_ops / t_q / alu_peak,
                "peak_basis": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x {mhz:.0f} MHz"},
    }
    return out


# --------------------------------------------------------------------------- CPU oracle
def oracle_step_sample(n_seqs, seed=4, threads=None):
    """Prepare a bounded sample of the serving step for the oracle: n_seqs
    sequences of the ragged mix with their packed cache (oracle-quantised)."""
    import numpy as np
    import torch
    import oracle as O
    from bit_kv_cache_quantize_gb300 import inputs as I

    w = I.ragged_32b(seed=seed)
    seqs = list(range(n_seqs))
    units = []
    for b in seqs:
        n = w.seq_lens[b]
        k = I.kv_sequence(w, "k", b, n + 1)
        v = I.kv_sequence(w, "v", b, n + 1)
        kb = k.view(torch.int16).numpy().view(np.uint16)
        vb = v.view(torch.int16).numpy().view(np.uint16)
        nf = (n + 1) // T
        for h in range(w.num_kv_heads):
            first = np.array([t * T * w.num_kv_heads * D + h * D for t in range(nf)], np.int64)
            kr, _ = O.quantize_batch(kb, "f16", first, w.num_kv_heads * D, False, nthreads=threads)
            vr, _ = O.quantize_batch(vb, "f16", first, w.num_kv_heads * D, True, nthreads=threads)
            units.append(dict(q=None, krec=list(kr), vrec=list(vr),
                              ktail=O.decode16(kb[nf * T:n + 1, h], "f16").reshape(-1, D),
                              vtail=O.decode16(vb[nf * T:n + 1, h], "f16").reshape(-1, D), b=b, h=h))
    q = I.queries(w, step=1)
    for u in units:
        u["q"] = O.decode16(q[u["b"], u["h"] * w.G:(u["h"] + 1) * w.G].contiguous().view(torch.int16).numpy()
                            .view(np.uint16), "f16")
    return w, units


def oracle_step(w, units, threads):
    import numpy as np
    import oracle as O
    G = w.G
    qa = np.stack([u["q"] for u in units])
    kt = np.zeros((len(units), T, D)); vt = np.zeros((len(units), T, D))
    nt = np.zeros(len(units), np.int32)
    for i, u in enumerate(units):
        m = u["ktail"].shape[0]
        kt[i, :m] = u["ktail"]; vt[i, :m] = u["vtail"]; nt[i] = m
    return O.attention_batch(qa, [u["krec"] for u in units], [u["vrec"] for u in units], kt, vt, nt, w.scale,
                             nthreads=threads)


def oracle_quantize_sample(n_seqs, threads):
    """The oracle quantiser on the first n_seqs sequences of the 32 x 16K
    bf16 prefill (every K and V tile of their 8 KV heads): (tile jobs per
    second, jobs, seconds).  Inputs are generated on the GPU when there is
    one (faster) and handed to the oracle as host bytes."""
    import numpy as np
    import torch
    import oracle as O
    from bit_kv_cache_quantize_gb300 import inputs as I
    w = I.prefill_32b()
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    n, H = w.seq_lens[0], w.num_kv_heads
    first = np.array([t * T * H * D + h * D for t in range(n // T) for h in range(H)], np.int64)
    srcs = []
    for b in range(n_seqs):
        for which in ("k", "v"):
            x = I.kv_sequence(w, which, b, n, gen).cpu()
            srcs.append((x.view(torch.int16).numpy().view(np.uint16).reshape(-1), which == "v"))
    t0 = time.perf_counter()
    for bits, is_v in srcs:
        O.quantize_batch(bits, "bf16", first, H * D, is_v, nthreads=threads)
    dt = time.perf_counter() - t0
    jobs = len(srcs) * len(first)
    return jobs / dt, jobs, dt


def cpu_baseline(n_seqs=4, reps=1, quant_seqs=4):
    threads = os.cpu_count() or 1
    w, units = oracle_step_sample(n_seqs, threads=threads)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(w, units, threads)
    dt = (time.perf_counter() - t0) / reps
    ctx = sum(w.seq_lens[:n_seqs])
    qrate, qjobs, qdt = oracle_quantize_sample(quant_seqs, threads)
    return {"value": n_seqs / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"decode step (attention over the packed cache + open tile, folded fp64 form) of "
                      f"{n_seqs} sequences x 8 KV heads x 8 queries of the ragged serving mix "
                      f"({ctx} context tokens); {dt:.2f} s per step on {threads} threads",
            "quantize_tiles_per_s": qrate,
            "quantize_sample": f"write path (rotation, 8 Sinkhorn iterations, scales, codes, packing) of every K and "
                               f"V tile of {quant_seqs} of the 32 x 16384-token bf16 prefill sequences x 8 KV heads "
                               f"({qjobs} tile jobs) in {qdt:.2f} s on {threads} threads"}


def serving_config(batch, mean_context, n_dec, parallelism):
    """The `config` object of the serving-step line (both arms)."""
    return {"workload": "ragged_32b_serving: 256 seqs, context U[128,32768] (never a multiple of 128), "
                        "Qwen3-32B layer 64 q / 8 KV heads, head_dim 128, fp16 inputs, K4/V2 "
                        "128-token tiles, 8 Sinkhorn iterations; step = append 1 token/seq "
                        "(close+quantise full tiles) + decode attention",
            "batch": batch, "mean_context": mean_context,
            "decode_steps_appended": n_dec, "l2": "inputs larger than L2 (packed cache ~3.5 GB)",
            "parallelism": parallelism}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    threads = os.cpu_count() or 1
    w, units = oracle_step_sample(args.ref_seqs, threads=threads)
    for _ in range(args.warmup):
        oracle_step(w, units, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, units, threads)
    dt = time.perf_counter() - t0
    v = args.ref_seqs * args.steps / dt
    sample = (f"{args.ref_seqs} sequences x 8 KV heads x 8 queries of the ragged serving mix per step, "
              f"CPU oracle (fp64 folded attention) on {threads} threads")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "strong" if world > 1 and args.shard == "heads" else "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": serving_config(len(w.seq_lens), statistics.mean(w.seq_lens), max(64, args.steps + args.warmup),
                                     "single GPU" if world == 1 else
                                     f"replicas x{world}" if args.shard == "replicas" else
                                     f"KV heads split {world} ways ({8 // world} KV / {64 // world} q heads per rank), "
                                     "no collective"),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_case(name, launches):
    """Small single-kernel workloads for ncu captures (each > L2, a few GB at
    most): the 16K decode (436 MB packed; 570 MB with the K4/V4 preset), the
    16-bit decode on the same shapes (2.1 GB), the quantiser on 4 of the 32
    prefill sequences, or the serving step's append (256 sequences x 8 KV
    heads with the ragged mix's open-tile fill, two of them closing a tile;
    134 MB of open tiles)."""
    import torch
    from bit_kv_cache_quantize_gb300 import build as B
    from bit_kv_cache_quantize_gb300 import inputs as I
    from bit_kv_cache_quantize_gb300 import kvarn as K
    from bit_kv_cache_quantize_gb300.cache import PagedCache
    B.build()
    dev = torch.device("cuda", 0)
    if name in ("decode16k", "decode16k_k4v4", "fp16"):
        w = I.qwen3_32b()
        if name == "decode16k_k4v4":
            w.v_bits = 4
        c = PagedCache(w, dev, fp16_pool=(name == "fp16"))
        c.prefill()
        q = I.queries(w, device=dev)
        o = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
        fn = (lambda: c.decode_fp16(q, o)) if name == "fp16" else (lambda: c.decode(q, o))
    elif name == "multiquery16k":
        w = I.qwen3_32b()
        c = PagedCache(w, dev)
        c.prefill()
        q = I.multi_queries(w, 16, device=dev)
        o = torch.empty(w.batch, 16, w.num_q_heads, D, dtype=torch.float32, device=dev)
        fn = lambda: c.multiquery(q, 16, o)
    elif name == "append":
        full = I.ragged_32b()
        r = [n % T for n in full.seq_lens]
        s = next(s for s in range(T) if sum((x + s) % T == T - 1 for x in r) == 2)
        lens = [T + (x + s) % T for x in r]  # the mix's open-tile fill s steps on, over one closed tile
        w = I.Workload("append_ragged_mix", full.batch, full.num_q_heads, full.num_kv_heads, full.dtype, lens,
                       seed=full.seed, decode_steps=1, max_tokens=2 * T, block_perm=True)
        c = PagedCache(w, dev)
        c.prefill()
        pos = torch.tensor(lens, dtype=torch.int32, device=dev)
        kn = torch.stack([I.kv_values(w, "k", b, lens[b], 1, dev)[0] for b in range(w.batch)])
        vn = torch.stack([I.kv_values(w, "v", b, lens[b], 1, dev)[0] for b in range(w.batch)])
        fn = lambda: c.append(kn, vn, pos)
    else:
        w = I.prefill_32b()
        w.batch = 4
        w.seq_lens = w.seq_lens[:4]
        c = PagedCache(w, dev)
        Bn, n = w.batch, w.seq_lens[0]
        k = torch.cat([I.kv_sequence(w, "k", b, n, dev) for b in range(Bn)])
        v = torch.cat([I.kv_sequence(w, "v", b, n, dev) for b in range(Bn)])
        nt = Bn * n // T
        first = torch.arange(nt, dtype=torch.int64, device=dev) * T
        dst = c.table[:, : n // T].reshape(-1).contiguous()
        fn = lambda: K.kvarn_quantize_tiles(c.cfg, k, v, w.num_kv_heads * D, Bn * n, first, dst, nt, c.pool, c.err)
    torch.cuda.synchronize()
    for _ in range(launches):
        fn()
    torch.cuda.synchronize()
    assert c.check_error() == 0
    print(json.dumps({"profile_case": name, "launches": launches}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="kvarn", choices=["kvarn", "reference"])
    ap.add_argument("--shard", default="heads", choices=["heads", "replicas"],
                    help="N > 1: split the step's KV heads over the ranks, or run N independent batches")
    ap.add_argument("--no-components", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seqs", type=int, default=16)
    ap.add_argument("--cpu-quant-seqs", type=int, default=8)
    ap.add_argument("--ref-seqs", type=int, default=4)
    ap.add_argument("--profile-case", choices=["decode16k", "decode16k_k4v4", "fp16", "quantize", "multiquery16k", "append"], default=None)
    ap.add_argument("--profile-launches", type=int, default=3)
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args.profile_case, args.profile_launches)
        return
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if world > 1 and args.impl != "reference":
        import torch
        torch.distributed.init_process_group("nccl")
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_gpu(args, rank, world)
        if rank == 0 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.cpu_seqs, quant_seqs=args.cpu_quant_seqs)
    if rank == 0 and res is not None:
        print(json.dumps(res))
    if world > 1 and args.impl != "reference":
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
