#!/usr/bin/env python
"""Benchmark of the paged KV cache hot path on GB300.

Headline: paged decode attention KV-read GB/s (and sequences/s) at the LLaMA-2-7B layer shape
-- 32 sequences, 32 query = 32 KV heads, head_dim 128, fp16, block_size 16, context lengths
uniform in [1, 4096], physical blocks from a seeded permutation of a pool sized 110% of need.
One step = one pass of the decode hot path over that batch: slot indexing of the 32 new tokens
-> paged append of their K/V -> split-K paged decode attention over L+1 tokens -> split merge.
value = KV bytes the attention reads per step (sum(L+1) x 32 heads x 128 x 2 B x 2) / step time.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): each rank runs its own batch (seed + rank), weak scaling,
no collective on the data path; value = all ranks' KV bytes / the slowest rank's time.
--impl reference times the CPU oracle (fp64 C) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import copy
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV-read GB/s and seqs/s at 7B shape; % of GB300 HBM peak"
WORKLOAD = ("LLaMA-2-7B-shape single-layer paged decode: 32 seqs, 32 q heads = 32 KV heads, head_dim 128, "
            "fp16, block_size 16, context U[1,4096] + 1 appended token, pool 110% of need, permuted block ids")


def _recorded_traffic(profile_md: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current kernel source."""
    import hashlib
    import re
    try:
        text = open(os.path.join(ROOT, "profiles", profile_md)).read()
        src, digest = re.search(r"counters-for: (\S+) sha256=([0-9a-f]{64})", text).groups()
        traffic = int(re.search(r"traffic_per_launch_bytes: (\d+)", text).group(1))
        with open(os.path.join(ROOT, src), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
        return traffic
    except Exception:
        return None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str):
        self.path = path
        self.proc = None
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def wait_running(self, limit_s: float = 10.0):
        """Until nvidia-smi has written its first sample (its start-up talks to the driver at length,
        which would otherwise fall into the timed region), or it has exited, or limit_s has passed."""
        if self.proc is None:
            return
        t0 = time.time()
        while time.time() - t0 < limit_s and self.proc.poll() is None:
            self.f.flush()
            try:
                if os.path.getsize(self.path) > 0:
                    break
            except OSError:
                break
            time.sleep(0.02)
        time.sleep(0.1) # past the first sample's own driver queries

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _reduce_max(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _reduce_sum(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(local_bytes: float, local_seqs: float, local_elapsed_s: float, ws: int):
    """Weak-scaling totals: (GB/s over all ranks, seqs/s over all ranks, slowest rank's seconds).

    Every rank runs its own batch; the job's throughput is all ranks' work over the slowest rank's
    time (the only cross-rank traffic is these three reductions, none on the data path)."""
    elapsed = _reduce_max(local_elapsed_s, ws)
    total_bytes = _reduce_sum(local_bytes, ws)
    total_seqs = _reduce_sum(local_seqs, ws)
    return total_bytes / elapsed / 1e9, total_seqs / elapsed, elapsed


def _barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------------------------- CPU oracle

def oracle_decode_rate(w, budget_s: float, max_seqs=None):
    """Time the fp64 CPU oracle on a decode pass over a subset of the batch.

    Returns (GB/s of KV read, seconds per pass, sequences in the sample, threads)."""
    import oracle
    from oracle import steps
    nseq = w.num_seqs if max_seqs is None else max(1, min(w.num_seqs, max_seqs))
    r = steps.decode_step(w)   # builds the oracle's own pool (slots + appends), untimed
    lens = w.decode_lens.copy()
    lens[nseq:] = 0
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.paged_decode(w.q, w.model_dtype, r["pool"], oracle.contiguous_strides(w.num_blocks, w.num_kv_heads,
                                                                                      w.block_size, w.head_dim),
                            w.kv_dtype, w.num_blocks, w.block_tables, lens, w.num_kv_heads, w.block_size,
                            float(w.scale), w.k_scale, w.v_scale)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = (time.perf_counter() - t0) / reps
    kv = int(lens.sum()) * w.num_kv_heads * w.head_dim * 2 * 2
    return kv / dt / 1e9, dt, nseq, oracle.num_threads(), reps


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_134_gb300 import workloads as W
    oracle.build()
    w = W.decode7b()
    # size each step: a subset of the sequences so that warmup + steps stay within ~60 s
    _, t_full, _, threads, _ = oracle_decode_rate(w, 0.0)
    per_step = 60.0 / max(1, args.steps + args.warmup)
    nseq = max(1, min(w.num_seqs, int(w.num_seqs * per_step / max(t_full, 1e-9))))
    from oracle import steps
    import oracle as O
    r = steps.decode_step(w)
    lens = w.decode_lens.copy()
    lens[nseq:] = 0
    st = O.contiguous_strides(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)

    def step():
        O.paged_decode(w.q, w.model_dtype, r["pool"], st, w.kv_dtype, w.num_blocks, w.block_tables, lens,
                       w.num_kv_heads, w.block_size, float(w.scale))

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    kv = int(lens.sum()) * w.num_kv_heads * w.head_dim * 2 * 2
    gbs = kv / dt / 1e9
    sample = f"decode attention of the first {nseq} of {w.num_seqs} sequences per step (KV {kv / 1e6:.1f} MB)"
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "seqs_per_s": round(nseq / dt, 3),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------------------------- GPU path

def _time_loop(fn, steps, stream):
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / 1e3


class L2Flush:
    """Reads a device buffer of twice the L2 size, so that the next kernel finds none of its inputs
    in L2.  A read leaves L2 holding clean lines: the dirty lines of the previous launch are written
    back during the flush, not during the next timed kernel (a flush that writes its buffer would
    leave 2 x L2 of dirty lines to be written back inside the timed launch).  Called between timed
    launches, outside the library's events around its kernels."""

    def __init__(self):
        l2 = int(getattr(torch.cuda.get_device_properties(torch.cuda.current_device()), "L2_cache_size", 0) or
                 (128 << 20))
        self.bytes = 2 * l2
        self.buf = torch.zeros(self.bytes // 4, dtype=torch.int32, device="cuda")
        self.acc = torch.zeros((), dtype=torch.int64, device="cuda")

    def __call__(self):
        torch.sum(self.buf, dim=0, dtype=torch.int64, out=self.acc)


def _kernel_loop_flushed(fn, reps, flush):
    """reps calls of fn, each after an L2 flush (the library's own events time its kernels)."""
    for _ in range(reps):
        flush()
        fn()
    torch.cuda.synchronize()


def secondary_prefill(P, W, gpu_path, peaks, reps=20, flush=None):
    """Packed causal prefill of 5256 tokens (lengths 128..2048), 32 heads, D=128, fp16, bs=16."""
    w = W.prefill()
    md = gpu_path.TORCH_DT[w.dtype]
    cache = gpu_path.new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.dtype, w.dtype)
    q, k, v = gpu_path.dev(w.q, md), gpu_path.dev(w.k, md), gpu_path.dev(w.v, md)
    cu, tables = gpu_path.dev(w.cu_seqlens), gpu_path.dev(w.block_tables)
    out = torch.empty_like(q)

    def step():
        P.packed_prefill_attention(q, k, v, cu, w.max_seqlen, tables, cache, float(w.scale), out=out)

    try:
        for _ in range(3):
            step()
        torch.cuda.synchronize()
    except Exception as e:  # reported, not hidden
        cache.close()
        return {"status": f"unavailable: {e}"}
    dt = _time_loop(step, reps, torch.cuda.current_stream()) / reps   # back to back, no events
    flush = flush or L2Flush()
    cache.profile_start(kinds=("prefill",))
    _kernel_loop_flushed(step, reps, flush)
    prof = cache.profile_read()
    err = cache.check_error()
    cache.close()
    kern = prof["prefill_ms"] / max(1, prof["prefill_launches"]) / 1e3
    tflops = w.flops() / kern / 1e12
    return {"workload": "packed causal prefill, lengths 128,200,512,1024,2048,256,64,1024 (5256 tokens), "
                        "32 heads, D=128, fp16, bs=16", "tokens_per_s": round(w.total_tokens / kern, 1),
            "ms_back_to_back": round(dt * 1e3, 4), "kernel_ms": round(kern * 1e3, 4), "tflops": round(tflops, 2),
            "causal_gflop": round(w.flops() / 1e9, 3), "l2": "flushed before each timed launch",
            "frac_of_bf16_peak": round(tflops / peaks[1], 4), "device_errors": err}


def secondary_decode(P, G, peaks, w, reps=50, unique_bytes=None, cascade=0):
    """Decode step (append_at + decode + merge) on another configuration; decode kernel timed by events.
    cascade > 0: the tables share that many tokens and the step runs the cascade decode (prefix phase
    on the tensor cores + suffix split-K decode + merge); its kernels are summed."""
    cache = G.new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, w.model_dtype,
                        w.k_scale, w.v_scale)
    G.fill_cache(cache, w)
    x = G.DecodeInputs(w)
    cache.reserve(w.num_seqs, w.num_q_heads, w.max_blocks)
    for _ in range(5):
        G.decode_step(cache, x, cascade_prefix=cascade)
    torch.cuda.synchronize()
    # the step without events (they would stop the kernels' overlap), then the kernels with events
    t = _time_loop(lambda: G.decode_step(cache, x, cascade_prefix=cascade), reps, torch.cuda.current_stream()) / reps
    cache.profile_start(kinds=("decode", "prefill") if cascade else ("decode",))
    _time_loop(lambda: G.decode_step(cache, x, cascade_prefix=cascade), reps, torch.cuda.current_stream())
    prof = cache.profile_read()
    err = cache.check_error()
    cache.close()
    kern = prof["decode_ms"] / max(1, prof["decode_launches"]) / 1e3
    if cascade:   # prefix phase (recorded as the prefill kind) + suffix decode kernel
        kern += prof["prefill_ms"] / max(1, prof["prefill_launches"]) / 1e3
    kv = w.kv_read_bytes()
    r = {"kv_dtype": w.kv_dtype, "block_size": w.block_size, "num_seqs": w.num_seqs,
         "heads": f"{w.num_q_heads}/{w.num_kv_heads}", "kv_bytes": kv, "step_us": round(t * 1e6, 2),
         "decode_kernel_us": round(kern * 1e6, 2), "kv_gbs": round(kv / kern / 1e9, 1),
         "frac_of_hbm": round(kv / kern / 1e9 / peaks[0], 4), "seqs_per_s": round(w.num_seqs / t, 1),
         "device_errors": err}
    if unique_bytes is not None:
        r["kv_gbs_label"] = "logical (shared prefix re-read per sequence, mostly L2 hits)"
        r["unique_kv_bytes"] = unique_bytes
        r["unique_kv_gbs"] = round(unique_bytes / kern / 1e9, 1)
        r["unique_frac_of_hbm"] = round(unique_bytes / kern / 1e9 / peaks[0], 4)
        r["unique_kv_gbs_per_step"] = round(unique_bytes / t / 1e9, 1)
    return r


def secondary_append(P, W, gpu_path, peaks, reps=20, flush=None):
    """Bulk paged append of 5256 tokens x 32 heads x 128 fp16 (86 MB read + 86 MB written)."""
    w = W.prefill()
    md = gpu_path.TORCH_DT[w.dtype]
    cache = gpu_path.new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.dtype, w.dtype)
    k, v = gpu_path.dev(w.k, md), gpu_path.dev(w.v, md)
    seq = np.repeat(np.arange(len(w.lengths), dtype=np.int32), w.lengths)
    pos = np.concatenate([np.arange(n, dtype=np.int32) for n in w.lengths])
    slots = P.paged_slot_mapping(gpu_path.dev(w.block_tables), gpu_path.dev(seq), gpu_path.dev(pos), w.block_size)
    for _ in range(3):
        P.paged_kv_append(cache, k, v, slots)
    torch.cuda.synchronize()
    flush = flush or L2Flush()
    cache.profile_start(kinds=("append",))
    _kernel_loop_flushed(lambda: P.paged_kv_append(cache, k, v, slots), reps, flush)
    prof = cache.profile_read()
    cache.close()
    kern = prof["append_ms"] / max(1, prof["append_launches"]) / 1e3
    nbytes = 2 * (k.numel() + v.numel()) * 2 + slots.numel() * 8
    return {"workload": "bulk append of 5256 tokens, 32 KV heads, D=128, fp16", "kernel_ms": round(kern * 1e3, 4),
            "gbs": round(nbytes / kern / 1e9, 1), "frac_of_hbm": round(nbytes / kern / 1e9 / peaks[0], 4),
            "algorithmic_bytes": nbytes, "l2": "flushed before each timed launch"}


def secondary_prefix_hit(P, W, G, peaks, reps=20, flush=None):
    """Prefill of 16 prompt tails (U{100..300} + 12 tokens) over a cached, shared 1488-token prefix,
    7B shape (32/32 heads, D=128, fp16, bs=16): ranged append of the tails + attention over the pool."""
    w = W.prefix_hit_prefill()
    cache = G.new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.dtype, w.dtype)
    G.fill_context(cache, w)
    x = G.ContextPrefillInputs(w)
    for _ in range(3):
        G.context_prefill_step(cache, x)
    torch.cuda.synchronize()
    dt = _time_loop(lambda: G.context_prefill_step(cache, x), reps, torch.cuda.current_stream()) / reps
    flush = flush or L2Flush()
    cache.profile_start(kinds=("prefill", "append"))
    _kernel_loop_flushed(lambda: G.context_prefill_step(cache, x), reps, flush)
    prof = cache.profile_read()
    err = cache.check_error()
    cache.close()
    kern = prof["prefill_ms"] / max(1, prof["prefill_launches"]) / 1e3
    app = prof["append_ms"] / max(1, prof["append_launches"]) / 1e3
    tflops = w.flops() / kern / 1e12
    return {"workload": "16 prompt tails (12 + U{100..300} tokens) over a cached 1488-token prefix shared by every "
                        "table, 32/32 heads, D=128, fp16, bs=16", "tail_tokens": w.total_tokens,
            "tokens_per_s": round(w.total_tokens / dt, 1), "ms_back_to_back": round(dt * 1e3, 4),
            "attention_kernel_ms": round(kern * 1e3, 4), "append_kernel_ms": round(app * 1e3, 4),
            "l2": "flushed before each timed call",
            "gflop": round(w.flops() / 1e9, 3), "tflops": round(tflops, 2),
            "frac_of_bf16_peak": round(tflops / peaks[1], 4), "device_errors": err}


def secondary_blocks(P, W, G, peaks, reps=20, nblocks=512, flush=None):
    """Whole-block copy (copy-on-write), swap-out to and swap-in from page-locked host memory:
    512 blocks of the 7B layer shape (256 KB each, 128 MB)."""
    nb = 2 * nblocks + 8
    cache = P.KVCache(nb, 16, 32, 128, "f16")
    cache.pool_elems().fill_(1)
    src = torch.arange(nblocks, dtype=torch.int32, device="cuda")
    dst = src + nblocks
    nbytes = nblocks * cache.block_bytes
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    res = {"workload": f"{nblocks} blocks of 16 tokens x 32 KV heads x 128 x fp16 (256 KB each)",
           "bytes_per_call": nbytes, "l2": "flushed before each timed launch"}
    # copy: HBM read + write; swaps: the bytes that cross to or from host memory
    for name, fn, moved in (("copy", lambda: P.paged_block_copy(cache, src, dst), 2 * nbytes),
                            ("swap_out_host", lambda: P.paged_block_swap_out(cache, src, host), nbytes),
                            ("swap_in_host", lambda: P.paged_block_swap_in(cache, dst, host), nbytes)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        flush = flush or L2Flush()
        if name == "copy":
            cache.profile_start(kinds=("copy",))
            _kernel_loop_flushed(fn, reps, flush)
            prof = cache.profile_read()
            kern = prof["copy_ms"] / max(1, prof["copy_launches"]) / 1e3
            gbs = moved / kern / 1e9
            res[name] = {"kernel_us": round(kern * 1e6, 2), "gbs_read_plus_write": round(gbs, 1),
                         "frac_of_hbm": round(gbs / peaks[0], 4)}
        else:
            # the whole call: a swap with host memory is gather/scatter kernels and copy-engine copies
            ts = []
            for _ in range(reps):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                e1.synchronize()
                ts.append(e0.elapsed_time(e1) / 1e3)
            call = sum(ts) / len(ts)
            res[name] = {"call_us": round(call * 1e6, 2), "host_gbs": round(moved / call / 1e9, 1)}
    res["device_errors"] = cache.check_error()
    cache.close()
    return res


def secondary_prefix_cache(P, reps=5):
    """Host prefix-cache work at the 13B shape's scale: 64 requests whose 4096-token prompts share
    the first 4064 tokens (bs=32): chained hashes of every full block, lookup, allocation of the
    misses, publication of the new blocks, release."""
    rng = np.random.default_rng(1010)
    shared = rng.integers(0, 32000, 4064).astype(np.int32)
    prompts = [np.concatenate([shared, rng.integers(0, 32000, 32).astype(np.int32)]) for _ in range(64)]
    best = None
    for _ in range(reps):
        pc = P.PrefixCache(64 * 128)
        t0 = time.perf_counter()
        held, nblk, hits = [], 0, 0
        for toks in prompts:
            hs = P.block_hashes(toks, 32, extra=b"llama-2-13b-fp16")
            hit = pc.match(hs)
            new = pc.allocate(len(hs) - len(hit))
            pc.insert(hs[len(hit):], new)
            held.append(np.concatenate([hit, new]))
            nblk += len(hs)
            hits += len(hit)
        for b in held:
            pc.release(b)
        dt = time.perf_counter() - t0
        pc.close()
        best = dt if best is None else min(best, dt)
    return {"workload": "64 prompts of 4096 tokens sharing 4064 (bs 32): hash, lookup, allocate, publish, release",
            "blocks": nblk, "hit_blocks": hits, "ms": round(best * 1e3, 3),
            "blocks_per_s": round(nblk / best, 1), "where": "host (C++), one thread"}


def compact_secondary(sec: dict) -> dict:
    """The secondary figures as they go on the bench line: numbers only, short keys, the kernels
    furthest from their roofline last (the full records, with workload descriptions, go to
    --detail-out).  fr = fraction of the measured peak (HBM for decode / append / copy, dense bf16
    for the prefills); us = mean kernel time; err = device error bits."""
    if not sec:
        return {}
    out = {}
    if "prefix13b" in sec:
        d = sec["prefix13b"]
        out["prefix13b"] = {"us": d["decode_kernel_us"], "gbs_logical": d["kv_gbs"], "gbs_unique": d["unique_kv_gbs"],
                            "err": d["device_errors"]}
    if "prefix13b_cascade" in sec:
        d = sec["prefix13b_cascade"]
        out["cascade13b"] = {"step_us": d["step_us"], "kernels_us": d["decode_kernel_us"],
                             "fr_unique": d["unique_frac_of_hbm"], "gbs_unique_step": d["unique_kv_gbs_per_step"],
                             "err": d["device_errors"]}
    if "stress" in sec:
        st = sec["stress"]
        out["stress"] = {k: {"us": v["decode_kernel_us"], "gbs": v["kv_gbs"], "fr": v["frac_of_hbm"],
                             "err": v["device_errors"]}
                         for k, v in st.items() if isinstance(v, dict)}
        out["stress"]["fp8_over_bf16_time"] = [st[f"bs{b}_fp8_over_bf16_time"] for b in (8, 16, 32)]
    if "prefix_cache_host" in sec:
        out["prefix_cache_blocks_per_s"] = sec["prefix_cache_host"]["blocks_per_s"]
    if "blocks" in sec:
        b = sec["blocks"]
        out["blocks"] = {"copy_fr": b["copy"]["frac_of_hbm"], "copy_us": b["copy"]["kernel_us"],
                         "swap_out_gbs": b["swap_out_host"]["host_gbs"], "swap_in_gbs": b["swap_in_host"]["host_gbs"],
                         "err": b["device_errors"]}
    if "prefix_hit_prefill" in sec:
        d = sec["prefix_hit_prefill"]
        out["prefix_hit"] = {"attn_us": round(d["attention_kernel_ms"] * 1e3, 2),
                             "append_us": round(d["append_kernel_ms"] * 1e3, 2), "tflops": d["tflops"],
                             "fr": d["frac_of_bf16_peak"], "err": d["device_errors"]}
    if "append" in sec:
        d = sec["append"]
        out["append5256"] = {"us": round(d["kernel_ms"] * 1e3, 2), "gbs": d["gbs"], "fr": d["frac_of_hbm"]}
    if "prefill" in sec:
        d = sec["prefill"]
        if "kernel_ms" in d:
            out["prefill5256"] = {"us": round(d["kernel_ms"] * 1e3, 2), "tflops": d["tflops"],
                                  "fr": d["frac_of_bf16_peak"], "err": d["device_errors"]}
        else:
            out["prefill5256"] = d
    out["l2"] = "flushed before each timed append / copy / prefill launch; decode inputs exceed L2"
    return out


def run_only(case: str):
    """One secondary case alone (a short run for ncu captures); prints {case: result}."""
    torch.cuda.set_device(0)
    import paged_kv_cache_134_gb300 as P
    from paged_kv_cache_134_gb300 import workloads as W
    from paged_kv_cache_134_gb300 import runner as G
    peaks = _peaks()
    if case == "prefill":
        r = secondary_prefill(P, W, G, peaks, reps=5)
    elif case == "append":
        r = secondary_append(P, W, G, peaks, reps=5)
    elif case == "prefix13b":
        r = secondary_decode(P, G, peaks, W.prefix13b(), reps=5)
    elif case == "prefix13b_cascade":
        w4 = W.prefix13b()
        r = secondary_decode(P, G, peaks, w4, reps=5, cascade=w4.shared_prefix_len)
    elif case == "prefix_hit":
        r = secondary_prefix_hit(P, W, G, peaks, reps=5)
    elif case == "blocks":
        r = secondary_blocks(P, W, G, peaks, reps=5)
    elif case == "prefix_cache":
        r = secondary_prefix_cache(P)
    elif case.startswith("stress_bs"):
        bs, kv = case[len("stress_bs"):].split("_")
        r = secondary_decode(P, G, peaks, W.stress(bs=int(bs), kv_dtype=kv), reps=5)
    else:
        raise SystemExit(f"unknown case {case}")
    print(json.dumps({case: r}), flush=True)


def run_ours(args):
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import paged_kv_cache_134_gb300 as P
    from paged_kv_cache_134_gb300 import workloads as W
    from paged_kv_cache_134_gb300 import runner as G

    peaks = _peaks()
    w = W.decode7b(seed=1002 + rank)
    cache = G.new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, w.model_dtype)
    G.fill_cache(cache, w)
    x = G.DecodeInputs(w)
    cache.reserve(w.num_seqs, w.num_q_heads, w.max_blocks)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    step = lambda: G.decode_step(cache, x)  # noqa: E731

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert cache.check_error() == 0

    # ---- timed region: inputs resident in HBM; KV (1.07 GB/step) is larger than L2 (129 MB)
    clock_dir = args.clocks_dir or tempfile.gettempdir()
    sampler = ClockSampler(local, os.path.join(clock_dir, f"pkv_clocks_rank{rank}.csv"))
    sampler.wait_running()
    launches0 = P.kernel_launches()
    # no events inside the timed region: an event between two kernels stops the append -> decode ->
    # merge overlap of programmatic dependent launch
    _barrier(ws)
    torch.cuda.synchronize()
    elapsed = _time_loop(step, args.steps, stream)
    torch.cuda.synchronize()
    _barrier(ws)
    launches = P.kernel_launches() - launches0
    assert cache.check_error() == 0
    # the decode kernel's own duration (the roofline's denominator): a second pass of at least 10
    # steps with events around every decode launch, still under the clock sampler
    rsteps = max(10, min(args.steps, 200))
    cache.profile_start(kinds=("decode",))
    _time_loop(step, rsteps, stream)
    torch.cuda.synchronize()
    prof = cache.profile_read()
    clocks = sampler.stop()
    assert cache.check_error() == 0

    kv_bytes = w.kv_read_bytes()
    value, seqs_per_s, elapsed_max = aggregate(float(kv_bytes) * args.steps, float(w.num_seqs) * args.steps, elapsed,
                                               ws)
    dec_kernel_s = prof["decode_ms"] / max(1, prof["decode_launches"]) / 1e3
    # per-kernel breakdown from a separate pass with events around every kernel (not the headline:
    # events between kernels stop their programmatic-launch overlap)
    cache.profile_start()
    bsteps = max(20, min(args.steps, 500))
    t_b = _time_loop(step, bsteps, stream)
    pb = cache.profile_read()
    breakdown = {"append_at_us": round(pb["append_ms"] / max(1, pb["append_launches"]) * 1e3, 2),
                 "decode_kernel_us": round(pb["decode_ms"] / max(1, pb["decode_launches"]) * 1e3, 2),
                 "merge_kernel_us": round(pb["merge_ms"] / max(1, pb["merge_launches"]) * 1e3, 2),
                 "step_us_all_kernels_bracketed": round(t_b / bsteps * 1e6, 2),
                 "step_us_timed_region": round(elapsed / args.steps * 1e6, 2)}
    achieved = kv_bytes / dec_kernel_s / 1e9

    # ---- end to end through the public API with host buffers (pinned), copies inside the timed region.
    # The step's inputs (q, the new token's K and V, tables, sequence ids, positions, lengths) sit in
    # one pinned host buffer laid out like a device buffer whose views the API calls read, so that
    # each step moves them with a single host-to-device copy; the output comes back with one more.
    # Two device input buffers and two outputs let a serving loop overlap: step i+1's input copy and
    # step i's output copy run on a copy stream while step i (and then i+1) computes.  Every step
    # still makes both of its copies inside the timed region.  The loop without overlap is timed too.
    fields = ("q", "new_k", "new_v", "tables", "seq_ids", "positions", "lens")
    offs, total = {}, 0
    for name in fields:
        t = getattr(x, name)
        offs[name] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    for name in fields:
        t = getattr(x, name)
        nb = t.numel() * t.element_size()
        h_in[offs[name]:offs[name] + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    d_in, xs = [], []
    for _ in range(2):
        buf = torch.empty(total, dtype=torch.uint8, device="cuda")
        xb = copy.copy(x)
        for name in fields:
            t = getattr(x, name)
            nb = t.numel() * t.element_size()
            setattr(xb, name, buf[offs[name]:offs[name] + nb].view(t.dtype).view(t.shape))
        xb.out = torch.empty_like(x.out)
        xb.slots = torch.empty_like(x.slots)
        d_in.append(buf)
        xs.append(xb)
    h_out = torch.empty(x.out.shape, dtype=x.out.dtype).pin_memory()
    h2d = total
    d2h = h_out.numel() * h_out.element_size()

    def e2e_serial_step():
        d_in[0].copy_(h_in, non_blocking=True)
        G.decode_step(cache, xs[0])
        h_out.copy_(xs[0].out, non_blocking=True)

    copy_stream = torch.cuda.Stream()

    def e2e_pipelined(n: int) -> float:
        cs, ps = stream, copy_stream
        ev_in = [torch.cuda.Event() for _ in range(2)]   # inputs of the step using buffer b have landed
        ev_k = [torch.cuda.Event() for _ in range(2)]    # kernels of the step using buffer b are done
        ev_out = [torch.cuda.Event() for _ in range(2)]  # output of the step using buffer b is on the host
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(cs)
        ps.wait_stream(cs)
        with torch.cuda.stream(ps):
            d_in[0].copy_(h_in, non_blocking=True)
            ev_in[0].record(ps)
        for i in range(n):
            b = i & 1
            if i + 1 < n:  # next step's inputs, once the step that last read that buffer is done
                with torch.cuda.stream(ps):
                    if i >= 1:
                        ps.wait_event(ev_k[b ^ 1])
                    d_in[b ^ 1].copy_(h_in, non_blocking=True)
                    ev_in[b ^ 1].record(ps)
            cs.wait_event(ev_in[b])
            if i >= 2:
                cs.wait_event(ev_out[b])  # the output buffer's previous copy to the host is done
            G.decode_step(cache, xs[b])
            ev_k[b].record(cs)
            with torch.cuda.stream(ps):
                ps.wait_event(ev_k[b])
                h_out.copy_(xs[b].out, non_blocking=True)
                ev_out[b].record(ps)
        cs.wait_stream(ps)
        t1.record(cs)
        t1.synchronize()
        return t0.elapsed_time(t1) / 1e3

    e2e_steps = max(10, min(args.steps, 1000))
    for _ in range(3):
        e2e_serial_step()
    e2e_pipelined(4)
    torch.cuda.synchronize()
    _barrier(ws)
    e2e_serial_t = _reduce_max(_time_loop(e2e_serial_step, e2e_steps, stream), ws)
    _barrier(ws)
    e2e_t = _reduce_max(e2e_pipelined(e2e_steps), ws)
    e2e_value = _reduce_sum(float(kv_bytes) * e2e_steps, ws) / e2e_t / 1e9
    e2e_serial_value = _reduce_sum(float(kv_bytes) * e2e_steps, ws) / e2e_serial_t / 1e9
    # the decode is deterministic: the output that came back to the host equals the device step's
    e2e_match = bool(torch.equal(h_out, x.out.cpu()))

    secondary = {}
    if rank == 0 and not args.skip_secondary:
        flush = L2Flush()
        w4 = W.prefix13b()
        uniq = (w4.shared_prefix_len + int((w4.context_lens - w4.shared_prefix_len + 1).sum())) * \
            w4.num_kv_heads * w4.head_dim * 2 * 2
        secondary["prefix13b"] = dict(workload="13B-shape decode, 64 seqs sharing a 4096-token prefix (128 blocks, "
                                               "ref count 64) + private suffix U{1..512}, 40/40 heads, bs=32, fp16",
                                      **secondary_decode(P, G, peaks, w4, unique_bytes=uniq))
        secondary["prefix13b_cascade"] = dict(
            workload="the same 13B-shape batch, cascade decode: the 4096-token shared prefix read once per "
                     "(head, prefix split) for all 64 sequences on the tensor cores, suffixes by split-K decode",
            **secondary_decode(P, G, peaks, w4, unique_bytes=uniq, cascade=w4.shared_prefix_len))
        del w4
        stress = {}
        for kv in ("bf16", "fp8"):
            for bs in (8, 16, 32):
                stress[f"bs{bs}_{kv}"] = secondary_decode(P, G, peaks, W.stress(bs=bs, kv_dtype=kv))
        for bs in (8, 16, 32):
            stress[f"bs{bs}_fp8_over_bf16_time"] = round(stress[f"bs{bs}_fp8"]["decode_kernel_us"] /
                                                         stress[f"bs{bs}_bf16"]["decode_kernel_us"], 3)
        secondary["stress"] = dict(workload="256 seqs, log-normal lengths (median 500, cap 8192), 32 q / 8 KV heads, "
                                            "D=128, churned free list; KV bf16 or FP8-E4M3 (per-head scales)", **stress)
        secondary["prefix_cache_host"] = secondary_prefix_cache(P)
        secondary["blocks"] = secondary_blocks(P, W, G, peaks, flush=flush)
        secondary["prefix_hit_prefill"] = secondary_prefix_hit(P, W, G, peaks, flush=flush)
        secondary["append"] = secondary_append(P, W, G, peaks, flush=flush)
        secondary["prefill"] = secondary_prefill(P, W, G, peaks, flush=flush)
        if args.detail_out:
            with open(args.detail_out, "w") as f:
                json.dump(secondary, f, indent=1)

    cpu = None
    if rank == 0 and ws == 1 and not args.skip_cpu:
        gbs, t_pass, nseq, threads, reps = oracle_decode_rate(w, budget_s=args.cpu_seconds)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"full decode attention pass over all {nseq} sequences, repeated {reps}x "
                         f"({t_pass:.2f} s per pass, fp64 C, OpenMP)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(elapsed_max / args.steps * 1e3, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
                       "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                       "num_blocks": w.num_blocks, "tokens_attended": int(w.decode_lens.sum()),
                       "kv_bytes_per_step": kv_bytes, "per_rank_seed": "1002 + rank",
                       "l2": "inputs larger than L2 (KV read per step 1.07 GB vs 129 MB L2)",
                       "split_tokens": int(os.environ.get("PAGEDKV_SPLIT_TOKENS", "256")),
                       "parallelism": f"replicas x{ws} (one independent batch per GPU)"},
            "seqs_per_s": round(seqs_per_s, 1),
            "seqs_per_s_32_layers": round(seqs_per_s / 32, 1),
            "hbm_frac": round(value / peaks[0], 4),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks[0], "unit": "GB/s",
                         "frac": round(achieved / peaks[0], 4),
                         "traffic": _recorded_traffic("decode_kernel_decode7b.md"),
                         "traffic_source": "profiles/decode_kernel_decode7b.md (ncu dram__bytes_read+write, one launch)",
                         "kernel": "pkv_decode::decode_kernel<128,1,f16,f16>",
                         "kernel_ms": round(dec_kernel_s * 1e3, 5),
                         "kernel_ms_samples": int(prof["decode_launches"]),
                         "peak_source": f"{peaks[3]} hbm_gbs (MEASURED_PEAKS.json)",
                         "algorithmic_bytes": "KV read: sum(L+1) x Hkv x D x 2 B x 2 (K and V) per launch"},
            "step_breakdown": breakdown,
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
                    "copies": "each step: one host-to-device copy of its packed inputs and one "
                              "device-to-host copy of its output, on a copy stream, overlapping the "
                              "neighbouring steps' kernels (double-buffered device inputs and outputs)",
                    "serial_value": round(e2e_serial_value, 2), "output_matches_device_step": e2e_match},
            "gpu_launches": int(launches),
            "clocks": clocks,
            "cpu_baseline": cpu,
            "secondary": compact_secondary(secondary),
        }
        print(json.dumps(line), flush=True)
    cache.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-secondary", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--clocks-dir", default=None,
                    help="folder for the nvidia-smi clock samples of the timed region (default: the temp dir)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--detail-out", default=None,
                    help="file for the full secondary records (workload descriptions included)")
    ap.add_argument("--only", default=None,
                    help="run one secondary case alone and print its JSON (for profiling): prefill, append, "
                         "prefix13b, prefix13b_cascade, prefix_hit, blocks, prefix_cache or stress_bs{8,16,32}_{bf16,fp8}")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args.only)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
