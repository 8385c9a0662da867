#!/usr/bin/env python3
"""Benchmark of the NVFP4 paged KV cache hot path on GB300.

Headline: NVFP4 paged decode attention KV-tokens/s (and HBM GB/s, % of 8 TB/s)
on the decode workload at the pages' shape: 32 sequences x 8192 cached tokens
(+1 appended), 64 query heads / 8 KV heads, head_dim 128, 16-token pages.
One step = quantize-append of the 32 new tokens + decode attention (with its
split combine), both through the C ABI.  Secondary lines of the same run: the
128K-token decode workload and one layer of the extend workload (FP8
workspace dequant and 2048-token quantize-write).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

`--impl reference` times the CPU oracle on the host cores instead (same
metric, bounded samples).  With torchrun (N > 1) every rank runs a replica.
"""
import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nvfp4_quantized_paged_quantize_gb300 import inputs  # noqa: E402

METRIC = "NVFP4 paged decode attention KV-tokens/s and HBM GB/s (% of 8 TB/s) on 1 GB300"
UNIT = "KV-tokens/s"
NOMINAL_HBM_GBS = 8000.0
L2_FLUSH_BYTES = 256 << 20


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def decode_source_hash():
    """sha256 of the decode kernel's sources (a committed ncu traffic figure is
    reported only while it still describes this code)."""
    import hashlib

    h = hashlib.sha256()
    for f in ("decode_attention.cu", "nvfp4kv_device.cuh"):
        with open(os.path.join(ROOT, "nvfp4_quantized_paged_quantize_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def committed_traffic(workload):
    """DRAM bytes per decode launch from profiles/decode_traffic.json (written
    from an ncu capture), or None if absent or taken on other code."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != decode_source_hash():
        return None
    return rec.get("traffic_bytes_per_launch", {}).get(workload)


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def world_max(torch, value, device):
    """The largest of one float over all ranks (the value itself without an
    initialised process group).  Replicas are timed separately; the slowest
    rank's total is the job's time."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_rank_step, steps, total_ms):
    """Whole-job units/s: every rank processed units_per_rank_step per step."""
    return world * units_per_rank_step * steps / (total_ms / 1e3)


# ---------------------------------------------------------------------------
# clocks sampled while the timed region runs
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"nvfp4kv_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = [[p.strip() for p in ln.split(",")] for ln in open(self.path)]
        lines = [p for p in lines if len(p) >= 9]
        if len({p[0] for p in lines}) > 1:          # several GPUs visible: keep ours
            lines = [p for p in lines if p[0] == str(self.gpu)]
        for parts in lines:
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": 0}
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": float(np.median(loaded)), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def _dev(torch, a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(dtype) if dtype is not None else t).cuda()


def _bf16(torch, bits):
    return _dev(torch, np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16), torch.bfloat16)


def _global_scales(torch, kv, wl, prompts, new):
    """1, or the library's calibration: nvfp4kv_tensor_amax folded over every K
    (every V) tensor on the device, then nvfp4kv_calibrated_global_scale."""
    pairs = wl.calibration_tensors(prompts, new)
    if not pairs:
        return 1.0, 1.0
    amax = torch.zeros(2, dtype=torch.float32, device="cuda")
    for p in pairs:
        for i in range(2):
            kv.nvfp4kv_tensor_amax(_bf16(torch, p[i]).reshape(-1), amax[i:i + 1], accumulate=True)
    a = amax.cpu().tolist()
    return kv.nvfp4kv_calibrated_global_scale(a[0]), kv.nvfp4kv_calibrated_global_scale(a[1])


def _fill_cache(torch, kv, wl, prompts, new):
    gk, gv = _global_scales(torch, kv, wl, prompts, new)
    cache = kv.Cache.empty(wl.num_pages, wl.num_kv_heads, k_global_scale=gk, v_global_scale=gv, zero=True)
    for b in range(wl.batch):
        k, v = prompts[b]
        kv.nvfp4kv_quantize_append(cache, _bf16(torch, k), _bf16(torch, v),
                                   _dev(torch, wl.slots(b, 0, k.shape[0])))
    torch.cuda.synchronize()
    return cache


def _fill_cache_streaming(torch, kv, wl, threads=16):
    """The cache of an uncalibrated workload (global scales 1), each sequence
    drawn by a worker thread and appended as soon as it is ready, so the host
    never holds the whole batch (the ragged workload is 7.4 GB of bf16)."""
    from concurrent.futures import ThreadPoolExecutor

    cache = kv.Cache.empty(wl.num_pages, wl.num_kv_heads, zero=True)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for b, (k, v) in enumerate(ex.map(wl.prompt_kv, range(wl.batch))):
            kv.nvfp4kv_quantize_append(cache, _bf16(torch, k), _bf16(torch, v),
                                       _dev(torch, wl.slots(b, 0, k.shape[0])))
    torch.cuda.synchronize()
    return cache


def variant_decode_lines(torch, kv, args, flush, hbm_peak):
    """Decode over each format variant's cache of the 8K workload (the pages'
    format comparison): the cache written by the variant's append from the
    workload's bf16 K/V, then the variant's decode timed like NVFP4's.  Bytes:
    144 per token and KV head (NVFP4, SR, Hadamard) or 136 (MXFP4), plus q and
    out."""
    from concurrent.futures import ThreadPoolExecutor

    wl = inputs.decode_config(2)
    steps = max(3, min(args.steps, 50))
    q, pt = _bf16(torch, wl.q()), _dev(torch, wl.page_table)
    lens = _dev(torch, wl.seq_lens.astype(np.int32))
    out = torch.empty((wl.batch, wl.num_q_heads, 128), dtype=torch.float32, device="cuda")
    nk, nv = wl.new_kv()
    res = {}
    for name, var in (("sr", kv.NVFP4KV_VARIANT_SR), ("hadamard", kv.NVFP4KV_VARIANT_HADAMARD),
                      ("mxfp4", kv.NVFP4KV_VARIANT_MXFP4)):
        mx = var == kv.NVFP4KV_VARIANT_MXFP4
        cache = kv.Cache.empty(wl.num_pages, wl.num_kv_heads, zero=True, mxfp4=mx)

        def draw(b):
            k, v = wl.prompt_kv(b)
            k = np.concatenate([k, nk[b:b + 1]])
            v = np.concatenate([v, nv[b:b + 1]])
            n = k.size
            r = (inputs.rounding_bytes(100 + 2 * b, n).reshape(k.shape),
                 inputs.rounding_bytes(101 + 2 * b, n).reshape(k.shape)) if var == kv.NVFP4KV_VARIANT_SR else None
            return k, v, r

        with ThreadPoolExecutor(max_workers=16) as ex:
            for b, (k, v, r) in enumerate(ex.map(draw, range(wl.batch))):
                slots = _dev(torch, wl.slots(b, 0, k.shape[0]))
                rk = _dev(torch, r[0]) if r is not None else None
                rv = _dev(torch, r[1]) if r is not None else None
                kv.nvfp4kv_quantize_append_variant(var, cache, _bf16(torch, k), _bf16(torch, v), slots, rk, rv)
        torch.cuda.synchronize()
        ws = torch.zeros(kv.nvfp4kv_decode_workspace_size(cache, wl.batch, wl.num_q_heads), dtype=torch.uint8,
                         device="cuda")
        ms, _ = time_steps(torch, steps, args.warmup,
                           lambda ev=None, c=cache, var=var: kv.nvfp4kv_decode_attention_variant(
                               var, c, q, out, pt, lens, wl.softmax_scale, ws), flush)
        t = float(np.mean(ms))
        per_token_head = 136 if mx else 144
        nbytes = wl.kv_tokens() * wl.num_kv_heads * per_token_head + q.numel() * 2 + out.numel() * 4
        gbs = nbytes / (t / 1e3) / 1e9
        res[f"decode_{name}_b32_ctx8k"] = {"kernel_ms": t, "kv_tokens_per_s": wl.kv_tokens() / (t / 1e3),
                                           "hbm_gbs": gbs, "frac_of_measured_peak": gbs / hbm_peak,
                                           "algorithmic_bytes": nbytes, "bytes_per_token_head": per_token_head}
        del cache, ws
        torch.cuda.empty_cache()
    return res


def _calibration_input(torch, wl):
    """One layer's K of a decode workload as one bf16 device tensor: the first
    sequence's prompt K drawn by the workload, repeated over the batch."""
    k, _ = wl.prompt_kv(0)
    x = _bf16(torch, k).reshape(-1).repeat(wl.batch)
    return x, torch.zeros(1, dtype=torch.float32, device="cuda")


class DecodeBench:
    """Device state and one step (append + decode) of a decode workload."""

    def __init__(self, torch, kv, wl):
        self.torch, self.kv, self.wl = torch, kv, wl
        self.new = wl.new_kv() if wl.append else None
        self.q_bits = wl.q()
        if wl.calibrated:
            prompts = wl.all_prompt_kv(threads=16)
            self.cache = _fill_cache(torch, kv, wl, prompts, self.new)
            del prompts
        else:
            self.cache = _fill_cache_streaming(torch, kv, wl)
        self.q = _bf16(torch, self.q_bits)
        self.pt = _dev(torch, wl.page_table)
        self.lens = _dev(torch, wl.seq_lens.astype(np.int32))
        if wl.append:
            self.k_new = _bf16(torch, self.new[0])
            self.v_new = _bf16(torch, self.new[1])
            self.slots = _dev(torch, wl.append_slots())
        self.out = torch.empty((wl.batch, wl.num_q_heads, 128), dtype=torch.float32, device="cuda")
        n = kv.nvfp4kv_decode_workspace_size(self.cache, wl.batch, wl.num_q_heads)
        self.ws = torch.zeros(n, dtype=torch.uint8, device="cuda")

    def append(self):
        if self.wl.append:
            self.kv.nvfp4kv_quantize_append(self.cache, self.k_new, self.v_new, self.slots)

    def decode(self):
        self.kv.nvfp4kv_decode_attention(self.cache, self.q, self.out, self.pt, self.lens,
                                         self.wl.softmax_scale, self.ws)

    def step(self):
        """One decode step: append the new tokens, then attend (one library call,
        the decode's set-up overlapping the append)."""
        if self.wl.append:
            self.kv.nvfp4kv_append_decode_attention(self.cache, self.k_new, self.v_new, self.slots, self.q,
                                                    self.out, self.pt, self.lens, self.wl.softmax_scale, self.ws)
        else:
            self.decode()

    def launches_per_step(self):
        return 2 if self.wl.append else 1


class PackedInputs:
    """A step's host inputs in one pinned buffer (each at a 256-byte offset)
    and its device twin: one H2D copy per step, device views for the call."""

    def __init__(self, torch, arrays):
        self.offsets, off = {}, 0
        raw = {name: np.ascontiguousarray(a).view(np.uint8).reshape(-1) for name, a in arrays.items()}
        for name, a in raw.items():
            self.offsets[name] = (off, a.size)
            off += (a.size + 255) // 256 * 256
        self.host = torch.empty(off, dtype=torch.uint8).pin_memory()
        hv = self.host.numpy()
        for name, a in raw.items():
            o, n = self.offsets[name]
            hv[o:o + n] = a
        self.dev = torch.empty(off, dtype=torch.uint8, device="cuda")
        self.nbytes = off                        # the bytes one upload copies (padding included)

    def view(self, name, dtype, shape):
        o, n = self.offsets[name]
        return self.dev[o:o + n].view(dtype).view(shape)

    def upload(self):
        self.dev.copy_(self.host, non_blocking=True)


def stream_probe_lines(torch, kv, b, steps, warmup, flush, hbm_peak, decode_ms):
    """Time the library's streaming probe over a decode bench's cache: the same
    page-heads the decode reads, with no attention math, in the decode's own
    pattern and as whole pages by bulk copy.  The decode's time is set beside."""
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv_bytes = b.wl.kv_tokens() * b.wl.num_kv_heads * 144
    out = {"kv_bytes": kv_bytes, "decode_kernel_ms": decode_ms,
           "decode_gbs_kv_only": kv_bytes / (decode_ms / 1e3) / 1e9}
    for name, mode in (("decode_pattern", kv.NVFP4KV_PROBE_DECODE_PATTERN),
                       ("whole_pages_bulk", kv.NVFP4KV_PROBE_WHOLE_PAGES)):
        ms, _ = time_steps(torch, steps, warmup,
                           lambda ev=None, mode=mode: kv.nvfp4kv_stream_probe(b.cache, b.pt, b.lens, sink, mode), flush)
        t = float(np.mean(ms))
        gbs = kv_bytes / (t / 1e3) / 1e9
        out[name] = {"kernel_ms": t, "hbm_gbs": gbs, "frac_of_measured_peak": gbs / hbm_peak,
                     "pct_of_8tbs": 100 * gbs / NOMINAL_HBM_GBS}
    return out


def make_l2_flush(torch):
    """Flush L2 between timed steps: write one buffer larger than L2, then read
    another.  The write evicts every line the step could reuse; the read then
    replaces the write's dirty lines with clean ones, so the timed step neither
    finds its inputs in L2 nor pays for writing the flush's data back (which
    a write-only flush leaves to the next kernel: ~120 MB of write-back)."""
    wbuf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    rbuf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush():
        wbuf.zero_()
        rbuf.sum()

    return flush


def time_steps(torch, steps, warmup, body, flush, split=None):
    """Run `warmup` untimed then `steps` timed iterations of body(); each timed
    iteration is bracketed by CUDA events on the current stream, with an L2
    flush (outside the events) before it.  split() may record an inner event
    pair around the dominant kernel.  Returns per-step ms and inner ms."""
    for _ in range(warmup):
        flush()
        body()
    torch.cuda.synchronize()
    E = torch.cuda.Event
    starts = [E(enable_timing=True) for _ in range(steps)]
    ends = [E(enable_timing=True) for _ in range(steps)]
    inner = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(steps)] if split else None
    torch.cuda.nvtx.range_push("timed")
    for i in range(steps):
        flush()
        starts[i].record()
        body(inner[i] if inner else None)
        ends[i].record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ims = [a.elapsed_time(b) for a, b in inner] if inner else None
    return ms, ims


def gpu_arm(args):
    import torch

    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    import nvfp4_quantized_paged_quantize_gb300 as kv

    kv.load()
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    flush = make_l2_flush(torch)

    wl = inputs.decode_config(2)
    bench = DecodeBench(torch, kv, wl)
    kv_tokens = wl.kv_tokens()
    alg_bytes = wl.algorithmic_bytes()

    def step(ev=None):
        bench.step()

    def decode_only(ev=None):
        if ev is not None:
            ev[0].record()
        bench.decode()
        if ev is not None:
            ev[1].record()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        step_ms, _ = time_steps(torch, args.steps, args.warmup, step, flush)
        # the decode call alone (its two kernels), for the roofline: inside the
        # step it overlaps the append, so it is timed in a loop of its own
        _, dec_ms = time_steps(torch, args.steps, args.warmup, decode_only, flush, split=True)
    torch.cuda.synchronize()
    total_ms = world_max(torch, float(sum(step_ms)), "cuda")
    ms_per_step = total_ms / args.steps
    value = job_throughput(world, kv_tokens, args.steps, total_ms)
    dec_avg_ms = float(np.mean(dec_ms))
    achieved = alg_bytes / (dec_avg_ms / 1e3) / 1e9

    # e2e through the public API with host buffers: per step one H2D copy of
    # the step's inputs (q, new K/V, slots, page table, lengths), packed in one
    # pinned buffer as a serving loop would stage them, the library call on
    # views of the device copy, and one D2H copy of the output into pinned memory
    packed = PackedInputs(torch, {"q": bench.q_bits, "k": bench.new[0], "v": bench.new[1],
                                  "slots": wl.append_slots(), "pt": wl.page_table,
                                  "lens": wl.seq_lens.astype(np.int32)})
    d_q = packed.view("q", torch.bfloat16, bench.q.shape)
    d_k = packed.view("k", torch.bfloat16, bench.k_new.shape)
    d_v = packed.view("v", torch.bfloat16, bench.v_new.shape)
    d_slots = packed.view("slots", torch.int64, bench.slots.shape)
    d_pt = packed.view("pt", torch.int32, bench.pt.shape)
    d_lens = packed.view("lens", torch.int32, bench.lens.shape)
    host_out = torch.empty(bench.out.shape, dtype=torch.float32).pin_memory()
    h2d = packed.nbytes
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step(ev=None):
        packed.upload()
        kv.nvfp4kv_append_decode_attention(bench.cache, d_k, d_v, d_slots, d_q, bench.out, d_pt, d_lens,
                                           wl.softmax_scale, bench.ws)
        host_out.copy_(bench.out, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 200))
    e2e_ms, _ = time_steps(torch, e2e_steps, args.warmup, e2e_step, flush)
    e2e_total = world_max(torch, float(sum(e2e_ms)), "cuda")
    e2e_value = job_throughput(world, kv_tokens, e2e_steps, e2e_total)
    probe = None
    if not args.skip_secondary:
        probe = stream_probe_lines(torch, kv, bench, max(3, min(args.steps, 200)), args.warmup, flush, hbm_peak,
                                   dec_avg_ms)
    del bench

    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 storage; f16 mma operands, f32 accumulate",
        "data": "synthetic (seeded numpy: K/V N(0,0.02) with 8 of every 4096 values = 6.0, q N(0,1))",
        "config": {
            "workload": wl.name, "batch": wl.batch, "ctx": int(wl.seq_lens[0]), "q_heads": wl.num_q_heads,
            "kv_heads": wl.num_kv_heads, "head_dim": 128, "page_size": 16,
            "step": "nvfp4kv_append_decode_attention: quantize-append of 32 new tokens + decode attention "
                    "(split-K decode + combine)",
            "l2": "flushed before every timed step, outside the step's events: a 256 MiB memset, then a read of "
                  "another 256 MiB (no input cached, no dirty flush lines left to write back)",
            "parallelism": f"replicas x{world}",
        },
        "decode": {
            "kernel_ms": dec_avg_ms,
            "kv_tokens_per_s": kv_tokens / (dec_avg_ms / 1e3),
            "hbm_gbs": achieved,
            "pct_of_8tbs": 100.0 * achieved / NOMINAL_HBM_GBS,
            "algorithmic_bytes": alg_bytes,
        },
        "roofline": {
            "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": committed_traffic(wl.name),
            "kernel": "decode_kernel + combine_kernel (one nvfp4kv_decode_attention call)",
            "peak_kind": f"{peak_kind} (copy bandwidth, burst)",
        },
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * 3,  # quantize-append, decode, split combine
        "clocks": clocks.summary(),
    }
    if not args.skip_secondary:
        line["secondary"] = secondary(torch, kv, args, flush, hbm_peak)
        line["secondary"]["stream_probe_b32_ctx8k"] = probe
        line["secondary"].update(variant_decode_lines(torch, kv, args, flush, hbm_peak))
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def secondary(torch, kv, args, flush, hbm_peak):
    out = {}
    steps = max(3, min(args.steps, 50))
    # long-context decode: 4 sequences x 131072 tokens, calibrated global scales
    wl = inputs.decode_config(3)
    b = DecodeBench(torch, kv, wl)
    ms, _ = time_steps(torch, steps, args.warmup, lambda ev=None: b.decode(), flush)
    t = float(np.mean(ms))
    gbs = wl.algorithmic_bytes() / (t / 1e3) / 1e9
    out["decode_b4_ctx128k"] = {"kernel_ms": t, "kv_tokens_per_s": wl.kv_tokens() / (t / 1e3), "hbm_gbs": gbs,
                                "pct_of_8tbs": 100 * gbs / NOMINAL_HBM_GBS, "frac_of_measured_peak": gbs / hbm_peak}
    out["stream_probe_b4_ctx128k"] = stream_probe_lines(torch, kv, b, steps, args.warmup, flush, hbm_peak, t)
    del b
    torch.cuda.empty_cache()
    # ragged continuous batching: 256 sequences, log-uniform lengths in [512,
    # 32768] (+1 appended), 32 q / 8 KV heads; the bytes are those of the
    # seeded lengths
    wl4 = inputs.decode_config(4)
    b = DecodeBench(torch, kv, wl4)
    ms, _ = time_steps(torch, steps, args.warmup, lambda ev=None: b.decode(), flush)
    t = float(np.mean(ms))
    gbs = wl4.algorithmic_bytes() / (t / 1e3) / 1e9
    out["decode_ragged_b256"] = {"kernel_ms": t, "kv_tokens_per_s": wl4.kv_tokens() / (t / 1e3), "hbm_gbs": gbs,
                                 "pct_of_8tbs": 100 * gbs / NOMINAL_HBM_GBS, "frac_of_measured_peak": gbs / hbm_peak,
                                 "algorithmic_bytes": wl4.algorithmic_bytes(), "kv_tokens": wl4.kv_tokens()}
    del b
    torch.cuda.empty_cache()
    # calibration: the amax pass over one layer's K of that workload (4 x 131072
    # tokens x 8 heads x 128 bf16 values, 1.07 GB), HBM-bound at 2 B per value
    x, amax = _calibration_input(torch, wl)
    ms, _ = time_steps(torch, steps, args.warmup, lambda ev=None: kv.nvfp4kv_tensor_amax(x, amax), flush)
    t = float(np.mean(ms))
    gbs = (2 * x.numel() + 4) / (t / 1e3) / 1e9
    out["calibrate_amax_b4_ctx128k_k"] = {"kernel_ms": t, "values": int(x.numel()), "hbm_gbs": gbs,
                                          "frac_of_measured_peak": gbs / hbm_peak}
    del x
    torch.cuda.empty_cache()
    # extend: one layer (16 x 16384-token prefix -> FP8 workspace; 16 x 2048 new tokens quantized)
    ew = inputs.extend_config(num_layers=1)
    cache = kv.Cache.empty(ew.num_pages, ew.num_kv_heads, zero=True)
    for s in range(ew.batch):
        k, v = ew.prefix_kv(0, s)
        kv.nvfp4kv_quantize_append(cache, _bf16(torch, k), _bf16(torch, v), _dev(torch, ew.slots(s, 0, ew.prefix_len)))
    ks, vs = zip(*[ew.chunk_kv(0, s) for s in range(ew.batch)])
    kc, vc = _bf16(torch, np.concatenate(ks)), _bf16(torch, np.concatenate(vs))
    slots = _dev(torch, ew.chunk_slots())
    pt, pl, cu = _dev(torch, ew.page_table), _dev(torch, ew.prefix_lens), _dev(torch, ew.cu_prefix)
    wk = torch.empty((ew.total_rows, ew.num_kv_heads, 128), dtype=torch.uint8, device="cuda")
    wv = torch.empty_like(wk)
    ms, _ = time_steps(torch, steps, args.warmup,
                       lambda ev=None: kv.nvfp4kv_dequant_to_fp8_workspace(cache, pt, pl, cu, wk, wv), flush)
    t = float(np.mean(ms))
    gbs = ew.dequant_bytes_per_layer() / (t / 1e3) / 1e9
    out["extend_dequant_fp8_per_layer"] = {"kernel_ms": t, "hbm_gbs": gbs, "frac_of_measured_peak": gbs / hbm_peak,
                                           "x80_layers_ms": 80 * t}
    ms, _ = time_steps(torch, steps, args.warmup,
                       lambda ev=None: kv.nvfp4kv_quantize_append(cache, kc, vc, slots), flush)
    t = float(np.mean(ms))
    gbs = ew.quantize_bytes_per_layer() / (t / 1e3) / 1e9
    out["extend_quantize_2048x16_per_layer"] = {"kernel_ms": t, "hbm_gbs": gbs, "frac_of_measured_peak": gbs / hbm_peak,
                                                "x80_layers_ms": 80 * t}
    # the chunk's own K/V into the workspace, then the extend attention over it
    rows = _dev(torch, ew.chunk_ws_rows())
    ms, _ = time_steps(torch, steps, args.warmup,
                       lambda ev=None: kv.nvfp4kv_bf16_to_fp8_workspace(kc, vc, rows, wk, wv), flush)
    t = float(np.mean(ms))
    vals = 2 * kc.numel()
    gbs = (3 * vals + 8 * ew.batch * ew.chunk_len) / (t / 1e3) / 1e9
    out["extend_chunk_to_fp8_per_layer"] = {"kernel_ms": t, "hbm_gbs": gbs, "frac_of_measured_peak": gbs / hbm_peak}
    # the same chunk written once into both the NVFP4 cache and the workspace
    ms, _ = time_steps(torch, steps, args.warmup,
                       lambda ev=None: kv.nvfp4kv_quantize_append_fp8(cache, kc, vc, slots, rows, wk, wv), flush)
    t = float(np.mean(ms))
    gbs = (vals * 2 + vals * 9 // 16 + vals + 16 * ew.batch * ew.chunk_len) / (t / 1e3) / 1e9
    out["extend_quantize_write_fp8_fused_per_layer"] = {"kernel_ms": t, "hbm_gbs": gbs,
                                                        "frac_of_measured_peak": gbs / hbm_peak}
    # the format variants' quantize-append of the same chunk (comparison paths)
    rk = _dev(torch, inputs.rounding_bytes(10, kc.numel())).view(kc.shape)
    rv = _dev(torch, inputs.rounding_bytes(11, vc.numel())).view(vc.shape)
    mxc = kv.Cache.empty(ew.num_pages, ew.num_kv_heads, zero=True, mxfp4=True)
    toks = ew.batch * ew.chunk_len
    # bytes besides the bf16 read: the pages written (and SR's random byte per value)
    for name, var, c_, other in (("sr", kv.NVFP4KV_VARIANT_SR, cache, vals * 9 // 16 + vals),
                                  ("hadamard", kv.NVFP4KV_VARIANT_HADAMARD, cache, vals * 9 // 16),
                                  ("mxfp4", kv.NVFP4KV_VARIANT_MXFP4, mxc, vals // 2 + vals // 32)):
        ms, _ = time_steps(torch, steps, args.warmup,
                           lambda ev=None, var=var, c_=c_: kv.nvfp4kv_quantize_append_variant(var, c_, kc, vc, slots,
                                                                                              rk, rv), flush)
        t = float(np.mean(ms))
        gbs = (2 * vals + other + 8 * toks) / (t / 1e3) / 1e9
        out[f"extend_quantize_variant_{name}_per_layer"] = {"kernel_ms": t, "hbm_gbs": gbs,
                                                             "frac_of_measured_peak": gbs / hbm_peak}
    q = _bf16(torch, ew.q(0))
    cq = _dev(torch, ew.cu_q)
    o = torch.empty((q.shape[0], ew.num_q_heads, 128), dtype=torch.float32, device="cuda")
    attn = lambda ev=None: kv.nvfp4kv_extend_attention(q, cq, ew.chunk_len, wk, wv, cu, pl, o, ew.softmax_scale)
    ms, _ = time_steps(torch, max(3, min(steps, 10)), args.warmup, attn, flush)
    t = float(np.mean(ms))
    tflops = ew.attention_flops_per_layer() / (t / 1e3) / 1e12
    peak = measured_peaks()[0]["bf16_tflops"]
    out["extend_attention_per_layer"] = {
        "kernel_ms": t, "tflops": tflops, "frac_of_measured_bf16_peak": tflops / peak,
        "flops": ew.attention_flops_per_layer(), "x80_layers_ms": 80 * t,
        "note": "f16 operands (the tensor-core rate of bf16), f32 accumulate; 16 x 2048 queries x 64 heads over "
                "16384 + causal chunk keys"}
    return out


# ---------------------------------------------------------------------------
# CPU oracle timings (the baseline, not the target)
# ---------------------------------------------------------------------------

class OracleSample:
    """One (sequence, KV head) pair of a decode workload, prepared for the oracle:
    its cached prompt quantized by the oracle (setup), then per step the append
    of the new token and the fp64 decode over the first n tokens."""

    def __init__(self, wl, b, h):
        import oracle

        self.oracle, self.wl, self.b, self.h = oracle, wl, b, h
        k, v = wl.prompt_kv(b)
        new = wl.new_kv() if wl.append else None
        if wl.append:
            k = np.concatenate([k, new[0][b:b + 1]])
            v = np.concatenate([v, new[1][b:b + 1]])
        self.k = np.ascontiguousarray(k[:, h:h + 1])
        self.v = np.ascontiguousarray(v[:, h:h + 1])
        L = self.k.shape[0]
        self.L = L
        npg = (L + 15) // 16
        self.cache = oracle.Cache(npg, 1)
        oracle.quantize_append(self.cache, self.k[:L - 1], self.v[:L - 1], np.arange(L - 1, dtype=np.int64))
        G = wl.num_q_heads // wl.num_kv_heads
        self.q = np.ascontiguousarray(wl.q()[b:b + 1, h * G:(h + 1) * G])
        self.pt = np.arange(npg, dtype=np.int32)[None]

    def step(self, n):
        """Append the last token, then decode over the first n tokens; returns KV-tokens done."""
        self.oracle.quantize_append(self.cache, self.k[-1:], self.v[-1:], np.array([self.L - 1], np.int64))
        self.oracle.decode_attention(self.cache, self.q, self.pt, np.array([n], np.int32), self.wl.softmax_scale)
        return n / self.wl.num_kv_heads


def _oracle_worker(args):
    """One host process: whole (sequence, KV head) pairs of a decode workload
    through the oracle for about budget_s; returns (KV-tokens, seconds, pairs)."""
    index, b, budget_s = args
    wl = inputs.decode_config(index)
    sample = OracleSample(wl, b % wl.batch, b % wl.num_kv_heads)
    t0 = time.perf_counter()
    done, pairs = 0.0, 0
    while time.perf_counter() - t0 < budget_s:
        done += sample.step(sample.L)
        pairs += 1
    return done, time.perf_counter() - t0, pairs


def cpu_baseline(wl, budget_s=12.0):
    """The oracle as it stands on a bounded sample: whole (sequence, KV head)
    pairs, one process per host core (spawned: this process has used the GPU),
    each running for about budget_s; KV-tokens are counted per layer over all
    KV heads (a pair of L tokens is L / Hkv KV-tokens).  The rate of one of the
    concurrent processes is reported beside the total."""
    import multiprocessing as mp

    cores = os.cpu_count() or 1
    index = 2 if wl.name.startswith("decode_b32") else 1
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_worker, [(index, b, budget_s) for b in range(cores)])
    done = sum(r[0] for r in res)
    wall = max(r[1] for r in res)
    pairs = sum(r[2] for r in res)
    per_process = res[0][0] / res[0][1]
    return {"value": done / wall, "unit": UNIT, "cores": cores, "kind": "oracle",
            "per_process_value": per_process,
            "sample": f"{pairs} (sequence, KV head) pairs of {wl.name} over {cores} processes: append 1 token + "
                      f"fp64 decode over {wl.seq_lens[0]} tokens x {wl.num_q_heads // wl.num_kv_heads} query "
                      f"heads each; {wall:.1f} s wall"}


def _reference_worker(index, b, n, warmup, steps, barrier, results):
    """One host process of the reference arm: the oracle on one (sequence, KV
    head) pair, n tokens per step; the timed steps start together in every
    process (barrier) and report (KV-tokens, seconds)."""
    wl = inputs.decode_config(index)
    sample = OracleSample(wl, b % wl.batch, b % wl.num_kv_heads)
    for _ in range(warmup):
        sample.step(n)
    barrier.wait()
    t0 = time.perf_counter()
    done = 0.0
    for _ in range(steps):
        done += sample.step(n)
    results.put((b, done, time.perf_counter() - t0))


def reference_arm(args):
    """The oracle timed as the reference arm: one process per host core, each on
    its own (sequence, KV head) pair of the headline workload, every step a
    bounded sample (n tokens) so the whole run takes about --cpu-total-s."""
    import multiprocessing as mp

    world, rank, _ = dist_info()
    if rank != 0:
        return
    wl = inputs.decode_config(2)
    sample = OracleSample(wl, 0, 0)
    t0 = time.perf_counter()
    sample.step(sample.L)
    t_full = time.perf_counter() - t0
    per_step = args.cpu_total_s / max(1, args.steps + args.warmup)
    n = int(min(sample.L, max(16, sample.L * per_step / max(t_full, 1e-6))))
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    barrier, results = ctx.Barrier(cores), ctx.Queue()
    procs = [ctx.Process(target=_reference_worker, args=(2, b, n, args.warmup, args.steps, barrier, results))
             for b in range(cores)]
    for p in procs:
        p.start()
    res = [results.get() for _ in procs]
    for p in procs:
        p.join()
    done = sum(r[1] for r in res)
    dt = max(r[2] for r in res)
    value = done / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": wl.name, "batch": wl.batch, "ctx": int(wl.seq_lens[0]), "q_heads": wl.num_q_heads,
                   "kv_heads": wl.num_kv_heads, "head_dim": 128, "page_size": 16,
                   "step": f"oracle in {cores} processes: each appends 1 token and decodes (fp64) over {n} "
                           f"tokens of its own (sequence, KV head)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{cores} (sequence, KV head) pairs, {n} of {sample.L} tokens per step each"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def only_arm(args):
    """Run one workload's kernels a few times (for profiler command lines)."""
    import torch

    import nvfp4_quantized_paged_quantize_gb300 as kv

    kv.load()
    flush = make_l2_flush(torch)
    if args.only == "calibrate":
        x, amax = _calibration_input(torch, inputs.decode_config(3))
        time_steps(torch, args.steps, args.warmup, lambda ev=None: kv.nvfp4kv_tensor_amax(x, amax), flush)
    elif args.only in ("decode8k", "decode128k", "ragged"):
        b = DecodeBench(torch, kv, inputs.decode_config({"decode8k": 2, "decode128k": 3, "ragged": 4}[args.only]))
        time_steps(torch, args.steps, args.warmup, lambda ev=None: (b.append(), b.decode()), flush)
    elif args.only == "stream-probe":
        b = DecodeBench(torch, kv, inputs.decode_config(2))
        peak = float(measured_peaks()[0]["hbm_gbs"])
        print(json.dumps({"stream_probe_b32_ctx8k": stream_probe_lines(torch, kv, b, args.steps, args.warmup, flush,
                                                                        peak, float("nan"))}))
    else:
        ew = inputs.extend_config(num_layers=1)
        cache = kv.Cache.empty(ew.num_pages, ew.num_kv_heads, zero=True)
        for s_ in range(ew.batch):
            k, v = ew.prefix_kv(0, s_)
            kv.nvfp4kv_quantize_append(cache, _bf16(torch, k), _bf16(torch, v),
                                       _dev(torch, ew.slots(s_, 0, ew.prefix_len)))
        ks, vs = zip(*[ew.chunk_kv(0, s_) for s_ in range(ew.batch)])
        kc, vc = _bf16(torch, np.concatenate(ks)), _bf16(torch, np.concatenate(vs))
        slots = _dev(torch, ew.chunk_slots())
        pt, pl, cu = _dev(torch, ew.page_table), _dev(torch, ew.prefix_lens), _dev(torch, ew.cu_prefix)
        wk = torch.empty((ew.total_rows, ew.num_kv_heads, 128), dtype=torch.uint8, device="cuda")
        wv = torch.empty_like(wk)
        rows = _dev(torch, ew.chunk_ws_rows())
        q = _bf16(torch, ew.q(0))
        cq = _dev(torch, ew.cu_q)
        o = torch.empty((q.shape[0], ew.num_q_heads, 128), dtype=torch.float32, device="cuda")
        time_steps(torch, args.steps, args.warmup,
                   lambda ev=None: (kv.nvfp4kv_dequant_to_fp8_workspace(cache, pt, pl, cu, wk, wv),
                                    kv.nvfp4kv_quantize_append(cache, kc, vc, slots),
                                    kv.nvfp4kv_bf16_to_fp8_workspace(kc, vc, rows, wk, wv),
                                    kv.nvfp4kv_extend_attention(q, cq, ew.chunk_len, wk, wv, cu, pl, o,
                                                                ew.softmax_scale)), flush)
    torch.cuda.synchronize()
    print(json.dumps({"only": args.only, "steps": args.steps, "warmup": args.warmup, "ok": True}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--skip-secondary", action="store_true", help="only the headline workload")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--cpu-total-s", type=float, default=90.0, help="reference arm: total oracle seconds")
    ap.add_argument("--only", choices=["decode8k", "decode128k", "ragged", "extend", "calibrate", "stream-probe"],
                    help="run just one workload's kernels (profiler command lines); no JSON metric line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.only:
        only_arm(args)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
