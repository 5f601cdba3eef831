"""Benchmark of the paged FP8 MLA decode step on GB300.

One step = the whole hot path over one batch: ``mla_kv_append`` of the step's
new tokens (Q per request) into their page slots, then ``mla_decode`` (split
kernel + log-sum-exp combine) over every request's pages. Inputs are seeded
synthetic workloads (``paged_mla_decode_gb300.workloads``) resident in HBM.

Default workload: single-user long context -- batch 1, 64 heads, one query
token, 100,000 cached tokens, FP8 e4m3 cache, page size 64. The cache (57.6 MB)
would fit in L2, so R independent copies of it (different shuffled pages,
R * size >= 4 x L2) are rotated step by step.

Output: one JSON line (rank 0). ``value`` is the algorithmic KV bandwidth in
GB/s (unique cache bytes read per step / step time); steps/s, tokens/s and the
fraction of the measured HBM peak ride along. ``--impl reference`` times the
float64 CPU oracle on the same workload instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_mla_decode_gb300 import accounting  # noqa: E402
from paged_mla_decode_gb300 import workloads as wl  # noqa: E402

METRIC = "paged FP8 MLA decode: KV HBM GB/s (% of GB300 peak) and decode steps/sec"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES_FALLBACK = 129 * 1024 * 1024

CONFIGS = {
    "long": (lambda: wl.long_context(), "e4m3",
             "single-user long context: B=1 H=64 Q=1 L=100000, FP8 e4m3 cache, page 64"),
    "tiny": (lambda: wl.tiny(), "e4m3", "tiny: B=2 H=16 Q=1 L={1024,777}, e4m3, page 64"),
    "concurrent": (lambda: wl.concurrent(), "e4m3",
                   "concurrent decode: B=32 H=64 Q=1 L~U[60k,140k], FP8 e4m3 cache"),
    "concurrent_bf16": (lambda: wl.concurrent(), "bf16",
                        "concurrent decode: B=32 H=64 Q=1 L~U[60k,140k], BF16 cache"),
    "prefix_shared": (lambda: wl.prefix_shared(), "e4m3",
                      "prefix-shared: 16 groups x 4 forks, 120k shared prefix, e4m3"),
    "speculative": (lambda: wl.speculative(), "e4m3",
                    "speculative decode: B=32 Q=4 causal drafts, L~logN(142k), e4m3"),
}


def _rank_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# Decoder layers of the served model ("How to serve trillions of tokens for
# trillion-parameter coding agents", section "Tensor parallel was the best
# parallelism strategy for maximum interactivity": 61 layers of 576-element
# latent entries); one model decode step runs mla_decode once per layer.
MODEL_LAYERS = 61

FALLBACK_BF16_TFLOPS = 1900.0
FP8_PER_BF16 = 2.0   # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak(operands: str):
    """Dense tensor peak (TFLOP/s) for the MMA operand type, and where it came from.

    The measured bf16 burst figure; e4m3 operands (tcgen05 kind::f8f6f4) take it
    times the nominal fp8/bf16 ratio.
    """
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16, src = float(json.load(f)["bf16_tflops"]), "measured bf16_tflops"
    except Exception:
        bf16, src = FALLBACK_BF16_TFLOPS, "fallback 1.9 PFLOP/s bf16"
    if operands == "fp8":
        return bf16 * FP8_PER_BF16, f"{src} x {FP8_PER_BF16:g} (nominal fp8/bf16)"
    return bf16, src


def slowest_rank_ms(elapsed_ms, dist=None):
    """The timed region's length on the slowest rank (max over the process group)."""
    if dist is None:
        return float(elapsed_ms)
    import torch
    tt = torch.tensor([float(elapsed_ms)], dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def aggregate(values_ms, units_per_rank):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    t = max(values_ms)
    return sum(units_per_rank) / (t / 1e3), t


def _norm_uuid(u) -> str:
    u = str(u).strip().lower()
    return u[4:] if u.startswith("gpu-") else u


class ClockSampler:
    """nvidia-smi clocks and throttle reasons of this process's GPU, every 50 ms.

    Every visible GPU is sampled and the rows of the one whose UUID matches
    ``gpu_uuid`` are kept (all rows when there is no match and only one GPU
    answers), so that neither a UUID format nor an index remapping by
    CUDA_VISIBLE_DEVICES can leave the record empty.
    """

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.proc = None
        self.uuid = _norm_uuid(gpu_uuid) if gpu_uuid else None
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "50"]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.summarise(out, self.uuid)

    @staticmethod
    def summarise(text: str, uuid: str | None):
        """Median SM clock, max clock and active throttle reasons of the matching rows."""
        by_gpu = {}
        for line in text.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                row = (float(parts[1]), float(parts[2]), parts[5:9])
            except ValueError:
                continue
            by_gpu.setdefault(_norm_uuid(parts[0]), []).append(row)
        if uuid and uuid in by_gpu:
            rows = by_gpu[uuid]
        elif len(by_gpu) == 1:
            rows = next(iter(by_gpu.values()))
        else:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, flags in rows for n, f in zip(names, flags)
                          if f.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


def _profile_traffic():
    """DRAM bytes per launch from the committed ncu record, if its kernel source is unchanged.

    ``profiles/decode_long_ncu.json`` names the source file it was taken from and
    that file's sha256; a mismatch (the kernel changed since) gives None.
    """
    path = os.path.join(ROOT, "profiles", "decode_long_ncu.json")
    try:
        with open(path) as f:
            prof = json.load(f)
        with open(os.path.join(ROOT, prof["source"]), "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except (OSError, KeyError, ValueError):
        return None
    if prof.get("source_sha256") != digest:
        return None
    return prof.get("dram_bytes_per_launch")


def rooflines(nbytes, flops, launch_us, hbm_peak, hbm_src, tc_peak, tc_src, traffic=None):
    """The call's HBM and tensor rooflines; the first one returned is the bound.

    ``nbytes`` and ``flops`` are the algorithmic bytes and flops of one call,
    ``launch_us`` its measured duration; the bound is the resource that needs
    the longer time at its peak (HBM GB/s, tensor TFLOP/s).
    """
    kernel = "mla_decode call (split decode kernel + LSE combine kernel)"
    gbs = nbytes / (launch_us * 1e-6) / 1e9
    tfs = flops / (launch_us * 1e-6) / 1e12
    hbm = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
           "frac": gbs / hbm_peak, "traffic": traffic, "kernel": kernel,
           "peak_source": hbm_src, "algorithmic_bytes_per_launch": nbytes,
           "avg_launch_us": launch_us}
    tc = {"bound": "tensor", "achieved": tfs, "peak": tc_peak, "unit": "TFLOP/s",
          "frac": tfs / tc_peak, "traffic": traffic, "kernel": kernel, "peak_source": tc_src,
          "algorithmic_flops_per_launch": flops, "avg_launch_us": launch_us}
    if flops / (tc_peak * 1e12) > nbytes / (hbm_peak * 1e9):
        return tc, hbm
    return hbm, tc


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline field)
# ---------------------------------------------------------------------------
def _oracle_sample_step(w, pages_ref, b, start_page, n_tokens):
    from oracle import attention as oatt
    table = w.block_table[b:b + 1, start_page:].copy()
    lens = np.array([n_tokens], np.int32)
    return oatt.decode(w.q_bits[b:b + 1, :1], pages_ref, table, lens, w.sm_scale, w.kv_scale)


def _oracle_pages(w, kv_dtype, max_tokens):
    """Oracle-encoded pages of request 0 (or as many tokens as max_tokens)."""
    from oracle import e4m3 as oe4m3
    pages = np.zeros((w.num_pages, 64, 576), dtype=np.uint8 if kv_dtype == "e4m3" else np.uint16)
    flat = pages.reshape(-1, 576)
    seg = w.request_segments[0][0]
    bits = w.segment_latent(seg)[:max_tokens]
    slots = w.segment_slots(seg)[:max_tokens]
    flat[slots] = oe4m3.encode(oe4m3.bf16_bits_to_f64(bits), w.kv_scale) if kv_dtype == "e4m3" \
        else bits
    return pages


def cpu_oracle_rate(w, kv_dtype, seconds=15.0, n_tokens=None, steps=None):
    """Oracle throughput on request 0 of the workload: GB/s of KV and seconds per token."""
    L0 = int(w.seq_lens[0])
    n = min(L0, n_tokens or L0)
    pages = _oracle_pages(w, kv_dtype, n)
    bpt = accounting.kv_bytes_per_token(kv_dtype)
    times = []
    t_start = time.perf_counter()
    k = 0
    while True:
        t0 = time.perf_counter()
        _oracle_sample_step(w, pages, 0, 0, n)
        times.append(time.perf_counter() - t0)
        k += 1
        if steps is not None and k >= steps:
            break
        if steps is None and time.perf_counter() - t_start >= seconds:
            break
    per = sum(times) / len(times)
    return n * bpt / per / 1e9, per / n, n, len(times)


def run_reference(args):
    rank, world, _ = _rank_env()
    if rank != 0:
        return 0
    make, kv_dtype, desc = CONFIGS[args.config]
    w = make()
    L0 = int(w.seq_lens[0])
    # calibrate: the whole run (warmup + steps) should take about two minutes
    _, sec_per_tok, _, _ = cpu_oracle_rate(w, kv_dtype, n_tokens=min(L0, 4096), steps=1)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(64, min(L0, budget / sec_per_tok)))
    from oracle import attention as oatt  # noqa: F401
    pages = _oracle_pages(w, kv_dtype, n)
    for _ in range(args.warmup):
        _oracle_sample_step(w, pages, 0, 0, n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_sample_step(w, pages, 0, 0, n)
    dt = time.perf_counter() - t0
    per_step = dt / args.steps
    bpt = accounting.kv_bytes_per_token(kv_dtype)
    value = n * bpt / per_step / 1e9
    sample = (f"{n} of the {L0} tokens of request 0, all {w.num_heads} heads, per step "
              f"(float64 numpy oracle, BLAS threads = default)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "kv_dtype": kv_dtype},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args):
    import torch

    from paged_mla_decode_gb300 import binding

    rank, world, local = _rank_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load_library()

    make, kv_dtype, desc = CONFIGS[args.config]
    if args.seq_len:
        if args.config != "long":
            raise SystemExit("--seq-len applies to the long-context workload only")
        w = wl.long_context(seq_len=args.seq_len)
        desc = desc.replace("L=100000", f"L={args.seq_len}")
    else:
        w = make()
    B, Q, H = w.batch, w.num_queries, w.num_heads
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", L2_BYTES_FALLBACK)
    bpt = accounting.kv_bytes_per_token(kv_dtype)
    unique_bytes = w.unique_tokens * bpt
    copies = args.copies or max(1, math.ceil(4 * l2 / unique_bytes))
    maps, tables = w.cache_copies(copies)

    # ---- resident inputs: R cache copies filled through mla_kv_append ----
    dt = torch.uint8 if kv_dtype == "e4m3" else torch.bfloat16
    kv_scale = w.kv_scale if kv_dtype == "e4m3" else 1.0
    pages = torch.zeros((copies * w.num_pages, 64, 576), dtype=dt, device=dev)
    chunk = 1 << 16
    for si in range(len(w.segments)):
        bits = w.segment_latent(si)
        for a in range(0, bits.shape[0], chunk):
            x = torch.from_numpy(bits[a:a + chunk].view(np.int16)).view(torch.bfloat16).to(dev)
            lat, rope = x[:, :512].contiguous(), x[:, 512:].contiguous()
            for r in range(copies):
                slots = torch.from_numpy(w.segment_slots(si, maps[r])[a:a + chunk]).to(dev)
                binding.mla_kv_append(lat, rope, slots, pages, kv_scale)
    torch.cuda.synchronize()
    del x, lat, rope

    q = torch.from_numpy(w.q_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    seq_lens = torch.from_numpy(w.seq_lens).to(dev)
    tables_d = [torch.from_numpy(t).to(dev) for t in tables]
    fresh = torch.from_numpy(w.fresh_token_latent().view(np.int16)).view(torch.bfloat16).to(dev)
    fresh_lat, fresh_rope = fresh[:, :512].contiguous(), fresh[:, 512:].contiguous()
    base_slots = w.fresh_token_slots().astype(np.int64)
    fresh_slots = []
    for r in range(copies):
        page, off = base_slots // 64, base_slots % 64
        fresh_slots.append(torch.from_numpy((maps[r][page] * 64 + off).astype(np.int32)).to(dev))
    out = torch.empty((B, Q, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Q, H), dtype=torch.float32, device=dev)
    ws = torch.zeros(binding.mla_decode_workspace_size(B, Q, H), dtype=torch.uint8, device=dev)
    f16_ops = args.operands == "f16"

    # Forked sessions (the prefix-shared workload) go through the grouped decode,
    # which reads each shared page once for its group, unless --plain-decode.
    grouped = bool(w.extra.get("forks")) and not args.plain_decode and not f16_ops
    if grouped:
        forks = int(w.extra["forks"])
        prefix_pages = torch.from_numpy(w.extra["prefix_pages"]).to(dev)
        ws = torch.zeros(binding.mla_decode_grouped_workspace_size(B, Q, H), dtype=torch.uint8,
                         device=dev)

    def decode_call(qq, table, lens, o, l):
        if grouped:
            binding.mla_decode_grouped(qq, pages, table, lens, forks, prefix_pages, w.sm_scale,
                                       kv_scale, o, l, ws)
        else:
            binding.mla_decode(qq, pages, table, lens, w.sm_scale, kv_scale, o, l, ws,
                               f16_operands=f16_ops)

    def step(r, ev=None):
        binding.mla_kv_append(fresh_lat, fresh_rope, fresh_slots[r], pages, kv_scale)
        if ev is not None:
            ev[0].record()
        decode_call(q, tables_d[r], seq_lens, out, lse)
        if ev is not None:
            ev[1].record()

    # ---- one CUDA graph per cache copy; decode bracketed by external events ----
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for r in range(copies):
            step(r)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True, external=True),
            torch.cuda.Event(enable_timing=True, external=True)) for _ in range(copies)]
    graphs = []
    for r in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(r, evs[r])
        graphs.append(g)
    torch.cuda.synchronize()

    try:
        gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_uuid = None
    sampler = ClockSampler(gpu_uuid)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % copies].replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record()
        for i in range(args.steps):
            graphs[i % copies].replay()
        t_end.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    # The decode call's own duration: the events captured around it in each graph
    # hold that graph's latest replay, so replay the graphs in rotation and read
    # every pair after each full rotation.
    decode_ms = []
    with torch.cuda.stream(stream):
        while len(decode_ms) < args.call_samples:
            for r in range(copies):
                graphs[r].replay()
            stream.synchronize()
            decode_ms += [a.elapsed_time(b) for a, b in evs]
    decode_us = 1e3 * sum(decode_ms) / len(decode_ms)
    decode_us_median = 1e3 * statistics.median(decode_ms)

    elapsed_ms = slowest_rank_ms(elapsed_ms, dist)

    status = binding.read_device_status(ws)
    steps_per_s = args.steps / (elapsed_ms / 1e3)
    sb = accounting.step_bytes(w.seq_lens, Q, H, kv_dtype, unique_tokens=w.unique_tokens)
    kv_gbs = world * sb["kv"] * steps_per_s / 1e9
    tokens_per_s = world * B * Q * steps_per_s

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        # A step's inputs (q, lengths, block table, the new tokens and their slots)
        # sit packed in one pinned host block per cache copy and go over in one
        # copy; out and lse come back in one copy. Copy, append, decode and the
        # read-back are captured in one CUDA graph per copy; every step replays it
        # and waits for the result on the host.
        parts = [("q", q), ("lens", seq_lens), ("table", tables_d[0]), ("lat", fresh_lat),
                 ("rope", fresh_rope), ("slots", fresh_slots[0])]
        offs, in_bytes = {}, 0
        for name, t in parts:
            offs[name] = in_bytes
            in_bytes += (t.numel() * t.element_size() + 255) // 256 * 256

        def view(buf, name, like):
            n = like.numel() * like.element_size()
            return buf[offs[name]:offs[name] + n].view(like.dtype).view(like.shape)

        h_in = []
        for r in range(copies):
            hb = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
            for name, t in parts:
                src = {"table": tables_d[r], "slots": fresh_slots[r]}.get(name, t)
                view(hb, name, t).copy_(src.cpu())
            h_in.append(hb)
        d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        d_q, d_lens, d_table, d_lat, d_rope, d_slots = (view(d_in, n, t) for n, t in parts)
        out_b = out.numel() * out.element_size()
        res_bytes = out_b + lse.numel() * lse.element_size()
        d_res = torch.empty(res_bytes, dtype=torch.uint8, device=dev)
        e_out = d_res[:out_b].view(torch.bfloat16).view(out.shape)
        e_lse = d_res[out_b:].view(torch.float32).view(lse.shape)
        h_res = torch.empty(res_bytes, dtype=torch.uint8).pin_memory()
        n_e2e = max(1, min(args.steps, args.e2e_steps))

        def issue(r):
            d_in.copy_(h_in[r], non_blocking=True)
            binding.mla_kv_append(d_lat, d_rope, d_slots, pages, kv_scale)
            decode_call(d_q, d_table, d_lens, e_out, e_lse)
            h_res.copy_(d_res, non_blocking=True)

        with torch.cuda.stream(stream):
            issue(0)
        stream.synchronize()
        e2e_graphs = []
        for r in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                issue(r)
            e2e_graphs.append(g)

        def e2e_step(r):
            with torch.cuda.stream(stream):
                e2e_graphs[r].replay()
            stream.synchronize()

        for i in range(min(args.warmup, 20)):
            e2e_step(i % copies)
        t0 = time.perf_counter()
        for i in range(n_e2e):
            e2e_step(i % copies)
        e2e_dt = (time.perf_counter() - t0) / n_e2e
        # the bytes read back are the last step's device result
        if not torch.equal(h_res, d_res.cpu()):
            raise RuntimeError("e2e: the result read back differs from the device result")
        e2e = {"value": world * sb["kv"] / e2e_dt / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": res_bytes, "steps": n_e2e,
               "ms_per_step": e2e_dt * 1e3,
               "mode": "per step: one pinned H2D copy of the packed inputs, kv append, decode, "
                       "one D2H copy of out+lse, replayed as a CUDA graph; host waits each step"}

    # ---- the integrity check ("Protecting a shared KV cache"): a separate pass
    # before decode; its time per call beside the decode call's ----
    kv_check = None
    if not args.no_check:
        rng = np.random.default_rng(5)
        tags = torch.from_numpy(rng.integers(-2**31, 2**31, size=pages.shape[0],
                                             dtype=np.int64).astype(np.int32)).to(dev)
        expected = tags[tables_d[0].clamp(min=0).long()].contiguous()
        chk_status = torch.full((B,), -1, dtype=torch.int32, device=dev)
        chk_lens = torch.empty_like(seq_lens)
        per_graph = 20
        with torch.cuda.stream(stream):
            binding.mla_kv_check(tags, tables_d[0], expected, seq_lens, chk_status, chk_lens)
        torch.cuda.synchronize()
        gck = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gck, stream=stream):
            for _ in range(per_graph):
                binding.mla_kv_check(tags, tables_d[0], expected, seq_lens, chk_status, chk_lens)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(3):
                gck.replay()
            c0.record()
            reps = 20
            for _ in range(reps):
                gck.replay()
            c1.record()
        torch.cuda.synchronize()
        check_us = 1e3 * c0.elapsed_time(c1) / (reps * per_graph)
        # The check guards one decode step of the model, which runs mla_decode once
        # per layer; the pages' model has 61 layers.
        kv_check = {"us_per_call": check_us, "fraction_of_decode_call": check_us / decode_us,
                    "model_layers": MODEL_LAYERS,
                    "fraction_of_model_step": check_us / (MODEL_LAYERS * decode_us),
                    "requests_failed": int((chk_status != 0).sum().item()),
                    "pages_checked": int(sum(-(-int(n) // 64) for n in w.seq_lens))}

    peak, peak_kind = measured_peaks()
    decode_bytes = sb["total"]
    traffic = _profile_traffic() if args.config == "long" and args.operands == "fp8" else None
    operands = "bf16" if kv_dtype == "bf16" else args.operands
    flops = accounting.step_flops(w.seq_lens, Q, H)
    tpeak, tsrc = tensor_peak(operands)
    roofline, roofline_other = rooflines(
        decode_bytes, flops, decode_us, peak,
        f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
        else "fallback 6.8 TB/s", tpeak, tsrc, traffic)
    tensor_bound = roofline["bound"] == "tensor"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, _, n_tok, n_steps = cpu_oracle_rate(w, kv_dtype, seconds=args.cpu_seconds)
        cpu = {"value": rate, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{n_steps} full oracle decode(s) of request 0 ({n_tok} tokens, "
                         f"{H} heads), float64 numpy, BLAS threads = default"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": kv_gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": kv_dtype, "data": "synthetic",
            "config": {"workload": desc, "batch": B, "queries": Q, "heads": H,
                       "mma_operands": "bf16" if kv_dtype == "bf16" else args.operands,
                       "decode": "mla_decode_grouped" if grouped else
                                 ("mla_decode_f16_operands" if f16_ops else "mla_decode"),
                       "seq_lens_total": int(w.seq_lens.sum()), "unique_tokens": w.unique_tokens,
                       "kv_dtype": kv_dtype, "page_size": 64,
                       "l2": f"rotating {copies} cache copies "
                             f"({copies * unique_bytes / 1e6:.0f} MB > L2 {l2 / 1e6:.0f} MB)",
                       "parallelism": f"replicas x{world}"},
            "steps_per_s": world * steps_per_s, "tokens_per_s": tokens_per_s,
            "kv_gbs": kv_gbs, "pct_of_hbm_peak": 100.0 * kv_gbs / peak,
            "roofline": roofline,
            ("roofline_hbm" if tensor_bound else "roofline_tensor"): roofline_other,
            "logical_kv_gbs": world * accounting.step_bytes(w.seq_lens, Q, H, kv_dtype)["kv"]
            * steps_per_s / 1e9,
            "cpu_baseline": cpu, "e2e": e2e, "kv_check": kv_check,
            # per step: KV append, then the decode call's kernels (query split, decode,
            # combine; the grouped decode also plans its row table first)
            "gpu_launches": (5 if grouped else 4) * args.steps, "clocks": clocks,
            "decode_call_us": {"mean": decode_us, "median": decode_us_median,
                               "samples": len(decode_ms)},
            "device_status": status,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(CONFIGS), default="long")
    ap.add_argument("--operands", choices=["fp8", "f16"], default="fp8",
                    help="tensor-core operands for an e4m3 cache: its bytes (mla_decode) or "
                         "f16 after widening (mla_decode_f16_operands, the ablation)")
    ap.add_argument("--copies", type=int, default=0, help="cache copies rotated (0 = auto)")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-check", action="store_true",
                    help="skip timing the integrity check (mla_kv_check) beside the decode")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--call-samples", type=int, default=400,
                    help="event-timed decode calls behind the roofline's avg_launch_us")
    ap.add_argument("--plain-decode", action="store_true",
                    help="decode forked sessions with mla_decode instead of mla_decode_grouped")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="cached tokens of the long-context workload (0 = 100,000)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
