#!/usr/bin/env python3
"""Benchmark: paged GQA decode attention on the 24-layer, 14 q / 2 KV head model shape.

One step = one decode token for 32 sequences at context 2048 through all 24
layers: per layer the new token's K/V go into the paged cache and the token
attends over its context (paged_decode_append_attention: append, split-context
decode and split merge in one kernel; --unfused times kv_append +
paged_decode_attention instead).  Inputs are seeded
synthetic data (N(0,1) fp16) resident in HBM; the K/V pools (768 MiB per
step) are larger than L2, so every step streams its cache from HBM.

value       KV-cache bytes read per step / device time per step (GB/s), all ranks
e2e         the same metric through the C ABI with host buffers: per step the
            copies of q, k_new, v_new, slots, block table and context lengths
            in from pinned host memory and of the outputs back are timed (host
            wall clock) with the 24 calls, overlapped with them (staging-copy
            kernels, harness.HostStep); the step is captured once in a CUDA
            graph and replayed, as a serving loop runs it; eager_value is the
            same step issued call by call from Python
roofline    the decode call (append + decode + split merge, one kernel) alone:
            algorithmic bytes per launch / CUDA-event launch time, against the
            measured HBM copy bandwidth
cpu_baseline the fp64 CPU oracle on a bounded sample of the same workload

--impl reference times the fp64 CPU oracle on the same workload instead.
--suite prints one JSON line per further listed workload (--suite-part picks a
part, --suite-multi-t one multi-token T); --profile-configs runs each listed
configuration's call a few times, a short command for a per-configuration ncu
launch list; --profile-only replays the headline step without printing.
Multi-GPU (torchrun): every rank runs its own replica (weak scaling), no
collective on the data path; the timing barrier and max-over-ranks use
torch.distributed.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged GQA decode attention: KV-cache GB/s (% HBM peak) and decode tokens/s"
WORKLOAD = ("decode step of a 24-layer model: 32 sequences x context 2048 (incl. the new token), 14 q / 2 KV "
            "heads, head_dim 64, fp16, block size 16, block tables permuted over a pool of 32 x 2048 tokens; "
            "per layer the new token's K/V appended to the paged cache, then paged GQA decode attention")
L, B, CTX, HQ, HKV, D = 24, 32, 2048, 14, 2, 64


def kv_bytes_per_step(ctx_total: int, layers: int) -> int:
    """Algorithmic KV-cache bytes read per step: every context token's K and V rows, every layer."""
    return ctx_total * HKV * D * 2 * 2 * layers


def decode_call_bytes(ctx_total: int, nblocks_total: int) -> int:
    """Algorithmic bytes of one paged_decode_attention call (one layer): K/V rows, q, out (fp16), table."""
    return kv_bytes_per_step(ctx_total, 1) + B * HQ * D * 2 * 2 + nblocks_total * 4 + B * 4


# DRAM traffic of one decode launch (dram__bytes_read.sum + dram__bytes_write.sum) from an ncu capture of
# `bench.py --profile-only`, valid only for the decode sources it was taken on (sha256 of the files below).
DECODE_SOURCES = ("paged_kv_cache_27_gb300/csrc/decode.cu", "paged_kv_cache_27_gb300/csrc/decode_common.cuh",
                  "paged_kv_cache_27_gb300/csrc/ptx.cuh", "paged_kv_cache_27_gb300/csrc/kvc_internal.h")
NCU_DECODE_TRAFFIC = {"sources_sha256": "e85d0f413793837192b265257551d14610c53f4d97d6bd88e0fd9f7395eef05d",
                      "bytes_per_launch": 33681920}


def decode_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic():
    """Bytes per launch from the ncu capture, or None once the decode sources have changed since."""
    rec = NCU_DECODE_TRAFFIC
    if rec["bytes_per_launch"] is None or rec["sources_sha256"] != decode_sources_sha256():
        return None
    return rec["bytes_per_launch"]


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.samples = []
        self.proc = None
        self.thread = None
        self.uuid = gpu_uuid

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.samples.append(parts)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        return self.summary()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in self.samples for n, v in zip(names, s[4:8]) if v.lower() == "active"})
        pw = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples),
                "power_w_median": float(np.median(pw)) if pw else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier_max(value: float, world: int, device) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms_per_step_max: float) -> float:
    """Units all ranks processed per second: every rank runs its own replica (weak scaling) and the step time
    is the slowest rank's."""
    return units_per_rank * world / (ms_per_step_max * 1e-3)


# ---------------------------------------------------------------------------
# reference arm / CPU baseline: the fp64 oracle as it stands
# ---------------------------------------------------------------------------
def oracle_sample(wl, seqs: int, layers, nthreads=None):
    """Time the oracle's decode on `seqs` sequences of the given layers; returns (seconds, kv bytes)."""
    import oracle
    from oracle import paging
    sub_table = wl.block_table[:seqs]
    sub_ctx = wl.ctx[:seqs]
    secs, nbytes = 0.0, 0
    for layer in layers:
        kc, vc = paging.fill_layer(wl, layer)
        oracle.append(kc, vc, wl.k_new[layer], wl.v_new[layer], paging.step_slots(wl.block_table, wl.ctx, wl.bs))
        t0 = time.perf_counter()
        oracle.decode(wl.q[layer][:seqs], kc, vc, sub_table, sub_ctx, wl.scale, nthreads=nthreads)
        secs += time.perf_counter() - t0
        nbytes += int(sub_ctx.astype(np.int64).sum()) * HKV * D * 2 * 2
    return secs, nbytes


def oracle_single_sequence_one_thread(seconds=1.0):
    """The oracle's decode of the single-sequence workload (context 256, 1 q / 1 KV head) on one thread: time per
    call over about `seconds` of repeated calls."""
    import oracle
    from oracle import paging
    import workloads
    wl = workloads.single_sequence_256()
    kc, vc = paging.fill_layer(wl, 0)
    oracle.append(kc, vc, wl.k_new[0], wl.v_new[0], paging.step_slots(wl.block_table, wl.ctx, wl.bs))
    n, t = 0, 0.0
    while t < seconds:
        t0 = time.perf_counter()
        oracle.decode(wl.q[0], kc, vc, wl.block_table, wl.ctx, wl.scale, nthreads=1)
        t += time.perf_counter() - t0
        n += 1
    us = t / n * 1e6
    return {"us_per_call": us, "GBps": wl.kv_tokens * wl.Hkv * wl.D * 2 * 2 / (us * 1e-6) / 1e9, "cores": 1,
            "calls": n}


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    import oracle
    import workloads
    wl = workloads.model_decode_step(L=1)
    seqs = 8
    cores = oracle.default_threads()
    for _ in range(args.warmup):
        oracle_sample(wl, seqs, [0])
    secs, nbytes = 0.0, 0
    for _ in range(args.steps):
        s, n = oracle_sample(wl, seqs, [0])
        secs += s
        nbytes += n
    gbs = nbytes / secs / 1e9
    sample = f"{seqs} of the 32 sequences of one layer per step (context 2048, 14 q / 2 KV heads)"
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    import paged_kv_cache_27_gb300 as kvc
    from paged_kv_cache_27_gb300.harness import DecodeSession, HostStep
    import workloads

    wl = workloads.model_decode_step()
    sess = DecodeSession(wl, device=device, out_dtype=torch.float16, blocks_per_split=args.blocks_per_split).fill()
    ctx_total = int(wl.ctx.astype(np.int64).sum())
    nblocks_total = int(sum(-(-int(c) // 16) for c in wl.ctx))
    step_bytes = kv_bytes_per_step(ctx_total, L)
    fused = not args.unfused
    kvc.kvc_set_launch_overlap(not args.no_overlap)
    # combine kernel only when the longest context needs more than one cluster (8 splits)
    combine = 1 if sess.nsplit > 8 else 0
    launches_per_step = L * ((1 if fused else 2) + combine)

    stream = torch.cuda.Stream(device)
    graph = sess.capture(fused=fused, stream=stream)
    dgraph = sess.capture(fused=fused, decode_only=True, stream=stream)
    assert kvc.kvc_device_error_flags(clear=True) == 0

    if args.profile_only:
        # a short fixed run for the ncu launch list
        for _ in range(args.warmup + args.steps):
            graph.replay()
        torch.cuda.synchronize()
        return 0

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid).start()
    cur = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(cur)
    for _ in range(args.steps):
        graph.replay()
    t1.record(cur)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms_step = t0.elapsed_time(t1) / args.steps
    # keep the same load running briefly if the timed region was too short for clock samples
    soak_until = time.time() + max(0.0, 1.5 - ms_step * args.steps / 1e3)
    while time.time() < soak_until:
        for _ in range(50):
            graph.replay()
        torch.cuda.synchronize()
    clocks = sampler.stop()
    ms_step = barrier_max(ms_step, world, device)

    # the decode call alone (roofline): all 24 layers back to back, so every launch streams from HBM
    reps = max(5, min(200, args.steps))
    for _ in range(3):
        dgraph.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(cur)
    for _ in range(reps):
        dgraph.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    us_decode = e0.elapsed_time(e1) * 1e3 / (reps * L)

    # end to end through the public API with host buffers: the step's inputs come from pinned host memory and its
    # output goes back there, the copies overlapped with the calls (HostStep)
    hs = HostStep(sess)
    h2d, d2h = hs.h2d_bytes, hs.d2h_bytes

    def e2e_step():
        hs.run(fused)

    # (a) the step as a serving loop runs it: the public-API calls and the copies captured once in a CUDA graph
    # and replayed per step (the inputs are read from the pinned host buffers at every replay, the outputs
    # land in the pinned host buffer); host wall clock around the replays
    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    egraph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device=device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        with torch.cuda.graph(egraph, stream=side):
            e2e_step()
    torch.cuda.synchronize()
    for _ in range(3):
        egraph.replay()
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for _ in range(e2e_steps):
        egraph.replay()
    torch.cuda.synchronize()
    ms_e2e = (time.perf_counter() - w0) * 1e3 / e2e_steps
    ms_e2e = barrier_max(ms_e2e, world, device)
    # (b) the same calls issued one by one from Python, no graph (prepared calls: ~4.5 us of host time each)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    ms_e2e_eager = (time.perf_counter() - w0) * 1e3 / e2e_steps
    ms_e2e_eager = barrier_max(ms_e2e_eager, world, device)

    # CPU baseline (rank 0, N = 1 only): the oracle on a bounded sample of the same workload
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        secs, nbytes, layers = 0.0, 0, 0
        while secs < 10.0 and layers < 20 * L:
            s, n = oracle_sample(wl, B, [layers % L])
            secs += s
            nbytes += n
            layers += 1
        cpu = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": oracle.default_threads(), "kind": "oracle",
               "sample": f"{layers} layer decodes of the 24-layer step (all 32 sequences, cycling layers), fp64, "
                         f"{secs:.1f} s of oracle time",
               "single_sequence_ctx256_one_thread": oracle_single_sequence_one_thread()}

    peak, peak_kind = load_peaks()
    # the other listed workloads, measured after the headline (rank 0 at N = 1; not part of the timed step)
    suite = None
    if rank == 0 and world == 1 and not args.no_suite:
        suite = config_summary(device, peak, load_tflops_peak()[0])
    gbs = whole_job_rate(step_bytes, world, ms_step) / 1e9
    call_bytes = decode_call_bytes(ctx_total, nblocks_total) + (B * HKV * D * 2 * 2 * 2 if fused else 0)
    achieved = call_bytes / (us_decode * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": L, "batch_per_gpu": B, "context": CTX, "q_heads": HQ,
                   "kv_heads": HKV, "head_dim": D, "block_size": 16, "num_splits": sess.nsplit,
                   "blocks_per_split": sess.bps, "l2": "inputs larger than L2: 768 MiB of K/V per step",
                   "launch": "CUDA graph of the 24-layer step" + ("" if args.no_overlap else
                                                                             ", programmatic dependent launch"),
                   "append": "fused into the decode kernel" if fused else "separate kv_append kernel"},
        "tokens_per_s": whole_job_rate(B, world, ms_step),
        "pct_hbm_peak": gbs / world / peak * 100.0,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": measured_traffic(), "peak_kind": peak_kind,
                     "kernel": ("paged_decode_append_attention" if fused else "paged_decode_attention")
                               + " call, one layer (split merge inside the kernel, on chip)",
                     "bytes_per_launch": call_bytes, "us_per_launch": us_decode},
        "cpu_baseline": cpu,
        "suite": suite,
        "e2e": {"value": whole_job_rate(step_bytes, world, ms_e2e) / 1e9, "unit": "GB/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "host wall clock per step: the step's inputs (block table, context lengths, slots, then "
                       "per layer q / k_new / v_new) read from one pinned host buffer and the outputs written back "
                       "to pinned host memory by kvc_copy_async staging kernels in the same stream as the 24 "
                       "public-API calls (header and layers 0-1 before the first call, later layers in pieces "
                       "alongside earlier calls, outputs eight layers at a time alongside a later call, the last "
                       "layer's after its call), captured once in a CUDA graph and replayed",
                "eager_value": whole_job_rate(step_bytes, world, ms_e2e_eager) / 1e9,
                "eager_ms_per_step": ms_e2e_eager},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    sess.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# --suite: one JSON line per further configuration (parity is the tests' job; these only measure)
# ---------------------------------------------------------------------------
class L2Flush:
    """Empties the L2 between timed calls: writes a 256 MiB buffer (nothing of the previous call stays in the
    129 MB L2), then reads a second 256 MiB buffer, so that the dirty lines of the write are written back before
    the timed call starts instead of competing with its reads."""

    def __init__(self, device):
        import torch
        self.w = torch.zeros(64 << 20, dtype=torch.float32, device=device)
        self.r = torch.zeros(64 << 20, dtype=torch.float32, device=device)
        self.out = torch.zeros(1, dtype=torch.float32, device=device)

    def __call__(self):
        import torch
        self.w.add_(1)
        torch.sum(self.r, dim=0, keepdim=True, out=self.out)


def _flush_l2(flush):
    flush()


def _timed_calls(fn, reps, flush_buf, stream):
    """Mean device time (us) of fn(), each call preceded by an L2 flush outside the timed span."""
    import torch
    total = 0.0
    for r in range(reps + 3):
        _flush_l2(flush_buf)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        if r >= 3:
            total += e0.elapsed_time(e1) * 1e3
    return total / reps


def _graph_of(fn, device):
    """fn() captured once in a CUDA graph with programmatic dependent launch between its kernels; returns the
    graph's replay (inputs must stay at the same addresses)."""
    import torch
    import paged_kv_cache_27_gb300 as kvc
    kvc.kvc_set_launch_overlap(True)
    try:
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                fn()
    finally:
        kvc.kvc_set_launch_overlap(False)
    return g.replay


def _decode_state(B, ctx, Hq, Hkv, D, device, seed):
    """Seeded synthetic decode state made on the device (K/V N(0,1) fp16, permuted block tables)."""
    import torch
    bs = 16
    nblk = -(-ctx // bs)
    NB = B * nblk
    gen = torch.Generator(device=device).manual_seed(seed)
    k_pool = torch.empty((NB, Hkv, bs, D), dtype=torch.float16, device=device)
    v_pool = torch.empty_like(k_pool)
    step = max(1, (1 << 24) // (Hkv * bs * D))
    for a in range(0, NB, step):
        for pool in (k_pool, v_pool):
            pool[a:a + step] = torch.randn(pool[a:a + step].shape, generator=gen, device=device).half()
    rng = np.random.default_rng(seed)
    table = torch.from_numpy(rng.permutation(NB).astype(np.int32).reshape(B, nblk)).to(device)
    ctx_t = torch.full((B,), ctx, dtype=torch.int32, device=device)
    q = torch.randn((B, Hq, D), generator=gen, device=device).half()
    kn = torch.randn((B, Hkv, D), generator=gen, device=device).half()
    vn = torch.randn((B, Hkv, D), generator=gen, device=device).half()
    return k_pool, v_pool, table, ctx_t, q, kn, vn


def _cfg1_us_per_call(device, stream):
    """Single sequence at context 256 (1 q / 1 KV head): the fused append + decode call, 100 back to back in a CUDA
    graph (latency-bound; the 64 KiB context stays in L2)."""
    import torch
    import workloads
    from paged_kv_cache_27_gb300 import harness
    wl = workloads.single_sequence_256()
    sess = harness.DecodeSession(wl, device=device, out_dtype=torch.float32).fill()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(100):
            sess.decode_append(0)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(10):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    sess.close()
    return e0.elapsed_time(e1) * 1e3 / 1000, wl.kv_tokens * wl.Hkv * wl.D * 2 * 2


def _cfg3_serving_mix(device, stream, flush):
    """The shared-prefix serving mix after its step's block management: the fused append + decode call with L2
    flushed, and attention alone through the plain decode and the cascade call."""
    import torch
    import paged_kv_cache_27_gb300 as kvc
    import workloads
    from paged_kv_cache_27_gb300 import harness
    mix = workloads.shared_prefix_mix()
    res = harness.serving_mix(mix, device=device, poison=False)
    table = torch.from_numpy(res["block_table"]).to(device)
    ctx = torch.from_numpy(mix.ctx).to(device)
    q = torch.from_numpy(mix.q).to(device)
    kn, vn = torch.from_numpy(mix.k_new).to(device), torch.from_numpy(mix.v_new).to(device)
    out = torch.empty((mix.B, mix.Hq, mix.D), dtype=torch.float16, device=device)
    max_ctx = int(mix.ctx.max())
    _, _, ws = kvc.paged_decode_plan(mix.B, mix.Hq, mix.Hkv, mix.D, max_ctx)
    wsb = torch.zeros(max(ws, 16), dtype=torch.uint8, device=device)
    step = lambda: kvc.paged_decode_append_attention(q, kn, vn, res["k_cache"], res["v_cache"], table, ctx,
                                                      mix.scale, out, wsb, max_ctx)
    us_step = _timed_calls(step, 20, flush, stream)
    pools = [(res["k_cache"], res["v_cache"])] + [(res["k_cache"].clone(), res["v_cache"].clone()) for _ in range(23)]
    calls = [lambda k=k, v=v: kvc.paged_decode_append_attention(q, kn, vn, k, v, table, ctx, mix.scale, out, wsb,
                                                                 max_ctx) for (k, v) in pools]
    us_graph = _layers_graph_us(calls, device, stream, flush)
    del pools, calls
    plain = lambda: kvc.paged_decode_attention(q, res["k_cache"], res["v_cache"], table, ctx, mix.scale, out, wsb,
                                               max_ctx)
    us_plain = _timed_calls(plain, 20, flush, stream)
    gs, sh, mxs = kvc.kv_cascade_groups(res["block_table"], mix.ctx)
    gs_d, sh_d = torch.from_numpy(gs).to(device), torch.from_numpy(sh).to(device)
    cws = kvc.paged_decode_cascade_plan(mix.B, mix.Hq, mix.Hkv, mix.D, max_ctx, len(gs) - 1, mxs)
    cwsb = torch.zeros(max(cws, 16), dtype=torch.uint8, device=device)
    casc = lambda: kvc.paged_decode_cascade_attention(q, res["k_cache"], res["v_cache"], table, ctx, gs_d, sh_d, mxs,
                                                      mix.scale, out, cwsb, max_ctx)
    us_casc = _timed_calls(casc, 20, flush, stream)
    row = 2 * mix.Hkv * mix.D * 2
    logical = int(mix.ctx.astype(np.int64).sum()) * row
    used = set()
    for b in range(mix.B):
        used.update(res["block_table"][b, :-(-int(mix.ctx[b]) // 16)].tolist())
    unique = len(used) * 16 * row
    return {"us_step": us_step, "us_step_graph24": us_graph, "logical_bytes": logical, "unique_bytes": unique,
            "tokens": mix.B,
            "us_decode_plain": us_plain, "us_decode_cascade": us_casc}


def _cfg4_cell_us(B, c, device, stream, flush):
    """One long-context cell: the fused append + decode call with L2 flushed; returns (us, splits, blocks/split)."""
    import torch
    import paged_kv_cache_27_gb300 as kvc
    kp, vp, tb, ct, q4, kn4, vn4 = _decode_state(B, c, 14, 2, 64, device, seed=B * 1000003 + c)
    o4 = torch.empty((B, 14, 64), dtype=torch.float16, device=device)
    ns, bps, ws = kvc.paged_decode_plan(B, 14, 2, 64, c)
    w4 = torch.zeros(max(ws, 16), dtype=torch.uint8, device=device)
    fn = lambda: kvc.paged_decode_append_attention(q4, kn4, vn4, kp, vp, tb, ct, 0.125, o4, w4, c)
    us = _timed_calls(fn, 20, flush, stream)
    del kp, vp
    return us, ns, bps


def _layers_graph_us(calls, device, stream, flush, reps=10):
    """Device time per call of `calls` (one per layer, each on its own pools) captured in one CUDA graph with
    launch overlap between consecutive kernels, as a model's decode step runs its layers; L2 flushed before each
    timed replay, so every layer reads its pools from HBM.  Returns us per layer."""
    import torch
    g = _graph_of(lambda: [c() for c in calls], device)
    for _ in range(3):
        g()
    torch.cuda.synchronize()
    total = 0.0
    for _ in range(reps):
        _flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g()
        e1.record(stream)
        e1.synchronize()
        total += e0.elapsed_time(e1) * 1e3
    return total / (reps * len(calls))


def _cfg4_cell_graph_us(B, c, device, stream, flush, layers=24):
    """One long-context cell as the layers of a decode step: `layers` fused append + decode calls, each on its own
    K/V pools (copies of one seeded pool, so no layer's reads hit another's lines in L2), in one CUDA graph with
    launch overlap; L2 flushed before each replay.  Returns us per layer."""
    import torch
    import paged_kv_cache_27_gb300 as kvc
    kp, vp, tb, ct, q4, kn4, vn4 = _decode_state(B, c, 14, 2, 64, device, seed=B * 1000003 + c)
    pools = [(kp, vp)] + [(kp.clone(), vp.clone()) for _ in range(layers - 1)]
    o4 = torch.empty((B, 14, 64), dtype=torch.float16, device=device)
    _, _, ws = kvc.paged_decode_plan(B, 14, 2, 64, c)
    w4 = torch.zeros(max(ws, 16), dtype=torch.uint8, device=device)
    calls = [lambda k=k, v=v: kvc.paged_decode_append_attention(q4, kn4, vn4, k, v, tb, ct, 0.125, o4, w4, c)
             for (k, v) in pools]
    us = _layers_graph_us(calls, device, stream, flush)
    del pools, kp, vp
    return us


def _prefill_us(seqlens, Hq, Hkv, D, causal, precise, device, stream, flush):
    """A varlen prefill call with L2 flushed, per call and replayed from a graph; returns (us, us_graph, flops)."""
    import torch
    import paged_kv_cache_27_gb300 as kvc
    T = sum(seqlens)
    gen = torch.Generator(device=device).manual_seed(T * 31 + Hq)
    qq = torch.randn((T, Hq, D), generator=gen, device=device).half()
    kk = torch.randn((T, Hkv, D), generator=gen, device=device).half()
    vv = torch.randn((T, Hkv, D), generator=gen, device=device).half()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32), device=device)
    oo = torch.empty((T, Hq, D), dtype=torch.float16, device=device)
    fn = lambda: kvc.prefill_attention(qq, kk, vv, cu, max(seqlens), 1.0 / np.sqrt(D), causal, oo, precise=precise)
    us = _timed_calls(fn, 20, flush, stream)
    us_g = _timed_calls(_graph_of(fn, device), 20, flush, stream)
    pairs = sum(s * (s + 1) // 2 for s in seqlens) if causal else sum(s * s for s in seqlens)
    return us, us_g, 4 * D * Hq * pairs


def _fp8_vs_fp16_graph(device, stream, Lq=24, Bq=32, Cq=2048):
    """24-layer decode-only CUDA graphs with launch overlap over the model step's shape (32 x 2048, 14 / 2 heads,
    D = 64): fp16 pools, and the same pools quantized to fp8 e4m3 with per-row scales through kv_append_fp8 (24
    different pools per form, more than L2).  Device time per layer of each form."""
    import torch
    import paged_kv_cache_27_gb300 as kvc
    kp0, vp0, tbq, ctq, _, _, _ = _decode_state(Bq, Cq, 14, 2, 64, device, seed=2024)
    NBq = kp0.shape[0]
    gen = torch.Generator(device=device).manual_seed(99)
    k16 = [kp0] + [torch.randn(kp0.shape, generator=gen, device=device).half() for _ in range(Lq - 1)]
    v16 = [vp0] + [torch.randn(vp0.shape, generator=gen, device=device).half() for _ in range(Lq - 1)]
    rec_bytes = kvc.kv_fp8_record_bytes(64)
    r8 = [torch.empty((NBq, 2, rec_bytes), dtype=torch.uint8, device=device) for _ in range(Lq)]
    all_slots = torch.arange(NBq * 16, dtype=torch.int64, device=device)
    for l in range(Lq):  # every pool row quantized through the library's append
        rows = lambda t: t.permute(0, 2, 1, 3).reshape(NBq * 16, 2, 64).contiguous()
        kvc.kv_append_fp8(rows(k16[l]), rows(v16[l]), all_slots, r8[l])
    qs = [torch.randn((Bq, 14, 64), generator=gen, device=device).half() for _ in range(Lq)]
    outq = torch.empty((Bq, 14, 64), dtype=torch.float16, device=device)
    _, _, wq = kvc.paged_decode_plan(Bq, 14, 2, 64, Cq)
    wsq = torch.zeros(max(wq, 16), dtype=torch.uint8, device=device)
    res_q = {}
    kvc.kvc_set_launch_overlap(True)
    try:
        for name in ("fp16", "fp8"):
            def body():
                for l in range(Lq):
                    if name == "fp16":
                        kvc.paged_decode_attention(qs[l], k16[l], v16[l], tbq, ctq, 0.125, outq, wsq, Cq)
                    else:
                        kvc.paged_decode_attention_fp8(qs[l], r8[l], tbq, ctq, 0.125, outq, wsq, Cq)
            body()
            torch.cuda.synchronize()
            gq = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(device)
            with torch.cuda.stream(side):
                with torch.cuda.graph(gq, stream=side):
                    body()
            for _ in range(5):
                gq.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(100):
                gq.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            res_q[name] = e0.elapsed_time(e1) * 1e3 / (100 * Lq)
    finally:
        kvc.kvc_set_launch_overlap(False)
    del k16, v16, r8
    toks = Bq * Cq
    b16 = toks * 2 * 2 * 64 * 2
    b8 = toks * 2 * 2 * 64 + toks * 2 * 2 * 4
    return {"us_per_layer_fp16": res_q["fp16"], "us_per_layer_fp8": res_q["fp8"],
            "speedup": res_q["fp16"] / res_q["fp8"],
            "GBps_fp16": b16 / (res_q["fp16"] * 1e-6) / 1e9, "GBps_fp8": b8 / (res_q["fp8"] * 1e-6) / 1e9,
            "tokens_per_s_fp16": Bq / (res_q["fp16"] * Lq * 1e-6), "tokens_per_s_fp8": Bq / (res_q["fp8"] * Lq * 1e-6),
            "bytes_per_layer_fp16": b16, "bytes_per_layer_fp8": b8}


def config_summary(device, peak, tflops_peak):
    """Compact figures for the other listed workloads, taken after the headline measurement (one GPU): single
    sequence, shared-prefix serving mix, the 12 long-context cells, and the two prefill shapes."""
    import torch
    t0 = time.perf_counter()
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(device)
    gbs = lambda nbytes, us: nbytes / (us * 1e-6) / 1e9
    out = {"timing": "device time (CUDA events) per call; L2 flushed before each timed call (256 MiB written, then "
                     "256 MiB of another buffer read, so the L2 holds no dirty lines), except the single sequence "
                     "(100 calls in a graph, L2-resident)"}
    us, nb = _cfg1_us_per_call(device, stream)
    out["single_sequence_ctx256"] = {"us_per_call": round(us, 3), "GBps": round(gbs(nb, us), 1), "kv_bytes": nb}
    c3 = _cfg3_serving_mix(device, stream, flush)
    out["serving_mix_B200"] = {
        "us_per_step": round(c3["us_step"], 2), "tokens_per_s": round(c3["tokens"] / (c3["us_step"] * 1e-6)),
        "logical_GBps": round(gbs(c3["logical_bytes"], c3["us_step"]), 1),
        "unique_GBps": round(gbs(c3["unique_bytes"], c3["us_step"]), 1),
        "pct_hbm_peak_unique": round(gbs(c3["unique_bytes"], c3["us_step"]) / peak * 100, 2),
        "us_per_layer_graph24": round(c3["us_step_graph24"], 2),
        "tokens_per_s_graph24": round(c3["tokens"] / (c3["us_step_graph24"] * 24e-6)),
        "logical_GBps_graph24": round(gbs(c3["logical_bytes"], c3["us_step_graph24"]), 1),
        "unique_GBps_graph24": round(gbs(c3["unique_bytes"], c3["us_step_graph24"]), 1),
        "pct_hbm_peak_unique_graph24": round(gbs(c3["unique_bytes"], c3["us_step_graph24"]) / peak * 100, 2),
        "us_decode_plain": round(c3["us_decode_plain"], 2), "us_decode_cascade": round(c3["us_decode_cascade"], 2),
        "cascade_speedup": round(c3["us_decode_plain"] / c3["us_decode_cascade"], 3),
        "logical_bytes": c3["logical_bytes"], "unique_bytes": c3["unique_bytes"]}
    cells = []
    for B in (1, 4, 16):
        for c in (4096, 16384, 65536, 131072):
            us, ns, bps = _cfg4_cell_us(B, c, device, stream, flush)
            usg = _cfg4_cell_graph_us(B, c, device, stream, flush)
            nb = B * c * 2 * 2 * 64 * 2
            cells.append({"B": B, "ctx": c, "us_per_call": round(us, 2), "GBps": round(gbs(nb, us), 1),
                          "pct_hbm_peak": round(gbs(nb, us) / peak * 100, 2), "splits": ns, "blocks_per_split": bps,
                          "us_per_layer_graph24": round(usg, 2), "GBps_graph24": round(gbs(nb, usg), 1),
                          "pct_hbm_peak_graph24": round(gbs(nb, usg) / peak * 100, 2)})
    out["long_context"] = cells
    out["long_context_timing"] = (
        "us_per_call: one call between CUDA events, L2 flushed before it; includes the launch gaps around a lone "
        "kernel (an event pair around a trivial kernel measures ~4 us on this GPU). *_graph24: the cell as the 24 "
        "layers of a decode step (each layer its own K/V pools), one CUDA graph with launch overlap, L2 flushed "
        "before each replay, device time per layer")
    for name, seqlens, hq, hkv in (("prefill_varlen_37_120_8_200_8x8_d64_causal", (37, 120, 8, 200), 8, 8),
                                   ("prefill_gqa_2x256_8x2_d64_causal", (256, 256), 8, 2)):
        us, us_g, fl = _prefill_us(seqlens, hq, hkv, 64, True, False, device, stream, flush)
        out[name] = {"us_per_call": round(us, 2), "us_per_call_graph": round(us_g, 2),
                     "TFLOPs_graph": round(fl / (us_g * 1e-6) / 1e12, 2),
                     "pct_tensor_peak_graph": round(fl / (us_g * 1e-6) / 1e12 / tflops_peak * 100, 3),
                     "flops": fl}
    q = _fp8_vs_fp16_graph(device, stream)
    out["quantized_cache_fp8_vs_fp16_24L_B32_ctx2048"] = {
        "us_per_layer_fp16": round(q["us_per_layer_fp16"], 3), "us_per_layer_fp8": round(q["us_per_layer_fp8"], 3),
        "speedup": round(q["speedup"], 3), "GBps_fp8": round(q["GBps_fp8"], 1),
        "pct_hbm_peak_fp8": round(q["GBps_fp8"] / peak * 100, 2),
        "timing": "24-layer decode-only CUDA graphs with launch overlap, device time per layer"}
    del flush
    torch.cuda.synchronize()
    out["seconds"] = round(time.perf_counter() - t0, 1)
    return out


def load_tflops_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 = fp16 tensor rate)"
    except Exception:
        return 1900.0, "fallback"


def run_profile_configs(args):
    """Each listed configuration's hot-path call four times (a warm-up call, then three with L2 flushed before
    each): a short command for a per-configuration ncu launch list.  One configuration's buffers at a time (at most
    ~2.2 GB on the device); prints one JSON line per configuration with the mean CUDA-event time of the three
    flushed calls and the number of library kernels one call launches."""
    import torch
    import paged_kv_cache_27_gb300 as kvc
    import workloads
    from paged_kv_cache_27_gb300 import harness
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(device)
    flush()  # the flush's own kernels load before the first timed call
    torch.cuda.synchronize()

    def once(name, fn, launches, algorithmic_bytes=None, flops=None, launches_before=0):
        fn()
        torch.cuda.synchronize()
        total = 0.0
        for _ in range(3):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            total += e0.elapsed_time(e1) * 1e3
        rec = {"profile_config": name, "us_mean_of_3": total / 3, "calls": 4, "kernels_per_call": launches,
               "library_launches_before": launches_before}
        if algorithmic_bytes is not None:
            rec["algorithmic_bytes"] = algorithmic_bytes
        if flops is not None:
            rec["flops"] = flops
        print(json.dumps(rec), flush=True)

    # 1: single sequence at context 256, fused append + decode
    wl = workloads.single_sequence_256()
    sess = harness.DecodeSession(wl, device=device, out_dtype=torch.float32).fill()
    once("1: single sequence, B=1, 1/1 heads, D=64, ctx 256",
         lambda: kvc.paged_decode_append_attention(sess.q[0], sess.k_new[0], sess.v_new[0], sess.k_pool[0],
                                                   sess.v_pool[0], sess.block_table, sess.context_lens, wl.scale,
                                                   sess.out[0], sess.workspace, sess.max_ctx), 1,
         algorithmic_bytes=256 * 2 * 64 * 2)
    sess.close()
    # 2: one layer of the 24-layer step (32 x 2048, 14 / 2 heads), fused append + decode
    kp, vp, tb, ct, q, kn, vn = _decode_state(32, 2048, 14, 2, 64, device, seed=5)
    o = torch.empty((32, 14, 64), dtype=torch.float16, device=device)
    _, _, ws = kvc.paged_decode_plan(32, 14, 2, 64, 2048)
    w = torch.zeros(max(ws, 16), dtype=torch.uint8, device=device)
    once("2: one layer of the decode step, B=32, 14/2 heads, D=64, ctx 2048",
         lambda: kvc.paged_decode_append_attention(q, kn, vn, kp, vp, tb, ct, 0.125, o, w, 2048), 1,
         algorithmic_bytes=32 * 2048 * 512)
    del kp, vp
    # 3: the shared-prefix serving mix after its step's block management, fused append + decode
    mix = workloads.shared_prefix_mix()
    res = harness.serving_mix(mix, device=device, poison=False)
    table = torch.from_numpy(res["block_table"]).to(device)
    ctx = torch.from_numpy(mix.ctx).to(device)
    q3 = torch.from_numpy(mix.q).to(device)
    kn3, vn3 = torch.from_numpy(mix.k_new).to(device), torch.from_numpy(mix.v_new).to(device)
    o3 = torch.empty((mix.B, mix.Hq, mix.D), dtype=torch.float16, device=device)
    mc = int(mix.ctx.max())
    ns3, _, ws3 = kvc.paged_decode_plan(mix.B, mix.Hq, mix.Hkv, mix.D, mc)
    w3 = torch.zeros(max(ws3, 16), dtype=torch.uint8, device=device)
    once("3: shared-prefix serving mix, B=200, 14/2 heads, D=64, ctx U{16..4096}",
         lambda: kvc.paged_decode_append_attention(q3, kn3, vn3, res["k_cache"], res["v_cache"], table, ctx,
                                                   mix.scale, o3, w3, mc), 1,
         algorithmic_bytes=int(mix.ctx.astype(np.int64).sum()) * 512, launches_before=1)  # the mix's own step
    del res
    # 4: the long-context cells, fused append + decode
    for B in (1, 4, 16):
        for c in (4096, 16384, 65536, 131072):
            kp, vp, tb, ct, q, kn, vn = _decode_state(B, c, 14, 2, 64, device, seed=B * 1000003 + c)
            o = torch.empty((B, 14, 64), dtype=torch.float16, device=device)
            ns, bps, ws = kvc.paged_decode_plan(B, 14, 2, 64, c)
            w = torch.zeros(max(ws, 16), dtype=torch.uint8, device=device)
            nblk = -(-c // 16)
            parts = -(-nblk // bps)
            once(f"4: B={B}, ctx={c}, 14/2 heads, D=64",
                 lambda: kvc.paged_decode_append_attention(q, kn, vn, kp, vp, tb, ct, 0.125, o, w, c),
                 2 if parts > 1 else 1, algorithmic_bytes=B * c * 512)
            del kp, vp, tb, ct, q, kn, vn, o, w
            torch.cuda.empty_cache()
    # 5: the two small prefills as their step runs: causal prefill, every token's K/V appended into a paged
    # cache, the next token's K/V appended, one decode step over the cache
    for name, wl5 in (("5: varlen prefill, seqlens 37/120/8/200, 8/8 heads, D=64, causal, then a decode step",
                       workloads.varlen_prefill()),
                      ("5: GQA prefill, B=2 x 256, 8/2 heads, D=64, causal, then a decode step",
                       workloads.gqa_prefill())):
        dv = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        q5, k5, v5, cu5 = dv(wl5.q), dv(wl5.k), dv(wl5.v), dv(wl5.cu_seqlens)
        T = q5.shape[0]
        n5 = len(wl5.seqlens)
        o5 = torch.empty((T, wl5.Hq, wl5.D), dtype=torch.float16, device=device)
        cfg5 = kvc.KvcConfig(num_layers=1, num_blocks=wl5.NB, num_kv_heads=wl5.Hkv, head_dim=wl5.D,
                             block_size=wl5.bs)
        kp5 = torch.zeros(cfg5.pool_shape, dtype=torch.float16, device=device)
        vp5 = torch.zeros_like(kp5)
        h5 = kvc.kv_cache_create(cfg5, kp5, vp5)
        seqlens = np.array(wl5.seqlens, np.int32)
        slots_all = dv(kvc.kv_slot_mapping(wl5.block_table, np.zeros(n5, np.int32), seqlens, wl5.bs))
        slots_new = dv(kvc.kv_slot_mapping(wl5.block_table, seqlens, np.ones(n5, np.int32), wl5.bs))
        qd, kd, vd = dv(wl5.q_dec), dv(wl5.k_dec), dv(wl5.v_dec)
        ctx5 = seqlens + 1
        tb5, ct5 = dv(wl5.block_table), dv(ctx5)
        od = torch.empty((n5, wl5.Hq, wl5.D), dtype=torch.float16, device=device)
        _, _, ws5 = kvc.paged_decode_plan(n5, wl5.Hq, wl5.Hkv, wl5.D, int(ctx5.max()))
        w5 = torch.zeros(max(ws5, 16), dtype=torch.uint8, device=device)

        def step5():
            kvc.prefill_attention(q5, k5, v5, cu5, max(wl5.seqlens), wl5.scale, True, o5)
            kvc.kv_append(h5, 0, k5, v5, slots_all)
            kvc.kv_append(h5, 0, kd, vd, slots_new)
            kvc.paged_decode_attention(qd, kp5[0], vp5[0], tb5, ct5, wl5.scale, od, w5, int(ctx5.max()))
        row = wl5.Hkv * wl5.D * 2 * 2  # K and V bytes of one token
        once(name, step5, 2,  # the prefill and the decode kernel (the appends are not in the list's filter)
             algorithmic_bytes=T * (wl5.Hq + 2 * wl5.Hkv) * wl5.D * 2 + (T + n5) * row + int(ctx5.sum()) * row,
             flops=4 * wl5.D * wl5.Hq * sum(s_ * (s_ + 1) // 2 for s_ in wl5.seqlens))
        kvc.kv_cache_destroy(h5)


def run_suite(args):
    import torch

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    peak, peak_kind = load_peaks()
    tflops_peak, tflops_kind = load_tflops_peak()
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(device)
    emit = lambda d: print(json.dumps(dict(suite=True, **d)), flush=True)

    if args.suite_part in ("all", "decode"):
        run_suite_decode(device, stream, flush, emit, peak)
    elif args.suite_part == "multi":
        run_suite_multi(device, stream, flush, emit, peak, args.suite_multi_t)
    elif args.suite_part == "cascade":
        run_suite_cascade(device, stream, flush, emit, peak)
    if args.suite_part in ("all", "prefill"):
        run_suite_prefill(device, stream, flush, emit, tflops_peak, tflops_kind)
    return 0


def run_suite_decode(device, stream, flush, emit, peak):
    import torch
    import paged_kv_cache_27_gb300 as kvc
    import workloads
    from paged_kv_cache_27_gb300 import harness

    # one sequence at context 256 (L2-resident, latency-bound)
    us, _ = _cfg1_us_per_call(device, stream)
    emit({"config": "single sequence: B=1, 1 q / 1 KV head, D=64, context 256", "us_per_decode": us,
          "note": "fused append + decode, 100 back-to-back calls in a CUDA graph; latency-bound, the 64 KiB context "
                  "sits in L2"})

    # shared-prefix serving mix: 200 sequences, groups of 8 share a 512-token prefix (refcounted blocks)
    c3 = _cfg3_serving_mix(device, stream, flush)
    us = c3["us_step"]
    logical, unique = c3["logical_bytes"], c3["unique_bytes"]
    emit({"config": "shared-prefix serving mix: B=200, 14 q / 2 KV heads, D=64, ctx ~ U{16..4096}, groups of 8 share a 512-token prefix",
          "us_per_step": us, "tokens_per_s": c3["tokens"] / (us * 1e-6),
          "logical_GBps": logical / (us * 1e-6) / 1e9, "unique_GBps": unique / (us * 1e-6) / 1e9,
          "logical_bytes": logical, "unique_bytes": unique, "pct_hbm_peak_unique": unique / (us * 1e-6) / 1e9 / peak * 100,
          "us_per_layer_graph24": c3["us_step_graph24"],
          "unique_GBps_graph24": unique / (c3["us_step_graph24"] * 1e-6) / 1e9,
          "pct_hbm_peak_unique_graph24": unique / (c3["us_step_graph24"] * 1e-6) / 1e9 / peak * 100,
          "us_decode_plain": c3["us_decode_plain"],
          "note": "fused append + decode per step, L2 flushed before each step; shared prefix blocks are read "
                  "once per sequence (logical) but may hit in L2 (unique = distinct blocks); graph24: the step as "
                  "the 24 layers of a CUDA graph, each on its own pools, L2 flushed per replay"})

    run_suite_cascade(device, stream, flush, emit, peak)

    run_suite_multi(device, stream, flush, emit, peak)

    # quantized cache (NEXT-4): 24-layer decode-only graphs with launch overlap, fp16 vs fp8
    qres = _fp8_vs_fp16_graph(device, stream)
    emit({"config": "quantized cache: 24-layer decode-only graph, 32 x 2048, 14 q / 2 KV heads, D=64, fp16 vs fp8 e4m3",
          **qres, "pct_hbm_peak_fp8": qres["GBps_fp8"] / peak * 100})
    # long contexts, where streaming dominates: B=16 x 65536, one call each with L2 flushed
    for (Bl, Cl) in ((16, 65536), (4, 131072)):
        kpl, vpl, tbl, ctl, ql, _, _ = _decode_state(Bl, Cl, 14, 2, 64, device, seed=Bl + Cl)
        NBl = kpl.shape[0]
        r8l = torch.empty((NBl, 2, kvc.kv_fp8_record_bytes(64)), dtype=torch.uint8, device=device)
        rows = lambda t: t.permute(0, 2, 1, 3).reshape(NBl * 16, 2, 64).contiguous()
        kvc.kv_append_fp8(rows(kpl), rows(vpl), torch.arange(NBl * 16, dtype=torch.int64, device=device), r8l)
        ol = torch.empty((Bl, 14, 64), dtype=torch.float16, device=device)
        _, _, wl_ = kvc.paged_decode_plan(Bl, 14, 2, 64, Cl)
        wsl = torch.zeros(max(wl_, 16), dtype=torch.uint8, device=device)
        us16 = _timed_calls(lambda: kvc.paged_decode_attention(ql, kpl, vpl, tbl, ctl, 0.125, ol, wsl, Cl), 20, flush,
                            stream)
        us8 = _timed_calls(lambda: kvc.paged_decode_attention_fp8(ql, r8l, tbl, ctl, 0.125, ol, wsl,
                                                                   Cl), 20, flush, stream)
        tl = Bl * Cl
        b16l, b8l = tl * 2 * 2 * 64 * 2, tl * 2 * 2 * 64 + tl * 2 * 2 * 4
        emit({"config": f"quantized cache: B={Bl} x ctx {Cl}, 14 q / 2 KV heads, D=64, one call, fp16 vs fp8 e4m3",
              "us_fp16": us16, "us_fp8": us8, "speedup": us16 / us8, "GBps_fp16": b16l / (us16 * 1e-6) / 1e9,
              "GBps_fp8": b8l / (us8 * 1e-6) / 1e9, "pct_hbm_peak_fp8": b8l / (us8 * 1e-6) / 1e9 / peak * 100})
        del kpl, vpl, r8l

    # head_dim 128 shapes: the 7B-class model (32 q / 8 KV heads) and the 32 x 32 x 128 MHA shape
    for Hq, Hkv in ((32, 8), (32, 32)):
        B, c, D = 32, 2048, 128
        kp, vp, tb, ct, qd, knd, vnd = _decode_state(B, c, Hq, Hkv, D, device, seed=Hq * 100 + Hkv)
        od = torch.empty((B, Hq, D), dtype=torch.float16, device=device)
        ns, bps, ws = kvc.paged_decode_plan(B, Hq, Hkv, D, c)
        wd = torch.zeros(max(ws, 16), dtype=torch.uint8, device=device)
        fn = lambda: kvc.paged_decode_append_attention(qd, knd, vnd, kp, vp, tb, ct, 1.0 / np.sqrt(D), od, wd, c)
        us = _timed_calls(fn, 20, flush, stream)
        nbytes = B * c * Hkv * D * 2 * 2
        emit({"config": f"head_dim 128: B={B}, ctx={c}, {Hq} q / {Hkv} KV heads, D={D} (one layer)",
              "us_per_call": us, "GBps": nbytes / (us * 1e-6) / 1e9,
              "pct_hbm_peak": nbytes / (us * 1e-6) / 1e9 / peak * 100, "splits": ns, "blocks_per_split": bps,
              "kv_bytes": nbytes})
        del kp, vp

    # long contexts, B in {1, 4, 16} x ctx in {4k, 16k, 64k, 128k}
    for B in (1, 4, 16):
        for c in (4096, 16384, 65536, 131072):
            us, ns, bps = _cfg4_cell_us(B, c, device, stream, flush)
            usg = _cfg4_cell_graph_us(B, c, device, stream, flush)
            nbytes = B * c * 2 * 2 * 64 * 2
            emit({"config": f"long context: B={B}, ctx={c}, 14 q / 2 KV heads, D=64", "us_per_call": us,
                  "GBps": nbytes / (us * 1e-6) / 1e9, "pct_hbm_peak": nbytes / (us * 1e-6) / 1e9 / peak * 100,
                  "us_per_layer_graph24": usg, "GBps_graph24": nbytes / (usg * 1e-6) / 1e9,
                  "pct_hbm_peak_graph24": nbytes / (usg * 1e-6) / 1e9 / peak * 100,
                  "splits": ns, "blocks_per_split": bps, "kv_bytes": nbytes})


def run_suite_cascade(device, stream, flush, emit, peak, mix=None, res=None):
    """Cascade decode against the plain decode: per call with L2 flushed, and the same call replayed from a CUDA
    graph (launch overlap between its kernels), L2 flushed before each replay."""
    import torch
    import paged_kv_cache_27_gb300 as kvc
    import workloads
    from paged_kv_cache_27_gb300 import harness

    if mix is None:
        mix = workloads.shared_prefix_mix()
        res = harness.serving_mix(mix, device=device, poison=False)
    table = torch.from_numpy(res["block_table"]).to(device)
    ctx = torch.from_numpy(mix.ctx).to(device)
    q = torch.from_numpy(mix.q).to(device)
    out = torch.empty((mix.B, mix.Hq, mix.D), dtype=torch.float16, device=device)
    max_ctx = int(mix.ctx.max())
    row = 2 * mix.Hkv * mix.D * 2  # K + V bytes per token
    logical = int(mix.ctx.astype(np.int64).sum()) * row
    # the shared-prefix mix, attention only: the plain decode vs the cascade (each group's shared prefix read once)
    _, _, pws = kvc.paged_decode_plan(mix.B, mix.Hq, mix.Hkv, mix.D, max_ctx)
    pwsb = torch.zeros(max(pws, 16), dtype=torch.uint8, device=device)
    plain = lambda: kvc.paged_decode_attention(q, res["k_cache"], res["v_cache"], table, ctx, mix.scale, out, pwsb,
                                               max_ctx)
    us_plain = _timed_calls(plain, 20, flush, stream)
    gs, sh, mxs = kvc.kv_cascade_groups(res["block_table"], mix.ctx)
    gs_d, sh_d = torch.from_numpy(gs).to(device), torch.from_numpy(sh).to(device)
    cws = kvc.paged_decode_cascade_plan(mix.B, mix.Hq, mix.Hkv, mix.D, max_ctx, len(gs) - 1, mxs)
    cwsb = torch.zeros(max(cws, 16), dtype=torch.uint8, device=device)
    casc = lambda: kvc.paged_decode_cascade_attention(q, res["k_cache"], res["v_cache"], table, ctx, gs_d, sh_d, mxs,
                                                      mix.scale, out, cwsb, max_ctx)
    us_casc = _timed_calls(casc, 20, flush, stream)
    us_plain_g = _timed_calls(_graph_of(plain, device), 20, flush, stream)
    us_casc_g = _timed_calls(_graph_of(casc, device), 20, flush, stream)
    shared_reads = int(sum(int(sh[b]) for b in range(mix.B)) - sum(int(sh[gs[g]]) for g in range(len(gs) - 1)))
    emit({"config": "shared-prefix mix, attention only: plain decode vs cascade (shared prefix blocks read once per group)",
          "us_plain": us_plain, "us_cascade": us_casc, "speedup": us_plain / us_casc,
          "us_plain_graph": us_plain_g, "us_cascade_graph": us_casc_g, "speedup_graph": us_plain_g / us_casc_g,
          "groups": len(gs) - 1, "max_shared_blocks": mxs,
          "block_reads_saved": shared_reads * mix.Hkv, "bytes_saved": shared_reads * 16 * row,
          "logical_GBps_plain": logical / (us_plain * 1e-6) / 1e9,
          "logical_GBps_cascade": logical / (us_casc * 1e-6) / 1e9})

    # a long shared prefix (not a listed config): 8 groups x 8 sequences share 8192 tokens, 1..200 private
    cw = workloads.cascade_decode(4242, [8] * 8, [512] * 8, list(np.random.default_rng(7).integers(1, 201, size=64)))
    cq, ckp, cvp = (torch.from_numpy(x).to(device) for x in (cw.q, cw.k_pool, cw.v_pool))
    ctb, cct = torch.from_numpy(cw.block_table).to(device), torch.from_numpy(cw.ctx).to(device)
    cgs, csh = torch.from_numpy(cw.group_start).to(device), torch.from_numpy(cw.shared_blocks).to(device)
    cout = torch.empty((64, cw.Hq, cw.D), dtype=torch.float16, device=device)
    cmax = int(cw.ctx.max())
    _, _, pws2 = kvc.paged_decode_plan(64, cw.Hq, cw.Hkv, cw.D, cmax)
    pw2 = torch.zeros(max(pws2, 16), dtype=torch.uint8, device=device)
    cws2 = kvc.paged_decode_cascade_plan(64, cw.Hq, cw.Hkv, cw.D, cmax, 8, 512)
    cw2 = torch.zeros(max(cws2, 16), dtype=torch.uint8, device=device)
    us_p = _timed_calls(lambda: kvc.paged_decode_attention(cq, ckp, cvp, ctb, cct, cw.scale, cout, pw2, cmax), 20,
                        flush, stream)
    plain2 = lambda: kvc.paged_decode_attention(cq, ckp, cvp, ctb, cct, cw.scale, cout, pw2, cmax)
    casc2 = lambda: kvc.paged_decode_cascade_attention(cq, ckp, cvp, ctb, cct, cgs, csh, 512, cw.scale, cout, cw2, cmax)
    us_c = _timed_calls(casc2, 20, flush, stream)
    us_pg = _timed_calls(_graph_of(plain2, device), 20, flush, stream)
    us_cg = _timed_calls(_graph_of(casc2, device), 20, flush, stream)
    lb = int(cw.ctx.astype(np.int64).sum()) * row
    ub = (8 * 512 * 16 + int(sum(int(c) - 8192 for c in cw.ctx))) * row
    emit({"config": "supplementary (not a listed config): 8 groups x 8 sequences sharing an 8192-token prefix, "
                    "1..200 private tokens each, 14 q / 2 KV heads, D=64",
          "us_plain": us_p, "us_cascade": us_c, "speedup": us_p / us_c,
          "us_plain_graph": us_pg, "us_cascade_graph": us_cg, "speedup_graph": us_pg / us_cg,
          "logical_bytes": lb, "unique_bytes": ub,
          "logical_GBps_plain": lb / (us_p * 1e-6) / 1e9, "unique_GBps_cascade": ub / (us_c * 1e-6) / 1e9})
    del ckp, cvp


def run_suite_multi(device, stream, flush, emit, peak, only_t=0):
    import torch
    import paged_kv_cache_27_gb300 as kvc

    # multi-token decode (speculative verification): T new tokens per sequence, B=32, context 2048; one call
    # with L2 flushed (host marshalling and launch included), and a 24-layer graph with launch overlap
    # (device time per layer; the pools of the 24 layers together exceed L2)
    Lm = 24
    kpm0, vpm0, tbm, ctm, _, _, _ = _decode_state(32, 2048, 14, 2, 64, device, seed=77)
    genm = torch.Generator(device=device).manual_seed(78)
    kml = [kpm0] + [torch.randn(kpm0.shape, generator=genm, device=device).half() for _ in range(Lm - 1)]
    vml = [vpm0] + [torch.randn(vpm0.shape, generator=genm, device=device).half() for _ in range(Lm - 1)]
    nbytes = 32 * 2048 * 2 * 2 * 64 * 2
    for T in ((only_t,) if only_t else (1, 2, 3, 4, 8)):
        qms = [torch.randn((32, T, 14, 64), generator=genm, device=device).half() for _ in range(Lm)]
        om = torch.empty((32, T, 14, 64), dtype=torch.float16, device=device)
        wsm = torch.zeros(max(kvc.paged_decode_multi_plan(32, 14, 2, 64, 2048, T), 16), dtype=torch.uint8,
                          device=device)
        us = _timed_calls(lambda: kvc.paged_decode_multi_attention(qms[0], kml[0], vml[0], tbm, ctm, 0.125, om, wsm,
                                                                   2048), 20, flush, stream)

        def body():
            for l in range(Lm):
                kvc.paged_decode_multi_attention(qms[l], kml[l], vml[l], tbm, ctm, 0.125, om, wsm, 2048)
        kvc.kvc_set_launch_overlap(True)
        try:
            body()
            torch.cuda.synchronize()
            gm = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(device)
            with torch.cuda.stream(side):
                with torch.cuda.graph(gm, stream=side):
                    body()
            for _ in range(5):
                gm.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(50):
                gm.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            us_g = e0.elapsed_time(e1) * 1e3 / (50 * Lm)
        finally:
            kvc.kvc_set_launch_overlap(False)
        emit({"config": f"multi-token decode: T={T} new tokens per sequence, B=32, ctx=2048, 14 q / 2 KV heads, D=64",
              "us_per_call": us, "GBps": nbytes / (us * 1e-6) / 1e9,
              "pct_hbm_peak": nbytes / (us * 1e-6) / 1e9 / peak * 100, "tokens_per_s": 32 * T / (us * 1e-6),
              "us_per_layer_graph": us_g, "GBps_graph": nbytes / (us_g * 1e-6) / 1e9,
              "pct_hbm_peak_graph": nbytes / (us_g * 1e-6) / 1e9 / peak * 100,
              "tokens_per_s_graph": 32 * T / (us_g * Lm * 1e-6)})
        del qms
    del kml, vml, kpm0, vpm0


def run_suite_prefill(device, stream, flush, emit, tflops_peak, tflops_kind):
    import torch
    import paged_kv_cache_27_gb300 as kvc

    # prefill shapes: causal varlen prefill on the tensor cores
    def prefill_case(name, seqlens, Hq, Hkv, D, causal=True, precise=False):
        us, us_g, flops = _prefill_us(seqlens, Hq, Hkv, D, causal, precise, device, stream, flush)
        tf = flops / (us * 1e-6) / 1e12
        emit({"config": name, "p_precision": "split (fp16 high part + residual)" if precise else "fp16",
              "us_per_call": us, "TFLOPs": tf, "pct_tensor_peak": tf / tflops_peak * 100,
              "us_per_call_graph": us_g, "TFLOPs_graph": flops / (us_g * 1e-6) / 1e12,
              "flops": flops, "peak_TFLOPs": tflops_peak, "peak_kind": tflops_kind,
              "note": "algorithmic flops (masked half not counted)" + (
                  "; the split form's tensor work is 1.5x that (P V runs for both parts of P)" if precise else "")})

    prefill_case("varlen prefill, seqlens 37/120/8/200, 8/8 heads, D=64, causal", (37, 120, 8, 200), 8, 8, 64)
    prefill_case("GQA prefill, B=2 x 256, 8/2 heads, D=64, causal", (256, 256), 8, 2, 64)
    prefill_case("supplementary (not a listed config): varlen x16, seqlens 592/1920/128/3200, 8/8, D=64, causal",
                 (592, 1920, 128, 3200), 8, 8, 64)
    prefill_case("supplementary (not a listed config): 4 x 4096 tokens, 32/8 heads, D=64, causal",
                 (4096,) * 4, 32, 8, 64)
    prefill_case("supplementary (not a listed config): 4 x 4096 tokens, 32/8 heads, D=128, causal",
                 (4096,) * 4, 32, 8, 128)
    prefill_case("supplementary (not a listed config): 4 x 4096 tokens, 32/8 heads, D=128, causal",
                 (4096,) * 4, 32, 8, 128, precise=True)
    prefill_case("supplementary (not a listed config): 4 x 4096 tokens, 32/8 heads, D=128, non-causal",
                 (4096,) * 4, 32, 8, 128, causal=False)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--blocks-per-split", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-suite", action="store_true", help="skip the other workloads' figures in the headline line")
    ap.add_argument("--unfused", action="store_true", help="separate kv_append + paged_decode_attention calls")
    ap.add_argument("--no-overlap", action="store_true", help="no programmatic dependent launch")
    ap.add_argument("--profile-only", action="store_true", help="replay warmup+steps graph steps, print nothing")
    ap.add_argument("--suite", action="store_true",
                    help="instead of the headline line: one JSON line per further configuration (1, 3, 4, 5)")
    ap.add_argument("--suite-part", choices=["all", "decode", "prefill", "multi", "cascade"], default="all",
                    help="decode: every decode configuration (multi-token and cascade included); multi / cascade: "
                         "those lines only")
    ap.add_argument("--profile-configs", action="store_true",
                    help="each listed configuration's call four times (a warm-up, three with L2 flushed): a short command for ncu")
    ap.add_argument("--suite-multi-t", type=int, default=0,
                    help="with --suite-part multi: only this number of new tokens per sequence (1..8)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if not 0 <= args.suite_multi_t <= 8:
        ap.error("--suite-multi-t must be in 1..8 (0: every listed T)")
    if args.impl == "reference":
        return run_reference(args)
    if args.suite:
        return run_suite(args)
    if args.profile_configs:
        return run_profile_configs(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
