"""Benchmark of the quantised KV-cache decode step on GB300.

Workload: Llama-3-8B-shaped decode attention, one layer (reported x32 for the
model step): batch 16, 32 query heads, 8 KV heads, head_dim 128, context
32768, bf16 activations, K 2-bit per channel / V 4-bit per token in 32-token
/ 32-channel groups, fp16 residual 32, sinks 4 + window 128. K channel (h, c)
is scaled by a seeded exp(U(0, ln 75)); V, q ~ N(0, 1). Inputs are synthetic
and generated on the device; the cache (543 MB per layer step) is larger
than L2, so no flush is needed between steps.

One step = kv_append of one new token (K, V) + kv_decode_attn, the whole
hot path of a decode step for one layer. Reported:
  value      effective bandwidth over the step's algorithmic bytes (GB/s)
  roofline   the decode kernels (split-KV partitions, then exact pools and
             LSE merge): algorithmic bytes / their average duration (CUDA
             events the library records on the launching stream around
             both), against the measured HBM peak
  e2e        the same step through the public API with host buffers
             (pinned host -> device inputs, device -> host output, copied
             on a second stream into double buffers so that they overlap
             the neighbouring steps' kernels)
  cpu_baseline  the CPU oracle timed on a bounded sample of the workload

--impl reference times the CPU oracle (the reference arm) on the same
workload, a bounded sample per step.
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

os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Quantised-KV decode attn: HBM GB/s (% of peak), µs/step; append tokens/s"
FALLBACK_HBM_GBS = 6800.0
APPEND_CALLS = 256  # kv_append calls timed on their own
WORKLOAD = dict(batch=16, n_q_heads=32, n_kv_heads=8, head_dim=128, context=32768, act_dtype="bf16",
                k_bits=2, v_bits=4, n_sink=4, window=128, layers_reported=32)
WORKLOAD_NAME = ("llama8b decode attention: B16 Hq32 Hkv8 D128 context 32768 bf16, "
                 "KIVI K2/V4 groups 32, residual 32, sinks 4 + window 128; one layer timed, x32 reported")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def slowest_rank(pg, values, device):
    """Every rank's timings replaced by the maximum over ranks (the job is
    as slow as its slowest replica); identity without a process group."""
    if pg is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_gbs(world, bytes_per_rank_step, ms_per_step):
    """Aggregate bandwidth of `world` replicas each moving bytes_per_rank_step
    per step of ms_per_step (the slowest rank's)."""
    return world * bytes_per_rank_step / (ms_per_step / 1e3) / 1e9


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampled every 20 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


DECODE_SOURCES = ("decode_kivi.cuh", "decode_common.cuh", "decode.cu", "decode_d128_k2.cu", "kvq_layout.h",
                  "kvq_internal.h", "kvq_device.cuh")
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "decode_traffic_llama8b.json")


def decode_sources_sha256():
    """sha256 of the decode kernels' sources, concatenated in DECODE_SOURCES order."""
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, "bit_kv_cache_append_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic():
    """DRAM bytes (read + write) of one decode at batch 16 from the ncu
    capture recorded in TRAFFIC_RECORD, if that capture was taken on the
    decode sources as they are now; None otherwise."""
    try:
        with open(TRAFFIC_RECORD) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    if rec.get("decode_sources_sha256") != decode_sources_sha256():
        return None
    return int(rec["dram_bytes_per_launch_b16"])


PREFILL_REPS = 5


def timed_prefill(torch, cache, k, v, stream, reps):
    """Median time (ms, CUDA events) of `reps` prefills of layer 0 with k, v;
    the cache is reset before every prefill after the first, and is left
    holding the last one."""
    times = []
    for r in range(reps):
        if r:
            cache.reset()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cache.prefill_quantize(0, k, v)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times)


def make_inputs(torch, w, seed, n_tokens, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    B, H, D = w["batch"], w["n_kv_heads"], w["head_dim"]
    fac = torch.exp(torch.rand((H, D), generator=g, device=device) * math.log(75.0))
    k = (torch.randn((B, H, n_tokens, D), generator=g, device=device) * fac[None, :, None, :]).to(torch.bfloat16)
    v = torch.randn((B, H, n_tokens, D), generator=g, device=device).to(torch.bfloat16)
    return k, v, fac


def algorithmic_bytes(stats, w):
    """Bytes the decode must read: every code, scale, zero and exact row it
    attends to, plus q in and the fp32 output."""
    B, Hq, D = w["batch"], w["n_q_heads"], w["head_dim"]
    cache = (stats["code_bytes"] + stats["kmeta_bytes"] + stats["vmeta_bytes"] + stats["sink_bytes"]
             + stats["tail_bytes"])
    return cache + B * Hq * D * 2 + B * Hq * D * 4


def warm_prefill(torch, binding, dev, cfg, dtype):
    """One small prefill on a scratch cache of the same configuration, so
    that the kernels the timed prefill runs are loaded and configured
    before it (the library's kernels load lazily on first launch)."""
    small = dict(cfg, batch=1, max_tokens=256)
    if small.get("rope_max_pos"):
        small["rope_max_pos"] = 256
    scratch = binding.KVCache(device=dev, **small)
    H, D = cfg["n_kv_heads"], cfg["head_dim"]
    x = torch.randn((1, H, 100, D), device=dev).to(dtype)
    scratch.prefill_quantize(0, x, x)
    torch.cuda.synchronize()
    del scratch


def append_bytes(w):
    """kv_append of one token: K and V read, written to the exact tail."""
    B, H, D = w["batch"], w["n_kv_heads"], w["head_dim"]
    return 2 * (B * H * D * 2) * 2


def oracle_sequence(seed=7):
    """One sequence of the workload (all 8 KV heads, 32767-token prefill and
    one append) in the CPU oracle."""
    import numpy as np
    import torch
    from oracle import CacheConfig, OracleCache
    w = WORKLOAD
    L, H, D = w["context"], w["n_kv_heads"], w["head_dim"]
    rng = np.random.default_rng(seed)
    fac = np.exp(rng.uniform(0, math.log(75.0), size=(H, D))).astype(np.float32)
    rb = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).float().numpy()
    k = rb(rng.standard_normal((1, H, L, D), dtype=np.float32) * fac[None, :, None, :])
    v = rb(rng.standard_normal((1, H, L, D), dtype=np.float32))
    q = rb(rng.standard_normal((1, w["n_q_heads"], D), dtype=np.float32))
    oc = OracleCache(CacheConfig(n_layers=1, batch=1, n_kv_heads=H, n_q_heads=w["n_q_heads"], head_dim=D,
                                 max_tokens=L + 64, k_bits=w["k_bits"], v_bits=w["v_bits"],
                                 n_sink=w["n_sink"], window=w["window"], act_dtype="bf16"))
    oc.prefill_quantize(0, k[:, :, : L - 1], v[:, :, : L - 1])
    oc.append(0, k[:, :, L - 1:], v[:, :, L - 1:])
    return oc, q


def unit_bytes(oc):
    """Algorithmic bytes of one (sequence, KV head) unit of the oracle cache."""
    s = oc.stats(0)
    H, D, g = oc.cfg.n_kv_heads, oc.cfg.head_dim, oc.g
    cache = s["code_bytes"] + s["kmeta_bytes"] + s["vmeta_bytes"] + s["sink_bytes"] + s["tail_bytes"]
    return cache / H + g * D * (2 + 4)


def cpu_baseline(repeats=6, seed=7):
    """The oracle as it stands, on a bounded sample: one sequence of the
    workload (8 KV-head units, 32 query heads) decoded `repeats` times on one
    host core. Returns (GB/s over the sample's algorithmic bytes, seconds,
    units)."""
    oc, q = oracle_sequence(seed)
    t0 = time.perf_counter()
    for _ in range(repeats):
        oc.decode_attn(0, q)
    t = time.perf_counter() - t0
    units = repeats * oc.cfg.n_kv_heads
    return units * unit_bytes(oc) / t / 1e9, t, units


def host_cpu_model():
    """The host CPU's model name (lscpu), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for line in out.splitlines():
            if line.split(":", 1)[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_worker(seed, repeats, barrier, queue):
    """One process of the all-cores leg: its own sequence of the workload in
    the oracle (built untimed), then, once every process is ready, `repeats`
    decodes of it. Puts (units, seconds, bytes per unit) on the queue."""
    oc, q = oracle_sequence(seed)
    barrier.wait()
    t0 = time.perf_counter()
    for _ in range(repeats):
        oc.decode_attn(0, q)
    queue.put((repeats * oc.cfg.n_kv_heads, time.perf_counter() - t0, unit_bytes(oc)))


def cpu_baseline_all_cores(repeats=2, n_proc=None):
    """The oracle on every host core: one spawned process per core, each
    decoding its own sequence (8 KV-head units) `repeats` times, all timed
    together. Returns (GB/s over all processes' algorithmic bytes, seconds of
    the slowest process, units, processes)."""
    import multiprocessing
    n_proc = n_proc or os.cpu_count() or 1
    ctx = multiprocessing.get_context("spawn")
    barrier, queue = ctx.Barrier(n_proc), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(100 + i, repeats, barrier, queue)) for i in range(n_proc)]
    for p in procs:
        p.start()
    res = [queue.get() for _ in procs]
    for p in procs:
        p.join()
    units = sum(r[0] for r in res)
    t = max(r[1] for r in res)
    return units * res[0][2] / t / 1e9, t, units, n_proc


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on the bench's workload; each step is
    the decode of one (sequence, KV head) unit with its 4 query heads."""
    if rank != 0:
        return
    oc, q = oracle_sequence(11)
    heads = [(0, j) for j in range(oc.g)]
    ts = []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oc.decode_attn(0, q, heads=heads)
        if s >= args.warmup:
            ts.append(time.perf_counter() - t0)
    ms = statistics.mean(ts) * 1e3
    value = unit_bytes(oc) / (ms / 1e3) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME,
                       "sample": "per step: decode of one (sequence, KV head) unit with its 4 query heads"},
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "one (sequence, KV head) unit per step, 32768-token context, decode only"},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local):
    import torch
    from bit_kv_cache_append_gb300 import binding
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = dist
    w = dict(WORKLOAD, batch=args.batch or WORKLOAD["batch"])
    L = w["context"]
    n_steps_total = args.warmup + args.steps + 2
    ccfg = dict(n_layers=1, batch=w["batch"], n_kv_heads=w["n_kv_heads"], n_q_heads=w["n_q_heads"],
                head_dim=w["head_dim"], max_tokens=L + 2 * n_steps_total + APPEND_CALLS + 64, k_bits=w["k_bits"],
                v_bits=w["v_bits"], n_sink=w["n_sink"], window=w["window"], act_dtype="bf16")
    warm_prefill(torch, binding, dev, ccfg, torch.bfloat16)
    cache = binding.KVCache(device=dev, **ccfg)
    stream = torch.cuda.current_stream()
    k, v, fac = make_inputs(torch, w, 1234 + rank, L - 1, dev)
    # prefill (append tokens/s of the bulk quantiser): the median of
    # PREFILL_REPS prefills of the whole context, the cache reset between them
    prefill_ms = timed_prefill(torch, cache, k, v, stream, PREFILL_REPS)
    prefill_tok_s = w["batch"] * (L - 1) / (prefill_ms / 1e3)
    del k, v
    g = torch.Generator(device=dev)
    g.manual_seed(99 + rank)
    B, H, Hq, D = w["batch"], w["n_kv_heads"], w["n_q_heads"], w["head_dim"]
    nk = (torch.randn((n_steps_total, B, H, 1, D), generator=g, device=dev) * fac[None, None, :, None, :]).to(torch.bfloat16)
    nv = torch.randn((n_steps_total, B, H, 1, D), generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn((B, Hq, D), generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)

    def step(i):
        cache.append(0, nk[i], nv[i])
        cache.decode_attn(0, q, out=out)

    # per-step events around the decode kernels (recorded by the library)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in kev:
        a.record(stream)
        b.record(stream)
    # clocks are sampled from here to the end of the timed region, all of it
    # under load: a ramp of untimed decodes of the same state (L unchanged)
    # for about 0.4 s, the warm-up steps, then the timed steps
    sampler = ClockSampler(local)
    sampler.start()
    t_ramp = time.perf_counter()
    while time.perf_counter() - t_ramp < 0.4:
        for _ in range(200):
            cache.decode_attn(0, q, out=out)
        torch.cuda.synchronize()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    stats0 = cache.stats(0)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    launches0 = binding.launch_count()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        cache.set_timing_events(*kev[i])
        step(args.warmup + i)
    t1.record(stream)
    torch.cuda.synchronize()
    launches = binding.launch_count() - launches0
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    cache.set_timing_events(None, None)
    ms_total = t0.elapsed_time(t1)
    stats1 = cache.stats(0)
    dec_bytes = (algorithmic_bytes(stats0, w) + algorithmic_bytes(stats1, w)) / 2
    step_bytes = dec_bytes + append_bytes(w)
    kernel_ms = [a.elapsed_time(b) for a, b in kev]
    kernel_avg_ms = statistics.mean(kernel_ms)
    cache.check_device_error()

    if args.skip_extras:
        if rank == 0:
            print(json.dumps({"ms_per_step": ms_total / args.steps, "kernel_us": kernel_avg_ms * 1e3,
                              "decode_bytes": int(dec_bytes), "launches": int(launches)}), flush=True)
        return
    # kv_append alone: APPEND_CALLS calls of one token each, back to back
    # (the tail write, and the group flush of every 32nd call)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a0.record(stream)
    for i in range(APPEND_CALLS):
        cache.append(0, nk[i % n_steps_total], nv[i % n_steps_total])
    a1.record(stream)
    torch.cuda.synchronize()
    append_tok_s = w["batch"] * APPEND_CALLS / (a0.elapsed_time(a1) / 1e3)

    # e2e: host buffers through the public API, every step's inputs copied
    # host -> device and its output read back inside the timed region. The
    # copies run on a second stream into double buffers: step i + 1's inputs
    # travel while step i's kernels run, and step i's output is read back
    # while step i + 1's run (a serving loop's pipelining; each step still
    # moves its own bytes, and the region ends when the last read-back has)
    hk = nk[: args.steps].cpu().pin_memory()
    hv = nv[: args.steps].cpu().pin_memory()
    hq = q.cpu().pin_memory()
    hout = torch.empty((B, Hq, D), dtype=torch.float32).pin_memory()
    dk = [torch.empty_like(nk[0]) for _ in range(2)]
    dv = [torch.empty_like(nv[0]) for _ in range(2)]
    dq = [torch.empty_like(q) for _ in range(2)]
    dout = [torch.empty_like(out) for _ in range(2)]
    cs = torch.cuda.Stream(device=dev)
    landed = [torch.cuda.Event() for _ in range(2)]  # buffer b's inputs are on the device
    used = [torch.cuda.Event() for _ in range(2)]    # buffer b's step has run (inputs free, output written)
    read = [torch.cuda.Event() for _ in range(2)]    # buffer b's output has been read back

    def put(i, b):  # step i's inputs into buffer b, once the step before on b has used them
        with torch.cuda.stream(cs):
            if i >= 2:
                cs.wait_event(used[b])
            dk[b].copy_(hk[i], non_blocking=True)
            dv[b].copy_(hv[i], non_blocking=True)
            dq[b].copy_(hq, non_blocking=True)
            landed[b].record(cs)

    cache2 = cache  # continue the same sequence
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    cs.wait_event(c0)
    put(0, 0)
    for i in range(args.steps):
        b = i & 1
        if i + 1 < args.steps:
            put(i + 1, b ^ 1)
        stream.wait_event(landed[b])
        if i >= 2:
            stream.wait_event(read[b])
        cache2.append(0, dk[b], dv[b])
        cache2.decode_attn(0, dq[b], out=dout[b])
        used[b].record(stream)
        with torch.cuda.stream(cs):
            cs.wait_event(used[b])
            hout.copy_(dout[b], non_blocking=True)
            read[b].record(cs)
    stream.wait_stream(cs)
    c1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = c0.elapsed_time(c1) / args.steps
    h2d = (dk[0].numel() + dv[0].numel() + dq[0].numel()) * 2
    d2h = hout.numel() * 4

    # in-process copy-kernel bandwidth (same kernel style, 1 GiB)
    src = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    for _ in range(3):
        binding.copy_bandwidth(src, dst)
    torch.cuda.synchronize()
    cts = []
    for _ in range(10):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.copy_bandwidth(src, dst)
        b.record(stream)
        torch.cuda.synchronize()
        cts.append(a.elapsed_time(b))
    copy_gbs = 2 * (1 << 30) / (statistics.median(cts) / 1e3) / 1e9
    del src, dst

    ms_step, e2e_ms = slowest_rank(pg, [ms_total / args.steps, e2e_ms], dev)
    value = whole_job_gbs(world, step_bytes, ms_step)
    peak, peak_kind = measured_peaks()
    achieved = dec_bytes / (kernel_avg_ms / 1e3) / 1e9
    if rank == 0:
        cpu_gbs, cpu_t, cpu_n = cpu_baseline(repeats=args.cpu_repeats)
        all_gbs, all_t, all_n, all_p = cpu_baseline_all_cores()
        cpu_model = host_cpu_model()
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME, "global_batch": w["batch"] * world, "seq_len": L,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (about 543 MB of cache read per step)",
                       "arith": "codes exact in f16 MMA operands; K scales folded into q as f16 value + residual, V scales into the f16 weights; f32 accumulate"},
            "us_per_step": round(ms_step * 1e3, 2),
            "us_per_model_step_x32": round(ms_step * 1e3 * w["layers_reported"], 1),
            "pct_of_peak": round(100 * achieved / peak, 2),
            "append_tokens_per_s": round(append_tok_s, 1),
            "append_note": f"kv_append alone, {APPEND_CALLS} one-token calls back to back (B tokens per call)",
            "prefill_tokens_per_s": round(prefill_tok_s, 1),
            "prefill_note": f"median of {PREFILL_REPS} prefills of {w['batch']} x {L - 1} tokens, the cache reset between",
            "copy_kernel_gbs": round(copy_gbs, 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": recorded_traffic() if w["batch"] == 16 else None,
                         "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of the decode "
                                           "kernels at batch 8, scaled by units to batch 16 (profiles/)",
                         "kernel": "decode_kivi_kernel<128,2,4> + merge_kernel<128> (split-KV partitions; exact pools and LSE merge)",
                         "algorithmic_bytes_per_launch": int(dec_bytes), "peak_kind": f"{peak_kind} hbm_gbs",
                         "kernel_us": round(kernel_avg_ms * 1e3, 2)},
            "cpu_baseline": {"value": round(all_gbs, 6), "unit": "GB/s", "cores": all_p, "kind": "oracle",
                             "sample": f"{all_n} (sequence, KV head) units with 4 query heads each over {all_p} "
                                       f"spawned processes (one sequence each), 32768-token context, decode only "
                                       f"({all_t:.1f} s, the slowest process)",
                             "cpu_model": cpu_model,
                             "one_core": {"value": round(cpu_gbs, 6), "unit": "GB/s", "cores": 1,
                                          "sample": f"{cpu_n} units of one sequence, decode only ({cpu_t:.1f} s)"}},
            "e2e": {"value": round(whole_job_gbs(world, step_bytes, e2e_ms), 3), "unit": "GB/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "copies": "second stream, double-buffered, overlapping the neighbouring steps"},
            "gpu_launches": int(launches),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


OTHER_WORKLOADS = {
    # name: cache shape, mode and bits, overlay, context, activation dtype
    "turboquant_k4v2": dict(batch=32, n_kv_heads=8, n_q_heads=32, head_dim=128, context=16384, act_dtype="f16",
                            mode="turboquant", k_bits=4, v_bits=2),
    "turboquant_k4v4": dict(batch=32, n_kv_heads=8, n_q_heads=32, head_dim=128, context=16384, act_dtype="f16",
                            mode="turboquant", k_bits=4, v_bits=4),
    "turboquant_k3v2": dict(batch=32, n_kv_heads=8, n_q_heads=32, head_dim=128, context=16384, act_dtype="f16",
                            mode="turboquant", k_bits=3, v_bits=2),
    "llama8b_q4_0v": dict(batch=16, n_kv_heads=8, n_q_heads=32, head_dim=128, context=32768, act_dtype="bf16",
                          mode="kivi", k_bits=2, v_bits=4, v_q4_0=True),
    "llama8b_k4v4": dict(batch=16, n_kv_heads=8, n_q_heads=32, head_dim=128, context=32768, act_dtype="bf16",
                         mode="kivi", k_bits=4, v_bits=4),
    "llama8b_k3v4": dict(batch=16, n_kv_heads=8, n_q_heads=32, head_dim=128, context=32768, act_dtype="bf16",
                         mode="kivi", k_bits=3, v_bits=4),
    "llama8b_k3v3": dict(batch=16, n_kv_heads=8, n_q_heads=32, head_dim=128, context=32768, act_dtype="bf16",
                         mode="kivi", k_bits=3, v_bits=3),
    "kvsink": dict(batch=4, n_kv_heads=8, n_q_heads=32, head_dim=128, context=131072, act_dtype="f16",
                   mode="kivi", k_bits=2, v_bits=2, n_dyn_sinks=5),
    "ring_int8": dict(batch=64, n_kv_heads=8, n_q_heads=8, head_dim=64, context=4100, act_dtype="f16",
                      mode="kivi", k_bits=8, v_bits=8, n_sink=4, evict_window=4096, rope_base=10000.0, layers=12),
    "ring_int4": dict(batch=64, n_kv_heads=8, n_q_heads=8, head_dim=64, context=4100, act_dtype="f16",
                      mode="kivi", k_bits=4, v_bits=4, n_sink=4, evict_window=4096, rope_base=10000.0, layers=12),
    "ring_int4_repos": dict(batch=64, n_kv_heads=8, n_q_heads=8, head_dim=64, context=4100, act_dtype="f16",
                            mode="kivi", k_bits=4, v_bits=4, n_sink=4, evict_window=4096, rope_base=10000.0,
                            rope_reposition=True, layers=12),
    "ring_int4_prerope": dict(batch=64, n_kv_heads=8, n_q_heads=8, head_dim=64, context=4100, act_dtype="f16",
                              mode="kivi", k_bits=4, v_bits=4, n_sink=4, evict_window=4096, rope_base=10000.0,
                              k_pre_rope=True, layers=12),
    "ring_int4_prerope_repos": dict(batch=64, n_kv_heads=8, n_q_heads=8, head_dim=64, context=4100,
                                    act_dtype="f16", mode="kivi", k_bits=4, v_bits=4, n_sink=4, evict_window=4096,
                                    rope_base=10000.0, k_pre_rope=True, rope_reposition=True, layers=12),
}


def run_workload(args):
    """One of the other workloads of the method on one GPU: prefill-quantise
    the context (tokens/s), then time steps of one append (with eviction for
    the ring) and one decode of one layer. Inputs are N(0, 1) drawn on the
    device (timing does not depend on the values). Prints one JSON line."""
    import torch
    from bit_kv_cache_append_gb300 import binding
    w = dict(OTHER_WORKLOADS[args.workload])
    if args.batch:
        w["batch"] = args.batch
    dev = torch.device("cuda", 0)
    dt = torch.float16 if w["act_dtype"] == "f16" else torch.bfloat16
    B, H, Hq, D, L = w["batch"], w["n_kv_heads"], w["n_q_heads"], w["head_dim"], w["context"]
    n_total = args.warmup + args.steps + 2
    ring = w.get("evict_window", 0) > 0
    cfg = dict(n_layers=1, batch=B, n_kv_heads=H, n_q_heads=Hq, head_dim=D,
               max_tokens=(w["evict_window"] + 64 if ring else L + n_total + 64), mode=w["mode"],
               k_bits=w["k_bits"], v_bits=w["v_bits"], n_sink=w.get("n_sink", 0), window=0,
               evict_window=w.get("evict_window", 0), n_dyn_sinks=w.get("n_dyn_sinks", 0), act_dtype=w["act_dtype"],
               rope_base=w.get("rope_base", 0.0), rope_max_pos=(L + n_total + 64 if w.get("rope_base") else 0),
               rope_reposition=w.get("rope_reposition", False), v_q4_0=w.get("v_q4_0", False),
               k_pre_rope=w.get("k_pre_rope", False))
    warm_prefill(torch, binding, dev, cfg, dt)
    cache = binding.KVCache(device=dev, **cfg)
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    k = torch.randn((B, H, L, D), generator=g, device=dev).to(dt)
    v = torch.randn((B, H, L, D), generator=g, device=dev).to(dt)
    stream = torch.cuda.current_stream()
    # the running KVSink selection lives on the device and is not cleared by a
    # reset, so that workload's prefill is timed once
    prefill_ms = timed_prefill(torch, cache, k, v, stream, 1 if cfg.get("n_dyn_sinks") else PREFILL_REPS)
    del k, v
    if ring:
        cache.evict(0)
    nk = torch.randn((n_total, B, H, 1, D), generator=g, device=dev).to(dt)
    nv = torch.randn((n_total, B, H, 1, D), generator=g, device=dev).to(dt)
    q = torch.randn((B, Hq, D), generator=g, device=dev).to(dt)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)

    def step(i):
        cache.append(0, nk[i], nv[i])
        if ring:
            cache.evict(0)
        cache.decode_attn(0, q, out=out)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    stats0 = cache.stats(0)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in kev:
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        cache.set_timing_events(*kev[i])
        step(args.warmup + i)
    t1.record(stream)
    torch.cuda.synchronize()
    cache.set_timing_events(None, None)
    cache.check_device_error()
    stats1 = cache.stats(0)
    ms_step = t0.elapsed_time(t1) / args.steps
    dec_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in kev)
    wb = dict(batch=B, n_q_heads=Hq, head_dim=D)
    dec_bytes = (algorithmic_bytes(stats0, wb) + algorithmic_bytes(stats1, wb)) / 2
    peak, peak_kind = measured_peaks()
    layers = w.get("layers", 1)
    line = {"workload": args.workload, "config": w, "data": "synthetic N(0,1) on the device",
            "prefill_tokens": B * L, "prefill_ms": round(prefill_ms, 3),
            "prefill_tokens_per_s": round(B * L / (prefill_ms / 1e3), 1),
            "prefill_note": "one prefill" if cfg.get("n_dyn_sinks") else f"median of {PREFILL_REPS} prefills, the cache reset between",
            "steps": args.steps, "warmup": args.warmup, "us_per_step": round(ms_step * 1e3, 2),
            "decode_us": round(dec_ms * 1e3, 2), "decode_bytes": int(dec_bytes),
            "decode_gbs": round(dec_bytes / (dec_ms / 1e3) / 1e9, 1),
            "decode_frac_of_peak": round(dec_bytes / (dec_ms / 1e3) / 1e9 / peak, 4), "peak_kind": peak_kind,
            "tokens_per_s": round(B / (ms_step / 1e3 * layers), 1),
            "tokens_per_s_note": f"B / (per-layer step x {layers} layers)" if layers > 1 else "B / step"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences (0: the workload's own; smaller values give profiling cases)")
    ap.add_argument("--skip-extras", action="store_true",
                    help="time the steps only (no e2e, copy or CPU legs); prints a short line")
    ap.add_argument("--cpu-repeats", type=int, default=6,
                    help="decodes of one oracle sequence (8 KV-head units each) in the CPU sample")
    ap.add_argument("--workload", choices=["llama8b"] + sorted(OTHER_WORKLOADS), default="llama8b",
                    help="llama8b is the benchmark line; the others print their own measurement line")
    args = ap.parse_args()
    rank, world, local = dist_env()
    if args.warmup < 3:
        args.warmup = 3
    if args.workload != "llama8b":
        run_workload(args)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
