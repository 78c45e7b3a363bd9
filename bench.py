"""Benchmark of packed variable-length GQA attention on GB300.

One step = one pva_forward (scheduler + prefill + decode kernels) over one
packed batch of the named workload, inputs resident in HBM.  Default
workload: bf16 causal GQA prefill, B=16, L_q=L_kv~U[128,2048], H=32, Hkv=8,
d=dv=128 (metric: TFLOP/s counting only unmasked (q,k) pairs at 2*H*(d+dv)
FLOPs each, 4*H*d when d == dv).  The decode workload reports KV-read GB/s instead.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl reference]

Prints ONE JSON line (rank 0).  Besides the cold-L2 headline it carries the
same steps with a warm L2 (``warm_l2``), median and minimum step times, and,
for the default workload on one GPU, the other configs each in its own timed
region (``other_configs``: chunked prefill, decode, long-context MQA with
softcap).  ``cpu_baseline`` times the fp64 oracle on the host cores (all of
them and one) and, for the default line, checks the fp32 workload against it.
``--impl reference`` times the fp64 CPU oracle (the only reference this
build has) on a bounded sample of the same workload.  Under torchrun every rank runs its own batch (seed = rank): the
work is independent per GPU (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD_TEXT = {
    "bf16_prefill": "bf16 causal GQA prefill: B=16, L_q=L_kv~U[128,2048], H=32, Hkv=8, d=dv=128, "
                    "default scale, softcap 0, N(0,1)",
    "bf16_chunked": "bf16 tail-aligned causal chunked prefill: B=32, L_q~U[1,512], "
                    "L_kv=L_q+U[0,4096], H=32, Hkv=8, d=128, N(0,1)",
    "bf16_decode": "bf16 decode: B=256, L_q=1, L_kv~U[512,8192], H=32, Hkv=8, d=128, causal",
    "bf16_longctx": "bf16 long-context MQA + softcap 50: B=4, L~logU[8192,32768], H=8, Hkv=1, "
                    "d=dv=256, causal, N(0,2)",
    "fp32_small": "fp32 non-causal: L={17,64,1,130}, H=Hkv=4, d=dv=64, scale 1/8",
    "bf16_mla": "bf16 causal prefill, q.k wider than v: B=8, L_q=L_kv~U[512,4096], H=Hkv=32, "
                "d=192, dv=128, N(0,1)",
    "bf16_decode_g16": "bf16 decode, 16 query heads per kv head: B=256, L_q=1, "
                       "L_kv~U[512,8192], H=32, Hkv=2, d=128, causal",
    "bf16_decode_mla": "bf16 decode, q.k wider than v: B=256, L_q=1, L_kv~U[512,8192], H=32, "
                       "Hkv=8, d=192, dv=128, causal",
    "bf16_window": "bf16 causal GQA prefill with a local window of 4096 keys: B=4, "
                   "L~logU[8192,32768], H=32, Hkv=8, d=dv=128, N(0,1)",
    "bf16_kvcache_decode": "bf16 GroupQueryAttention decode step on a BNSH KV cache of capacity "
                           "8192: B=256, keys after the append ~U[512,8192], H=32, Hkv=8, "
                           "d=128, rotary on 128 dims (half-split, f32 tables), append + "
                           "rotary + attention",
}
METRIC = "varlen attn TFLOP/s (prefill) & KV-read GB/s (decode), % of roofline"
L2_FLUSH_BYTES = 256 << 20


def visible_keys(a: int, b: int, is_causal: bool, window: int = 0):
    """Keys each of the a query rows of a sequence sees (b keys): row i, causal
    limit c = i + b - a, sees [max(0, c + 1 - window) if window > 0 else 0,
    min(b, c + 1) if causal else b)."""
    import numpy as np
    c = np.arange(a, dtype=np.int64) + (b - a)
    hi = np.minimum(b, c + 1) if is_causal else np.full(a, b, dtype=np.int64)
    lo = np.maximum(0, c + 1 - window) if window > 0 else np.zeros(a, dtype=np.int64)
    return np.maximum(hi - lo, 0)


def unmasked_pairs(lq, lkv, is_causal: bool, window: int = 0) -> int:
    """(query, key) pairs the mask leaves visible, summed over sequences (one
    head)."""
    return int(sum(int(visible_keys(int(a), int(b), is_causal, window).sum())
                   for a, b in zip(lq, lkv)))


def work_units(w):
    """Algorithmic work of one step: (FLOPs, KV bytes)."""
    pairs = unmasked_pairs(w["lq"], w["lkv"], w["is_causal"], w.get("window", 0))
    # 2 FLOP per multiply-add: q.k over d and p.v over dv for every unmasked
    # (query, key) pair and head (4 H d when d == dv)
    flops = pairs * 2 * w["num_heads"] * (w["head_size"] + w["v_head_size"])
    kv_bytes = sum(w["lkv"]) * w["kv_num_heads"] * (w["head_size"] + w["v_head_size"]) * \
        (2 if w["dtype"] != "f32" else 4)
    return flops, kv_bytes


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def recorded_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel_key)
    if not rec:
        return None
    h = hashlib.sha256()
    for src in rec.get("sources", []):
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("sources_sha256"):
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

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
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x: float, world: int, device) -> float:
    """Largest per-rank value (step time) across the job; identity at N=1."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: int, world: int, device) -> int:
    """Job-wide total of a per-rank count (work of independent batches)."""
    if world <= 1:
        return int(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([int(x)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return int(t.item())


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class OracleSampler:
    """Times the fp64 CPU oracle on bounded samples of a workload: sequences
    of the workload's own length draw, materialised one at a time with the
    same value recipe, and a uniform sample of their (token, head) output
    rows.  Work is counted like the GPU arm's (visible pairs x 4 d FLOPs, or
    K/V bytes for decode)."""

    def __init__(self, w_name: str, seed: int = 0, threads: int = 0):
        import numpy as np
        import torch

        from gqa_attention_cu_gb300 import workloads
        self.np, self.torch, self.wl = np, torch, workloads
        self.threads = threads  # 0: every host core (OpenMP default)
        self.name = w_name
        self.spec = workloads.WORKLOADS[w_name]
        gen = torch.Generator("cpu").manual_seed(seed)
        self.lq, self.lkv = workloads.draw_lengths(self.spec, gen)
        self.rng = np.random.default_rng(seed + 7)
        self.gen = torch.Generator("cpu").manual_seed(seed + 11)
        self.per_pair = None

    def _one(self, pair_budget: int):
        np, sp = self.np, self.spec
        import oracle
        H, Hkv = sp.num_heads, sp.kv_num_heads
        cand = [b for b in range(len(self.lq)) if self.lq[b] > 0]
        b = int(self.rng.choice(cand))
        lq, lkv = self.lq[b], self.lkv[b]
        q, k, v, cq, ck = self.wl.make_packed([lq], [lkv], H, Hkv, sp.head_size, sp.v_head_size,
                                              sp.dtype, sp.sigma, gen=self.gen)
        vis = visible_keys(lq, lkv, sp.is_causal, sp.window)
        avg = max(1.0, float(vis.mean()))
        n_rows = int(max(1, min(lq * H, pair_budget / avg)))
        rows = np.sort(self.rng.choice(lq * H, size=n_rows, replace=False))
        pairs = int(vis[rows // H].sum())
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, cq, ck, rows, H, Hkv, sp.scale, sp.is_causal, sp.softcap,
                              threads=self.threads, local_window=sp.window)
        return time.perf_counter() - t0, pairs, n_rows

    def run(self, seconds: float):
        """Oracle work for about `seconds`; returns (seconds, pairs, rows)."""
        if self.per_pair is None:
            dt, pairs, _ = self._one(200_000)
            self.per_pair = dt / max(pairs, 1)
        tot_t = tot_p = tot_r = 0
        while tot_t < seconds:
            budget = max(10_000, int(min(seconds - tot_t, seconds / 2) / self.per_pair))
            dt, pairs, n = self._one(budget)
            tot_t, tot_p, tot_r = tot_t + dt, tot_p + pairs, tot_r + n
        self.per_pair = tot_t / max(tot_p, 1)
        return tot_t, tot_p, tot_r

    def value(self, secs: float, pairs: int):
        sp = self.spec
        if self.name.startswith("bf16_decode"):
            # every visible pair of a kv head's G query rows reads one K and V row;
            # count each K/V row once per kv head, as the GPU arm does
            kv = pairs / (sp.num_heads // sp.kv_num_heads) * (sp.head_size + sp.v_head_size) * 2
            return kv / secs / 1e9, "GB/s"
        return pairs * 2 * (sp.head_size + sp.v_head_size) / secs / 1e12, "TFLOP/s"


class CacheStepSampler:
    """Times the cache-step oracle (metadata, append, rotary, fp64 attention)
    on bounded samples: a few sequences of the workload's total-length draw
    per call, each with its own small cache.  Work is the K/V bytes of the
    valid cache rows, counted as the GPU arm counts them."""

    def __init__(self, w_name: str, seed: int = 0):
        import torch

        from gqa_attention_cu_gb300 import workloads
        self.torch, self.wl, self.name = torch, workloads, w_name
        self.spec = workloads.WORKLOADS[w_name]
        # the totals make_cache_step draws for this seed
        self.totals = torch.randint(self.spec.params["lo"], self.spec.params["hi"] + 1,
                                    (self.spec.B,),
                                    generator=torch.Generator("cpu").manual_seed(seed)).tolist()
        self.gen = torch.Generator("cpu").manual_seed(seed + 11)
        self.cos, self.sin = workloads.rotary_tables(self.spec.params["cache_rows"],
                                                     self.spec.params["rotary_dim"])
        self.next = 0

    def _one(self):
        from oracle import gqa_cache
        torch, sp = self.torch, self.spec
        tot = [self.totals[(self.next + i) % len(self.totals)] for i in range(2)]
        self.next += 2
        cap, H, Hkv, d = max(tot), sp.num_heads, sp.kv_num_heads, sp.head_size
        td = self.wl.DTYPES[sp.dtype]
        r = lambda *shape: torch.randn(shape, generator=self.gen).to(td)  # noqa: E731
        q, kn, vn = r(2, 1, H, d), r(2, 1, Hkv, d), r(2, 1, Hkv, d)
        kc, vc = r(2, Hkv, cap, d), r(2, Hkv, cap, d)
        t0 = time.perf_counter()
        gqa_cache.gqa_cache_step(q, kn, vn, kc, vc, [t - 1 for t in tot], H, Hkv, self.cos,
                                 self.sin)
        return time.perf_counter() - t0, sum(tot) * Hkv * 2 * d * 2

    def run(self, seconds: float):
        tot_t = tot_b = n = 0
        while tot_t < seconds:
            dt, nb = self._one()
            tot_t, tot_b, n = tot_t + dt, tot_b + nb, n + 2
        return tot_t, tot_b, n

    def value(self, secs: float, kv_bytes: int):
        return kv_bytes / secs / 1e9, "GB/s"


def make_sampler(w_name: str, threads: int = 0):
    if w_name == "bf16_kvcache_decode":
        return CacheStepSampler(w_name)
    return OracleSampler(w_name, threads=threads)


def cpu_model() -> str:
    """Host CPU model (lscpu, else /proc/cpuinfo), for the baseline record."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for ln in r.stdout.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def run_reference(args, w_name):
    """The fp64 CPU oracle, timed on the host cores, on a bounded sample of the
    workload per step (rank 0 only; other ranks exit without work)."""
    rank, world, _ = dist_info()
    if rank != 0:
        return
    import oracle
    smp = make_sampler(w_name)
    for _ in range(args.warmup):
        smp.run(args.ref_seconds / 4)
    secs = pairs = rows = 0
    for _ in range(args.steps):
        t, p, r = smp.run(args.ref_seconds)
        secs, pairs, rows = secs + t, pairs + p, rows + r
    value, unit = smp.value(secs, pairs)
    sample = (f"~{args.ref_seconds:g} s of oracle work per step: {rows // args.steps} random "
              f"(token, head) output rows per step from sequences of the workload's length draw"
              if w_name != "bf16_kvcache_decode" else
              f"~{args.ref_seconds:g} s of oracle work per step: {rows // args.steps} sequences "
              f"of the workload's length draw per step, whole cache step each")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[w_name], "name": w_name, "sample": sample},
        "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w_name, seconds=12.0, single_thread_seconds=4.0):
    """The oracle as it stands on the host cores, on a bounded sample, plus a
    shorter single-thread sample of the same recipe."""
    import oracle
    smp = make_sampler(w_name)
    secs, pairs, rows = smp.run(seconds)
    value, unit = smp.value(secs, pairs)
    what = ("sequences of the workload's length draw, whole cache step each"
            if w_name == "bf16_kvcache_decode" else
            "random (token, head) output rows from sequences of the workload's length draw")
    rec = {"value": value, "unit": unit, "cores": oracle.max_threads(), "kind": "oracle",
           "cpu_model": cpu_model(), "sample": f"{rows} {what}, {secs:.1f} s"}
    if w_name != "bf16_kvcache_decode" and single_thread_seconds > 0:
        one = make_sampler(w_name, threads=1)
        s1, p1, r1 = one.run(single_thread_seconds)
        v1, _ = one.value(s1, p1)
        rec["single_thread"] = {"value": v1, "unit": unit, "cores": 1,
                                "sample": f"{r1} {what}, {s1:.1f} s"}
    return rec


def fp32_oracle_check(pva, dev):
    """The fp32_small workload through pva_forward, against the fp64 oracle
    (which is timed too): the accuracy figure of the fp32 path."""
    import numpy as np
    import torch

    import oracle
    from gqa_attention_cu_gb300 import workloads
    w = workloads.make("fp32_small")
    args = [w[k_].to(dev) for k_ in ("q", "k", "v", "cu_q", "cu_kv")]
    out = torch.empty(w["q"].shape[0], w["num_heads"], w["v_head_size"], dtype=torch.float32,
                      device=dev)
    pva.pva_forward(*args, out, w["B"], w["num_heads"], w["kv_num_heads"], w["head_size"],
                    w["v_head_size"], w["scale"], int(w["is_causal"]), w["softcap"])
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    ref = oracle.attention(w["q"], w["k"], w["v"], w["cu_q"], w["cu_kv"], w["num_heads"],
                           w["kv_num_heads"], w["scale"], w["is_causal"], w["softcap"])
    t_oracle = time.perf_counter() - t0
    err = np.abs(out.double().cpu().numpy() - ref)
    return {"max_abs_vs_oracle": float(err.max()), "tolerance": 2e-5,
            "oracle_ms_full": 1e3 * t_oracle}


def bench_kvcache(args, rank, world, local, dev):
    """One GroupQueryAttention decode step per timed step (pva_gqa_kvcache):
    metadata, append + rotary, scheduler and split-KV decode straight from the
    BNSH caches.  The step is repeatable: with the same seqlens_k it rewrites
    the same cache row each time.  Metric: K/V bytes of the valid cache rows
    per second (each row read once for its kv head's G query heads)."""
    import torch

    import gqa_attention_cu_gb300 as pva
    from gqa_attention_cu_gb300 import workloads

    w_name = args.workload
    c = workloads.make_cache_step(w_name, seed=rank, B=args.batch, device=str(dev))
    H, Hkv, d = c["num_heads"], c["kv_num_heads"], c["head_size"]
    kv_bytes = sum(c["totals"]) * Hkv * 2 * d * 2
    stream = torch.cuda.Stream(device=dev)
    out = torch.empty_like(c["q"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(q, kn, vn, sk, s):
        pva.pva_gqa_kvcache(q, kn, vn, c["k_cache"], c["v_cache"], sk, out, H, Hkv, c["cos"],
                            c["sin"], stream=s)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(c["q"], c["k_new"], c["v_new"], c["seqlens_k"], stream)
    torch.cuda.synchronize(dev)
    if pva.pva_get_status(stream) != 0:
        raise SystemExit("device status bits set during warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)

    def fwd(s):
        step(c["q"], c["k_new"], c["v_new"], c["seqlens_k"], s)
    wall0 = time.perf_counter()
    step_ms, _ = time_steps(pva, fwd, stream, dev, args.steps, flush)
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    _, kernel_ms = time_steps(pva, fwd, stream, dev, args.steps, flush, profile=True)
    clk = clocks.stop()
    ms = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    job_kv = sum_over_ranks(kv_bytes, world, dev)
    if pva.pva_get_status(stream) != 0:
        raise SystemExit("device status bits set during the timed steps")

    # end to end: this step's new token (q, k, v) and lengths from pinned host
    # memory, the output back; the caches stay resident, as in serving
    host = {k: c[k].cpu().pin_memory() for k in ("q", "k_new", "v_new", "seqlens_k")}
    dbuf = {k: torch.empty_like(c[k]) for k in host}
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()
    e2e_ms = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            flush.fill_(i & 0xff)
            a.record(stream)
            for k_ in host:
                dbuf[k_].copy_(host[k_], non_blocking=True)
            step(dbuf["q"], dbuf["k_new"], dbuf["v_new"], dbuf["seqlens_k"], stream)
            out_host.copy_(out, non_blocking=True)
            b.record(stream)
            b.synchronize()
            if i >= args.warmup:
                e2e_ms.append(a.elapsed_time(b))
    e2e = max_over_ranks(sum(e2e_ms) / len(e2e_ms), world, dev)
    if pva.pva_get_status(stream) != 0:
        raise SystemExit("device status bits set during the end-to-end steps")

    peaks = measured_peaks()
    dec_ms = [k[2] for k in kernel_ms if k[2] >= 0]
    front_ms = [k[0] for k in kernel_ms]
    dom_ms = sum(dec_ms) / len(dec_ms)
    achieved = kv_bytes / (dom_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": job_kv / (ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[w_name], "name": w_name,
                   **({"batch_override": args.batch} if args.batch else {}),
                   "l2": "flushed between steps; caches (8.6 GB) exceed L2",
                   "kv_bytes_per_step": kv_bytes,
                   "kernel_ms": {"front_and_scheduler": sum(front_ms) / len(front_ms),
                                 "decode": dom_ms},
                   "parallelism": f"replicas x{world} (independent caches per GPU)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": recorded_traffic("decode_kvcache_bf16_d128_g4"),
                     "kernel": "pva_decode_kernel (cache planes)",
                     "peak_source": peaks["source"] + " hbm_gbs"},
        "e2e": {"value": job_kv / (e2e * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e},
        # metadata, append + rotary, scheduler, prefill (no items), decode
        "gpu_launches": 5 * args.steps,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w_name)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def dominant_kernel(w):
    if w["dtype"] == "f32":
        return "pva_prefill_f32_kernel"
    if w["head_size"] == w["v_head_size"] and w["head_size"] in (64, 128):
        return "pva_prefill_pair_kernel"
    return "pva_prefill_tc_kernel"


def launches_per_step(w):
    """Kernels one pva_forward launches: scheduler, prefill, and the split-KV
    decode kernel for the shapes it serves."""
    G = w["num_heads"] // w["kv_num_heads"]
    dec = w["dtype"] != "f32" and G in (1, 2, 4, 8, 16)
    return 3 if dec else 2


def time_steps(pva, forward, stream, dev, steps, flush, profile=False):
    """`steps` device-timed calls (CUDA events on the launching stream); with
    `flush` a 256 MB buffer is written between calls (cold L2).  Returns the
    per-step times and, with `profile`, the per-kernel times of each call
    (the library then records events between its kernels, which keeps a
    kernel from starting its set-up while the one before it finishes, so
    step times of a profiled pass are not the step rate)."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    kernel_ms = []
    torch.cuda.synchronize(dev)
    if profile:
        pva.pva_profile(True)
    with torch.cuda.stream(stream):
        for i in range(steps):
            if flush is not None:
                flush.fill_(i & 0xff)
            starts[i].record(stream)
            forward(stream)
            ends[i].record(stream)
            if profile:
                kernel_ms.append(pva.pva_kernel_times())
    torch.cuda.synchronize(dev)
    if profile:
        pva.pva_profile(False)
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], kernel_ms


def step_stats(ms):
    return {"mean": sum(ms) / len(ms), "median": statistics.median(ms), "min": min(ms)}


def summarize(w, w_name, step_ms, kernel_ms, peaks):
    """Whole-step rate and the dominant kernel's roofline for one timed run."""
    flops, kv_bytes = work_units(w)
    is_decode = w_name.startswith("bf16_decode")
    pre = [k[1] for k in kernel_ms]
    dec = [k[2] for k in kernel_ms if k[2] >= 0]
    ms = sum(step_ms) / len(step_ms)
    if is_decode:
        # Single-row sequences of the tuned shapes go to the split-KV decode
        # kernel; those of other shapes, when they are many, to the
        # tensor-core prefill kernel: the roofline is the busier kernel's.
        dom_dec = sum(dec) / len(dec) if dec else 0.0
        dom_pre = sum(pre) / len(pre)
        dom = max(dom_dec, dom_pre)
        kern = "pva_decode_kernel" if dom_dec >= dom_pre else dominant_kernel(w)
        achieved = kv_bytes / (dom * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "kernel": kern,
                "peak_source": peaks["source"] + " hbm_gbs"}
        value, unit = kv_bytes / (ms * 1e-3) / 1e9, "GB/s"
    else:
        dom = sum(pre) / len(pre)
        achieved = flops / (dom * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "kernel": dominant_kernel(w),
                "peak_source": peaks["source"] + " bf16_tflops (burst: kernel timed alone)"}
        value, unit = flops / (ms * 1e-3) / 1e12, "TFLOP/s"
    kms = {"scheduler": sum(k[0] for k in kernel_ms) / len(kernel_ms),
           "prefill": sum(pre) / len(pre), "decode": (sum(dec) / len(dec)) if dec else None}
    kmed = {"prefill": statistics.median(pre), "decode": statistics.median(dec) if dec else None}
    return {"value": value, "unit": unit, "ms_per_step": ms, "step_ms": step_stats(step_ms),
            "kernel_ms": kms, "kernel_ms_median": kmed, "roofline": roof,
            "flops_per_step": flops, "kv_bytes_per_step": kv_bytes}


def make_forward(pva, w, out):
    H, Hkv, d, dv = w["num_heads"], w["kv_num_heads"], w["head_size"], w["v_head_size"]

    def forward(q, k, v, cq, ck, o, s):
        if w["window"] > 0:
            pva.pva_forward_local(q, k, v, cq, ck, o, w["B"], H, Hkv, d, dv, w["scale"],
                                  int(w["is_causal"]), w["softcap"], w["window"], stream=s)
        else:
            pva.pva_forward(q, k, v, cq, ck, o, w["B"], H, Hkv, d, dv, w["scale"],
                            int(w["is_causal"]), w["softcap"], stream=s)

    def step(s):
        forward(w["q"], w["k"], w["v"], w["cu_q"], w["cu_kv"], out, s)
    return forward, step


def bench_other_config(pva, w_name, dev, steps, warmup, flush, peaks, local):
    """One more workload in the same process (device-timed steps only), for
    the record beside the headline line."""
    import torch

    from gqa_attention_cu_gb300 import workloads
    w = workloads.make(w_name, seed=0, device=str(dev))
    out = torch.empty(w["q"].shape[0], w["num_heads"], w["v_head_size"], dtype=w["q"].dtype,
                      device=dev)
    stream = torch.cuda.Stream(device=dev)
    _, step = make_forward(pva, w, out)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step(stream)
    torch.cuda.synchronize(dev)
    if pva.pva_get_status(stream) != 0:
        raise SystemExit(f"device status bits set during {w_name} warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    step_ms, _ = time_steps(pva, step, stream, dev, steps, flush)
    _, kernel_ms = time_steps(pva, step, stream, dev, steps, flush, profile=True)
    clk = clocks.stop()
    if pva.pva_get_status(stream) != 0:
        raise SystemExit(f"device status bits set during {w_name}")
    rec = summarize(w, w_name, step_ms, kernel_ms, peaks)
    rec["workload"] = WORKLOAD_TEXT[w_name]
    rec["clocks"] = clk
    rec["gpu_launches"] = launches_per_step(w) * steps
    del w, out
    torch.cuda.empty_cache()
    return rec


OTHER_CONFIGS = ("bf16_chunked", "bf16_decode", "bf16_longctx")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="bf16_prefill", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-seconds", type=float, default=4.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the other configs measured beside the default line")
    ap.add_argument("--batch", type=int, default=None,
                    help="draw only this many sequences of the workload's recipe "
                         "(smaller cases for profiler captures; not a bench line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        run_reference(args, args.workload)
        return

    import torch
    import torch.distributed as dist

    import gqa_attention_cu_gb300 as pva
    from gqa_attention_cu_gb300 import workloads

    rank, world, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pva.build()
    pva.load_library()

    w_name = args.workload
    if w_name == "bf16_kvcache_decode":
        bench_kvcache(args, rank, world, local, dev)
        return
    w = workloads.make(w_name, seed=rank, device=str(dev), B=args.batch)
    H, dv = w["num_heads"], w["v_head_size"]
    flops, kv_bytes = work_units(w)
    is_decode = w_name.startswith("bf16_decode")
    stream = torch.cuda.Stream(device=dev)
    out = torch.empty(w["q"].shape[0], H, dv, dtype=w["q"].dtype, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    forward, step = make_forward(pva, w, out)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(stream)
    torch.cuda.synchronize(dev)
    if pva.pva_get_status(stream) != 0:
        raise SystemExit("device status bits set during warm-up")

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    step_ms, _ = time_steps(pva, step, stream, dev, args.steps, flush)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    job_flops = sum_over_ranks(flops, world, dev)
    job_kv = sum_over_ranks(kv_bytes, world, dev)
    if pva.pva_get_status(stream) != 0:
        raise SystemExit("device status bits set during the timed steps")
    # Per-kernel times (the roofline's denominator) from a separate pass of
    # the same steps with the library's kernel events on.
    _, kernel_ms = time_steps(pva, step, stream, dev, args.steps, flush, profile=True)
    peaks = measured_peaks()
    rec = summarize(w, w_name, step_ms, kernel_ms, peaks)

    # The same steps without the L2 flush (inputs partly L2-resident from the
    # previous step): reported beside the cold-L2 figures, never as `value`.
    warm_ms, _ = time_steps(pva, step, stream, dev, args.steps, None)
    _, warm_kernel_ms = time_steps(pva, step, stream, dev, args.steps, None, profile=True)
    warm = summarize(w, w_name, warm_ms, warm_kernel_ms, peaks)

    # ---- end to end through the public API with host buffers ---------------
    # pva_forward_from_host: the batch in pinned host memory, copied in and
    # the output copied back by the call, chunk by chunk, overlapped with the
    # attention (windowed workloads: the copies around pva_forward_local).
    host = {k: w[k].cpu().pin_memory() for k in ("q", "k", "v", "cu_q", "cu_kv")}
    dbuf = {k: torch.empty_like(w[k]) for k in ("q", "k", "v", "cu_q", "cu_kv")}
    cu_scratch = torch.zeros(4 * w["B"] + 34, dtype=torch.int32, device=dev)
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()
    e2e_ms = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            flush.fill_(i & 0xff)
            a.record(stream)
            if w["window"] > 0:
                for k_ in host:
                    dbuf[k_].copy_(host[k_], non_blocking=True)
                forward(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["cu_q"], dbuf["cu_kv"], out, stream)
                out_host.copy_(out, non_blocking=True)
            else:
                pva.pva_forward_from_host(host["q"], host["k"], host["v"], host["cu_q"],
                                          host["cu_kv"], out_host, dbuf["q"], dbuf["k"],
                                          dbuf["v"], out, cu_scratch, w["B"], w["num_heads"],
                                          w["kv_num_heads"], w["head_size"], w["v_head_size"],
                                          w["scale"], int(w["is_causal"]), w["softcap"],
                                          stream=stream)
            b.record(stream)
            b.synchronize()
            if i >= args.warmup:
                e2e_ms.append(a.elapsed_time(b))
    e2e = max_over_ranks(sum(e2e_ms) / len(e2e_ms), world, dev)

    unit = rec["unit"]
    if is_decode:
        value = job_kv / (ms * 1e-3) / 1e9
        e2e_v = job_kv / (e2e * 1e-3) / 1e9
        traffic_key = "decode_bf16_d128_g4" if w_name == "bf16_decode" else f"decode_{w_name}"
    else:
        value = job_flops / (ms * 1e-3) / 1e12
        e2e_v = job_flops / (e2e * 1e-3) / 1e12
        traffic_key = f"prefill_{w_name}"
    roof = dict(rec["roofline"])
    roof["traffic"] = recorded_traffic(traffic_key)
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[w_name], "name": w_name,
                   **({"batch_override": args.batch} if args.batch else {}),
                   "l2": "flushed between steps (256 MB write); inputs also exceed L2"
                   if not is_decode else "flushed between steps; K/V (4.6 GB) exceed L2",
                   "tokens_q": int(w["cu_q"][-1]), "tokens_kv": int(w["cu_kv"][-1]),
                   "flops_per_step": flops, "kv_bytes_per_step": kv_bytes,
                   "kernel_ms": rec["kernel_ms"], "kernel_ms_median": rec["kernel_ms_median"],
                   "step_ms": rec["step_ms"],
                   "parallelism": f"replicas x{world} (independent batches per GPU)"},
        "roofline": roof,
        "warm_l2": {"value": warm["value"], "unit": unit, "step_ms": warm["step_ms"],
                    "kernel_ms": warm["kernel_ms"], "frac": warm["roofline"]["frac"],
                    "note": "same steps without the L2 flush; not the headline"},
        "e2e": {"value": e2e_v, "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e,
                "call": "pva_forward_local with the copies around it" if w["window"] > 0
                else "pva_forward_from_host (copies overlapped with the attention)"},
        "gpu_launches": launches_per_step(w) * args.steps,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    del host, dbuf, out_host
    # The other configs, each in its own timed region, beside the headline.
    if (rank == 0 and world == 1 and w_name == "bf16_prefill" and not args.batch
            and not args.no_other_configs):
        del w, out
        torch.cuda.empty_cache()
        others = {}
        for name in OTHER_CONFIGS:
            others[name] = bench_other_config(pva, name, dev, args.steps, args.warmup, flush,
                                              peaks, local)
        line["other_configs"] = others
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w_name)
        if w_name == "bf16_prefill" and world == 1:
            line["cpu_baseline"]["fp32_small"] = fp32_oracle_check(pva, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
