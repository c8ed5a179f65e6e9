#!/usr/bin/env python
"""Benchmark of the paged KV-cache hot path on one B300 (or N independent replicas).

Default workload: Qwen3-8B-shaped decode -- 1024 sequences, context = input U{100..1024} +
generated U{100..1024}, 32 query / 8 KV heads, head_dim 128, block_size 256, 36 layer caches with
random physical block placement. One step = for each of the 36 layers: the store of the newest
token of every sequence (pkv_kv_store) and paged decode attention over the whole context
(pkv_paged_decode); the first layer's decode call plans on the device and the later ones reuse
that plan (--replan: every layer plans; --fused: one pkv_paged_decode_store per layer).

Prints one JSON line (rank 0). `--impl reference` times the fp64 CPU oracle on a bounded sample of
the same workload instead (the only reference implementation of this path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged-decode KV GB/s (% of HBM peak) and decode tokens/s at Qwen3-8B shapes"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6400.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def source_digest(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled(kernel_key, source):
    """The committed ncu figures of one kernel launch (profiles/traffic.json), or None once the
    kernel source has changed since they were captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel_key)
    if not d or d.get("source_sha") != source_digest(source):
        return None
    return d


def profiled_traffic(kernel_key, source):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    d = profiled(kernel_key, source)
    return None if d is None else d.get("dram_bytes_per_launch")


PREFILL_SRC = os.path.join(ROOT, "paged_kv_cache_496_b300", "csrc", "paged_prefill.cu")
DECODE_SRC = os.path.join(ROOT, "paged_kv_cache_496_b300", "csrc", "paged_decode.cu")
DECODE_TC_SRC = os.path.join(ROOT, "paged_kv_cache_496_b300", "csrc", "paged_decode_tc.cu")


def decode_engine_name(pk, engine):
    return "tensor_core" if engine == pk.DECODE_ENGINE_TENSOR_CORE else "cuda_core"


def decode_profile(pk, engine, workload_key):
    """(profile key, kernel source) of the decode kernel an engine runs, for profiles/traffic.json
    lookups: the CUDA-core kernel's entries are paged_decode_<workload>, the tensor-core kernel's
    paged_decode_tc_<workload>."""
    if engine == pk.DECODE_ENGINE_TENSOR_CORE:
        return "paged_decode_tc_" + workload_key, DECODE_TC_SRC
    return "paged_decode_" + workload_key, DECODE_SRC
STORE_SRC = os.path.join(ROOT, "paged_kv_cache_496_b300", "csrc", "kv_store.cu")


def prefill_profile_keys():
    """traffic and tensor-pipe utilisation of the prefix-prefill launch, from ncu (or None)."""
    d = profiled("paged_prefill_prefix", PREFILL_SRC) or {}
    return {"traffic": d.get("dram_bytes_per_launch"),
            "tensor_pipe_active_pct": d.get("tensor_pipe_active_pct"),
            "ncu_source_sha": d.get("source_sha")}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join("/tmp", f"pkv_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "50"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 300.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r[2] for r in rows)}


def max_over_ranks(x, world, device=None):
    """The slowest rank's value (timing is taken as the maximum over ranks)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, seconds_max, world):
    """Whole-job throughput of independent replicas: all ranks' units over the slowest time."""
    return units_per_rank * world / seconds_max


# ------------------------------------------------------------------------------------------------
# Workload set-up on the device
# ------------------------------------------------------------------------------------------------


class DecodeStep:
    """All layers of one decode step, resident in HBM."""

    def __init__(self, name, torch, pk, device, log_fill=True, num_seqs=None, num_layers=None,
                 fused=False, engine=None, reuse_plan=True):
        self.w = w = W.WORKLOADS[name]
        self.torch, self.pk = torch, pk
        self.ctx = W.decode_lengths(name)
        if num_seqs:
            self.ctx = self.ctx[:num_seqs]
        self.B, self.L = len(self.ctx), (num_layers or w.num_layers)
        self.bt, self.nb = W.place_blocks(W.rng_for(w.seed, 10, 0), self.ctx, w.block_size)
        self.slots = W.slots_for_positions(self.bt, np.arange(self.B), self.ctx - 1, w.block_size)
        pool_shape = (self.nb, w.block_size, w.num_kv_heads, w.head_dim)
        pool_bytes = 2 * int(np.prod(pool_shape)) * 2
        free, _ = torch.cuda.mem_get_info(device)
        per_layer_io = self.B * (2 * w.num_q_heads + 2 * w.num_kv_heads) * w.head_dim * 2
        budget = free - 6 * (1 << 30) - self.L * per_layer_io
        self.n_pools = int(max(1, min(self.L, budget // pool_bytes)))
        t0 = time.time()
        self.pools = []
        for l in range(self.n_pools):
            kc = torch.empty(pool_shape, dtype=torch.bfloat16, device=device)
            vc = torch.empty(pool_shape, dtype=torch.bfloat16, device=device)
            W.fill_normal_bf16_(kc, w.seed, 20 + l, 1)
            W.fill_normal_bf16_(vc, w.seed, 20 + l, 2)
            self.pools.append((kc, vc))
        torch.cuda.synchronize()
        if log_fill:
            log(f"[bench] {self.n_pools} layer pools of {pool_bytes / 1e9:.2f} GB filled in "
                f"{time.time() - t0:.1f} s")
        mk = lambda shape, s: W.fill_normal_bf16_(  # noqa: E731
            torch.empty(shape, dtype=torch.bfloat16, device=device), w.seed, 1000 + s)
        self.q = [mk((self.B, w.num_q_heads, w.head_dim), 3 * l) for l in range(self.L)]
        self.k_new = [mk((self.B, w.num_kv_heads, w.head_dim), 3 * l + 1) for l in range(self.L)]
        self.v_new = [mk((self.B, w.num_kv_heads, w.head_dim), 3 * l + 2) for l in range(self.L)]
        self.out = [torch.empty_like(x) for x in self.q]
        self.bt_dev = torch.from_numpy(self.bt).to(device)
        self.ctx_dev = torch.from_numpy(self.ctx).to(device)
        self.slots_dev = torch.from_numpy(self.slots).to(device)
        self.scale = 1.0 / np.sqrt(w.head_dim)
        self.plan = pk.decode_plan(self.B, w.num_q_heads, self.pools[0][0], int(self.ctx.max()), 0,
                                   engine)
        self.ws = torch.empty(max(256, self.plan.workspace_bytes), dtype=torch.uint8,
                              device=device)
        self.kv_bytes_per_layer = int(self.ctx.sum()) * w.kv_bytes_per_token
        self.fused = fused
        # Layers after the first run on the device plan the first one wrote (same lengths): with
        # the store fused, every layer launches the plan-or-store grid and the decode kernel;
        # without, kv_store and the decode kernel, plus the first layer's plan kernel.
        self.reuse = reuse_plan
        self.launches_per_step = (2 * self.L if fused else
                                  (2 * self.L + 1 if reuse_plan else 3 * self.L))

    def layer(self, l, pre=None, post=None):
        """Store the newest token of every sequence and decode layer l."""
        pk = self.pk
        kc, vc = self.pools[l % self.n_pools]
        if not self.fused:
            pk.kv_store(self.k_new[l], self.v_new[l], self.slots_dev, kc, vc)
        if pre is not None:
            pre.record()
        reuse = self.reuse and l > 0
        if self.fused:
            pk.paged_decode_store(self.q[l], self.k_new[l], self.v_new[l], self.slots_dev, kc, vc,
                                  self.bt_dev, self.ctx_dev, self.scale, out=self.out[l],
                                  plan=self.plan, workspace=self.ws, reuse_plan=reuse)
        else:
            pk.paged_decode(self.q[l], kc, vc, self.bt_dev, self.ctx_dev, self.scale,
                            out=self.out[l], plan=self.plan, workspace=self.ws,
                            reuse_plan=reuse)
        if post is not None:
            post.record()

    def run(self, events=None):
        for l in range(self.L):
            if events is None:
                self.layer(l)
            else:
                self.layer(l, events[l][0], events[l][1])


class PrefillStep:
    """The prefix-cache prefill workload: store the new tokens, then varlen causal prefill."""

    def __init__(self, torch, pk, device):
        self.torch, self.pk = torch, pk
        self.w = w = W.WORKLOADS["prefix_prefill"]
        ql = W.prefix_prefill_suffix_lengths(w.num_seqs)
        c = W.prefix_prefill_case(w.seed, w.num_seqs, 1024, 100, 1024, w.num_q_heads,
                                  w.num_kv_heads, w.head_dim, w.block_size, suffix_lens=ql)
        self.case = c
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(  # noqa
            torch.bfloat16).to(device)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)  # noqa
        self.q, self.k, self.v = bf(c.q), bf(c.k), bf(c.v)
        self.kc, self.vc = bf(c.k_cache), bf(c.v_cache)
        self.cu_q, self.cu_k = i32(c.cu_seqlens_q), i32(c.cu_seqlens_k)
        self.bt, self.slots = i32(c.block_tables), i32(c.slot_mapping)
        self.out = torch.empty_like(self.q)
        self.max_q = int(c.q_lens.max())
        qn = c.q_lens.astype(np.float64)
        pre = (c.k_lens - c.q_lens).astype(np.float64)
        pairs = float(np.sum(qn * pre + qn * (qn + 1) / 2))  # (query, key) pairs under the mask
        self.flops = 4.0 * w.head_dim * w.num_q_heads * pairs   # QK^T and PV, 2 flops per MAC
        self.tokens = int(qn.sum())

    def store(self):
        self.pk.kv_store(self.k, self.v, self.slots, self.kc, self.vc)

    def prefill(self):
        self.pk.paged_prefill(self.q, self.k, self.v, self.cu_q, self.cu_k, self.bt,
                              self.case.scale, k_cache=self.kc, v_cache=self.vc, out=self.out,
                              max_seqlen_q=self.max_q)


def measured_tensor_peak(sustained=False):
    """The bf16 GEMM peak: the burst figure (a kernel timed alone) or the sustained one (a
    kernel run back to back for seconds, under the power limit)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
        if key in d:
            return float(d[key]), "measured"
    return (1400.0 if sustained else 1800.0), "fallback"


def store_arm(args, torch, pk, device):
    """--workload kv_store_decode | kv_store_prefill: the KV store alone (a component, not the
    headline), at the decode step's size (1024 tokens, one per Qwen3-8B sequence) or the
    prefix-cache prefill's (35,968 new tokens), into a Qwen3-8B-shaped layer pool (8 kv heads,
    head_dim 128, block_size 256). GB/s counts the bytes read and written."""
    T = 1024 if args.workload == "kv_store_decode" else 35968
    nb = 5200
    kc = W.fill_normal_bf16_(torch.empty((nb, 256, 8, 128), dtype=torch.bfloat16, device=device),
                             6, 1)
    vc = W.fill_normal_bf16_(torch.empty_like(kc), 6, 2)
    slots = torch.from_numpy(W.rng_for(6, 3).permutation(nb * 256)[:T].astype(np.int32)).to(
        device)
    k = W.fill_normal_bf16_(torch.empty((T, 8, 128), dtype=torch.bfloat16, device=device), 6, 4)
    v = W.fill_normal_bf16_(torch.empty_like(k), 6, 5)
    for _ in range(args.warmup):
        pk.kv_store(k, v, slots, kc, vc)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        pk.kv_store(k, v, slots, kc, vc)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    moved = 2 * 2 * T * 8 * 128 * 2  # K and V, read and written
    peak, kind = measured_peaks()
    gbs = moved / ms / 1e6
    line = {"metric": "KV store GB/s (read + written)", "value": gbs, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "tokens": T, "num_kv_heads": 8,
                       "head_dim": 128, "block_size": 256},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "peak_source": kind,
                         "traffic": profiled_traffic(args.workload, STORE_SRC)},
            "device_error_flags": pk.get_device_error()}
    print(json.dumps(line), flush=True)
    return 0


def prefill_arm(args, torch, pk, device):
    """--workload prefix_prefill: TFLOP/s of the prefill kernel (a component, not the headline)."""
    ps = PrefillStep(torch, pk, device)
    for _ in range(args.warmup):
        ps.store()
        ps.prefill()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        ps.store()
        a.record()
        ps.prefill()
        b.record()
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    peak, kind = measured_tensor_peak()
    tf = ps.flops / (ms / 1e3) / 1e12
    line = {"metric": "prefix-cache prefill TFLOP/s (causal, algorithmic)", "value": tf,
            "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16", "accumulate": "fp32",
            "data": "synthetic", "config": {"workload": "prefix_prefill", "num_seqs": 64,
                                            "new_tokens": ps.tokens, "prefix": 1024},
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / peak, "peak_source": kind, **prefill_profile_keys()},
            "device_error_flags": pk.get_device_error()}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------
# CPU oracle arm
# ------------------------------------------------------------------------------------------------


def oracle_sample_case(name, n_seqs):
    """A host-side sample of the workload: n_seqs sequences of one layer, drawn on the host."""
    w = W.WORKLOADS[name]
    ctx = W.decode_lengths(name)[:n_seqs]
    return W.random_decode_case(w.seed, n_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                w.block_size, 0, 0, context_lens=ctx)


def time_oracle(name, target_s=10.0, max_seqs=1024):
    """Time the oracle (store + decode of one layer) on a host sample: as many sequences as make
    one run take about a second (at most one layer's worth), repeated to about target_s."""
    import oracle
    orc = oracle.default()
    w = W.WORKLOADS[name]
    n = 8

    def one(case):
        t0 = time.perf_counter()
        kc, vc, _ = orc.kv_store(case.k_new, case.v_new, case.slot_mapping, case.k_cache,
                                 case.v_cache)
        orc.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.scale)
        return time.perf_counter() - t0

    while True:
        case = oracle_sample_case(name, n)
        dt = one(case)
        if dt >= 1.0 or n >= max_seqs:
            break
        n = min(max_seqs, max(n + 1, int(n * 1.2 / max(dt, 1e-3))))
    runs, total = [dt], dt
    while total < target_s:
        runs.append(one(case))
        total += runs[-1]
    dt = sum(runs) / len(runs)
    kv = int(case.context_lens.sum()) * w.kv_bytes_per_token
    return dict(n_seqs=n, seconds=dt, runs=len(runs), kv_bytes=kv, cores=orc.max_threads(),
                gbs=kv / dt / 1e9, tokens_per_s=n / (dt * w.num_layers))


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    orc = oracle.default()
    w = W.WORKLOADS[args.workload]
    probe = time_oracle(args.workload, target_s=2.0, max_seqs=64)
    n = probe["n_seqs"]
    case = oracle_sample_case(args.workload, n)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        kc, vc, _ = orc.kv_store(case.k_new, case.v_new, case.slot_mapping, case.k_cache,
                                 case.v_cache)
        orc.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.scale)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    kv = int(case.context_lens.sum()) * w.kv_bytes_per_token
    dt = sum(times) / len(times)
    value = kv / dt / 1e9
    sample = (f"{n} of {w.num_seqs} sequences of one of {w.num_layers} layers per step "
              f"(store of the newest token + decode, fp64)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "decode_tokens_per_s": n / (dt * w.num_layers),
        "config": {"workload": args.workload, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": orc.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_8b_decode")
    ap.add_argument("--no-extras", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--fused", action="store_true",
                    help="one pkv_paged_decode_store per layer (the step's store in the decode "
                         "call's first grid) instead of pkv_kv_store then pkv_paged_decode")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: fewer layers than the workload (not a bench number)")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="profiling only: the first N sequences (not a bench number)")
    ap.add_argument("--engine", default="auto", choices=["auto", "cuda_core", "tensor_core"],
                    help="decode engine (auto: the library's choice for the shape)")
    ap.add_argument("--replan", action="store_true",
                    help="plan on the device in every layer's decode call instead of reusing the "
                         "first layer's plan")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import paged_kv_cache_496_b300 as pk

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    props = torch.cuda.get_device_properties(device)
    gpu_uuid = str(getattr(props, "uuid", "") or "")
    if gpu_uuid and not gpu_uuid.startswith("GPU-"):
        gpu_uuid = "GPU-" + gpu_uuid

    if args.workload == "prefix_prefill":
        return prefill_arm(args, torch, pk, device)
    if args.workload in ("kv_store_decode", "kv_store_prefill"):
        return store_arm(args, torch, pk, device)
    engine = {"auto": None, "cuda_core": pk.DECODE_ENGINE_CUDA_CORE,
              "tensor_core": pk.DECODE_ENGINE_TENSOR_CORE}[args.engine]
    step = DecodeStep(args.workload, torch, pk, device, num_seqs=args.num_seqs,
                      num_layers=args.layers, fused=args.fused, engine=engine,
                      reuse_plan=not args.replan)
    engine_name = decode_engine_name(pk, step.plan.engine)
    reduced = bool(args.num_seqs or args.layers)
    w = step.w

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def ranks_max(x):
        return max_over_ranks(x, world, device)

    # ---- warm-up, then the timed region ----
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    assert pk.get_device_error() == 0, "device error flag raised during warm-up"
    # CUDA events around every decode call of every fifth timed step (and of the last one): an
    # event between two kernels costs the stream a few microseconds, so bracketing every call
    # of every step would slow the step being measured by ~0.5-0.9%.
    sampled = [i % 5 == 4 or i == args.steps - 1 for i in range(args.steps)]
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(step.L)]
           if sampled[i] else None for i in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_uuid) as clocks:
        start.record()
        for i in range(args.steps):
            step.run(evs[i])
        stop.record()
        torch.cuda.synchronize()
    barrier()
    ms = ranks_max(start.elapsed_time(stop) / args.steps)
    decode_ms = [e[0].elapsed_time(e[1]) for s in evs if s is not None for e in s]
    decode_ms_mean = ranks_max(sum(decode_ms) / len(decode_ms))
    flags = pk.get_device_error()
    if flags:
        log(f"[bench] device error flags {flags:#x}")

    kv_step = step.kv_bytes_per_layer * step.L
    value = job_throughput(kv_step, ms / 1e3, world) / 1e9
    tokens_per_s = job_throughput(step.B, ms / 1e3, world)
    peak, peak_kind = measured_peaks()
    achieved = step.kv_bytes_per_layer / (decode_ms_mean / 1e3) / 1e9
    prof_key, prof_src = decode_profile(pk, step.plan.engine, "qwen3_8b")
    traffic = profiled_traffic(prof_key, prof_src) if args.workload == "qwen3_8b_decode" else None

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        h_q = [pin(x) for x in step.q]
        h_k = [pin(x) for x in step.k_new]
        h_v = [pin(x) for x in step.v_new]
        h_bt, h_ctx, h_sl = pin(step.bt_dev), pin(step.ctx_dev), pin(step.slots_dev)
        h_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in step.out]
        h2d = sum(x.numel() * x.element_size() for x in h_q + h_k + h_v + [h_bt, h_ctx, h_sl])
        d2h = sum(x.numel() * x.element_size() for x in h_out)

        # Copies overlap compute, in groups of 6 layers pipelined across steps: group g of step
        # i + 1 is copied in (stream s_in) as soon as step i has finished with group g, and group
        # g's outputs are copied out (stream s_out) as soon as they are done. The small per-step
        # tensors (tables, lengths, slots), which every layer reads, alternate between two sets.
        main = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        groups = [list(range(g, min(g + 6, step.L))) for g in range(0, step.L, 6)]
        small = [{"bt_dev": step.bt_dev, "ctx_dev": step.ctx_dev, "slots_dev": step.slots_dev},
                 {n: torch.empty_like(getattr(step, n))
                  for n in ("bt_dev", "ctx_dev", "slots_dev")}]
        ev_in = [torch.cuda.Event() for _ in groups]
        ev_done = [torch.cuda.Event() for _ in groups]
        ev_out = [torch.cuda.Event() for _ in groups]
        ev_step = [torch.cuda.Event() for _ in range(2)]

        def copy_small(i):  # step i's tables, lengths and slots into set i % 2
            k = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_step[k])  # step i - 2 no longer reads this set
                small[k]["bt_dev"].copy_(h_bt, non_blocking=True)
                small[k]["ctx_dev"].copy_(h_ctx, non_blocking=True)
                small[k]["slots_dev"].copy_(h_sl, non_blocking=True)

        def copy_group(i, g):  # step i's q, k_new, v_new of group g
            with torch.cuda.stream(s_in):
                if i >= 1:
                    s_in.wait_event(ev_done[g])  # step i - 1 has finished group g
                for l in groups[g]:
                    step.q[l].copy_(h_q[l], non_blocking=True)
                    step.k_new[l].copy_(h_k[l], non_blocking=True)
                    step.v_new[l].copy_(h_v[l], non_blocking=True)
                ev_in[g].record(s_in)

        def e2e_steps(n):
            s_in.wait_stream(main)
            copy_small(0)
            for g in range(len(groups)):
                copy_group(0, g)
            for i in range(n):
                for name, t in small[i % 2].items():
                    setattr(step, name, t)
                if i + 1 < n:
                    copy_small(i + 1)
                for g in range(len(groups)):
                    main.wait_event(ev_in[g])
                    if i >= 1:
                        main.wait_event(ev_out[g])  # step i - 1's outputs of group g are out
                    for l in groups[g]:
                        step.layer(l)
                    ev_done[g].record(main)
                    with torch.cuda.stream(s_out):
                        s_out.wait_event(ev_done[g])
                        for l in groups[g]:
                            h_out[l].copy_(step.out[l], non_blocking=True)
                        ev_out[g].record(s_out)
                    if i + 1 < n:
                        copy_group(i + 1, g)
                ev_step[i % 2].record(main)
            main.wait_stream(s_out)
            for name, t in small[0].items():  # the step's own tensors again
                setattr(step, name, t)

        e2e_steps(args.warmup)
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        e2e_steps(args.steps)
        e1.record()
        torch.cuda.synchronize()
        barrier()
        e2e_ms = ranks_max(e0.elapsed_time(e1) / args.steps)
        e2e = {"value": kv_step * world / (e2e_ms / 1e3) / 1e9, "unit": UNIT,
               "ms_per_step": e2e_ms, "decode_tokens_per_s": step.B * world / (e2e_ms / 1e3),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "overlap": "copies in groups of 6 layers, pipelined across steps"}

    extras = {}
    if not args.no_extras:
        extras = secondary_measurements(torch, pk, device, step)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not reduced:
        r = time_oracle(args.workload)
        cpu = {"value": r["gbs"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
               "sample": f"{r['n_seqs']} sequences x 1 layer (store + decode), "
                         f"{r['runs']} runs of {r['seconds']:.2f} s, KV GB/s of the sample",
               "decode_tokens_per_s": r["tokens_per_s"]}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "accumulate": "fp32", "data": "synthetic",
            "decode_tokens_per_s": tokens_per_s, "pct_of_hbm_peak": 100.0 * value / world / peak,
            "config": {"workload": args.workload, "num_seqs": step.B, "num_layers": step.L,
                       "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
                       "head_dim": w.head_dim, "block_size": w.block_size,
                       "context": w.description,
                       "mean_context": float(step.ctx.mean()),
                       "kv_bytes_per_step": kv_step, "distinct_layer_pools": step.n_pools,
                       "l2": "inputs larger than L2 (KV read per layer >> 126 MB), no flush",
                       "step": ("per layer: one pkv_paged_decode_store (a grid that stores the "
                                "newest token of every sequence and, in the first layer, plans; "
                                "then the persistent decode kernel)" if step.fused else
                                "per layer: kv_store (1 token/seq), then paged_decode") +
                               ("; layers after the first reuse the first layer's device plan"
                                if step.reuse else "; every layer plans"),
                       "decode_engine": engine_name,
                       "parallelism": f"replicas x{world}",
                       "reduced_for_profiling": reduced},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": "paged_decode (plan%s + %s)"
                                   % (" grid with the step's store" if step.fused else "",
                                      "paged_decode_tc_kernel" if engine_name == "tensor_core"
                                      else "paged_decode_kernel"),
                         "algorithmic_bytes_per_launch": step.kv_bytes_per_layer,
                         "mean_launch_ms": decode_ms_mean, "peak_source": peak_kind,
                         "decode_calls_timed": len(decode_ms),
                         "timed_calls": "every decode call of every fifth timed step and of the "
                                        "last one, CUDA events on the launching stream"},
            "clocks": clocks.summary(),
            "gpu_launches": step.launches_per_step * args.steps,
            "device_error_flags": flags,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "components": extras,
            "gpu": props.name,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def secondary_measurements(torch, pk, device, main_step):
    """Other rows of the hot path, each timed on its own (not part of the step above)."""
    res = {}

    def timed(fn, reps=10):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    # the same step through the other API: the store fused into the decode kernel, or not
    was = main_step.fused
    main_step.fused = not was
    ms = timed(main_step.run, reps=3)
    main_step.fused = was
    res["fused_step" if not was else "unfused_step"] = {
        "ms": ms, "GB/s": main_step.kv_bytes_per_layer * main_step.L / ms / 1e6}

    # the same step planning in every layer instead of reusing the first layer's device plan
    was = main_step.reuse
    main_step.reuse = not was
    ms = timed(main_step.run, reps=3)
    main_step.reuse = was
    res["step_planning_every_layer" if was else "step_reusing_plan"] = {
        "ms": ms, "GB/s": main_step.kv_bytes_per_layer * main_step.L / ms / 1e6}

    # the same step on the other decode engine (the library picks one per shape)
    plan = main_step.plan
    other = (pk.DECODE_ENGINE_CUDA_CORE if plan.engine == pk.DECODE_ENGINE_TENSOR_CORE
             else pk.DECODE_ENGINE_TENSOR_CORE)
    try:
        main_step.plan = pk.decode_plan(main_step.B, main_step.w.num_q_heads,
                                        main_step.pools[0][0], int(main_step.ctx.max()), 0, other)
        ms = timed(main_step.run, reps=5)
        res["step_on_" + decode_engine_name(pk, other)] = {
            "ms": ms, "GB/s": main_step.kv_bytes_per_layer * main_step.L / ms / 1e6}
    except Exception as e:  # the other engine may not support the shape: report it
        res["step_on_" + decode_engine_name(pk, other)] = {"error": repr(e)}
    finally:
        main_step.plan = plan

    # kv_store alone at the decode size (launch-bound) and at the prefill size (bandwidth-bound)
    kc, vc = main_step.pools[0]
    ms = timed(lambda: pk.kv_store(main_step.k_new[0], main_step.v_new[0], main_step.slots_dev,
                                   kc, vc))
    row = main_step.w.kv_bytes_per_token // 2
    res["kv_store_1024_tokens"] = {"ms": ms, "GB/s": 2 * 2 * main_step.B * row / ms / 1e6,
                                   "traffic": profiled_traffic("kv_store_decode", STORE_SRC)}
    T = 35968
    rng = W.rng_for(4, 300)
    slots = torch.from_numpy(rng.permutation(main_step.nb * 256)[:T].astype(np.int32)).to(device)
    kn = W.fill_normal_bf16_(torch.empty((T, 8, 128), dtype=torch.bfloat16, device=device),
                             4, 301)
    ms = timed(lambda: pk.kv_store(kn, kn, slots, kc, vc))
    res["kv_store_35968_tokens"] = {"ms": ms, "GB/s": 2 * 2 * T * row / ms / 1e6,
                                    "traffic": profiled_traffic("kv_store_prefill", STORE_SRC)}

    # whole-block moves on the decode pool: 512 copy-on-write copies and a 512-block swap-out
    perm = torch.from_numpy(W.rng_for(3, 500).permutation(main_step.nb)[:1024].astype(np.int32))
    pairs = perm.view(512, 2).contiguous().to(device)
    ids = perm[:512].contiguous().to(device)
    blk_bytes = 256 * main_step.w.num_kv_heads * main_step.w.head_dim * 2 * 2  # K and V
    ms = timed(lambda: pk.copy_blocks(kc, vc, pairs))
    res["copy_blocks_512"] = {"ms": ms, "GB/s": 2 * 512 * blk_bytes / ms / 1e6}
    gk, gv = pk.gather_blocks(kc, vc, ids)
    ms = timed(lambda: pk.gather_blocks(kc, vc, ids, out_k=gk, out_v=gv))
    res["gather_blocks_512"] = {"ms": ms, "GB/s": 2 * 512 * blk_bytes / ms / 1e6}
    del gk, gv

    # chained block hashes of the decode batch's token ids (prefix-cache lookup)
    ctx = main_step.ctx
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)).to(device)
    tok = torch.from_numpy(W.rng_for(3, 600).integers(0, 151936, int(ctx.sum()))
                           .astype(np.int32)).to(device)
    mb = int(ctx.max()) // 256
    hashes = torch.empty((len(ctx), mb), dtype=torch.int64, device=device)
    ms = timed(lambda: pk.block_hashes(tok, cu, 256, mb, out=hashes))
    nfull = int((ctx // 256).sum())
    res["block_hashes_qwen3_8b_batch"] = {"ms": ms, "full_blocks": nfull,
                                          "GB/s": nfull * 256 * 4 / ms / 1e6}

    # long-context split decode (one layer)
    try:
        layer = _decode_layer("long_splitk_decode", torch, device)
        ms = timed(lambda: pk.paged_decode(layer["q"], layer["kc"], layer["vc"], layer["bt"],
                                           layer["ctx"], layer["scale"], out=layer["out"],
                                           plan=layer["plan"], workspace=layer["ws"]))
        # the same call reusing the plan a first call made, as the layers of a step after the
        # first do (the plan kernel then drops out of the call)
        ms_reused = timed(lambda: pk.paged_decode(
            layer["q"], layer["kc"], layer["vc"], layer["bt"], layer["ctx"], layer["scale"],
            out=layer["out"], plan=layer["plan"], workspace=layer["ws"], reuse_plan=True))
        lp = profiled(*decode_profile(pk, layer["plan"].engine, "long_splitk")) or {}
        res["long_splitk_decode"] = {"ms": ms, "GB/s": layer["kv"] / ms / 1e6,
                                     "ms_plan_reused": ms_reused,
                                     "GB/s_plan_reused": layer["kv"] / ms_reused / 1e6,
                                     "decode_engine": decode_engine_name(pk, layer["plan"].engine),
                                     "frac_of_hbm_peak": layer["kv"] / ms / 1e6 /
                                     measured_peaks()[0],
                                     "traffic": lp.get("dram_bytes_per_launch"),
                                     "dram_throughput_pct": lp.get("dram_throughput_pct_of_peak")}
        del layer
    except Exception as e:  # report, do not hide
        res["long_splitk_decode"] = {"error": repr(e)}
    ps = None
    try:
        ps = PrefillStep(torch, pk, device)
        ps.store()
        # Burst: a few calls timed alone after the memory-bound work above, against the burst
        # GEMM peak. The sustained figure is taken last (below): seconds at the power limit
        # would lower the clock of whatever is timed after them. (An idle pause before the
        # burst does not help: the clock drops to idle and the warm-up calls do not restore it.)
        ms = timed(ps.prefill)
        peak, _ = measured_tensor_peak()
        tf = ps.flops / (ms / 1e3) / 1e12
        res["prefix_prefill"] = {"ms": ms, "TFLOP/s": tf, "frac_of_bf16_peak": tf / peak,
                                 "timing": "burst: a few calls timed alone",
                                 "new_tokens": ps.tokens, **prefill_profile_keys()}
    except Exception as e:
        res["prefix_prefill"] = {"error": repr(e)}
    try:
        res["mixed_prefill_decode"] = _mixed_batch(torch, pk, device, timed)
    except Exception as e:
        res["mixed_prefill_decode"] = {"error": repr(e)}
    try:
        res["qwen3_0p6b_step"] = _qwen3_0p6b_step(torch, pk, device)
    except Exception as e:
        res["qwen3_0p6b_step"] = {"error": repr(e)}
    try:
        if ps is not None and "error" not in res["prefix_prefill"]:
            # sustained: after two seconds of back-to-back calls, against the sustained peak
            t_end = time.time() + 2.0
            while time.time() < t_end:
                for _ in range(20):
                    ps.prefill()
                torch.cuda.synchronize()
            ms_sus = timed(ps.prefill, reps=200)
            peak_sus, _ = measured_tensor_peak(sustained=True)
            tf_sus = ps.flops / (ms_sus / 1e3) / 1e12
            res["prefix_prefill"].update({"ms_sustained": ms_sus, "TFLOP/s_sustained": tf_sus,
                                          "frac_of_sustained_bf16_peak": tf_sus / peak_sus})
    except Exception as e:
        res["prefix_prefill"]["sustained_error"] = repr(e)
    del ps
    return res


def _qwen3_0p6b_step(torch, pk, device, steps=10):
    """The whole Qwen3-0.6B-shaped decode step: 28 layers x (kv_store of the newest token of 256
    sequences, then paged decode), one distinct layer pool each (while memory allows), timed like
    the headline step: CUDA events around the step and around every decode call."""
    st = DecodeStep("qwen3_0p6b_decode", torch, pk, device, log_fill=False)
    for _ in range(3):
        st.run()
    torch.cuda.synchronize()
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(st.L)]
           for _ in range(steps)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(steps):
        st.run(evs[i])
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    dec = [e[0].elapsed_time(e[1]) for s_ in evs for e in s_]
    dec_ms = sum(dec) / len(dec)
    peak, _ = measured_peaks()
    kv_step = st.kv_bytes_per_layer * st.L
    achieved = st.kv_bytes_per_layer / (dec_ms / 1e3) / 1e9
    out = {"ms_per_step": ms, "GB/s": kv_step / ms / 1e6,
           "decode_tokens_per_s": st.B / (ms / 1e3), "frac_of_hbm_peak": kv_step / ms / 1e6 / peak,
           "decode_mean_launch_ms": dec_ms, "decode_frac": achieved / peak,
           "num_seqs": st.B, "num_layers": st.L, "distinct_layer_pools": st.n_pools,
           "decode_engine": decode_engine_name(pk, st.plan.engine),
           "kv_bytes_per_step": kv_step, "flags": pk.get_device_error()}
    del st
    torch.cuda.empty_cache()
    return out


def _mixed_batch(torch, pk, device, timed):
    """One varlen call mixing 960 decode rows (one new token each) and 64 prefill chunks of 256
    tokens after a 512-token cached prefix, at Qwen3-8B head geometry, block size 256."""
    import paged_kv_cache_496_b300 as pkm
    rng = W.rng_for(7, 400)
    n_dec, n_pre = 960, 64
    dec_ctx = W.decode_context_lengths(rng, n_dec)
    ql = np.concatenate([np.ones(n_dec, np.int32), np.full(n_pre, 256, np.int32)])
    prefix = np.concatenate([dec_ctx - 1, np.full(n_pre, 512, np.int32)]).astype(np.int32)
    kl = ql + prefix
    BS, Hq, Hkv, D = 256, 32, 8, 128
    bt, nb = W.place_blocks(rng, kl, BS)
    mk = lambda shape, s: W.fill_normal_bf16_(  # noqa: E731
        torch.empty(shape, dtype=torch.bfloat16, device=device), 7, s)
    kc, vc = mk((nb, BS, Hkv, D), 1), mk((nb, BS, Hkv, D), 2)
    T = int(ql.sum())
    q, k, v = mk((T, Hq, D), 3), mk((T, Hkv, D), 4), mk((T, Hkv, D), 5)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)  # noqa
    cu_q = i32(np.concatenate([[0], np.cumsum(ql)]))
    cu_k = i32(np.concatenate([[0], np.cumsum(kl)]))
    seq = np.concatenate([np.full(n, b) for b, n in enumerate(ql)])
    pos = np.concatenate([prefix[b] + np.arange(n) for b, n in enumerate(ql)])
    slots = i32(W.slots_for_positions(bt, seq, pos, BS))
    btd = i32(bt)
    out = torch.empty_like(q)
    pkm.kv_store(k, v, slots, kc, vc)

    def call():
        pkm.paged_prefill(q, k, v, cu_q, cu_k, btd, 1 / np.sqrt(D), k_cache=kc, v_cache=vc,
                          out=out, max_seqlen_q=256)
    ms = timed(call)
    qn, pre = ql.astype(np.float64), prefix.astype(np.float64)
    flops = 4.0 * D * Hq * float(np.sum(qn * pre + qn * (qn + 1) / 2))
    kv = float(kl.sum()) * Hkv * D * 4
    return {"ms": ms, "TFLOP/s": flops / ms / 1e9, "KV GB/s": kv / ms / 1e6,
            "rows": "960 decode + 64 x 256 prefill", "timing": "burst: a few calls timed alone"}


def _decode_layer(name, torch, device):
    import paged_kv_cache_496_b300 as pk
    w = W.WORKLOADS[name]
    ctx = W.decode_lengths(name)
    bt, nb = W.place_blocks(W.rng_for(w.seed, 10, 0), ctx, w.block_size)
    shape = (nb, w.block_size, w.num_kv_heads, w.head_dim)
    kc = W.fill_normal_bf16_(torch.empty(shape, dtype=torch.bfloat16, device=device), w.seed, 1)
    vc = W.fill_normal_bf16_(torch.empty(shape, dtype=torch.bfloat16, device=device), w.seed, 2)
    q = W.fill_normal_bf16_(torch.empty((len(ctx), w.num_q_heads, w.head_dim),
                                        dtype=torch.bfloat16, device=device), w.seed, 3)
    plan = pk.decode_plan(len(ctx), w.num_q_heads, kc, int(ctx.max()), 0)
    return dict(q=q, kc=kc, vc=vc, bt=torch.from_numpy(bt).to(device),
                ctx=torch.from_numpy(ctx).to(device), scale=1.0 / np.sqrt(w.head_dim),
                out=torch.empty_like(q), plan=plan,
                ws=torch.empty(max(256, plan.workspace_bytes), dtype=torch.uint8, device=device),
                kv=int(ctx.sum()) * w.kv_bytes_per_token)


if __name__ == "__main__":
    sys.exit(main())
