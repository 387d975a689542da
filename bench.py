#!/usr/bin/env python
"""Benchmark of the fused ZeRO-2 step: mean reduce-scatter of n_dp bf16 gradient
buffers + fp32 AdamW + bf16 cast + gather write, on one GB300 per process.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the whole path over the workload: the bucket loop of
zero_reduce_scatter_adamw launches over every owned shard.  Default workload:
GPT-2-XL shapes (N = 1,557,611,200 parameters, 48 blocks, d 1600, ffn 6400,
vocab 50257) flattened for n_dp = 8 simulated ranks, 5e8-element buckets.  The
Llama-7B single-shard workload (S = 842,301,952, 8 gradient slices with 1 %
outliers x100) is measured in the same run and reported under "workloads".

Printed: one JSON line (rank 0).  `value` = parameters updated per second over
all ranks (each rank runs its own replica: the simulated ranks live in one
GPU's memory, nothing is exchanged between GPUs, so N GPUs are N independent
replicas -> weak scaling).  Inputs are larger than L2 (tens of GB), so no L2
flush is needed between steps.  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "params updated/s for fused reduce+AdamW+cast+gather; HBM GB/s vs GB300 peak"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
SEED = 0
HP = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
CPU_SAMPLE = 1 << 25          # elements of the cpu_baseline sample
CPU_BASELINE_SECONDS = 10.0   # CPU work for the cpu_baseline leg
REF_SAMPLE = 1 << 23          # elements per step of the reference arm (bounded CPU sample)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["gpt2xl", "llama7b-shard", "probe"], default="gpt2xl",
                    help="probe: N = 2^26 at n_dp = 8 in one launch (about 2 GB on the device, "
                         "larger than L2), the case used for ncu section captures")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the second workload")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# distributed plumbing (replicas: a barrier and a max over ranks, nothing else)
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, local):
    import torch
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float, device) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        self.sel = []
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, pw, reasons = [], [], [], set()
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                pw.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------

def _peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _kernel_source_hash():
    h = hashlib.sha256()
    for name in ("zero_rs_adamw.cu", "zero_common.cuh"):
        with open(os.path.join(ROOT, "zero_sharded_mixed_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic_per_elem(n_src):
    """DRAM bytes per element of the fused kernel from a committed ncu summary,
    or None when the kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "rs_adamw_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("kernel_source_sha") != _kernel_source_hash():
            return None
        return float(rec["dram_bytes_per_element"][str(n_src)])
    except Exception:
        return None


class Workload:
    """Device buffers and the step of one configuration."""

    def __init__(self, name, device):
        import torch
        from zero_sharded_mixed_gb300 import binding as zb
        from zero_sharded_mixed_gb300 import inputs
        from zero_sharded_mixed_gb300.step import bucket_ranges
        self.name = name
        self.zb = zb
        self.device = device
        n_dp = 8
        if name == "gpt2xl":
            numels = inputs.gpt2xl_numels()
            L = zb.zero_layout(numels, n_dp, 8, 500_000_000)
            self.owner = None
            lo, hi = 0, L.padded_n
            self.rank_begin, self.rank_end, self.src_base = 0, n_dp, 0
            src_len, outlier = L.padded_n, 0.0
            self.desc = {"workload": "gpt2xl_zero2_all_shards", "model": "GPT-2-XL shapes",
                         "N": L.n, "n_dp": n_dp, "shard": L.shard, "padded_n": L.padded_n,
                         "bucket": L.bucket, "buckets": L.n_buckets}
        elif name == "probe":
            L = zb.zero_layout([1 << 26], n_dp, 8, 500_000_000)
            self.owner = None
            lo, hi = 0, L.padded_n
            self.rank_begin, self.rank_end, self.src_base = 0, n_dp, 0
            src_len, outlier = L.padded_n, 0.0
            self.desc = {"workload": "probe_flat_2p26_ndp8", "model": "flat vector",
                         "N": L.n, "n_dp": n_dp, "shard": L.shard, "padded_n": L.padded_n,
                         "bucket": L.bucket, "buckets": L.n_buckets}
        else:
            numels = inputs.llama7b_numels()
            L = zb.zero_layout(numels, n_dp, 8, 500_000_000)
            o = 0
            self.owner = o
            lo, hi = o * L.shard, (o + 1) * L.shard
            self.rank_begin, self.rank_end, self.src_base = o, o + 1, lo
            src_len, outlier = L.shard, 0.01
            self.desc = {"workload": "llama7b_zero2_one_shard", "model": "Llama-7B shapes",
                         "N": L.n, "n_dp": n_dp, "shard": L.shard, "owner": o,
                         "bucket": L.bucket, "outliers": "1% x100"}
        self.L = L
        self.ranges = bucket_ranges(L, lo, hi)
        self.elems = hi - lo
        self.n_src = n_dp
        self.bytes_per_elem = 26 + 2 * n_dp
        g = torch.empty((n_dp, src_len), dtype=torch.bfloat16, device=device)
        n_real = max(0, min(L.n, hi) - lo)
        for r in range(n_dp):
            inputs.grad_bf16_into(g[r], n_real, SEED, step=1, rank=r, outlier_p=outlier)
        self.grads = g
        self.grad_list = [g[r] for r in range(n_dp)]
        w = torch.zeros(self.elems, dtype=torch.float32, device=device)
        if n_real:
            w[:n_real].normal_(0.0, 0.02, generator=torch.Generator(device=device).manual_seed(
                inputs.derive_seed(SEED, 1)))
        self.master = w
        self.m = torch.zeros_like(w)
        self.v = torch.zeros_like(w)
        self.out = torch.zeros(L.padded_n, dtype=torch.bfloat16, device=device)
        self.launches_per_step = len(self.ranges)
        self.device_bytes = (g.numel() * 2 + 3 * w.numel() * 4 + self.out.numel() * 2)

    def hp(self, t):
        return self.zb.ZeroAdamW.make(step=t, **HP)

    def step(self, t, events=None):
        zb = self.zb
        hp = self.hp(t)
        for j, (s, e) in enumerate(self.ranges):
            if events is not None:
                events[j][0].record()
            zb.zero_reduce_scatter_adamw(self.L, self.grad_list, zb.ZERO_BF16, self.src_base,
                                         float(self.L.n_dp), self.rank_begin, self.rank_end, s, e,
                                         self.master, self.m, self.v, self.out, zb.ZERO_OUT_FULL, hp)
            if events is not None:
                events[j][1].record()

    def free(self):
        for k in ("grads", "grad_list", "master", "m", "v", "out"):
            setattr(self, k, None)


def time_workload(wl, steps, warmup, dist, device, sampler=None):
    import torch
    t = 1
    for _ in range(warmup):
        wl.step(t)
        t += 1
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in wl.ranges] for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.15)
    start.record()
    for k in range(steps):
        wl.step(t, ev[k])
        t += 1
    end.record()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    total_ms = start.elapsed_time(end)
    kernel_ms = sum(a.elapsed_time(b) for step_ev in ev for a, b in step_ev)
    return total_ms, kernel_ms, clocks, t


def time_e2e(wl, steps, warmup, t0, dist):
    """The same step through the public binding with host buffers: every step
    copies the n_dp gradient buffers from pinned host memory to the device and
    reads the updated bf16 weights back to pinned host memory."""
    import torch
    host_g = torch.empty(wl.grads.shape, dtype=wl.grads.dtype, pin_memory=True)
    host_g.copy_(wl.grads)
    host_out = torch.empty(wl.out.shape, dtype=wl.out.dtype, pin_memory=True)
    t = t0

    def one():
        nonlocal t
        wl.grads.copy_(host_g, non_blocking=True)
        wl.step(t)
        host_out.copy_(wl.out, non_blocking=True)
        t += 1

    for _ in range(warmup):
        one()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(dist)
    start.record()
    for _ in range(steps):
        one()
    end.record()
    torch.cuda.synchronize()
    barrier(dist)
    ms = start.elapsed_time(end) / steps
    return ms, host_g.numel() * 2, host_out.numel() * 2


def cpu_sample(wl, n):
    """A contiguous sample of the workload copied to the host: (grads, w, m, v)."""
    import numpy as np
    import torch
    n = min(n, wl.elems)
    g = wl.grads[:, :n].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    w = wl.master[:n].cpu().numpy().copy()
    m = wl.m[:n].cpu().numpy().copy()
    v = wl.v[:n].cpu().numpy().copy()
    return g, w, m, v


def time_oracle(sample, seconds, n_dp):
    import oracle
    g, w, m, v = sample
    hp = oracle.AdamW(**HP)
    t = 1
    done = 0
    t0 = time.perf_counter()
    while True:
        _, w, m, v = oracle.rs_adamw_reference(g, n_dp, w, m, v, hp, t)
        t += 1
        done += g.shape[1]
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return done / el, el, done


# --------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------

def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, local)
    from zero_sharded_mixed_gb300 import binding as zb
    from zero_sharded_mixed_gb300 import build as zbuild
    if rank == 0 or not os.path.exists(zb.lib_path):
        zbuild.build()
    barrier(dist)
    zb.load()

    peak, peak_kind = _peak()
    primary = args.workload
    extra = [w for w in ("gpt2xl", "llama7b-shard") if w != primary]
    order = [primary] + ([] if args.no_extra or primary == "probe" else extra)
    results = {}
    line = None
    for name in order:
        wl = Workload(name, device)
        torch.cuda.synchronize()
        sampler = ClockSampler(local) if name == primary else None
        total_ms, kernel_ms, clocks, t_next = time_workload(wl, args.steps, args.warmup, dist, device, sampler)
        ms_step = max_over_ranks(dist, total_ms / args.steps, device)
        kern_ms = max_over_ranks(dist, kernel_ms / args.steps, device)
        value = wl.elems * world / (ms_step / 1e3)
        launches = wl.launches_per_step
        bytes_step = wl.elems * wl.bytes_per_elem
        achieved = bytes_step / (kern_ms / 1e3) / 1e9
        tpe = _traffic_per_elem(wl.n_src)
        res = {
            "value": value, "ms_per_step": ms_step,
            "hbm_gbs_step": bytes_step / (ms_step / 1e3) / 1e9,
            "config": dict(wl.desc, l2="inputs %.1f GB > 129 MB L2, no flush" % (wl.device_bytes / 1e9)),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": (tpe * wl.elems / launches) if tpe is not None else None,
                         "algorithmic_bytes_per_launch": bytes_step / launches,
                         "bytes_per_param": wl.bytes_per_elem,
                         "kernel": "zgb::rs_adamw_vec_kernel<%d,true>" % wl.n_src},
            "gpu_launches": launches * args.steps,
        }
        if name == primary:
            res["clocks"] = clocks
            if not args.no_e2e:
                e2e_steps = max(1, min(args.steps, 10))
                e_ms, h2d, d2h = time_e2e(wl, e2e_steps, 1, t_next + 1, dist)
                e_ms = max_over_ranks(dist, e_ms, device)
                res["e2e"] = {"value": wl.elems * world / (e_ms / 1e3), "unit": UNIT,
                              "ms_per_step": e_ms, "steps": e2e_steps,
                              "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
            if not args.no_cpu_baseline and world == 1 and rank == 0:
                sample = cpu_sample(wl, CPU_SAMPLE)
                rate, secs, done = time_oracle(sample, CPU_BASELINE_SECONDS, wl.n_src)
                res["cpu_baseline"] = {
                    "value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                    "sample": "first %d owned elements of the workload (all %d gradient slices), "
                              "%d oracle steps, %.1f s single-threaded" % (sample[1].size, wl.n_src,
                                                                          done // sample[1].size, secs)}
        results[name] = res
        wl.free()
        del wl
        torch.cuda.empty_cache()

    if rank == 0:
        p = results[primary]
        line = {
            "metric": METRIC, "value": p["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": p["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "storage": "bf16 gradients and weights, fp32 master/m/v",
            "data": "synthetic (seeded normal gradients and weights, model shapes only)",
            "config": dict(p["config"], parallelism="replicas x%d (simulated n_dp=%d per GPU)"
                           % (world, p["config"]["n_dp"])),
            "hbm_gbs_step": p["hbm_gbs_step"],
            "roofline": p["roofline"],
            "gpu_launches": p["gpu_launches"],
            "clocks": p.get("clocks"),
            "e2e": p.get("e2e"),
            "cpu_baseline": p.get("cpu_baseline"),
            "impl": "ours",
            "workloads": {k: {kk: v[kk] for kk in ("value", "ms_per_step", "hbm_gbs_step", "roofline", "config")}
                          for k, v in results.items() if k != primary},
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle, as it stands, on a bounded sample of the same workload:
    each step updates REF_SAMPLE owned elements from all n_dp gradient slices."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from zero_sharded_mixed_gb300 import inputs
    n_dp = 8
    n = REF_SAMPLE
    g = inputs.grads_bf16(n_dp, n, n, seed=SEED, step=1,
                          outlier_p=0.01 if args.workload == "llama7b-shard" else 0.0)
    gb = inputs.bf16_bits(g)
    w = inputs.master_weights(n, n, seed=SEED).numpy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    hp = oracle.AdamW(**HP)
    t = 1
    for _ in range(args.warmup):
        _, w, m, v = oracle.rs_adamw_reference(gb, n_dp, w, m, v, hp, t)
        t += 1
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _, w, m, v = oracle.rs_adamw_reference(gb, n_dp, w, m, v, hp, t)
        t += 1
    el = time.perf_counter() - t0
    ms = el * 1e3 / max(1, args.steps)
    value = n / (ms / 1e3)
    wl_name = {"gpt2xl": "gpt2xl_zero2_all_shards", "llama7b-shard": "llama7b_zero2_one_shard",
               "probe": "probe_flat_2p26_ndp8"}[args.workload]
    sample = "%d owned elements per step (a bounded sample of %s), %d gradient slices" % (n, wl_name, n_dp)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
        "config": {"workload": wl_name, "n_dp": n_dp, "sample_elements": n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
