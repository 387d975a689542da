#!/usr/bin/env python
"""Benchmark of the ZeRO step on one GB300 per process: the fused mean
reduce-scatter of n_dp bf16 gradient buffers + fp32 AdamW + bf16 cast + gather
write, plus the accumulation and ZeRO-3 paths.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the path over the workload.  The headline workload
(the last JSON line) is GPT-2-XL shapes (N = 1,557,611,200 parameters, 48
blocks, d 1600, ffn 6400, vocab 50257) flattened for n_dp = 8 simulated ranks
with 5e8-element buckets, every owned shard updated each step.  Measured in the
same run with fewer steps, each printed on a JSON line of its own before the
headline (key "workload_result"):
  llama7b-shard       one owned shard of Llama-7B shapes (S = 842,301,952), 8 slices
                      with 1 % outliers x100 (also summarised in the headline's
                      "target_7b": the fused update's fraction of the copy peak);
  gpt2xl-clip         the GPT-2-XL step with clipping by the global gradient norm
                      (a norm pass, then the clipped fused update);
  gpt2xl-qgrad        the GPT-2-XL step with ZeRO++ 8-bit gradients;
  accum-zero1/2       gradient accumulation, GPT-2-XL shapes, n_dp = 4, 4
                      micro-batches, in the stage-1 and stage-2 orders;
  zero3               the per-unit gather / reduce-scatter / update path over the
                      34 Llama-7B units at n_dp = 8;
  zero3-fused         the same with each unit's reduce-scatter and update in one
                      pass; zero3-fused-graph: that step captured in a CUDA graph;
  zero3-prefetch      each unit's gather issued one unit ahead on a side stream;
  zero3-int8[-fused]  8-bit weight gathers (ZeRO++);
  zero3-zeropp[-fused] both ZeRO++ 8-bit paths;
  cast                the bf16 cast of GPT-2-XL-sized master weights on its own
                      (zero_cast_bf16, the engines' set-up and restore step);
  checkpoint          a save / restore of one Llama-7B block unit's shards.
Only with --with-compute: zero3-compute and zero3-prefetch-compute, the
unfused step with a stand-in layer matmul (cuBLAS) per unit, gathers in line
and one unit ahead.  Each workload carries the oracle timed on the same kind of
step beside it (cpu_baseline).  Every launch is timed with CUDA events on its
stream; `roofline` uses the dominant kernel's algorithmic bytes per launch over
its average launch time.

`value` = parameters updated per second over all ranks.  The simulated ranks
live in one GPU's memory and nothing is exchanged between GPUs, so N GPUs run
N independent replicas (weak scaling).  Inputs are tens of GB, larger than L2,
so no L2 flush is needed between steps.  --impl reference times the CPU oracle
on a bounded sample of the same workload instead.
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
QGRAD_BLOCK = 256        # block of the 8-bit gradient format in the ZeRO++ workloads
HP = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
CPU_SAMPLE = 1 << 25          # elements of the cpu_baseline sample
CPU_BASELINE_SECONDS = 6.0    # wall seconds of the all-cores cpu_baseline leg (plus a quarter on one core)
HEADLINE_MAX_CHARS = 2000     # the headline JSON line stays short enough to survive a tail of the log
TARGET_FRAC_7B = 0.8          # the bandwidth fraction asked of the fused update on the Llama-7B shard
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e nominal bandwidth, beside the measured copy peak
REF_SAMPLE = 1 << 25          # elements per step of the reference arm (bounded CPU sample)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["gpt2xl", "gpt2xl-clip", "gpt2xl-qgrad", "llama7b-shard",
                                           "probe", "accum-zero1", "accum-zero2", "cast", "zero3",
                                           "zero3-int8", "zero3-prefetch", "zero3-zeropp",
                                           "zero3-fused", "zero3-int8-fused", "zero3-zeropp-fused",
                                           "zero3-fused-graph", "zero3-compute", "zero3-prefetch-compute"],
                    default="gpt2xl",
                    help="probe: N = 2^26 at n_dp = 8 in one launch (about 2 GB on the device, "
                         "larger than L2), the case used for ncu section captures")
    ap.add_argument("--elems", type=int, default=0,
                    help="replace the model shape by a flat vector of this many elements "
                         "(small cases for profiling; not a headline workload)")
    ap.add_argument("--bucket", type=int, default=500_000_000,
                    help="reduce bucket in elements of the ZeRO-1/2 workloads run with --elems "
                         "(small cases for profiling; the model workloads keep 5e8)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--with-compute", action="store_true",
                    help="also time the two ZeRO-3 workloads with a stand-in layer matmul (cuBLAS) per unit")
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


def replica_value(elems_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job parameters updated per second: every rank updates its own
    replica's elements; the slowest rank's step time counts."""
    return elems_per_rank * world / (ms_per_step / 1e3)


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
    """Hash of the fused update's code: its sources with // comments and blank
    lines removed, so that an edit of a comment keeps a traffic record valid."""
    import re
    h = hashlib.sha256()
    for name in ("zero_rs_adamw.cu", "zero_common.cuh", "zero_update.cuh", "zero_quant.cuh"):
        with open(os.path.join(ROOT, "zero_sharded_mixed_gb300", "csrc", name)) as f:
            for line in f:
                code = re.sub(r"//.*", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
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


class Op:
    """One timed call of a step: kernel kind, algorithmic bytes, the call, and
    how many of the library's kernels the call launches."""
    __slots__ = ("kind", "bytes", "fn", "kernels")

    def __init__(self, kind, nbytes, fn, kernels=1):
        self.kind, self.bytes, self.fn, self.kernels = kind, nbytes, fn, kernels


class Workload:
    """Device buffers and the step (a list of Ops) of one configuration."""

    n_src = 8
    kernel_label = "zgb::rs_adamw_vec_kernel<0,8> (bf16 sources x 8)"

    def __init__(self, device):
        from zero_sharded_mixed_gb300 import binding as zb
        self.zb = zb
        self.device = device

    def hp(self, t):
        return self.zb.ZeroAdamW.make(step=t, **HP)

    def ops(self, t):
        raise NotImplementedError

    def free(self):
        for k in list(vars(self)):
            if k not in ("zb", "device", "desc", "elems", "device_bytes", "name", "bytes_per_elem",
                         "dominant"):
                setattr(self, k, None)


def _owners(L, begin, end):
    """Launches of one 8-bit gradient call over [begin, end) (aligned buffers):
    one for a range of several whole shards (the owners share one grid) or of
    several owners whose boundaries lie on the range's 8-element grid (one
    stream over the range), else one per owner whose shard the range meets."""
    if end <= begin:
        return 0
    owners = (end - 1) // L.shard - begin // L.shard + 1
    if owners > 1 and begin % L.shard == 0 and end % L.shard == 0:
        return 1
    if owners > 1 and L.shard % 8 == 0 and begin % 8 == 0:
        return 1
    return owners


def _master(n_real, n, device):
    import torch
    from zero_sharded_mixed_gb300 import inputs
    w = torch.zeros(n, dtype=torch.float32, device=device)
    if n_real:
        w[:n_real].normal_(0.0, 0.02, generator=torch.Generator(device=device).manual_seed(
            inputs.derive_seed(SEED, 1)))
    return w


class Zero2Workload(Workload):
    """ZeRO-2 step: the bucketed fused update of every owned element in
    [lo, hi) from n_dp bf16 gradient buffers."""

    def __init__(self, name, device, elems=0, bucket=500_000_000):
        import torch
        from zero_sharded_mixed_gb300 import inputs
        from zero_sharded_mixed_gb300.step import bucket_ranges
        super().__init__(device)
        zb = self.zb
        n_dp = 8
        self.name = name
        self.clip = name == "gpt2xl-clip"
        self.qgrad = name == "gpt2xl-qgrad"
        if name in ("gpt2xl", "gpt2xl-clip", "gpt2xl-qgrad"):
            numels = [elems] if elems else inputs.gpt2xl_numels()
            L = zb.zero_layout(numels, n_dp, 8, bucket if elems else 500_000_000)
            lo, hi, self.rank_begin, self.rank_end = 0, L.padded_n, 0, n_dp
            src_len, outlier = L.padded_n, 0.0
            self.desc = {"workload": ("flat%d_zero2" % elems if elems else "gpt2xl_zero2_all_shards")
                         + ("_clip1.0" if self.clip else "") + ("_int8_grads" if self.qgrad else ""),
                         "model": "flat vector" if elems else "GPT-2-XL shapes",
                         "N": L.n, "n_dp": n_dp, "shard": L.shard, "padded_n": L.padded_n,
                         "bucket": L.bucket, "buckets": L.n_buckets}
        elif name == "probe":
            L = zb.zero_layout([1 << 26], n_dp, 8, 500_000_000)
            lo, hi, self.rank_begin, self.rank_end = 0, L.padded_n, 0, n_dp
            src_len, outlier = L.padded_n, 0.0
            self.desc = {"workload": "probe_flat_2p26_ndp8", "model": "flat vector",
                         "N": L.n, "n_dp": n_dp, "shard": L.shard, "padded_n": L.padded_n,
                         "bucket": L.bucket, "buckets": L.n_buckets}
        else:
            L = zb.zero_layout(inputs.llama7b_numels(), n_dp, 8, 500_000_000)
            o = 0
            lo, hi, self.rank_begin, self.rank_end = o * L.shard, (o + 1) * L.shard, o, o + 1
            src_len, outlier = L.shard, 0.01
            self.desc = {"workload": "llama7b_zero2_one_shard", "model": "Llama-7B shapes",
                         "N": L.n, "n_dp": n_dp, "shard": L.shard, "owner": o,
                         "bucket": L.bucket, "outliers": "1% x100"}
        self.L, self.src_base = L, lo
        self.ranges = bucket_ranges(L, lo, hi)
        self.elems = hi - lo
        self.bytes_per_elem = 26 + 2 * n_dp + (2 * n_dp if self.clip else 0)
        self.dominant = "rs_adamw_clip" if self.clip else "rs_adamw"
        if self.clip:
            from zero_sharded_mixed_gb300.step import NormBuffers
            self.norm = NormBuffers(device)
            self.kernel_label = "zgb::norm_partial_kernel<true,8> + zgb::rs_adamw_vec_kernel<0,8> (clip)"
        g = torch.empty((n_dp, src_len), dtype=torch.bfloat16, device=device)
        n_real = max(0, min(L.n, hi) - lo)
        for r in range(n_dp):
            inputs.grad_bf16_into(g[r], n_real, SEED, step=1, rank=r, outlier_p=outlier)
        self.grads = g
        self.grad_list = [g[r] for r in range(n_dp)]
        self.master = _master(n_real, self.elems, device)
        self.m = torch.zeros_like(self.master)
        self.v = torch.zeros_like(self.master)
        self.out = torch.zeros(L.padded_n, dtype=torch.bfloat16, device=device)
        self.device_bytes = g.numel() * 2 + 3 * self.elems * 4 + self.out.numel() * 2
        if self.qgrad:
            from zero_sharded_mixed_gb300.step import Int8Grads
            self.qg = Int8Grads(L, n_dp, QGRAD_BLOCK, device)
            self.desc["quant_block"] = QGRAD_BLOCK
            sb = n_dp * 4 / QGRAD_BLOCK            # scale bytes per element of all sources
            # every rank quantizes its gradient (2 B read + 1 B written + scales),
            # then the fused update reads 1 B per source plus its scale
            self.bytes_per_elem = n_dp * 3 + sb + 26 + n_dp + sb
            self.dominant = "rs_adamw_int8"
            self.kernel_label = "zgb::qgrad_vec_kernel<8,true> + zgb::quantize_group_kernel<8,4> x 8 ranks"
            self.device_bytes += self.qg.q.numel() + self.qg.scales.numel() * 4

    def ops(self, t):
        zb, hp = self.zb, self.hp(t)
        n_dp = self.L.n_dp
        out = []
        if self.qgrad:
            P = self.L.padded_n
            sb = n_dp * 4 / QGRAD_BLOCK

            def quant():
                self.qg.quantize(self.grad_list)          # every simulated rank at once
            out.append(Op("quantize_grad", int(n_dp * P * (3 + 4 / QGRAD_BLOCK)), quant, kernels=n_dp))
            qs, ss = self.qg.sources()
            for s, e in self.ranges:
                def fn(s=s, e=e):
                    zb.zero_reduce_scatter_adamw_int8(self.L, qs, ss, QGRAD_BLOCK, float(n_dp), 0,
                                                      n_dp, s, e, self.master, self.m, self.v,
                                                      self.out, zb.ZERO_OUT_FULL, hp)
                out.append(Op("rs_adamw_int8", int((e - s) * (26 + n_dp + sb)), fn,
                              kernels=_owners(self.L, s, e)))
            return out
        if self.clip:
            for j, (s, e) in enumerate(self.ranges):
                def fn(s=s, e=e, j=j):
                    zb.zero_grad_norm_sq(self.L, self.grad_list, zb.ZERO_BF16, self.src_base,
                                         float(n_dp), s, e, self.norm.workspace, self.norm.norm_sq,
                                         j > 0)
                out.append(Op("grad_norm", (e - s) * 2 * n_dp, fn, kernels=2))   # partial sums + finalize
            for s, e in self.ranges:
                def fn(s=s, e=e):
                    zb.zero_reduce_scatter_adamw_clip(
                        self.L, self.grad_list, zb.ZERO_BF16, self.src_base, float(n_dp),
                        self.rank_begin, self.rank_end, s, e, self.master, self.m, self.v, self.out,
                        zb.ZERO_OUT_FULL, hp, self.norm.norm_sq, 1.0)
                out.append(Op("rs_adamw_clip", (e - s) * (26 + 2 * n_dp), fn))
            return out
        for s, e in self.ranges:
            def fn(s=s, e=e):
                zb.zero_reduce_scatter_adamw(self.L, self.grad_list, zb.ZERO_BF16, self.src_base,
                                             float(n_dp), self.rank_begin, self.rank_end,
                                             s, e, self.master, self.m, self.v, self.out,
                                             zb.ZERO_OUT_FULL, hp)
            out.append(Op("rs_adamw", (e - s) * self.bytes_per_elem, fn))
        return out


class AccumWorkload(Workload):
    """Gradient accumulation, GPT-2-XL shapes, n_dp = 4, K = 4 micro-batches.
    zero1: each rank adds its full bf16 micro-batch gradient into its own fp32
    buffer for the first K-1 micro-batches; the last one is fused with the
    update (sum over ranks of acc_r + g_r, divisor n_dp*K).
    zero2: the first K-1 micro-batches are reduce-scattered (summed) into the
    owners' fp32 shard buffer; the last is fused with the update (A + sum over
    ranks of g_r).  The same n_dp gradient buffers serve every micro-batch
    (each read is larger than L2, so the traffic is that of fresh data)."""

    n_src = 4

    def __init__(self, name, device, elems=0):
        import torch
        from zero_sharded_mixed_gb300 import inputs
        from zero_sharded_mixed_gb300.step import bucket_ranges
        super().__init__(device)
        zb = self.zb
        self.name = name
        n_dp, K = 4, 4
        self.K = K
        self.order = "zero1" if name == "accum-zero1" else "zero2"
        L = zb.zero_layout([elems] if elems else inputs.gpt2xl_numels(), n_dp, 8, 500_000_000)
        self.L = L
        P = L.padded_n
        self.ranges = bucket_ranges(L)
        self.elems = P
        g = torch.empty((n_dp, P), dtype=torch.bfloat16, device=device)
        for r in range(n_dp):
            inputs.grad_bf16_into(g[r], L.n, SEED, step=1, rank=r)
        self.grads = [g[r] for r in range(n_dp)]
        self._g = g
        self.master = _master(L.n, P, device)
        self.m = torch.zeros(P, device=device)
        self.v = torch.zeros(P, device=device)
        self.out = torch.zeros(P, dtype=torch.bfloat16, device=device)
        if self.order == "zero1":
            self.acc = [torch.empty(P, device=device) for _ in range(n_dp)]
            per = n_dp * (6 + (K - 2) * 10) + (6 * n_dp + 26)
            self.kernel_label = "zgb::acc_vec_kernel<1,true,true> + zgb::rs_adamw_vec_kernel<2,4> (fused finish)"
            self.dominant = "accumulate_local"
        else:
            self.A = torch.empty(P, device=device)
            per = (2 * n_dp + 4) + (K - 2) * (2 * n_dp + 8) + (4 + 2 * n_dp + 26)
            self.kernel_label = "zgb::acc_vec_kernel<4,true,false> + zgb::rs_adamw_vec_kernel<3,4> (fused finish)"
            self.dominant = "accumulate_reduce"
        self.bytes_per_elem = per
        self.desc = {"workload": ("flat%d" % elems if elems else "gpt2xl") + "_accumulation_%s" % self.order,
                     "model": "flat vector" if elems else "GPT-2-XL shapes",
                     "N": L.n, "n_dp": n_dp, "micro_batches": K, "bucket": L.bucket}
        self.device_bytes = (g.numel() * 2 + 3 * P * 4 + P * 2 +
                             (n_dp * P * 4 if self.order == "zero1" else P * 4))

    def ops(self, t):
        zb, hp, L, K = self.zb, self.hp(t), self.L, self.K
        n_dp = L.n_dp
        out = []
        if self.order == "zero1":
            for k in range(K - 1):
                for r in range(n_dp):
                    def fn(r=r, k=k):
                        zb.zero_accumulate(L, zb.ZERO_ACC_LOCAL, [self.grads[r]], zb.ZERO_BF16, 0,
                                           self.acc[r], 0, 0, L.padded_n, k == 0)
                    out.append(Op("accumulate_local", L.padded_n * (6 if k == 0 else 10), fn))
            for s, e in self.ranges:
                def fn(s=s, e=e):
                    zb.zero_accumulate_adamw(L, zb.ZERO_ACC_LOCAL, self.acc, 0, self.grads, 0,
                                             float(n_dp * K), 0, n_dp, s, e, self.master, self.m,
                                             self.v, self.out, zb.ZERO_OUT_FULL, hp)
                out.append(Op("accumulate_adamw", (e - s) * (6 * n_dp + 26), fn))
        else:
            for k in range(K - 1):
                for s, e in self.ranges:
                    def fn(s=s, e=e, k=k):
                        zb.zero_accumulate(L, zb.ZERO_ACC_REDUCE, self.grads, zb.ZERO_BF16, 0, self.A, 0,
                                           s, e, k == 0)
                    out.append(Op("accumulate_reduce", (e - s) * (2 * n_dp + (4 if k == 0 else 8)), fn))
            for s, e in self.ranges:
                def fn(s=s, e=e):
                    zb.zero_accumulate_adamw(L, zb.ZERO_ACC_REDUCE, [self.A], 0, self.grads, 0,
                                             float(n_dp * K), 0, n_dp, s, e, self.master, self.m,
                                             self.v, self.out, zb.ZERO_OUT_FULL, hp)
                out.append(Op("accumulate_adamw", (e - s) * (4 + 2 * n_dp + 26), fn))
        return out


class CastWorkload(Workload):
    """The cast of freshly initialised master weights to bf16 on its own
    (zero_cast_bf16), GPT-2-XL shapes: 4 bytes read and 2 written per element.
    The engines run it once at set-up and after a restore; it is timed here so
    that it, too, stands against the copy peak."""

    n_src = 0
    kernel_label = "zgb::cast_bf16_vec_kernel"

    def __init__(self, name, device, elems=0):
        import torch
        from zero_sharded_mixed_gb300 import inputs
        super().__init__(device)
        numels = [elems] if elems else inputs.gpt2xl_numels()
        n = sum(numels)
        self.name = name
        self.master = _master(n, n, device)
        self.out = torch.empty(n, dtype=torch.bfloat16, device=device)
        self.elems = n
        self.bytes_per_elem = 6
        self.dominant = "cast_bf16"
        self.desc = {"workload": ("flat%d" % elems if elems else "gpt2xl") + "_cast_master_bf16",
                     "model": "flat vector" if elems else "GPT-2-XL shapes", "N": n}
        self.device_bytes = n * 6

    def ops(self, t):
        def fn():
            self.zb.zero_cast_bf16(self.master, self.out)
        return [Op("cast_bf16", self.elems * 6, fn)]


class Zero3Workload(Workload):
    """ZeRO-3 per-unit path, Llama-7B units at n_dp = 8 (embedding, 32 blocks,
    head).  Per unit and step: gather the bf16 shards into a ring buffer for
    forward, release; gather again for backward; reduce-scatter the unit
    gradient (8 bf16 buffers -> fp32 owned shards); release; update the owned
    shards, bf16 into each rank's own shard.  One set of 8 unit-gradient
    buffers (sized for the largest unit) serves every unit."""

    def __init__(self, name, device, elems=0):
        import torch
        from zero_sharded_mixed_gb300 import inputs
        from zero_sharded_mixed_gb300 import step as zstep
        super().__init__(device)
        zb = self.zb
        self.name = name
        self.zstep = zstep
        self.zeropp = name in ("zero3-zeropp", "zero3-zeropp-fused")
        self.graph = name == "zero3-fused-graph"
        self.fused = name in ("zero3-fused", "zero3-int8-fused", "zero3-zeropp-fused", "zero3-fused-graph")
        self.int8 = name in ("zero3-int8", "zero3-zeropp", "zero3-int8-fused", "zero3-zeropp-fused")
        self.prefetch = name in ("zero3-prefetch", "zero3-prefetch-compute")
        # a stand-in for each layer's own work, to show what the prefetch hides
        self.with_compute = name in ("zero3-compute", "zero3-prefetch-compute")
        n_dp = 8
        self.units = []
        total = 0
        # the update that writes 8-bit shards itself needs 256-element slices
        align = 256 if name in ("zero3-int8-fused", "zero3-zeropp-fused") else 8
        for i, numels in enumerate([[elems]] if elems else inputs.llama7b_units()):
            L = zb.zero_layout(numels, n_dp, align=align)
            P = L.padded_n
            w = _master(L.n, P, device)
            shards = torch.empty(P, dtype=torch.bfloat16, device=device)
            zb.zero_cast_bf16(w, shards)
            self.units.append(zstep.Zero3Unit(L, shards.view(n_dp, L.shard), w,
                                              torch.zeros(P, device=device), torch.zeros(P, device=device)))
            total += P
        cap = max(u.layout.padded_n for u in self.units)
        self.ring = zstep.GatherRing(cap, device=str(device))
        g = torch.empty((n_dp, cap), dtype=torch.bfloat16, device=device)
        for r in range(n_dp):
            inputs.grad_bf16_into(g[r], cap, SEED, step=1, rank=r)
        self._g = g
        self.A = torch.empty(cap, device=device)
        self.elems = total
        if self.int8:
            self.qs = [zstep.Int8Shards(u.layout, 256, device) for u in self.units]
            for u, q in zip(self.units, self.qs):
                zstep.zero3_quantize(u, q)
            # two 8-bit gathers (1 B read + 2 B written), RS, update, re-quantize (2 B read + 1 B written)
            self.bytes_per_elem = 3 + 3 + (2 * n_dp + 4) + 30 + 3
            self.kernel_label = ("zgb::dequant_gather_vec_kernel, quantize_group_kernel<8,4>, "
                                 "acc_vec_kernel<8,1,0>, rs_adamw_vec_kernel<1,1>")
        else:
            self.bytes_per_elem = 4 + 4 + (2 * n_dp + 4) + 30
            self.kernel_label = "zgb::gather_vec_kernel, acc_vec_kernel<8,1,0>, rs_adamw_vec_kernel<1,1>"
        self.dominant = "rs_adamw"
        if self.fused and not self.int8:
            # two gathers, then the reduce-scatter and the update in one pass (42 B)
            self.bytes_per_elem = 4 + 4 + 26 + 2 * n_dp
            self.dominant = "rs_adamw_fused"
            self.kernel_label = "zgb::gather_vec_kernel, rs_adamw_vec_kernel<0,8> (own-shard output)"
        if self.fused and self.int8 and not self.zeropp:
            # two 8-bit gathers, then reduce-scatter + update + quantization in one pass
            self.bytes_per_elem = 3 + 3 + 2 * n_dp + 24 + 1 + 3 * 4 / 256
            self.dominant = "rs_adamw_fused_q8"
            self.kernel_label = "zgb::dequant_gather_vec_kernel, rs_adamw_vec_kernel<0,8,q8>"
        if self.zeropp:
            self.qg = zstep.Int8Grads(zb.zero_layout([cap], n_dp, align=align), n_dp, QGRAD_BLOCK, device)
            self.side = zstep.side_streams(n_dp, device)
            sb = n_dp * 4 / QGRAD_BLOCK
            # + every rank quantizes its unit gradient; the RS reads 1 B per source (+ scales)
            self.bytes_per_elem = 3 + 3 + (n_dp * 3 + sb) + (n_dp + sb + 4) + 30 + 3
            self.kernel_label = ("zgb::dequant_gather_vec_kernel, quantize_group_kernel<8,4>, "
                                 "qgrad_vec_kernel<8,false>, rs_adamw_vec_kernel<1,1>")
            if self.fused:
                # two 8-bit gathers, every rank quantizes its gradient, then one pass:
                # 8-bit gradients in, AdamW, 8-bit shards out
                self.bytes_per_elem = 3 + 3 + (n_dp * 3 + sb) + (n_dp + sb) + 24 + 1 + 4 / 256
                self.dominant = "rs_adamw_int8_q8"
                self.kernel_label = ("zgb::dequant_gather_vec_kernel, quantize_group_kernel<8,4>, "
                                     "qgrad_vec_kernel<8,true,q8>")
        if self.graph:
            # the fused step captured once in a CUDA graph: the schedule's advance
            # kernel, then every unit's two gathers and its fused reduce-scatter +
            # update, replayed as one launch per step (lr and the bias corrections
            # read from device memory)
            self.sched = zstep.StepSchedule(n_steps=1 << 16, **HP)
            unit_ops = self._step_ops(self.sched.hp())

            def step_fn():
                self.sched.advance()
                for op in unit_ops:
                    op.fn()
            self.gs = zstep.GraphStep(step_fn)
            self.graph_kernels = 1 + sum(op.kernels for op in unit_ops)
            self.dominant = "zero3_graph_step"
            self.kernel_label = ("one CUDA graph: zgb::schedule_advance_kernel, gather_vec_kernel, "
                                 "rs_adamw_vec_kernel<0,8> (own-shard output)")
        if self.with_compute:
            # forward: X[T, 4096] @ W once; backward: twice (data and weight gradients),
            # with W the gathered unit's first 4096 x cols elements (cols = P / 4096
            # rounded down to a multiple of 64, so the rows stay 128-byte aligned)
            self.X = torch.randn(COMPUTE_TOKENS, 4096, device=device).to(torch.bfloat16)
            self.Y = torch.empty(COMPUTE_TOKENS * (cap // 4096), device=device, dtype=torch.bfloat16)

            def compute(i, buf, phase):
                cols = self.units[i].layout.padded_n // 4096 // 64 * 64
                W = buf[:4096 * cols].view(4096, cols)
                Y = self.Y[:COMPUTE_TOKENS * cols].view(COMPUTE_TOKENS, cols)
                for _ in range(1 if phase == "fwd" else 2):
                    torch.mm(self.X, W, out=Y)
            self.compute_fn = compute
            self.compute_flops = sum(3 * 2 * COMPUTE_TOKENS * 4096 * (u.layout.padded_n // 4096 // 64 * 64)
                                     for u in self.units)
        if self.prefetch:
            self.dominant = "zero3_step_prefetched"
            self.kernel_label = "gathers on a side stream one unit ahead of RS + update"
            self.pf = zstep.Zero3Prefetcher(self.units, self.ring, device=device)
        if self.with_compute:
            # the step's HBM bytes over the whole step, matmuls included: not a kernel roofline
            self.bound = "mixed"
            self.dominant = "zero3_step"
            self.kernel_label = ("gather, stand-in layer matmuls (cuBLAS), layer RS, update"
                                 + (", gathers one unit ahead on a side stream" if self.prefetch else ""))
        self.desc = {"workload": "llama7b_zero3_units" + ("_int8_gather" if self.int8 else "")
                     + ("_int8_grads" if self.zeropp else "")
                     + ("_fused_rs_update" if self.fused else "")
                     + ("_align256" if align == 256 else "")
                     + ("_prefetch" if self.prefetch else "")
                     + ("_with_layer_compute" if self.with_compute else "")
                     + ("_cuda_graph" if self.graph else ""),
                     "model": "Llama-7B shapes",
                     "units": len(self.units), "N": sum(u.layout.n for u in self.units), "n_dp": n_dp,
                     "ring_slots": 2}
        if self.int8:
            self.desc["quant_block"] = 256
        if self.with_compute:
            self.desc["layer_compute"] = ("stand-in: bf16 X[%d, 4096] @ unit[4096, cols], once forward, "
                                          "twice backward (cuBLAS), %.3g FLOP per step"
                                          % (COMPUTE_TOKENS, self.compute_flops))
        self.device_bytes = total * (12 + 2) + 2 * cap * 2 + g.numel() * 2 + cap * 4
        if self.zeropp:
            self.device_bytes += self.qg.q.numel() + self.qg.scales.numel() * 4

    def ops(self, t):
        if self.graph:
            return [Op("zero3_graph_step", self.elems * self.bytes_per_elem, self.gs.replay,
                       kernels=self.graph_kernels)]
        return self._step_ops(self.hp(t))

    def _step_ops(self, hp):
        zb, zs = self.zb, self.zstep
        out = []
        grads_of = lambda i: [self._g[r, :self.units[i].layout.padded_n] for r in range(self.units[i].layout.n_dp)]
        if self.prefetch:
            def step_all():
                zs.zero3_step_prefetched(self.pf, grads_of, self.A, hp,
                                         compute=self.compute_fn if self.with_compute else None)
            out.append(Op("zero3_step" if self.with_compute else "zero3_step_prefetched",
                          self.elems * self.bytes_per_elem, step_all, kernels=4 * len(self.units)))
            return out
        if self.with_compute:
            def step_seq():
                for i, u in enumerate(self.units):
                    self.compute_fn(i, zs.zero3_gather(u, self.ring, ("fwd", i)), "fwd")
                    self.ring.release(("fwd", i))
                for i in reversed(range(len(self.units))):
                    u = self.units[i]
                    P = u.layout.padded_n
                    self.compute_fn(i, zs.zero3_gather(u, self.ring, ("bwd", i)), "bwd")
                    zs.zero3_layer_reduce_scatter(u, grads_of(i), self.A[:P])
                    self.ring.release(("bwd", i))
                    zs.zero3_update(u, self.A[:P], hp)
            out.append(Op("zero3_step", self.elems * self.bytes_per_elem, step_seq, kernels=4 * len(self.units)))
            return out
        for i, u in enumerate(self.units):
            P = u.layout.padded_n
            grads = [self._g[r, :P] for r in range(u.layout.n_dp)]
            q = self.qs[i] if self.int8 else None

            def fwd(u=u, i=i, q=q):
                if q is not None:
                    zs.zero3_gather_int8(u, q, self.ring, ("fwd", i))
                else:
                    zs.zero3_gather(u, self.ring, ("fwd", i))
                self.ring.release(("fwd", i))

            def bwd_gather(u=u, i=i, q=q):
                if q is not None:
                    zs.zero3_gather_int8(u, q, self.ring, ("bwd", i))
                else:
                    zs.zero3_gather(u, self.ring, ("bwd", i))

            def rs(u=u, i=i, P=P, grads=grads):
                zs.zero3_layer_reduce_scatter(u, grads, self.A[:P])
                self.ring.release(("bwd", i))

            def quant_grads(u=u, P=P, grads=grads):
                # every simulated rank at once, on side streams joined back (step.quantize_ranks)
                zs.quantize_ranks(u.layout, grads, [self.qg.q[r, :P] for r in range(u.layout.n_dp)],
                                  [self.qg.scales[r] for r in range(u.layout.n_dp)], QGRAD_BLOCK, self.side)

            def rs_int8(u=u, i=i, P=P):
                zb.zero_accumulate_int8(u.layout, [self.qg.q[r, :P] for r in range(u.layout.n_dp)],
                                        [self.qg.scales[r] for r in range(u.layout.n_dp)],
                                        QGRAD_BLOCK, self.A[:P], 0, 0, P, True)
                self.ring.release(("bwd", i))

            def upd(u=u, P=P):
                zs.zero3_update(u, self.A[:P], hp)

            gkind, gbytes = ("gather_int8", P * 3 + q.nb * u.layout.n_dp * 4) if q is not None \
                else ("gather", P * 4)
            out.append(Op(gkind, gbytes, fwd))
            out.append(Op(gkind, gbytes, bwd_gather))
            if self.fused and self.zeropp:
                n = u.layout.n_dp
                sbytes = n * (-(-u.layout.shard // QGRAD_BLOCK)) * 4

                def rs_upd_int8_q8(u=u, i=i, P=P, q=q, n=n):
                    zb.zero_reduce_scatter_adamw_int8_q8(
                        u.layout, [self.qg.q[r, :P] for r in range(n)], [self.qg.scales[r] for r in range(n)],
                        QGRAD_BLOCK, float(n), 0, n, 0, P, u.master, u.m, u.v, q.q.view(-1),
                        q.scales.view(-1), 256, hp)
                    self.ring.release(("bwd", i))
                out.append(Op("quantize_grad", n * (P * 3 + sbytes), quant_grads, kernels=n))
                # a call over the unit's whole shards is one launch (blockIdx.y = owner)
                out.append(Op("rs_adamw_int8_q8", P * (n + 25) + n * sbytes + (P // 256) * 4, rs_upd_int8_q8))
                continue
            if self.fused and q is not None:
                def rs_upd_q8(u=u, i=i, grads=grads, q=q):
                    zs.zero3_reduce_scatter_update_q8(u, grads, q, hp)
                    self.ring.release(("bwd", i))
                out.append(Op("rs_adamw_fused_q8", P * (2 * u.layout.n_dp + 25) + (P // 256) * 4, rs_upd_q8))
                continue
            if self.fused:
                def rs_upd(u=u, i=i, grads=grads):
                    zs.zero3_reduce_scatter_update(u, grads, hp)
                    self.ring.release(("bwd", i))
                out.append(Op("rs_adamw_fused", P * (26 + 2 * u.layout.n_dp), rs_upd))
                continue
            if self.zeropp:
                n = u.layout.n_dp
                sbytes = n * (-(-u.layout.shard // QGRAD_BLOCK)) * 4
                out.append(Op("quantize_grad", n * (P * 3 + sbytes), quant_grads, kernels=n))
                out.append(Op("accumulate_int8", P * (n + 4) + n * sbytes, rs_int8))   # one launch per unit
            else:
                out.append(Op("accumulate_reduce", P * (2 * u.layout.n_dp + 4), rs))
            out.append(Op("rs_adamw", P * 30, upd))
            if q is not None:
                def quant(u=u, q=q):
                    zs.zero3_quantize(u, q)
                out.append(Op("quantize_int8", P * 3 + q.nb * u.layout.n_dp * 4, quant))
        return out


def make_workload(name, device, elems=0, bucket=500_000_000):
    if name in ("gpt2xl", "gpt2xl-clip", "gpt2xl-qgrad"):
        return Zero2Workload(name, device, elems, bucket)
    if name in ("llama7b-shard", "probe"):
        return Zero2Workload(name, device)
    if name in ("accum-zero1", "accum-zero2"):
        return AccumWorkload(name, device, elems)
    if name == "cast":
        return CastWorkload(name, device, elems)
    if name in ("zero3", "zero3-int8", "zero3-prefetch", "zero3-zeropp", "zero3-fused",
                "zero3-int8-fused", "zero3-zeropp-fused", "zero3-fused-graph", "zero3-compute",
                "zero3-prefetch-compute"):
        return Zero3Workload(name, device, elems)
    raise ValueError(name)


def time_workload(wl, steps, warmup, dist, device, sampler=None):
    """W untimed steps, then K timed steps with a CUDA event pair around every
    launch (on the launching stream) and one pair around the whole region."""
    import torch
    t = 1
    for _ in range(warmup):
        for op in wl.ops(t):
            op.fn()
        t += 1
    plan = [wl.ops(t + k) for k in range(steps)]
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in ops] for ops in plan]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.15)
    start.record()
    for ops, evs in zip(plan, ev):
        for op, (a, b) in zip(ops, evs):
            a.record()
            op.fn()
            b.record()
    end.record()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    per_kind = {}
    step_ms = []
    for ops, evs in zip(plan, ev):
        step_ms.append(evs[0][0].elapsed_time(evs[-1][1]))     # first launch's start to last's end
        for op, (a, b) in zip(ops, evs):
            d = per_kind.setdefault(op.kind, {"ms": 0.0, "bytes": 0, "launches": 0, "kernels": 0})
            d["ms"] += a.elapsed_time(b)
            d["bytes"] += op.bytes
            d["launches"] += 1
            d["kernels"] += op.kernels
    per_kind["_steps"] = step_ms
    return start.elapsed_time(end), per_kind, clocks, t + steps


def e2e_host_bytes(wl, shared_rows=False):
    """Pinned host bytes the e2e leg holds: every rank's gradients (or one row
    that every simulated rank's copy reads) and the result."""
    rows = 1 if shared_rows else wl.grads.shape[0]
    return rows * wl.grads.shape[1] * wl.grads.element_size() + wl.out.numel() * wl.out.element_size()


def host_fits(nbytes) -> bool:
    """Whether nbytes fit in 85 % of the host memory available now."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return nbytes <= 0.85 * int(line.split()[1]) * 1024
    except OSError:
        pass
    return True


def all_ranks_agree(dist, flag: bool, device) -> bool:
    """True when the flag is true on every rank."""
    if dist is None:
        return flag
    import torch
    t = torch.tensor([1 if flag else 0], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return bool(t.item())


def time_e2e(wl, steps, warmup, t0, dist, shared_rows=False):
    """The same step through the public API with host buffers: every step copies
    the n_dp gradient buffers from pinned host memory to the device and reads the
    updated bf16 weights back into pinned host memory (step.HostPipeline, which
    overlaps bucket b's copies with bucket b-1's update, and the result copies
    with the gradient copies).  shared_rows: when the host cannot pin every
    rank's gradients (several GPUs per host), each simulated rank's copy reads
    one shared pinned row (rank 0's gradient) -- the same bytes move each step."""
    import torch
    from zero_sharded_mixed_gb300.step import HostPipeline
    if shared_rows:
        row = torch.empty(wl.grads.shape[1], dtype=wl.grads.dtype, pin_memory=True)
        row.copy_(wl.grads[0])
        host_g = row.expand(wl.grads.shape)         # every rank's row is the same host memory
    else:
        host_g = torch.empty(wl.grads.shape, dtype=wl.grads.dtype, pin_memory=True)
        host_g.copy_(wl.grads)
    host_out = torch.empty(wl.out.shape, dtype=wl.out.dtype, pin_memory=True)
    # the pipeline's two modes: result copies overlapped with the gradient copies,
    # or deferred until every gradient copy has landed.  `warmup` timed steps of
    # each; the timed steps run the one whose warm-up steps took less (the max
    # over ranks, so that every rank picks the same).  On most boxes overlapping
    # is faster (125 against 134 ms); on some, steps of the overlapped pipeline
    # alternated between 128 and 370 ms.
    pipes = {"overlap": HostPipeline(wl.L, device=wl.device),
             "deferred": HostPipeline(wl.L, device=wl.device, defer_out=True)}
    t = t0
    warm = {}
    for name, pipe in pipes.items():
        warm[name] = []
        for _ in range(max(1, warmup)):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            pipe.step(host_g, wl.grads, wl.master, wl.m, wl.v, wl.out, host_out, wl.hp(t))
            b.record()
            torch.cuda.synchronize()
            warm[name].append(a.elapsed_time(b))
            t += 1
    cost = {name: max_over_ranks(dist, sum(v), wl.device) for name, v in warm.items()}
    mode = min(cost, key=cost.get)
    pipe = pipes[mode]
    print("e2e warm-up (ms): " + "; ".join("%s %s" % (k, " ".join("%.1f" % x for x in v))
                                          for k, v in warm.items()) + "; timed: " + mode,
          file=sys.stderr, flush=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    barrier(dist)
    marks[0].record()
    for k in range(steps):
        pipe.step(host_g, wl.grads, wl.master, wl.m, wl.v, wl.out, host_out, wl.hp(t))
        marks[k + 1].record()
        t += 1
    torch.cuda.synchronize()
    barrier(dist)
    ms = marks[0].elapsed_time(marks[-1]) / steps
    steps_ms = [marks[k].elapsed_time(marks[k + 1]) for k in range(steps)]
    print("e2e steps (ms): " + " ".join("%.1f" % x for x in steps_ms), file=sys.stderr, flush=True)
    per_step = sorted(steps_ms)
    # the host link on this machine: plain copies of the step's gradients, pinned host to device;
    # the fastest of three (the link's rate varies from moment to moment on a shared host)
    link_gbs = 0.0
    for _ in range(3):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for r in range(host_g.shape[0]):
            wl.grads[r].copy_(host_g[r], non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        link_gbs = max(link_gbs, host_g.numel() * 2 / (a.elapsed_time(b) / 1e3) / 1e9)
    return ms, host_g.numel() * 2, host_out.numel() * 2, link_gbs, per_step, mode


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


def host_cores() -> int:
    """The host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(sample, seconds, n_dp, threads=1):
    """The oracle, as it stands, stepping over the sample for about `seconds`:
    with threads > 1 the sample is cut into that many contiguous chunks, each
    stepped by its own thread (the oracle's C routines release the interpreter
    lock).  Returns (elements per second, seconds, elements updated)."""
    import numpy as np
    import oracle
    oracle.build()                       # compiled before the timed region, if stale
    g, w, m, v = sample
    hp = oracle.AdamW(**HP)
    n = g.shape[1]
    bounds = [n * k // threads for k in range(threads + 1)]
    done = [0] * threads
    t0 = time.perf_counter()

    def run(k):
        a, b = bounds[k], bounds[k + 1]
        gc, wc, mc, vc = np.ascontiguousarray(g[:, a:b]), w[a:b].copy(), m[a:b].copy(), v[a:b].copy()
        t = 1
        while True:
            _, wc, mc, vc = oracle.rs_adamw_reference(gc, n_dp, wc, mc, vc, hp, t)
            t += 1
            done[k] += b - a
            if time.perf_counter() - t0 >= seconds:
                return

    if threads == 1:
        run(0)
    else:
        ts = [threading.Thread(target=run, args=(k,)) for k in range(threads)]
        for th in ts:
            th.start()
        for th in ts:
            th.join()
    el = time.perf_counter() - t0
    return sum(done) / el, el, sum(done)


COMPUTE_TOKENS = 1024         # tokens of the stand-in layer compute of the ZeRO-3 overlap workloads
WORKLOAD_SAMPLE = 1 << 19     # elements of each extra workload's oracle sample
WORKLOAD_ORACLE_SECONDS = 0.2  # each extra workload's oracle timing on every core (half that on one)


def oracle_workload_step(name, n):
    """The oracle's statement of one step of workload `name` over a seeded host
    sample of n owned elements with the workload's rank count and structure
    (gathers, quantization, accumulation, clipping, update): returns (step(t),
    elements updated per step, a description).  Runs on the host only."""
    import numpy as np
    import oracle
    from zero_sharded_mixed_gb300 import inputs
    if name == "cast":
        w = inputs.master_weights(n, n, seed=SEED).numpy()

        def cast_step(t):
            oracle.cast_bf16(w)
        return cast_step, n, "%d owned elements, the bf16 cast of master weights" % n
    hp = oracle.AdamW(**HP)
    n_dp = 4 if name.startswith("accum") else 8
    n -= n % (n_dp * 256)
    K = 4 if name.startswith("accum") else 1
    st = {"w": inputs.master_weights(n, n, seed=SEED).numpy(), "m": np.zeros(n, np.float32),
          "v": np.zeros(n, np.float32)}
    outlier = 0.01 if name == "llama7b-shard" else 0.0
    grads = [inputs.bf16_bits(inputs.grads_bf16(n_dp, n, n, seed=SEED, step=1, micro=k, outlier_p=outlier))
             for k in range(K)]
    g = grads[0]
    st["shards"] = oracle.cast_bf16(st["w"]).reshape(n_dp, -1)
    int8w = name in ("zero3-int8", "zero3-int8-fused", "zero3-zeropp", "zero3-zeropp-fused")
    int8g = name in ("gpt2xl-qgrad", "zero3-zeropp", "zero3-zeropp-fused")
    zero3 = name.startswith("zero3")
    if int8w:
        st["q"] = [oracle.quantize_int8(st["shards"][o], 256) for o in range(n_dp)]

    def step(t):
        if zero3:                            # gather before forward and before backward
            for _ in range(2):
                if int8w:
                    oracle.all_gather(np.stack([oracle.dequantize_int8(q, sc, 256) for q, sc in st["q"]]))
                else:
                    oracle.all_gather(st["shards"])
        clip = None
        if int8g:
            q, sc = oracle.quantize_grad_int8(g, n_dp, 256)
            src = oracle.accumulate_reduce_int8(None, q, sc, n_dp, 256, True)[None, :]
        elif name == "accum-zero1":
            acc = [None] * n_dp
            for k in range(K):
                acc = [oracle.accumulate_local(acc[r], grads[k][r], k == 0) for r in range(n_dp)]
            src = np.stack(acc)
        elif name == "accum-zero2" or (zero3 and "fused" not in name):
            A = None
            for k in range(K):
                A = oracle.accumulate_reduce(A, grads[k], k == 0)
            src = A[None, :]
        else:
            src = g
        if name == "gpt2xl-clip":
            clip = (oracle.grad_norm_sq(src, n_dp * K), 1.0)
        out, st["w"], st["m"], st["v"] = oracle.rs_adamw_reference(src, n_dp * K, st["w"], st["m"],
                                                                   st["v"], hp, t, clip=clip)
        st["shards"] = out.reshape(n_dp, -1)
        if int8w:
            st["q"] = [oracle.quantize_int8(st["shards"][o], 256) for o in range(n_dp)]

    what = ("%d owned elements, %d gradient slices%s%s%s%s" %
            (n, n_dp, ", %d micro-batches" % K if K > 1 else "", ", two gathers" if zero3 else "",
             ", 8-bit weights" if int8w else "", ", 8-bit gradients" if int8g else ""))
    return step, n, what


def time_oracle_workload(name, seconds, threads=1):
    """The oracle's statement of workload `name` on every host core: each
    thread steps its own copy of the step over 1/threads of the sample, after
    one untimed step."""
    import oracle
    oracle.build()                       # compiled before the timed region, if stale
    per = max(WORKLOAD_SAMPLE // threads, 8 * 256)
    steps = [oracle_workload_step(name, per) for _ in range(threads)]
    for step, _, _ in steps:
        step(1)                          # one untimed step each (first-touch allocations)
    done = [0] * threads
    t0 = time.perf_counter()

    def run(k):
        step, n, _ = steps[k]
        t = 2
        while time.perf_counter() - t0 < seconds:
            step(t)
            t += 1
            done[k] += n

    ts = [threading.Thread(target=run, args=(k,)) for k in range(threads)]
    for th in ts:
        th.start()
    for th in ts:
        th.join()
    el = time.perf_counter() - t0
    what = steps[0][2]
    return {"value": sum(done) / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "%d threads, each its own copy of the step over %s; %.1f s" % (threads, what, el)}


def time_checkpoint(device):
    """Save and restore one Llama-7B block unit's sharded state (n_dp = 8: fp32
    master, m, v and the bf16 shards, one file per rank with its CRC-32) in a
    temporary directory, through checkpoint.save / restore; the restored state
    must equal the saved one bit for bit.  Host-bound: device-to-host copies,
    the CRC and the file system."""
    import shutil
    import tempfile

    import torch
    from zero_sharded_mixed_gb300 import binding as zb
    from zero_sharded_mixed_gb300 import checkpoint as ck
    from zero_sharded_mixed_gb300 import inputs
    numels = inputs.llama7b_block_numels()
    L = zb.zero_layout(numels, 8)
    P = L.padded_n
    st = [_master(L.n, P, device), torch.randn(P, device=device) * 1e-4, torch.rand(P, device=device) * 1e-8]
    shards = torch.empty(P, dtype=torch.bfloat16, device=device)
    zb.zero_cast_bf16(st[0], shards)
    hp = zb.ZeroAdamW.make(step=7, **HP)
    nbytes = P * 14
    d = tempfile.mkdtemp(prefix="zgb_ckpt_")
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ck.save(d, L, numels, *st, 7, hp, out_bf16=shards)
        t_save = time.perf_counter() - t0
        back = [torch.empty_like(x) for x in st]
        back_w = torch.empty_like(shards)
        t0 = time.perf_counter()
        step = ck.restore(d, L, *back, out_bf16=back_w)
        torch.cuda.synchronize()
        t_restore = time.perf_counter() - t0
        same = step == 7 and all(torch.equal(a.view(torch.int32), b.view(torch.int32)) for a, b in zip(st, back)) \
            and torch.equal(shards.view(torch.int16), back_w.view(torch.int16))
        host = torch.zeros(L.shard * 12, dtype=torch.uint8)          # one rank's fp32 payload
        t0 = time.perf_counter()
        ck.crc32(host.numpy())
        crc_gbs = host.numel() / (time.perf_counter() - t0) / 1e9
    except OSError as e:
        return {"unavailable": "checkpoint directory: %s" % e}
    finally:
        shutil.rmtree(d, ignore_errors=True)
    return {"workload": "llama7b_block_unit_checkpoint", "params": L.n, "n_dp": 8, "files": 8,
            "bytes": nbytes, "save_s": t_save, "restore_s": t_restore,
            "save_gbs": nbytes / t_save / 1e9, "restore_gbs": nbytes / t_restore / 1e9,
            "crc_gbs_one_core": crc_gbs, "round_trip_bit_exact": bool(same),
            "threads": ck._workers(8),
            "bound": "host: the CRC-32 (crc_gbs_one_core per thread), page-cache copies, "
                     "device-host copies"}


# --------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------

def _kernels_summary(per_kind, steps):
    out = {}
    for kind, d in per_kind.items():
        out[kind] = {"launches_per_step": d["kernels"] // steps,
                     "ms_per_step": d["ms"] / steps,
                     "bytes_per_step": d["bytes"] // steps,
                     "achieved_gbs": d["bytes"] / (d["ms"] / 1e3) / 1e9 if d["ms"] > 0 else None}
    return out


EXTRA_WORKLOADS = ("gpt2xl", "llama7b-shard", "gpt2xl-clip", "gpt2xl-qgrad", "accum-zero1", "accum-zero2",
                   "zero3", "zero3-fused", "zero3-fused-graph", "zero3-prefetch", "zero3-int8",
                   "zero3-int8-fused", "zero3-zeropp", "zero3-zeropp-fused", "cast")
COMPUTE_WORKLOADS = ("zero3-compute", "zero3-prefetch-compute")


def workload_order(args):
    """The primary workload, then (unless --no-extra or --elems) every other
    workload; the two with stand-in layer matmuls only under --with-compute."""
    primary = args.workload
    if args.elems or args.no_extra or primary == "probe":
        return [primary]
    extras = EXTRA_WORKLOADS + (COMPUTE_WORKLOADS if args.with_compute else ())
    return [primary] + [w for w in extras if w != primary]


def workload_line(name, res):
    """One JSON line for a workload other than the headline one.  It carries
    no "metric" or "value" key, so that the headline line printed last is the
    only line with the contract's keys."""
    line = {"impl": "ours", "workload_result": name, "params_per_s": res["value"]}
    for k in ("ms_per_step", "steps", "step_ms_median", "hbm_gbs_step", "bytes_per_param_step", "config",
              "roofline", "kernels", "gpu_launches", "cpu_baseline", "overlap"):
        if k in res:
            line[k] = res[k]
    return _rounded(line)


def _rounded(x, digits=6):
    """Floats to `digits` significant digits, recursively (the printed lines
    stay short; no figure here is known to more digits than that)."""
    if isinstance(x, float):
        return float("%.*g" % (digits, x))
    if isinstance(x, dict):
        return {k: _rounded(v, digits) for k, v in x.items()}
    if isinstance(x, list):
        return [_rounded(v, digits) for v in x]
    return x


def _compact_roofline(r):
    return {k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac", "peak_kind", "traffic",
                              "algorithmic_bytes_per_launch", "kernel") if k in r}


def target_7b(res):
    """The fused update on one owned shard of the Llama-7B shapes: its step
    time, rate and fraction of the measured copy peak (and of the nominal HBM
    bandwidth), against the 80 % asked of it."""
    if res is None:
        return None
    r = res["roofline"]
    return {"workload": res["config"]["workload"], "ms_per_step": res["ms_per_step"],
            "params_per_s": res["value"], "hbm_gbs_step": res["hbm_gbs_step"],
            "frac": r["frac"], "frac_step": res["hbm_gbs_step"] / r["peak"],
            "frac_nominal": r["achieved"] / NOMINAL_HBM_GBS, "target_frac": TARGET_FRAC_7B,
            "met": min(r["frac"], r["achieved"] / NOMINAL_HBM_GBS) >= TARGET_FRAC_7B}


def headline_line(p, args, world, seven_b=None):
    """The headline JSON line: the contract's keys for the primary workload,
    compact (the other workloads have lines of their own)."""
    cfg = dict(p["config"], parallelism="replicas x%d, n_dp=%d simulated per GPU"
               % (world, p["config"].get("n_dp", 8)))
    e2e = p.get("e2e")
    if e2e is not None:
        e2e = {k: e2e[k] for k in ("value", "unit", "ms_per_step", "steps", "step_ms_min", "step_ms_median",
                                   "h2d_bytes_per_step", "d2h_bytes_per_step", "host_rows", "mode", "unavailable")
               if k in e2e}
        if "link" in p["e2e"]:
            e2e["link_h2d_gbs"] = p["e2e"]["link"]["h2d_gbs"]
            e2e["link_frac"] = p["e2e"]["link"]["frac"]
    line = {
        "metric": METRIC, "value": p["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": p["ms_per_step"],
        "step_ms_median": p["step_ms_median"], "step_ms_min": p["step_ms_min"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded normal draws, model shapes)",
        "config": cfg,
        "hbm_gbs_step": p["hbm_gbs_step"],
        "bytes_per_param_step": p["bytes_per_param_step"],
        "roofline": _compact_roofline(p["roofline"]),
        "gpu_launches": p["gpu_launches"],
        "clocks": p.get("clocks"),
        "e2e": e2e,
        "cpu_baseline": p.get("cpu_baseline"),
        "target_7b": seven_b,
        "impl": "ours",
    }
    line = _rounded(line)
    # never let an optional field push the line past the limit
    for k in ("bytes_per_param_step", "step_ms_median"):
        if len(json.dumps(line)) <= HEADLINE_MAX_CHARS:
            break
        line.pop(k, None)
    if len(json.dumps(line)) > HEADLINE_MAX_CHARS and line.get("cpu_baseline"):
        line["cpu_baseline"] = {k: line["cpu_baseline"][k] for k in ("value", "unit", "cores", "kind")}
    return line


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, local)
    from zero_sharded_mixed_gb300 import binding as zb
    from zero_sharded_mixed_gb300 import build as zbuild
    # one builder per node (ranks share the tree); every rank learns whether it worked
    err = None
    if local == 0:
        try:
            zbuild.build()
        except Exception as e:        # reported on every rank below
            err = e
    if not all_ranks_agree(dist, err is None, device):
        raise RuntimeError("building libzero_gb300.so failed on a node's first rank") from err
    zb.load()

    peak, peak_kind = _peak()
    primary = args.workload
    results = {}
    for name in workload_order(args):
        wl = make_workload(name, device, args.elems if name == primary else 0, args.bucket)
        torch.cuda.synchronize()
        is_primary = name == primary
        # the other workloads: up to 20 timed steps after up to 3 warm-up steps
        steps = args.steps if is_primary else max(1, min(args.steps, 20))
        warm = args.warmup if is_primary else max(1, min(args.warmup, 3))
        sampler = ClockSampler(local) if is_primary else None
        total_ms, per_kind, clocks, t_next = time_workload(wl, steps, warm, dist, device, sampler)
        step_list = sorted(per_kind.pop("_steps"))
        ms_step = max_over_ranks(dist, total_ms / steps, device)
        kernels = _kernels_summary(per_kind, steps)
        dom = per_kind[wl.dominant]
        dom_ms = max_over_ranks(dist, dom["ms"] / dom["launches"], device)   # average launch
        dom_bytes = dom["bytes"] / dom["launches"]                           # per launch
        achieved = dom_bytes / (dom_ms / 1e3) / 1e9
        bytes_step = wl.elems * wl.bytes_per_elem
        tpe = _traffic_per_elem(wl.n_src) if wl.dominant == "rs_adamw" and \
            name in ("gpt2xl", "llama7b-shard", "probe") else None
        res = {
            "value": replica_value(wl.elems, world, ms_step), "ms_per_step": ms_step, "steps": steps,
            "step_ms_median": step_list[len(step_list) // 2], "step_ms_min": step_list[0],
            "hbm_gbs_step": bytes_step / (ms_step / 1e3) / 1e9,
            "bytes_per_param_step": wl.bytes_per_elem,
            "config": dict(wl.desc, l2="%.1f GB > L2, no flush" % (wl.device_bytes / 1e9)),
            "roofline": {"bound": getattr(wl, "bound", "hbm"), "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": (tpe * dom_bytes / wl.bytes_per_elem) if tpe is not None else None,
                         "algorithmic_bytes_per_launch": dom_bytes,
                         "kernel": wl.dominant, "kernel_symbols": wl.kernel_label},
            "kernels": kernels,
            "gpu_launches": sum(d["kernels"] for d in per_kind.values()),
        }
        if is_primary:
            res["clocks"] = clocks
            if not args.no_e2e and isinstance(wl, Zero2Workload):
                local = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
                need = e2e_host_bytes(wl)
                shared = not all_ranks_agree(dist, host_fits(need * local), device)
                fits = not shared or all_ranks_agree(dist, host_fits(e2e_host_bytes(wl, True) * local), device)
                if fits:
                    e2e_steps = max(1, min(args.steps, 10))
                    e_ms, h2d, d2h, link_gbs, per_step, mode = time_e2e(wl, e2e_steps, 2, t_next + 1, dist,
                                                                        shared)
                    e_ms = max_over_ranks(dist, e_ms, device)
                    link_ms = h2d / (link_gbs * 1e9) * 1e3
                    res["e2e"] = {"value": replica_value(wl.elems, world, e_ms), "unit": UNIT,
                                  "ms_per_step": e_ms, "steps": e2e_steps,
                                  "step_ms_min": per_step[0], "step_ms_median": per_step[len(per_step) // 2],
                                  "host_rows": "shared" if shared else "per rank", "mode": mode,
                                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                                  "link": {"h2d_gbs": link_gbs, "h2d_ms_per_step": link_ms,
                                           "frac": link_ms / e_ms}}
                else:
                    res["e2e"] = {"value": None, "unit": UNIT,
                                  "unavailable": "host memory: %d local ranks x %.1f GB of pinned "
                                  "step inputs and results exceed 85%% of the available host memory"
                                  % (local, e2e_host_bytes(wl, True) / 1e9)}
            if not args.no_cpu_baseline and world == 1 and rank == 0 and isinstance(wl, Zero2Workload):
                sample = cpu_sample(wl, CPU_SAMPLE)
                cores = host_cores()
                rate1, _, _ = time_oracle(sample, CPU_BASELINE_SECONDS / 4, wl.n_src, threads=1)
                rate, secs, done = time_oracle(sample, CPU_BASELINE_SECONDS, wl.n_src, threads=cores)
                res["cpu_baseline"] = {
                    "value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                    "single_core_value": rate1,
                    "sample": "first %d owned elements (all %d gradient slices), %d chunks, one thread "
                              "each; %.1f passes in %.1f s" % (sample[1].size, wl.n_src, cores,
                                                              done / sample[1].size, secs)}
        if not is_primary and not args.no_cpu_baseline and world == 1 and rank == 0:
            one = time_oracle_workload(name, WORKLOAD_ORACLE_SECONDS / 2, threads=1)
            every = time_oracle_workload(name, WORKLOAD_ORACLE_SECONDS, threads=host_cores())
            # the faster of one thread and every core (the 8-bit steps' oracle is interpreter-bound,
            # and its threads contend)
            res["cpu_baseline"] = dict(every if every["value"] >= one["value"] else one,
                                       single_core_value=one["value"])
        if name == "zero3-prefetch-compute" and "zero3-compute" in results:
            seq = results["zero3-compute"]["ms_per_step"]
            gathers = results["zero3"]["kernels"]["gather"]["ms_per_step"] if "zero3" in results else None
            res["overlap"] = {"sequential_ms": seq, "prefetched_ms": res["ms_per_step"],
                              "hidden_ms": seq - res["ms_per_step"], "gather_ms_alone": gathers}
        results[name] = res
        if not is_primary and rank == 0:
            print(json.dumps(workload_line(name, res)), flush=True)
        wl.free()
        del wl
        torch.cuda.empty_cache()

    if rank == 0 and not args.no_extra and not args.elems and primary != "probe":
        print(json.dumps({"impl": "ours", "workload_result": "checkpoint", "checkpoint": time_checkpoint(device)}),
              flush=True)

    if rank == 0:
        seven = results.get("llama7b-shard")
        print(json.dumps(headline_line(results[primary], args, world, target_7b(seven))), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle, as it stands, on a bounded sample of the same workload:
    each step updates REF_SAMPLE owned elements from all n_dp gradient slices,
    cut into one contiguous chunk per host core, each chunk stepped by its own
    thread (the oracle's C routines release the interpreter lock)."""
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
    oracle.build()
    cores = host_cores()
    bounds = [n * k // cores for k in range(cores + 1)]
    chunks = [[np.ascontiguousarray(gb[:, a:b]), w[a:b].copy(), m[a:b].copy(), v[a:b].copy()]
              for a, b in zip(bounds[:-1], bounds[1:])]

    def step_chunk(k, t):
        c = chunks[k]
        _, c[1], c[2], c[3] = oracle.rs_adamw_reference(c[0], n_dp, c[1], c[2], c[3], hp, t)

    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(cores) as ex:
        t = 1
        for _ in range(args.warmup):
            list(ex.map(step_chunk, range(cores), [t] * cores))
            t += 1
        t0 = time.perf_counter()
        for _ in range(args.steps):
            list(ex.map(step_chunk, range(cores), [t] * cores))
            t += 1
        el = time.perf_counter() - t0
    ms = el * 1e3 / max(1, args.steps)
    value = n / (ms / 1e3)
    wl_name = {"gpt2xl": "gpt2xl_zero2_all_shards", "llama7b-shard": "llama7b_zero2_one_shard",
               "probe": "probe_flat_2p26_ndp8"}.get(args.workload, args.workload)
    sample = ("%d owned elements per step (a bounded sample of %s), %d gradient slices, in %d "
              "contiguous chunks, one thread each" % (n, wl_name, n_dp, cores))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
        "config": {"workload": wl_name, "n_dp": n_dp, "sample_elements": n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
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
