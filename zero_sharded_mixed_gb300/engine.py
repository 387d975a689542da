"""A ZeRO optimizer driven by a configuration: the step sequence chosen from it.

The engines own the sharded state of the simulated ranks and pick, for the
configured stage, accumulation steps, clipping and ZeRO++ switches, the
sequence of library calls (step.py) that one training step needs:

* ``ZeroEngine`` (stages 1 and 2): ``backward(grads)`` once per micro-batch
  with every rank's bf16 gradient ([n_dp, P]); ``step()`` after the last one.
  Stage 1 accumulates each rank's full gradient locally and reduce-scatters
  once; stage 2 reduce-scatters every micro-batch ("ZeRO and FSDP", the
  paragraph on gradient accumulation).  The last micro-batch is fused into the
  update unless clipping needs the whole gradient's norm first.
* ``Zero3Engine`` (stage 3, per unit): ``gather(i, phase)`` before a unit's
  forward (phase "fwd") or backward ("bwd"), ``release(i, phase)`` after,
  ``backward(i, grads, micro)`` with the unit's gradient, ``step()`` at the
  end.  With one micro-batch and no clipping a unit is updated as soon as its
  gradient is reduced (one pass); otherwise the reduced gradients wait in fp32
  until ``step()``.  With ``overlap_comm`` each gather also starts the next
  unit's gather on a side stream (forward in order, then backward in reverse:
  "DeepSpeed ZeRO", "Stage 3 step by step", prefetching), when a ring slot is
  free.

Every element is computed by the library's kernels; the engines only hold
buffers and order the calls.
"""
from __future__ import annotations

import torch

from . import binding as zb
from . import checkpoint as ck
from . import step as zs
from .config import ZeroConfig


def _hp(cfg: ZeroConfig, t: int) -> zb.ZeroAdamW:
    return zb.ZeroAdamW.make(cfg.lr_at(t), cfg.betas[0], cfg.betas[1], cfg.eps, cfg.weight_decay, t)


class _Tracing:
    """Step time, gradient norm and the memory estimate ("DeepSpeed ZeRO",
    "Monitoring": track step time and memory use, log gradient norms; "Reading
    the memory report": the engine can report an estimate of memory per GPU at
    startup, to compare with what a run reaches)."""

    def _trace_init(self):
        self._ev = None

    def _step_begin(self):
        self._ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        self._ev[0].record()

    def _step_end(self):
        self._ev[1].record()

    def last_step_ms(self) -> float | None:
        """Device time of the last step() (CUDA events on the caller's stream;
        waits for it to finish)."""
        if self._ev is None:
            return None
        self._ev[1].synchronize()
        return self._ev[0].elapsed_time(self._ev[1])

    def grad_norm(self) -> float | None:
        """The global L2 norm of the last step's mean gradient, before clipping
        (only kept when gradient_clipping is configured; reads the device)."""
        if self.norm is None or self.t == 0:
            return None
        return float(self.norm.norm_sq.item()) ** 0.5

    def memory_estimate(self) -> dict:
        """Model-state bytes per GPU of a real n_dp-GPU job at every stage by the
        pages' formula (2 + 2 + 12 bytes per parameter, sharded by stage), and
        the bytes this process holds for all simulated ranks."""
        n = self._n_params()
        est = {f"stage{s}": zb.zero_memory_bytes(n, self._n_dp(), s) for s in range(4)}
        est["params"] = n
        est["this_process_bytes"] = sum(t.numel() * t.element_size() for t in self._held())
        return est


class ZeroEngine(_Tracing):
    """Stages 1 and 2 over n_dp simulated ranks of one flat parameter vector."""

    def __init__(self, numels, n_dp: int, config: ZeroConfig, master: torch.Tensor | None = None,
                 device="cuda", align: int = 8):
        if config.stage not in (1, 2):
            raise ValueError("ZeroEngine runs stages 1 and 2; use Zero3Engine for stage 3")
        self.cfg = config
        self.numels = [int(x) for x in numels]
        self.K = config.gradient_accumulation_steps
        if config.zero_quantized_gradients and config.stage == 1 and self.K > 1:
            raise ValueError("stage 1 accumulates locally before it communicates: quantized "
                             "gradients apply to stage 2 or to one micro-batch")
        self.L = L = zb.zero_layout(numels, n_dp, align, config.reduce_bucket_size)
        P = L.padded_n
        self.master = torch.zeros(P, device=device) if master is None else master
        self.m = torch.zeros(P, device=device)
        self.v = torch.zeros(P, device=device)
        self.out = torch.empty(P, dtype=torch.bfloat16, device=device)
        zb.zero_cast_bf16(self.master, self.out, P)         # the initial bf16 weights
        self.acc = [torch.empty(P, device=device) for _ in range(n_dp)] \
            if (config.stage == 1 and self.K > 1) else None
        self.A = torch.empty(P, device=device) if (config.stage == 2 and self.K > 1) else None
        self.norm = zs.NormBuffers(device) if config.gradient_clipping > 0 else None
        self.qg = zs.Int8Grads(L, n_dp, config.quant_block, device) \
            if config.zero_quantized_gradients else None
        self.t = 0
        self.micro = 0
        self._last = None
        self._trace_init()

    def _n_params(self):
        return self.L.n

    def _n_dp(self):
        return self.L.n_dp

    def _held(self):
        held = [self.master, self.m, self.v, self.out] + (self.acc or []) + ([self.A] if self.A is not None else [])
        if self.qg is not None:
            held += [self.qg.q, self.qg.scales]
        return held

    @property
    def weights(self) -> torch.Tensor:
        """The full flat bf16 weights every rank holds after a step."""
        return self.out

    def backward(self, grads: torch.Tensor):
        """Take one micro-batch: grads[r] is rank r's bf16 gradient (P elements)."""
        if self.micro >= self.K:
            raise RuntimeError("step() is due: all accumulation micro-batches were given")
        rows = [grads[r] for r in range(self.L.n_dp)]
        first = self.micro == 0
        last = self.micro == self.K - 1
        if self.K == 1 or (last and self.norm is None):
            self._last = rows             # fused into step(), or the one micro-batch of a step
        elif self.cfg.stage == 1:
            zs.zero1_accumulate_micro(self.L, rows, self.acc, first)
        elif self.qg is not None:
            self.qg.quantize(rows)
            q, s = self.qg.sources()
            zb.zero_accumulate_int8(self.L, q, s, self.qg.block, self._acc_buffer(), 0, 0,
                                    self.L.padded_n, first)
        else:
            zs.zero2_accumulate_micro(self.L, rows, self.A, first)
        self.micro += 1

    def _acc_buffer(self):
        if self.A is None:
            self.A = torch.empty(self.L.padded_n, device=self.master.device)
        return self.A

    def step(self):
        if self.micro != self.K:
            raise RuntimeError(f"step() after {self.micro} of {self.K} micro-batches")
        self._step_begin()
        L, cfg, K = self.L, self.cfg, self.K
        hp = _hp(cfg, self.t + 1)
        n = L.n_dp
        if self.norm is not None:
            # clipping: the norm of the whole mean gradient first, then the clipped update
            if K == 1 and self.qg is None:
                zs.zero12_step_clipped(L, self._last, self.master, self.m, self.v, self.out, hp,
                                       cfg.gradient_clipping, self.norm)
            else:
                # the reduced gradient: the ranks' local sums (stage 1), else the owners'
                srcs = [self._acc_buffer()] if (cfg.stage == 2 or self.qg is not None) else self.acc
                if K == 1:                                     # quantized, one micro-batch
                    self.qg.quantize(self._last)
                    q, s = self.qg.sources()
                    zb.zero_accumulate_int8(L, q, s, self.qg.block, srcs[0], 0, 0, L.padded_n, True)
                div = float(n * K)
                ranges = zs.bucket_ranges(L)
                for j, (s0, e0) in enumerate(ranges):
                    zb.zero_grad_norm_sq(L, srcs, zb.ZERO_F32, 0, div, s0, e0, self.norm.workspace,
                                         self.norm.norm_sq, j > 0)
                for s0, e0 in ranges:
                    zb.zero_reduce_scatter_adamw_clip(L, srcs, zb.ZERO_F32, 0, div, 0, n, s0, e0,
                                                      self.master, self.m, self.v, self.out,
                                                      zb.ZERO_OUT_FULL, hp, self.norm.norm_sq,
                                                      cfg.gradient_clipping)
        elif self.qg is not None and K == 1:
            self.qg.quantize(self._last)
            zs.zero12_step_int8(L, self.qg, self.master, self.m, self.v, self.out, hp)
        elif self.qg is not None:                              # stage 2, K > 1, quantized
            self.qg.quantize(self._last)
            q, s = self.qg.sources()
            zb.zero_accumulate_int8(L, q, s, self.qg.block, self._acc_buffer(), 0, 0, L.padded_n,
                                    False)
            zs.zero2_finish(L, self.A, K, self.master, self.m, self.v, self.out, hp)
        elif K == 1:
            zs.zero12_step(L, self._last, self.master, self.m, self.v, self.out, hp)
        elif cfg.stage == 1:
            zs.zero1_finish_fused(L, self.acc, self._last, K, self.master, self.m, self.v, self.out, hp)
        else:
            zs.zero2_finish_fused(L, self.A, self._last, K, self.master, self.m, self.v, self.out, hp)
        self._step_end()
        self.t += 1
        self.micro = 0
        self._last = None

    # -- checkpoints ("ZeRO Optimizer, in depth", "Checkpoints: sharded on the
    # way in, consolidated on the way out")

    def save_checkpoint(self, dirpath):
        """Every rank's shard of master / m / v and its bf16 weights, one file
        per rank, with the step count."""
        if self.micro:
            raise RuntimeError("save_checkpoint() between micro-batches: finish the step first")
        return ck.save(dirpath, self.L, self.numels, self.master, self.m, self.v, self.t,
                       _hp(self.cfg, max(1, self.t)), out_bf16=self.out)

    def load_checkpoint(self, dirpath) -> int:
        """Restore the state saved by save_checkpoint; returns the step count."""
        self.t = ck.restore(dirpath, self.L, self.master, self.m, self.v, out_bf16=self.out)
        self.micro = 0
        self._last = None
        return self.t

    def save_16bit_model(self, dirpath):
        """The full bf16 weights (every rank holds them after a step) as one file."""
        return ck.save_16bit_model(dirpath, self.out, self.numels)


class Zero3Engine(_Tracing):
    """Stage 3 over a list of units, each flattened, padded and sharded alone.
    last_step_ms() times step() itself: the updates that wait for it (with
    accumulation or clipping), not the per-unit fused updates of backward()."""

    def __init__(self, units_numels, n_dp: int, config: ZeroConfig, masters=None, device="cuda"):
        if config.stage != 3:
            raise ValueError("Zero3Engine runs stage 3")
        self.cfg = config
        self.numels = [[int(x) for x in u] for u in units_numels]
        self.K = config.gradient_accumulation_steps
        # the update that writes 8-bit shards itself needs 256-element slices
        self.fused = self.K == 1 and config.gradient_clipping == 0
        align = config.quant_block if config.zero_quantized_weights else 8
        self.units = []
        for i, numels in enumerate(units_numels):
            L = zb.zero_layout(numels, n_dp, align)
            P = L.padded_n
            w = torch.zeros(P, device=device) if masters is None else masters[i]
            shards = torch.empty(P, dtype=torch.bfloat16, device=device)
            zb.zero_cast_bf16(w, shards, P)                 # the initial bf16 shards
            self.units.append(zs.Zero3Unit(L, shards.view(n_dp, L.shard), w,
                                           torch.zeros(P, device=device), torch.zeros(P, device=device)))
        cap = max(u.layout.padded_n for u in self.units)
        self.ring = zs.GatherRing(cap, device=str(device))
        self.q8 = None
        if config.zero_quantized_weights:
            self.q8 = [zs.Int8Shards(u.layout, config.quant_block, device) for u in self.units]
            for u, q in zip(self.units, self.q8):
                zs.zero3_quantize(u, q)
        self.qg = [zs.Int8Grads(u.layout, n_dp, config.quant_block, device) for u in self.units] \
            if config.zero_quantized_gradients else None
        self.A = None if self.fused else [torch.empty(u.layout.padded_n, device=device)
                                          for u in self.units]
        self.norm = zs.NormBuffers(device) if config.gradient_clipping > 0 else None
        self.pf = zs.Zero3Prefetcher(self.units, self.ring, int8=self.q8, device=device) \
            if config.overlap_comm else None
        self.t = 0
        self._trace_init()

    def _n_params(self):
        return sum(u.layout.n for u in self.units)

    def _n_dp(self):
        return self.units[0].layout.n_dp if self.units else 1

    def _held(self):
        held = [x for u in self.units for x in (u.master, u.m, u.v, u.shards)] + self.ring.buffers
        held += self.A or []
        if self.q8 is not None:
            held += [x for q in self.q8 for x in (q.q, q.scales)]
        if self.qg is not None:
            held += [x for q in self.qg for x in (q.q, q.scales)]
        return held

    def _next(self, i: int, phase: str):
        """The gather that follows unit i's in the step's traversal, or None."""
        n = len(self.units)
        if phase == "fwd":
            return (i + 1, "fwd") if i + 1 < n else (n - 1, "bwd")
        if phase == "bwd" and i > 0:
            return (i - 1, "bwd")
        return None

    def _cancel_prefetches(self):
        """Drop pending prefetches: the caller's stream waits for them, then
        their ring slots are free for reuse."""
        for (tag, i) in list(self.pf.pending):
            self.pf.get(i, tag)
            self.ring.release((tag, i))

    def gather(self, i: int, phase="fwd") -> torch.Tensor:
        """Unit i's full bf16 weights in a ring slot, until release(i, phase)."""
        u = self.units[i]
        if self.pf is not None and (phase, i) in self.pf.pending:
            buf = self.pf.get(i, phase)
        else:
            if self.pf is not None:
                self._cancel_prefetches()
            if self.q8 is not None:
                buf = zs.zero3_gather_int8(u, self.q8[i], self.ring, (phase, i))
            else:
                buf = zs.zero3_gather(u, self.ring, (phase, i))
        if self.pf is not None:
            nxt = self._next(i, phase)
            if nxt is not None and self.ring.resident < self.ring.slots:
                self.pf.prefetch(nxt[0], nxt[1])
        return buf

    def release(self, i: int, phase="fwd"):
        self.ring.release((phase, i))

    def backward(self, i: int, grads: torch.Tensor, micro: int = 0):
        """Unit i's gradient of one micro-batch: grads[r] is rank r's bf16 gradient."""
        u = self.units[i]
        rows = [grads[r] for r in range(u.layout.n_dp)]
        if self.qg is not None:
            self.qg[i].quantize(rows)
        if self.fused:
            hp = _hp(self.cfg, self.t + 1)
            if self.qg is not None and self.q8 is not None:
                zs.zero3_reduce_scatter_update_int8_q8(u, self.qg[i], self.q8[i], hp)
            elif self.qg is not None:
                q, s = self.qg[i].sources()
                zb.zero_reduce_scatter_adamw_int8(u.layout, q, s, self.qg[i].block, float(u.layout.n_dp),
                                                  0, u.layout.n_dp, 0, u.layout.padded_n, u.master,
                                                  u.m, u.v, u.shards.view(-1), zb.ZERO_OUT_SHARD, hp)
            elif self.q8 is not None:
                zs.zero3_reduce_scatter_update_q8(u, rows, self.q8[i], hp)
            else:
                zs.zero3_reduce_scatter_update(u, rows, hp)
        elif self.qg is not None:
            zs.zero3_layer_reduce_scatter_int8(u, self.qg[i], self.A[i], first=(micro == 0))
        else:
            zs.zero3_layer_reduce_scatter(u, rows, self.A[i], first=(micro == 0))

    def step(self):
        if self.pf is not None:
            self._cancel_prefetches()
        self._step_begin()
        hp = _hp(self.cfg, self.t + 1)
        if not self.fused:
            if self.norm is not None:
                zs.zero3_clipped_updates(self.units, self.A, hp, self.cfg.gradient_clipping, self.norm,
                                         n_micro=self.K)
                if self.q8 is not None:
                    for u, q in zip(self.units, self.q8):
                        zs.zero3_quantize(u, q)
            else:
                for i, u in enumerate(self.units):
                    if self.q8 is not None:
                        zs.zero3_update_q8(u, self.A[i], self.q8[i], hp, n_micro=self.K)
                    else:
                        zs.zero3_update(u, self.A[i], hp, n_micro=self.K)
        self._step_end()
        self.t += 1

    # -- checkpoints: one sharded checkpoint per unit

    def _bf16_shards_current(self):
        """With 8-bit weights the update writes only the 8-bit shards; the bf16
        shards are brought back to bf16(master) by the library's cast, round to
        nearest even like the update's own."""
        if self.q8 is not None:
            for u in self.units:
                zb.zero_cast_bf16(u.master, u.shards.view(-1), u.layout.padded_n)

    def save_checkpoint(self, dirpath):
        """Every unit's shards of master / m / v and its owners' bf16 shards."""
        if self.pf is not None:
            self._cancel_prefetches()
        self._bf16_shards_current()
        ck.save_units(dirpath, self.units, self.numels, self.t, _hp(self.cfg, max(1, self.t)),
                      with_bf16=True)

    def load_checkpoint(self, dirpath) -> int:
        """Restore the state saved by save_checkpoint (the 8-bit shards are
        re-derived from the bf16 ones); returns the step count."""
        if self.pf is not None:
            self._cancel_prefetches()
        self.t = ck.restore_units(dirpath, self.units, with_bf16=True)
        if self.q8 is not None:
            for u, q in zip(self.units, self.q8):
                zs.zero3_quantize(u, q)
        return self.t

    def save_16bit_model(self, dirpath):
        """With stage3_gather_16bit_weights_on_model_save: every unit's bf16
        shards gathered (by the library's gather, unit by unit through the ring)
        into one file of the model's weights, padding dropped."""
        if not self.cfg.stage3_gather_16bit_weights_on_model_save:
            raise RuntimeError("save_16bit_model at stage 3 needs "
                               "zero_optimization.stage3_gather_16bit_weights_on_model_save")
        if self.pf is not None:
            self._cancel_prefetches()
        self._bf16_shards_current()
        parts = []
        for i, u in enumerate(self.units):
            buf = zs.zero3_gather(u, self.ring, ("save", i))     # the bf16 shards, not the 8-bit copies
            parts.append(buf[:u.layout.n].to("cpu"))
            self.ring.release(("save", i))
        flat = torch.cat(parts) if parts else torch.empty(0, dtype=torch.bfloat16)
        return ck.save_16bit_model(dirpath, flat, [x for u in self.numels for x in u])
