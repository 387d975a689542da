"""Sharded checkpoints of the ZeRO state: save per rank, consolidate, reshard.

"ZeRO Optimizer, in depth", "Checkpoints: sharded on the way in, consolidated
on the way out": every rank writes its own shard of model and optimizer state
plus a small metadata file, so saving needs no gather; a consolidation utility
rebuilds one plain full-precision state ("DeepSpeed ZeRO", "Saving and
loading": a utility consolidates sharded checkpoints into a single
full-precision file); a resume on another GPU count needs a conversion first.

Layout of a checkpoint directory:
* ``meta.json`` -- the layout (N, n_dp, S, P, alignment, bucket), the tensors'
  element counts and flat offsets, the step, the AdamW hyper-parameters, and
  the CRC-32 of every rank file;
* ``rank_00000.bin`` ... -- one file per rank, written by the library
  (``zero_ckpt_write_shard``): that rank's fp32 master / m / v shard and,
  optionally, its bf16 weights, with a CRC-32 over the payload.

The file IO and the CRC run in the native library; this module only copies
shards between device and (pinned) host memory and lays out the files.  The
rank files of one call are written or read by up to ``MAX_WORKERS`` threads at
once (the library releases the interpreter lock while it hashes and moves
bytes), each with its own host staging buffers.
"""
from __future__ import annotations

import ctypes
import json
import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from . import binding as zb

META = "meta.json"
FORMAT = "zero_gb300 sharded checkpoint"
MAX_WORKERS = 8        # threads writing or reading rank files at once (each stages one shard)


def _workers(n_ranks: int) -> int:
    return max(1, min(n_ranks, MAX_WORKERS, os.cpu_count() or 1))


def _rank_file(rank: int) -> str:
    return f"rank_{rank:05d}.bin"


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def write_shard(path, header: zb.ZeroCkptHeader, master, m, v, w_bf16=None):
    """Write one rank's shard from host numpy arrays (fp32, and uint16 bf16 bits)."""
    arrs = [np.ascontiguousarray(x, dtype=np.float32) for x in (master, m, v)]
    w = None if w_bf16 is None else np.ascontiguousarray(w_bf16, dtype=np.uint16)
    for a in arrs + ([w] if w is not None else []):
        if a.size != header.shard:
            raise ValueError(f"shard arrays must hold {header.shard} elements, got {a.size}")
    rc = zb.load().zero_ckpt_write_shard(os.fsencode(path), ctypes.byref(header),
                                         *[_ptr(a) for a in arrs], _ptr(w) if w is not None else None)
    zb._check(rc, "zero_ckpt_write_shard")


def read_shard(path, with_bf16=False):
    """Read one rank's shard: (header, master, m, v, w_bf16 or None), host arrays."""
    lib = zb.load()
    h = zb.ZeroCkptHeader()
    has = ctypes.c_int32()
    zb._check(lib.zero_ckpt_read_header(os.fsencode(path), ctypes.byref(h), ctypes.byref(has)),
              "zero_ckpt_read_header")
    s = h.shard
    master, m, v = (np.empty(s, np.float32) for _ in range(3))
    w = np.empty(s, np.uint16) if (with_bf16 and has.value) else None
    zb._check(lib.zero_ckpt_read_shard(os.fsencode(path), ctypes.byref(h), _ptr(master), _ptr(m),
                                       _ptr(v), _ptr(w) if w is not None else None, s),
              "zero_ckpt_read_shard")
    return h, master, m, v, w


def crc32(data) -> int:
    a = np.ascontiguousarray(data)
    return int(zb.load().zero_crc32(_ptr(a) if a.size else None, a.nbytes))


def payload_crc(path) -> int:
    """The payload CRC-32 a shard file's header records (computed when written)."""
    c = ctypes.c_uint32()
    zb._check(zb.load().zero_ckpt_payload_crc(os.fsencode(path), ctypes.byref(c)), "zero_ckpt_payload_crc")
    return int(c.value)


def save(dirpath, L: zb.ZeroLayout, numels, master, m, v, step: int, hp: zb.ZeroAdamW,
         out_bf16=None, rank_begin: int = 0):
    """Save the owners rank_begin.. of layout L: ``master``/``m``/``v`` hold their
    shards back to back (device or host tensors); ``out_bf16`` (optional, the
    full flat bf16 buffer) adds each rank's bf16 weights.  Returns the metadata."""
    os.makedirs(dirpath, exist_ok=True)
    S = L.shard
    n_ranks = master.numel() // S if S else 0
    if master.numel() != n_ranks * S:
        raise ValueError("master must hold whole shards")
    pin = torch.cuda.is_available()
    local = threading.local()

    def write_rank(k):
        if not hasattr(local, "host"):        # this worker's staging buffers
            local.host = [torch.empty(S, dtype=torch.float32, pin_memory=pin) for _ in range(3)]
            local.hw = torch.empty(S, dtype=torch.bfloat16, pin_memory=pin) if out_bf16 is not None else None
        r = rank_begin + k
        for dst, src in zip(local.host, (master, m, v)):
            dst.copy_(src[k * S:(k + 1) * S])
        if local.hw is not None:
            local.hw.copy_(out_bf16[r * S:(r + 1) * S])
        h = zb.ZeroCkptHeader(L.n, L.padded_n, S, L.align, int(step), L.n_dp, r, hp.lr, hp.beta1,
                              hp.beta2, hp.eps, hp.weight_decay, 0)
        arrs = [x.numpy() for x in local.host]
        wb = local.hw.view(torch.int16).numpy().view(np.uint16) if local.hw is not None else None
        path = os.path.join(dirpath, _rank_file(r))
        write_shard(path, h, *arrs, wb)
        return _rank_file(r), payload_crc(path)

    with ThreadPoolExecutor(_workers(n_ranks)) as ex:
        crcs = dict(ex.map(write_rank, range(n_ranks)))
    offsets = np.concatenate([[0], np.cumsum(numels)[:-1]]).astype(int).tolist() if len(numels) else []
    meta_path = os.path.join(dirpath, META)
    meta = {}
    if os.path.exists(meta_path):
        with open(meta_path) as f:
            meta = json.load(f)
    meta.update({
        "format": FORMAT, "version": 1, "n": L.n, "n_dp": L.n_dp, "shard": S, "padded_n": L.padded_n,
        "align": L.align, "bucket": L.bucket, "step": int(step), "numels": [int(x) for x in numels],
        "offsets": offsets, "bf16_weights": out_bf16 is not None,
        "adamw": {"lr": hp.lr, "beta1": hp.beta1, "beta2": hp.beta2, "eps": hp.eps,
                  "weight_decay": hp.weight_decay},
    })
    meta.setdefault("crc32", {}).update(crcs)
    with open(meta_path, "w") as f:
        json.dump(meta, f, indent=1)
    return meta


def load_meta(dirpath):
    with open(os.path.join(dirpath, META)) as f:
        meta = json.load(f)
    if meta.get("format") != FORMAT:
        raise ValueError(f"{dirpath}: not a {FORMAT}")
    return meta


def restore(dirpath, L: zb.ZeroLayout, master, m, v, rank_begin: int = 0, out_bf16=None) -> int:
    """Load the shards of owners rank_begin.. into ``master``/``m``/``v`` (and the
    bf16 weights into ``out_bf16``); the layout must match the checkpoint's.
    Returns the step to continue from."""
    meta = load_meta(dirpath)
    if (meta["n"], meta["n_dp"], meta["shard"]) != (L.n, L.n_dp, L.shard):
        raise ValueError("the checkpoint was saved for another layout: reshard it first")
    S = L.shard
    n_ranks = master.numel() // S if S else 0

    def read_rank(k):
        r = rank_begin + k
        h, ms, mm, mv, w = read_shard(os.path.join(dirpath, _rank_file(r)),
                                      with_bf16=out_bf16 is not None)
        if h.rank != r or h.step != meta["step"]:
            raise ValueError(f"rank file {r} does not match the metadata")
        for dst, src in zip((master, m, v), (ms, mm, mv)):
            dst[k * S:(k + 1) * S].copy_(torch.from_numpy(src))
        if out_bf16 is not None and w is not None:
            out_bf16[r * S:(r + 1) * S].copy_(torch.from_numpy(w.view(np.int16)).view(torch.bfloat16))

    with ThreadPoolExecutor(_workers(n_ranks)) as ex:
        list(ex.map(read_rank, range(n_ranks)))
    return int(meta["step"])


def consolidate(dirpath, split: bool = False):
    """The plain full-precision state: master / m / v as flat fp32 vectors of the
    N real elements (padding dropped), or, with split, a dict per tensor."""
    meta = load_meta(dirpath)
    N, S, n_dp = meta["n"], meta["shard"], meta["n_dp"]
    out = {k: np.empty(n_dp * S, np.float32) for k in ("master", "m", "v")}
    for r in range(n_dp):
        h, ms, mm, mv, _ = read_shard(os.path.join(dirpath, _rank_file(r)))
        if h.rank != r:
            raise ValueError(f"rank file {r} holds rank {h.rank}")
        for k, a in zip(("master", "m", "v"), (ms, mm, mv)):
            out[k][r * S:(r + 1) * S] = a
    flat = {k: a[:N].copy() for k, a in out.items()}
    flat["step"] = meta["step"]
    if not split:
        return flat
    tensors = []
    for off, cnt in zip(meta["offsets"], meta["numels"]):
        tensors.append({k: flat[k][off:off + cnt] for k in ("master", "m", "v")})
    return {"step": meta["step"], "tensors": tensors}


def reshard(dir_in, dir_out, n_dp: int, align: int | None = None, bucket: int | None = None):
    """Write the same state laid out for another number of ranks."""
    meta = load_meta(dir_in)
    flat = consolidate(dir_in)
    numels = meta["numels"] or [meta["n"]]
    L = zb.zero_layout(numels, n_dp, align or meta["align"], bucket or meta["bucket"])
    padded = {k: np.zeros(L.padded_n, np.float32) for k in ("master", "m", "v")}
    for k in padded:
        padded[k][:L.n] = flat[k]
    a = meta["adamw"]
    hp = zb.ZeroAdamW.make(a["lr"], a["beta1"], a["beta2"], a["eps"], a["weight_decay"],
                           max(1, meta["step"]))
    return save(dir_out, L, numels, *(torch.from_numpy(padded[k]) for k in ("master", "m", "v")),
                meta["step"], hp)


# --------------------------------------------------------------------------
# stage 3: one checkpoint per unit ("ZeRO and FSDP", "FSDP, ZeRO-3 inside
# PyTorch": every unit is flattened, padded and sharded on its own)
# --------------------------------------------------------------------------

UNITS = "units.json"


def _unit_dir(dirpath, i: int) -> str:
    return os.path.join(dirpath, f"unit_{i:05d}")


def save_units(dirpath, units, numels_per_unit, step: int, hp: zb.ZeroAdamW, with_bf16: bool = False):
    """Save every stage-3 unit (step.Zero3Unit: its layout, fp32 master / m / v
    over all owners, and the owners' bf16 shards) as its own sharded
    checkpoint in unit_00000/, unit_00001/, ...; units.json lists them."""
    os.makedirs(dirpath, exist_ok=True)
    for i, (u, numels) in enumerate(zip(units, numels_per_unit)):
        save(_unit_dir(dirpath, i), u.layout, numels, u.master, u.m, u.v, step, hp,
             out_bf16=u.shards.reshape(-1) if with_bf16 else None)
    with open(os.path.join(dirpath, UNITS), "w") as f:
        json.dump({"format": FORMAT, "units": len(units), "step": int(step)}, f, indent=1)


def _n_units(dirpath) -> int:
    with open(os.path.join(dirpath, UNITS)) as f:
        meta = json.load(f)
    if meta.get("format") != FORMAT:
        raise ValueError(f"{dirpath}: not a {FORMAT}")
    return int(meta["units"])


def restore_units(dirpath, units, with_bf16: bool = False) -> int:
    """Load every unit's shards back (the layouts must match); returns the step."""
    n = _n_units(dirpath)
    if n != len(units):
        raise ValueError(f"the checkpoint holds {n} units, not {len(units)}")
    steps = {restore(_unit_dir(dirpath, i), u.layout, u.master, u.m, u.v,
                     out_bf16=u.shards.reshape(-1) if with_bf16 else None)
             for i, u in enumerate(units)}
    if len(steps) != 1:
        raise ValueError("the units were saved at different steps")
    return steps.pop()


def consolidate_units(dirpath):
    """The plain full-precision state of the whole model: every unit's real
    elements (padding dropped), units in order, as flat fp32 vectors."""
    parts = [consolidate(_unit_dir(dirpath, i)) for i in range(_n_units(dirpath))]
    out = {k: np.concatenate([p[k] for p in parts]) if parts else np.empty(0, np.float32)
           for k in ("master", "m", "v")}
    out["step"] = parts[0]["step"] if parts else 0
    return out


def reshard_units(dir_in, dir_out, n_dp: int, align: int | None = None):
    """Every unit laid out for another number of ranks."""
    n = _n_units(dir_in)
    for i in range(n):
        reshard(_unit_dir(dir_in, i), _unit_dir(dir_out, i), n_dp, align)
    with open(os.path.join(dir_in, UNITS)) as f:
        meta = json.load(f)
    with open(os.path.join(dir_out, UNITS), "w") as f:
        json.dump(meta, f, indent=1)


# --------------------------------------------------------------------------
# one full 16-bit weight file ("ZeRO Optimizer, in depth": with
# stage3_gather_16bit_weights_on_model_save, save_16bit_model gathers the
# 16-bit weights at save time, for inference or sharing)
# --------------------------------------------------------------------------

MODEL16 = "model_16bit.bin"
MODEL16_META = "model_16bit.json"


def save_16bit_model(dirpath, weights_bf16, numels):
    """Write the model's bf16 weights as one file: ``weights_bf16`` is the flat
    vector of the N real elements in flattening order (device or host); the
    metadata lists the tensors' element counts and the CRC-32 of the file."""
    os.makedirs(dirpath, exist_ok=True)
    n = int(sum(numels))
    w = weights_bf16.reshape(-1)[:n]
    host = w.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
    if host.size != n:
        raise ValueError(f"the weights hold {host.size} elements, the tensors {n}")
    path = os.path.join(dirpath, MODEL16)
    host.tofile(path)
    meta = {"format": FORMAT + " (16-bit weights)", "version": 1, "dtype": "bf16", "n": n,
            "numels": [int(x) for x in numels], "crc32": crc32(host.view(np.uint8))}
    with open(os.path.join(dirpath, MODEL16_META), "w") as f:
        json.dump(meta, f, indent=1)
    return meta


def load_16bit_model(dirpath, split: bool = False):
    """The saved bf16 weights as uint16 bit patterns (the flat vector, or a list
    per tensor with split); the CRC-32 is checked."""
    with open(os.path.join(dirpath, MODEL16_META)) as f:
        meta = json.load(f)
    w = np.fromfile(os.path.join(dirpath, MODEL16), dtype=np.uint16)
    if w.size != meta["n"] or crc32(w.view(np.uint8)) != meta["crc32"]:
        raise ValueError(f"{dirpath}: the 16-bit weight file does not match its metadata")
    if not split:
        return w
    offs = np.concatenate([[0], np.cumsum(meta["numels"])]).astype(int)
    return [w[a:b] for a, b in zip(offs[:-1], offs[1:])]
