"""Sharded checkpoints on the host (no GPU): the shard file round trip, the
CRC-32 against zlib's (a library routine), corruption detection, consolidation
(padding dropped, tensors split at their offsets) and resharding to another
number of ranks."""
import ctypes
import os
import zlib as zlib_ref

import numpy as np
import pytest
import torch

from zero_sharded_mixed_gb300 import binding as zb
from zero_sharded_mixed_gb300 import checkpoint as ck


def _state(P, seed):
    rng = np.random.default_rng(seed)
    return [torch.from_numpy((rng.standard_normal(P) * s).astype(np.float32)) for s in (0.02, 1e-4, 1e-8)]


def test_crc32_matches_zlib(zlib):
    """Every length 0..40 (the 8-byte loop and the byte tail), start offsets off
    the 8-byte grid, and long buffers."""
    buf = np.random.default_rng(0).integers(0, 256, 1 << 20, dtype=np.uint8)
    for n in list(range(41)) + [4096, 100_003, 1 << 20]:
        for off in (0, 1, 3, 7):
            data = buf[off:off + n]
            assert ck.crc32(data) == (zlib_ref.crc32(data.tobytes()) & 0xFFFFFFFF), (n, off)
    assert ck.crc32(np.zeros(8, np.uint8)) == (zlib_ref.crc32(bytes(8)) & 0xFFFFFFFF)
    assert ck.crc32(np.full(9, 255, np.uint8)) == (zlib_ref.crc32(b"\xff" * 9) & 0xFFFFFFFF)


def test_the_header_records_the_payload_crc(zlib, tmp_path):
    S = 777
    h = zb.ZeroCkptHeader(3100, 3108, S, 1, 2, 4, 1, 1e-4, 0.9, 0.999, 1e-8, 0.1, 0)
    rng = np.random.default_rng(1)
    a = [rng.standard_normal(S).astype(np.float32) for _ in range(3)]
    w = rng.integers(0, 1 << 16, S).astype(np.uint16)
    p = str(tmp_path / "r.bin")
    ck.write_shard(p, h, *a, w)
    payload = b"".join(x.tobytes() for x in a + [w])
    assert ck.payload_crc(p) == (zlib_ref.crc32(payload) & 0xFFFFFFFF)
    with pytest.raises(zb.ZeroError):
        ck.payload_crc(str(tmp_path / "missing.bin"))


def test_shard_round_trip_and_corruption(zlib, tmp_path):
    S = 1000
    h = zb.ZeroCkptHeader(3990, 4000, S, 8, 7, 4, 2, 1e-4, 0.9, 0.999, 1e-8, 0.1, 0)
    rng = np.random.default_rng(0)
    a = [rng.standard_normal(S).astype(np.float32) for _ in range(3)]
    w = rng.integers(0, 1 << 16, S).astype(np.uint16)
    p = str(tmp_path / "r.bin")
    ck.write_shard(p, h, *a, w)
    h2, m, mm, v, w2 = ck.read_shard(p, with_bf16=True)
    for x, y in zip(a + [w], [m, mm, v, w2]):
        np.testing.assert_array_equal(x, y)
    assert (h2.rank, h2.step, h2.n_dp, h2.shard, h2.n) == (2, 7, 4, S, 3990)
    # reading without the bf16 part still checks the whole payload
    assert ck.read_shard(p)[4] is None
    # one flipped byte anywhere in the payload is caught
    raw = bytearray(open(p, "rb").read())
    for pos in (len(raw) - 1, len(raw) - 2 * S - 5, len(raw) // 2):
        bad = bytearray(raw)
        bad[pos] ^= 0x40
        open(p, "wb").write(bad)
        with pytest.raises(zb.ZeroError) as e:
            ck.read_shard(p)
        assert e.value.code == zb.ZERO_ECORRUPT
    open(p, "wb").write(b"not a shard file at all, definitely not")
    with pytest.raises(zb.ZeroError) as e:
        ck.read_shard(p)
    assert e.value.code == zb.ZERO_ECORRUPT
    with pytest.raises(zb.ZeroError) as e:
        ck.read_shard(str(tmp_path / "missing.bin"))
    assert e.value.code == zb.ZERO_EIO


def test_header_validation(zlib, tmp_path):
    x = np.zeros(8, np.float32)
    for bad in [dict(rank=4), dict(n_dp=0), dict(padded_n=31), dict(n=33), dict(step=-1)]:
        kw = dict(n=30, padded_n=32, shard=8, align=8, step=1, n_dp=4, rank=0)
        kw.update(bad)
        h = zb.ZeroCkptHeader(kw["n"], kw["padded_n"], kw["shard"], kw["align"], kw["step"],
                              kw["n_dp"], kw["rank"], 0, 0, 0, 0, 0, 0)
        with pytest.raises(zb.ZeroError) as e:
            ck.write_shard(str(tmp_path / "x.bin"), h, x, x, x)
        assert e.value.code == zb.ZERO_EINVAL


def test_header_whose_size_overflows_is_refused(zlib, tmp_path):
    """A header with shard * n_dp past int64 (2^62 * 4 wraps to the padded_n 0
    given) is refused by the writer before any byte count is formed; the
    arrays passed are never read."""
    x = np.zeros(8, np.float32)
    h = zb.ZeroCkptHeader(0, 0, 1 << 62, 8, 1, 4, 0, 0, 0, 0, 0, 0, 0)
    path = tmp_path / "x.bin"
    rc = zb.load().zero_ckpt_write_shard(os.fsencode(str(path)), ctypes.byref(h), *[x.ctypes.data] * 3, None)
    assert rc == zb.ZERO_EINVAL
    assert not path.exists()


def test_save_consolidate_reshard(zlib, tmp_path):
    numels = [1000, 3, 4097, 50]
    L = zb.zero_layout(numels, 4, align=8)
    P, N = L.padded_n, L.n
    master, m, v = _state(P, 1)
    for t in (master, m, v):
        t[N:] = 0
    hp = zb.ZeroAdamW.make(step=5)
    meta = ck.save(str(tmp_path / "a"), L, numels, master, m, v, 5, hp)
    assert meta["n_dp"] == 4 and len(meta["crc32"]) == 4
    flat = ck.consolidate(str(tmp_path / "a"))
    assert flat["step"] == 5
    for k, t in (("master", master), ("m", m), ("v", v)):
        np.testing.assert_array_equal(flat[k], t[:N].numpy())
    per = ck.consolidate(str(tmp_path / "a"), split=True)
    assert [x["master"].size for x in per["tensors"]] == numels
    np.testing.assert_array_equal(per["tensors"][2]["m"], m[1003:1003 + 4097].numpy())
    # another GPU count: 4 -> 3 -> 7 ranks, the consolidated state is unchanged
    ck.reshard(str(tmp_path / "a"), str(tmp_path / "b"), 3)
    ck.reshard(str(tmp_path / "b"), str(tmp_path / "c"), 7, align=1)
    for d in ("b", "c"):
        again = ck.consolidate(str(tmp_path / d))
        for k in ("master", "m", "v"):
            np.testing.assert_array_equal(again[k], flat[k])
    assert ck.load_meta(str(tmp_path / "c"))["n_dp"] == 7
    # restoring into the original layout gives back every element, padding included
    got = [torch.empty(P) for _ in range(3)]
    assert ck.restore(str(tmp_path / "a"), L, *got) == 5
    for a, b in zip(got, (master, m, v)):
        assert torch.equal(a, b)
    # and a layout mismatch is refused
    with pytest.raises(ValueError):
        ck.restore(str(tmp_path / "b"), L, *got)


def test_stage3_units_save_consolidate_reshard_restore(zlib, tmp_path):
    """Stage-3 units, each its own layout: one checkpoint per unit; the
    consolidated model state is every unit's real elements in order; resharding
    to another rank count keeps it; a restore gives back every element."""
    from zero_sharded_mixed_gb300.step import Zero3Unit
    n_dp = 5
    numels_per_unit = [[1], [4097], [1000, 24, 3, 5000]]
    units = []
    for i, numels in enumerate(numels_per_unit):
        L = zb.zero_layout(numels, n_dp)
        master, m, v = _state(L.padded_n, 10 + i)
        for t in (master, m, v):
            t[L.n:] = 0
        shards = master.to(torch.bfloat16).view(n_dp, L.shard)
        units.append(Zero3Unit(L, shards, master, m, v))
    hp = zb.ZeroAdamW.make(step=3)
    ck.save_units(str(tmp_path / "u"), units, numels_per_unit, 3, hp, with_bf16=True)
    flat = ck.consolidate_units(str(tmp_path / "u"))
    assert flat["step"] == 3
    for k in ("master", "m", "v"):
        want = np.concatenate([getattr(u, k)[:u.layout.n].numpy() for u in units])
        np.testing.assert_array_equal(flat[k], want)
    ck.reshard_units(str(tmp_path / "u"), str(tmp_path / "u3"), 3, align=1)
    again = ck.consolidate_units(str(tmp_path / "u3"))
    for k in ("master", "m", "v"):
        np.testing.assert_array_equal(again[k], flat[k])
    fresh = [Zero3Unit(u.layout, torch.zeros_like(u.shards), torch.empty_like(u.master),
                       torch.empty_like(u.m), torch.empty_like(u.v)) for u in units]
    assert ck.restore_units(str(tmp_path / "u"), fresh, with_bf16=True) == 3
    for a, b in zip(fresh, units):
        for k in ("master", "m", "v"):
            assert torch.equal(getattr(a, k), getattr(b, k))
        assert torch.equal(a.shards.view(torch.int16), b.shards.view(torch.int16))
    with pytest.raises(ValueError):
        ck.restore_units(str(tmp_path / "u"), fresh[:2])


def test_16bit_model_round_trip_and_corruption(zlib, tmp_path):
    """The 16-bit weight file: the real elements only, split back per tensor;
    a flipped byte or a truncated file is refused."""
    numels = [5, 1, 4097, 33]
    n = sum(numels)
    bits = np.random.default_rng(3).integers(0, 1 << 16, size=n + 11, dtype=np.uint16)  # + padding
    w = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    d = str(tmp_path / "w16")
    meta = ck.save_16bit_model(d, w, numels)
    assert meta["n"] == n and meta["numels"] == numels
    flat = ck.load_16bit_model(d)
    assert np.array_equal(flat, bits[:n])
    parts = ck.load_16bit_model(d, split=True)
    assert [p.size for p in parts] == numels
    assert np.array_equal(np.concatenate(parts), bits[:n])
    with pytest.raises(ValueError):
        ck.save_16bit_model(str(tmp_path / "short"), w[:n - 1], numels)
    path = tmp_path / "w16" / ck.MODEL16
    raw = bytearray(path.read_bytes())
    raw[1234] ^= 0x10
    path.write_bytes(bytes(raw))
    with pytest.raises(ValueError):
        ck.load_16bit_model(d)
    raw[1234] ^= 0x10
    path.write_bytes(bytes(raw[:-2]))
    with pytest.raises(ValueError):
        ck.load_16bit_model(d)
    path.write_bytes(bytes(raw))
    assert np.array_equal(ck.load_16bit_model(d), bits[:n])
