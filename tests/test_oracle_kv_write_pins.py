"""Pins for the oracle's DCP KV-cache writer and its E4M3 encoder (CPU only).

The encoder is tied to the E4M3 format definition (every code round-trips, midpoints go to
the even code, values past 448 saturate) and to an independent library routine (torch's
float8_e4m3fn cast).  The writer is tied to the owner rule by enumeration (the rank of a
slot among its shard's slots, not the oracle's closed form), to hand-built FP8 blocks whose
codes and scale are known exactly, and to the skip / shard-filter contract.
"""
import numpy as np
import pytest
import torch

P = 64


def finite_codes():
    return [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_e4m3_encode_round_trips_every_code(orc):
    for c in finite_codes():
        v = np.float32(orc.e4m3_decode(c))
        assert orc.e4m3_encode(float(v)) == c, c


def test_e4m3_encode_midpoints_go_to_even_code(orc):
    for c in range(0, 0x7E):
        lo, hi = orc.e4m3_decode(c), orc.e4m3_decode(c + 1)
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # exact in fp32 (at most 5 significant bits)
        even = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode(float(mid)) == even, (c, float(mid))
        assert orc.e4m3_encode(float(np.nextafter(mid, np.float32(0)))) == c
        assert orc.e4m3_encode(float(np.nextafter(mid, np.float32(1e9)))) == c + 1
        assert orc.e4m3_encode(-float(mid)) == even | 0x80


def test_e4m3_encode_saturates_at_448(orc):
    for v in (448.0, 448.5, 464.0, 479.9, 1e6, 3e38):
        assert orc.e4m3_encode(v) == 0x7E
        assert orc.e4m3_encode(-v) == 0xFE
    assert orc.e4m3_encode(0.0) == 0x00 and orc.e4m3_encode(-0.0) == 0x80


def test_e4m3_encode_matches_torch_cast(orc):
    g = torch.Generator().manual_seed(5)
    v = torch.cat([torch.randn(4000, generator=g) * 100,
                   torch.randn(2000, generator=g) * 0.01,        # subnormal E4M3 range
                   (torch.rand(2000, generator=g) - 0.5) * 896]).clamp(-448, 448)
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(x)) for x in v.numpy()], dtype=np.uint8)
    assert np.array_equal(got, ref)


def enum_owner_local(T, dcp, interleave):
    owner = np.empty(T, dtype=np.int64)
    local = np.empty(T, dtype=np.int64)
    seen = [0] * dcp
    for t in range(T):
        s = (t // interleave) % dcp
        owner[t] = s
        local[t] = seen[s]
        seen[s] += 1
    return owner, local


def _tables(dcp, num_seqs, pages_per, rng):
    """Block tables [dcp][num_seqs][pages_per] over a random permutation of the pool."""
    num_pages = dcp * num_seqs * pages_per
    perm = rng.permutation(num_pages).astype(np.int32)
    return perm.reshape(dcp, num_seqs, pages_per), num_pages


@pytest.mark.parametrize("dcp,interleave", [(1, 1), (2, 1), (4, 1), (2, 64), (8, 64)])
def test_kv_write_bf16_places_rows_by_enumerated_owner(orc, dcp, interleave):
    rng = np.random.default_rng(dcp * 100 + interleave)
    num_seqs, T = 3, 700
    pages_per = -(-(-(-T // dcp)) // P) + 2
    bt, num_pages = _tables(dcp, num_seqs, pages_per, rng)
    pool = np.zeros((num_pages, P, 1152), dtype=np.uint8)
    n = 200
    seq = rng.integers(0, num_seqs, n).astype(np.int32)
    pos = rng.choice(T, n, replace=False).astype(np.int32)
    kv = rng.integers(0, 256, (n, 1152)).astype(np.uint8)
    out, written, skipped = orc.kv_write(kv, seq, pos, pool, 0, bt, dcp, interleave)
    assert written == n and skipped == 0
    owner, local = enum_owner_local(T, dcp, interleave)
    expect = pool.copy()
    for i in range(n):
        s, l = owner[pos[i]], local[pos[i]]
        expect[bt[s, seq[i], l // P], l % P] = kv[i]
    assert np.array_equal(out, expect)


def _bf16_bytes(vals):
    return torch.tensor(np.asarray(vals, np.float32)).to(torch.bfloat16).view(torch.uint8).numpy()


def test_kv_write_fp8_blocks_with_known_codes(orc):
    rng = np.random.default_rng(7)
    codes = rng.choice([c for c in finite_codes() if c not in (0x00, 0x80)], 128)
    codes[5] = 0x7E  # amax exactly 448 * scale
    codes[9] = 0xFE
    table = orc.e4m3_table()
    row = np.zeros(576, np.float32)
    row[0:128] = 0.0                                     # all-zero block: scale 0, codes 0
    row[128:256] = table[codes] * 0.125                  # scale = 56 / 448 = 0.125 exactly
    row[256:384] = rng.standard_normal(128) * 3
    row[384:512] = -np.abs(rng.standard_normal(128)) * 1e-3
    row[512:576] = rng.standard_normal(64)
    kv = _bf16_bytes(row)[None, :]
    bt = np.zeros((1, 1, 1), np.int32)
    pool = np.full((1, P, 656), 0xAA, np.uint8)
    out, written, _ = orc.kv_write(kv, np.array([0], np.int32), np.array([3], np.int32), pool, 1, bt, 1, 1)
    assert written == 1
    r = out[0, 3]
    scales = r[512:528].view(np.float32)
    assert scales[0] == 0.0 and np.all(r[0:128] == 0)
    assert scales[1] == np.float32(0.125) and np.array_equal(r[128:256], codes.astype(np.uint8))
    vb = torch.tensor(_bf16_bytes(row)).view(torch.bfloat16).float().numpy()
    for blk in (2, 3):
        v = vb[128 * blk:128 * blk + 128]
        assert scales[blk] == np.float32(np.float32(np.abs(v).max()) / np.float32(448))
        deq = table[r[128 * blk:128 * blk + 128]] * scales[blk]
        # E4M3 keeps 3 mantissa bits: half an ulp is 2^-4 relative (2^-10 * scale absolute
        # in the subnormal range)
        assert np.all(np.abs(deq - v) <= np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10 * scales[blk]) * (1 + 1e-6))
    assert np.array_equal(r[528:656], kv[0, 1024:1152])
    assert np.all(out[0, :3] == 0xAA) and np.all(out[0, 4:] == 0xAA)   # no other row touched


def test_kv_write_shard_filter_and_skips(orc):
    rng = np.random.default_rng(11)
    dcp, T, num_seqs = 4, 512, 2
    bt, num_pages = _tables(dcp, num_seqs, 3, rng)
    bt[2, 1, 0] = -1                                     # a missing page
    pool = np.zeros((num_pages, P, 1152), np.uint8)
    pos = np.array([0, 1, 2, 3, 4, 5, 6, 7, -1, 10], np.int32)
    seq = np.array([0, 0, 1, 1, 1, 1, 0, 0, 0, 5], np.int32)   # seq 5 out of range
    kv = rng.integers(1, 256, (10, 1152)).astype(np.uint8)
    full, written, skipped = orc.kv_write(kv, seq, pos, pool, 0, bt, dcp, 1)
    # token 2 (seq 1, shard 2, local 0) hits the missing page; -1 and seq 5 are skipped too
    assert (written, skipped) == (7, 3)
    acc = pool.copy()
    for s in range(dcp):
        part, w, _ = orc.kv_write(kv, seq, pos, acc, 0, bt, dcp, 1, shard=s)
        changed = np.flatnonzero(np.any(part != acc, axis=(1, 2)))
        assert set(changed.tolist()) <= set(bt[s].reshape(-1).tolist())
        acc = part
    assert np.array_equal(acc, full)
