"""GPU parity of the DCP KV-cache write (dcp_kv_cache_write) against the oracle.

The pool bytes a call writes (E4M3 codes, fp32 scales, bf16 RoPE, or the bf16 row) are
integer results of fp32 decisions both sides take identically, so they must be
bit-identical to the oracle's.  Also: the shard filter, the checked-mode error bits, a
bench-sized call checked on sampled rows, and a round trip through the fused decode."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
P = 64


@pytest.fixture(scope="module")
def dcp():
    import decode_context_sparse_gb300 as d
    from decode_context_sparse_gb300 import build
    build.build()
    d.load()
    return d


def _rows(n, gen):
    """Token rows with the cases that matter for the quantiser: N(0,1), wide dynamic range,
    all-zero blocks, tiny values (E4M3 subnormals after scaling), exact ties."""
    x = torch.randn((n, 576), generator=gen) * torch.exp(torch.randn((n, 1), generator=gen) * 2)
    z = torch.rand((n, 4), generator=gen) < 0.05
    for b in range(4):
        x[:, 128 * b:128 * b + 128][z[:, b]] = 0.0
    x[: n // 8, 0:128] *= 1e-4
    return x.to(torch.bfloat16)


def _case(n, seqs, T, dcp_, interleave, kv_dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    pages_per = -(-(-(-T // dcp_)) // P) + 1
    num_pages = dcp_ * seqs * pages_per + 3
    perm = torch.randperm(num_pages, generator=gen)[: dcp_ * seqs * pages_per].to(torch.int32)
    bt = perm.view(dcp_, seqs, pages_per).contiguous()
    tb = synth.TOKEN_BYTES[kv_dtype]
    pool = torch.randint(0, 256, (num_pages, P, tb), generator=gen, dtype=torch.uint8)
    flat = torch.randperm(seqs * T, generator=gen)[:n]
    seq = (flat // T).to(torch.int32)
    pos = (flat % T).to(torch.int32)
    pos[:: 97] = -1                    # padding rows
    return _rows(n, gen), seq, pos, pool, bt


@pytest.mark.parametrize("kv_dtype", [synth.KV_FP8, synth.KV_BF16])
@pytest.mark.parametrize("dcp_,interleave", [(1, 1), (2, 1), (8, 1), (4, 64)])
def test_kv_write_matches_oracle_bytes(dcp, orc, kv_dtype, dcp_, interleave):
    kv, seq, pos, pool, bt = _case(1003, 3, 3000, dcp_, interleave, kv_dtype, seed=dcp_ * 10 + interleave)
    ref, written, skipped = orc.kv_write(kv, seq, pos, pool, kv_dtype, bt, dcp_, interleave)
    assert skipped == int((pos < 0).sum()) and written == int((pos >= 0).sum())
    d_pool = pool.cuda()
    dcp.dcp_kv_cache_write(kv.cuda(), seq.cuda(), pos.cuda(), d_pool, kv_dtype, bt.cuda(), dcp_, interleave)
    torch.cuda.synchronize()
    assert np.array_equal(d_pool.cpu().numpy(), ref)


def test_kv_write_shard_filter(dcp, orc):
    kv, seq, pos, pool, bt = _case(500, 2, 2000, 4, 1, synth.KV_FP8, seed=3)
    for s in range(4):
        ref, _, _ = orc.kv_write(kv, seq, pos, pool, synth.KV_FP8, bt, 4, 1, shard=s)
        d_pool = pool.cuda()
        dcp.dcp_kv_cache_write(kv.cuda(), seq.cuda(), pos.cuda(), d_pool, synth.KV_FP8, bt.cuda(), 4, 1,
                               shard=s)
        torch.cuda.synchronize()
        assert np.array_equal(d_pool.cpu().numpy(), ref), s


def test_kv_write_checked_mode_flags_and_skips(dcp, orc):
    kv, seq, pos, pool, bt = _case(300, 2, 1000, 2, 1, synth.KV_BF16, seed=4)
    bt[1, 0, 0] = 10 ** 6          # a page past the pool
    seq[5] = 7                     # a sequence past the tables
    ref, _, skipped = orc.kv_write(kv, seq, pos, pool, synth.KV_BF16, bt, 2, 1)
    assert skipped >= 2
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_pool = pool.cuda()
    dcp.dcp_kv_cache_write(kv.cuda(), seq.cuda(), pos.cuda(), d_pool, synth.KV_BF16, bt.cuda(), 2, 1,
                           checked=True, err_flag=err)
    torch.cuda.synchronize()
    assert np.array_equal(d_pool.cpu().numpy(), ref)
    e = int(err.item())
    assert e & dcp.DCP_ERRBIT_PAGE_RANGE and e & dcp.DCP_ERRBIT_SLOT_RANGE


def test_kv_write_bench_size_sampled(dcp, orc):
    """64 sequences x 2048 new tokens (the bench's cache-fill call), FP8, D = 8: every row
    lands where the owner rule puts it; 1500 sampled rows are byte-identical to the oracle."""
    seqs, T, D = 64, 2048, 8
    gen = torch.Generator(device="cuda").manual_seed(9)
    pages_per = T // D // P
    num_pages = D * seqs * pages_per
    bt = torch.randperm(num_pages, device="cuda", generator=gen).to(torch.int32).view(D, seqs, pages_per)
    kv = (torch.randn((seqs * T, 576), device="cuda", generator=gen)).to(torch.bfloat16)
    seq = torch.arange(seqs, device="cuda", dtype=torch.int32).repeat_interleave(T)
    pos = torch.arange(T, device="cuda", dtype=torch.int32).repeat(seqs)
    pool = torch.zeros((num_pages, P, 656), dtype=torch.uint8, device="cuda")
    dcp.dcp_kv_cache_write(kv, seq, pos, pool, synth.KV_FP8, bt, D, 1)
    torch.cuda.synchronize()
    pick = torch.randperm(seqs * T, generator=torch.Generator().manual_seed(1))[:1500]
    kv_s, seq_s, pos_s = kv[pick.cuda()].cpu(), seq[pick.cuda()].cpu(), pos[pick.cuda()].cpu()
    blank = np.zeros((num_pages, P, 656), np.uint8)
    ref, written, _ = orc.kv_write(kv_s, seq_s, pos_s, blank, synth.KV_FP8, bt.cpu(), D, 1)
    assert written == 1500
    got = pool.cpu().numpy()
    s = (pos_s.numpy() // 1) % D
    l = pos_s.numpy() // D
    pages = bt.cpu().numpy()[s, seq_s.numpy(), l // P]
    assert np.array_equal(got[pages, l % P], ref[pages, l % P])


def test_kv_write_then_fused_decode_round_trip(dcp, orc):
    """Fill an FP8 cache with the GPU writer, decode it with the fused kernel, and compare with
    the oracle's attention over the oracle-written cache (the same bytes)."""
    from parity import check_lse, check_out
    seqs, T, D, H, K = 2, 1500, 4, 128, 256
    gen = torch.Generator().manual_seed(21)
    pages_per = -(-(-(-T // D)) // P)
    num_pages = D * seqs * pages_per
    bt = torch.randperm(num_pages, generator=gen).to(torch.int32).view(D, seqs, pages_per).contiguous()
    kv = torch.randn((seqs * T, 576), generator=gen).to(torch.bfloat16)
    seq = torch.arange(seqs, dtype=torch.int32).repeat_interleave(T)
    pos = torch.arange(T, dtype=torch.int32).repeat(seqs)
    pool0 = torch.zeros((num_pages, P, 656), dtype=torch.uint8)
    d_pool = pool0.cuda()
    dcp.dcp_kv_cache_write(kv.cuda(), seq.cuda(), pos.cuda(), d_pool, synth.KV_FP8, bt.cuda(), D, 1)
    ref_pool, _, _ = orc.kv_write(kv, seq, pos, pool0, synth.KV_FP8, bt, D, 1)
    torch.cuda.synchronize()
    assert np.array_equal(d_pool.cpu().numpy(), ref_pool)
    rows = 4
    row_seq = torch.tensor([0, 0, 1, 1], dtype=torch.int32)
    q = torch.randn((rows, H, 576), generator=gen).to(torch.bfloat16)
    lens = torch.full((rows,), T, dtype=torch.int32)
    topk = synth.sample_topk(lens, K, gen)
    out, lse = dcp.mla_decode_dcp_fused(q.cuda(), d_pool, synth.KV_FP8, bt.cuda(), row_seq.cuda(),
                                        1 / 192 ** 0.5, D, 1, idx=topk.cuda())
    torch.cuda.synchronize()
    ref_o, ref_l = orc.attention(q, torch.from_numpy(ref_pool), bt, row_seq, D, 1, synth.KV_FP8,
                                 1 / 192 ** 0.5, topk=topk, row_len=lens)
    check_out(out, ref_o, "round trip")
    check_lse(lse, ref_l, "round trip")


def _reciprocal_traps(limit=8):
    """(amax, v) with bf16 values for which v * (1/scale) and the IEEE quotient v / scale
    (scale = amax / 448, fp32) round to different E4M3 codes: a writer that multiplies by the
    reciprocal without checking gets these wrong.  Found by exhaustive search over bf16 v."""
    bits = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    vals = bits[np.isfinite(bits)]

    def e4(x):
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
            torch.float8_e4m3fn).view(torch.uint8).numpy()
    out = []
    for amax in vals[(vals >= 0.5) & (vals <= 300)][::97]:
        s = np.float32(amax) / np.float32(448)
        r = np.float32(1) / s
        v = vals[np.abs(vals) <= amax]
        bad = e4((v / s).astype(np.float32)) != e4((v * r).astype(np.float32))
        for x in v[bad][:2]:
            out.append((float(amax), float(x)))
        if len(out) >= limit:
            break
    return out


def test_kv_write_quotients_near_e4m3_boundaries(dcp, orc):
    """Rows built from values whose reciprocal product rounds to another code than the exact
    quotient: the written codes must still be those of the IEEE quotients (the oracle's)."""
    traps = _reciprocal_traps()
    assert traps, "the search found no trap values"
    n = len(traps)
    kv = torch.zeros((n, 576))
    for i, (amax, v) in enumerate(traps):
        for b in range(4):
            kv[i, 128 * b] = amax
            kv[i, 128 * b + 1:128 * b + 128] = v * (1 if b % 2 == 0 else -1)
    kv = kv.to(torch.bfloat16)
    assert all(float(kv[i, 1].abs()) == abs(v) for i, (_, v) in enumerate(traps))
    seq = torch.zeros(n, dtype=torch.int32)
    pos = torch.arange(n, dtype=torch.int32)
    bt = torch.arange(2, dtype=torch.int32).view(1, 1, 2)
    pool = torch.zeros((2, P, 656), dtype=torch.uint8)
    ref, written, _ = orc.kv_write(kv, seq, pos, pool, synth.KV_FP8, bt, 1, 1)
    assert written == n
    d_pool = pool.cuda()
    dcp.dcp_kv_cache_write(kv.cuda(), seq.cuda(), pos.cuda(), d_pool, synth.KV_FP8, bt.cuda(), 1, 1)
    torch.cuda.synchronize()
    assert np.array_equal(d_pool.cpu().numpy(), ref)


def test_kv_write_signed_zeros_and_extreme_scales(dcp, orc):
    """Blocks the quotient method treats with care: -0 and +0 beside nonzero values (the sign
    of a zero decides its code), bf16 subnormals, a block of zeros of both signs (scale 0),
    blocks whose scale lies below 2^-100 or near the top of the fp32 range (exact divisions),
    and quotients just around the smallest E4M3 subnormal's rounding midpoint."""
    gen = torch.Generator().manual_seed(21)
    rows = []
    base = torch.randn((8, 576), generator=gen)
    r = base.clone()
    r[0, 1:64:2] = -0.0
    r[0, 2:64:2] = 0.0
    r[1, 0:128] = torch.randn(128, generator=gen) * 2.0 ** -128   # bf16 subnormals
    r[1, 128:256] = 0.0
    r[1, 128:256:3] = -0.0                                      # all-zero block, both signs
    r[2, 0:128] = torch.randn(128, generator=gen) * 2.0 ** -95  # scale below 2^-100
    r[2, 128:256] = torch.randn(128, generator=gen) * 2.0 ** 126  # scale near 2^118
    r[3, 0] = 448.0                                             # scale exactly 1
    r[3, 1:128] = torch.linspace(2.0 ** -11, 2.0 ** -9, 127)      # around 2^-10, the midpoint
    r[3, 128] = -448.0
    r[3, 129:256] = -torch.linspace(2.0 ** -11, 2.0 ** -9, 127)
    rows.append(r)
    kv = torch.cat(rows).to(torch.bfloat16)
    assert bool(torch.signbit(kv[0, 1])) and kv[0, 1] == 0
    n = kv.shape[0]
    seq = torch.zeros(n, dtype=torch.int32)
    pos = torch.arange(n, dtype=torch.int32)
    bt = torch.arange(1, dtype=torch.int32).view(1, 1, 1)
    pool = torch.zeros((1, P, 656), dtype=torch.uint8)
    ref, written, _ = orc.kv_write(kv, seq, pos, pool, synth.KV_FP8, bt, 1, 1)
    assert written == n
    d_pool = pool.cuda()
    dcp.dcp_kv_cache_write(kv.cuda(), seq.cuda(), pos.cuda(), d_pool, synth.KV_FP8, bt.cuda(), 1, 1)
    torch.cuda.synchronize()
    got = d_pool.cpu().numpy()
    assert (ref[0, 0, 1:64:2] == 0x80).all() and (ref[0, 0, 2:64:2] == 0x00).all()
    assert np.array_equal(got, ref)
