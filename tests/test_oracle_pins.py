"""Pins for the oracle: it is checked against things other than itself.

Each test ties an oracle function to a closed form, a hand-worked fixture in
tests/golden/, a brute-force enumeration, an independent library routine, or an
invariant the pages fix (merge of shard partials equals unsharded attention; an empty
shard gives zero output and -inf LSE; the merge of all-empty shards is zero; the remap
keeps exactly the owned slots in their order).  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
P = 64


# ----------------------------------------------------------------------------- helpers
def enum_owner_local(T, dcp, interleave):
    """Owner by the workload statement (block of `interleave` slots, mod D) and local id
    by enumeration: the rank of the slot among the slots its shard holds."""
    owner = np.empty(T, dtype=np.int64)
    local = np.empty(T, dtype=np.int64)
    seen = [0] * dcp
    for t in range(T):
        s = (t // interleave) % dcp
        owner[t] = s
        local[t] = seen[s]
        seen[s] += 1
    return owner, local


def bf16_bits(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy()


def place_bf16(seqs, dcp, interleave, rng=None):
    """Paged BF16 pool built by enumeration (not by the oracle's closed form).

    seqs: list of float arrays [L_b, 576] whose values are exact in bf16.
    Returns pool [pages, 64, 1152] uint8 and block_table [D, B, maxp] int32."""
    B = len(seqs)
    per = []
    for X in seqs:
        own, loc = enum_owner_local(len(X), dcp, interleave)
        per.append((own, loc))
    need = [[int(np.sum(own == s) + P - 1) // P for (own, _) in per] for s in range(dcp)]
    maxp = max(1, max(max(r) for r in need))
    total = sum(sum(r) for r in need)
    order = np.arange(total)[::-1].copy() if rng is None else rng.permutation(total)
    bt = np.full((dcp, B, maxp), -1, dtype=np.int32)
    c = 0
    for s in range(dcp):
        for b in range(B):
            bt[s, b, :need[s][b]] = order[c:c + need[s][b]]
            c += need[s][b]
    pool = np.zeros((max(total, 1), P, 576), dtype=np.int16)
    for b, X in enumerate(seqs):
        own, loc = per[b]
        bits = bf16_bits(X)
        for t in range(len(X)):
            page = bt[own[t], b, loc[t] // P]
            pool[page, loc[t] % P] = bits[t]
    return pool.view(np.uint8).reshape(pool.shape[0], P, 1152), bt


def place_fp8(codes, scales, rope, dcp, interleave):
    """FP8 pool for one sequence by enumeration; codes [L,512] u8, scales [L,4] f32,
    rope [L,64] (bf16-exact)."""
    L = codes.shape[0]
    own, loc = enum_owner_local(L, dcp, interleave)
    need = [int(np.sum(own == s) + P - 1) // P for s in range(dcp)]
    maxp = max(need)
    bt = np.full((dcp, 1, maxp), -1, dtype=np.int32)
    c = 0
    for s in range(dcp):
        bt[s, 0, :need[s]] = np.arange(c, c + need[s])[::-1]
        c += need[s]
    pool = np.zeros((c, P, 656), dtype=np.uint8)
    rb = bf16_bits(rope).view(np.uint8).reshape(L, 128)
    for t in range(L):
        row = pool[bt[own[t], 0, loc[t] // P], loc[t] % P]
        row[:512] = codes[t]
        row[512:528] = np.asarray(scales[t], dtype=np.float32).view(np.uint8)
        row[528:656] = rb[t]
    return pool, bt


def q_bits(q):
    return bf16_bits(q)


def run_attn(orc, q, pool, bt, dcp, interleave, kv_dtype, sm, topk=None, row_len=None,
             shard=-1, row_seq=None):
    R = q.shape[0]
    rs = np.zeros(R, dtype=np.int32) if row_seq is None else np.asarray(row_seq, np.int32)
    return orc.attention(q_bits(q), pool, bt, rs, dcp, interleave, kv_dtype, sm,
                         topk=None if topk is None else np.asarray(topk, np.int32),
                         row_len=None if row_len is None else np.asarray(row_len, np.int32),
                         shard=shard)


# ----------------------------------------------------------------------------- E4M3
def test_e4m3_spot_values_from_format(orc):
    # OCP FP8 E4M3 ("fn"): max normal 448, min normal 2^-6, subnormal step 2^-9, NaN S.1111.111
    assert orc.e4m3_decode(0x00) == 0.0
    assert math.copysign(1.0, orc.e4m3_decode(0x80)) == -1.0
    assert orc.e4m3_decode(0x01) == 2.0 ** -9
    assert orc.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert orc.e4m3_decode(0x08) == 2.0 ** -6
    assert orc.e4m3_decode(0x38) == 1.0
    assert orc.e4m3_decode(0x3C) == 1.5
    assert orc.e4m3_decode(0x7E) == 448.0
    assert orc.e4m3_decode(0xFE) == -448.0
    assert math.isnan(orc.e4m3_decode(0x7F)) and math.isnan(orc.e4m3_decode(0xFF))


def test_e4m3_all_codes_match_torch_and_are_monotone(orc):
    tab = orc.e4m3_table()
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(tab), ~finite)
    assert np.array_equal(tab[finite], ref[finite])
    pos = tab[0:127]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(tab[128:255], -pos)


# ----------------------------------------------------------------------------- owner / local
@pytest.mark.parametrize("dcp,interleave", [(1, 1), (2, 1), (3, 1), (4, 1), (8, 1), (2, 64),
                                            (4, 64), (8, 64), (3, 5)])
def test_owner_local_match_enumeration(orc, dcp, interleave):
    T = 3 * dcp * interleave * 7 + 11
    own, loc = enum_owner_local(T, dcp, interleave)
    for t in range(T):
        assert orc.owner(t, dcp, interleave) == own[t]
        assert orc.local(t, dcp, interleave) == loc[t]


@pytest.mark.parametrize("dcp,interleave", [(2, 1), (4, 1), (8, 1), (2, 64), (8, 64)])
def test_count_owned_closed_form(orc, dcp, interleave):
    ID = dcp * interleave
    for L in [0, 1, 5, 63, 64, 65, 255, 256, 1000, 4099]:
        for s in range(dcp):
            closed = (L // ID) * interleave + min(max(L % ID - s * interleave, 0), interleave)
            assert orc.count_owned(L, dcp, interleave, s) == closed


# ----------------------------------------------------------------------------- remap
def _read_remap_golden():
    cases = []
    for line in open(os.path.join(GOLDEN, "remap_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = [p.strip() for p in line.split("|")]
        d, i = map(int, parts[0].split())
        g = list(map(int, parts[1].split()))
        shards = []
        for grp in parts[2:]:
            ids, cnt = grp.split(";")
            shards.append((list(map(int, ids.split())), int(cnt)))
        cases.append((d, i, g, shards))
    return cases


@pytest.mark.parametrize("case", _read_remap_golden())
def test_remap_golden(orc, case):
    d, i, g, shards = case
    loc, cnt = orc.remap(np.array([g], dtype=np.int32), d, i)
    assert len(shards) == d
    for s, (ids, c) in enumerate(shards):
        assert loc[s, 0].tolist() == ids
        assert cnt[s, 0] == c
        one, onec = orc.remap(np.array([g], dtype=np.int32), d, i, shard=s)
        assert one[0, 0].tolist() == ids and onec[0, 0] == c


@pytest.mark.parametrize("dcp", [2, 4, 8])
def test_remap_invariants_on_stress_rows(orc, dcp):
    import synth
    prob = synth.cfg4_remap_merge(dcp, rows=48, k=512, seq_len=20000, with_partials=False)
    g = prob.topk.numpy()
    I = prob.interleave
    loc, cnt = orc.remap(g, dcp, I)
    for r in range(g.shape[0]):
        valid = [t for t in g[r] if t >= 0]
        assert int(cnt[:, r].sum()) == len(valid)
        back = []
        for s in range(dcp):
            c = cnt[s, r]
            assert np.all(loc[s, r, c:] == -1) and np.all(loc[s, r, :c] >= 0)
            # invert local -> global independently: block j of I slots on shard s is
            # global block j*D + s
            gl = [(l // I) * I * dcp + s * I + l % I for l in loc[s, r, :c]]
            pos = [valid.index(t) for t in gl]
            assert pos == sorted(pos)          # original order kept
            back += gl
        assert sorted(back) == sorted(valid)   # exactly the owned slots, nothing else
    assert cnt[:, 48 // 2].sum() == 0           # the all-padding row


def test_remap_stress_has_empty_shard_rows(orc):
    import synth
    prob = synth.cfg4_remap_merge(4, rows=256, k=512, seq_len=20000, with_partials=False)
    _, cnt = orc.remap(prob.topk.numpy(), 4, prob.interleave)
    some_empty = ((cnt == 0).any(axis=0) & (cnt.sum(axis=0) > 0)).sum()
    assert some_empty >= 3


# ----------------------------------------------------------------------------- attention
SM = 1.0 / math.sqrt(192.0)


def _rand_int_tokens(rng, L):
    return rng.integers(-4, 5, size=(L, 576)).astype(np.float32) / 4.0  # exact in bf16


def test_attention_fetches_the_right_slot(orc):
    # each token's dim 0 holds its global slot id; q = e0, scale 1 -> lse = slot id
    for dcp, I in [(1, 1), (2, 1), (4, 1), (2, 64), (3, 64)]:
        L = 200
        X = np.zeros((L, 576), np.float32)
        X[:, 0] = np.arange(L)
        X[:, 1] = -np.arange(L) / 2.0
        pool, bt = place_bf16([X], dcp, I, rng=np.random.default_rng(dcp * 7 + I))
        slots = [0, 1, 63, 64, 65, 127, 128, 199, 150]
        q = np.zeros((len(slots), 1, 576), np.float32)
        q[:, 0, 0] = 1.0
        topk = np.array([[t, -1, -1] for t in slots], np.int32)
        out, lse = run_attn(orc, q, pool, bt, dcp, I, 0, 1.0, topk=topk,
                            row_seq=np.zeros(len(slots)))
        assert np.array_equal(lse[:, 0], np.array(slots, dtype=np.float64))
        assert np.array_equal(out[:, 0, 0], np.array(slots, dtype=np.float64))
        assert np.array_equal(out[:, 0, 1], -np.array(slots, dtype=np.float64) / 2.0)


def test_attention_zero_query_is_mean_and_log_count(orc):
    rng = np.random.default_rng(1)
    X = _rand_int_tokens(rng, 300)
    pool, bt = place_bf16([X], 2, 1, rng=rng)
    slots = [3, 17, 200, 299, 0, 150, 151]
    q = np.zeros((1, 2, 576), np.float32)
    out, lse = run_attn(orc, q, pool, bt, 2, 1, 0, SM, topk=[slots + [-1]])
    assert np.allclose(lse, math.log(len(slots)), atol=1e-14, rtol=0)
    assert np.allclose(out[0, 0], X[slots, :512].astype(np.float64).mean(axis=0), atol=1e-14, rtol=0)


def test_attention_two_logits_quarter_three_quarters(orc):
    # logits {0, ln 3} -> weights {1/4, 3/4}, lse = ln 4
    X = np.zeros((10, 576), np.float32)
    X[4, 520] = 1.0          # key marker in a RoPE dim, outside the value dims
    X[2, 5] = 4.0
    X[4, 5] = 8.0
    pool, bt = place_bf16([X], 2, 1)
    q = np.zeros((1, 1, 576), np.float32)
    q[0, 0, 520] = 1.0
    out, lse = run_attn(orc, q, pool, bt, 2, 1, 0, math.log(3.0), topk=[[2, 4]])
    assert abs(lse[0, 0] - math.log(4.0)) < 1e-15
    assert abs(out[0, 0, 5] - 7.0) < 1e-14
    assert np.count_nonzero(out[0, 0]) == 1


def test_attention_single_slot_and_equal_keys(orc):
    rng = np.random.default_rng(2)
    X = _rand_int_tokens(rng, 64)
    pool, bt = place_bf16([X], 1, 1)
    q = rng.integers(-3, 4, size=(1, 3, 576)).astype(np.float32) / 2.0
    out, lse = run_attn(orc, q, pool, bt, 1, 1, 0, SM, topk=[[37]])
    for h in range(3):
        assert abs(lse[0, h] - SM * float(np.dot(q[0, h].astype(np.float64), X[37]))) < 1e-12
        assert np.array_equal(out[0, h], X[37, :512].astype(np.float64))
    Y = np.tile(X[5], (40, 1))
    pool, bt = place_bf16([Y], 2, 1)
    out, lse = run_attn(orc, q, pool, bt, 2, 1, 0, SM, row_len=[40])
    for h in range(3):
        s = SM * float(np.dot(q[0, h].astype(np.float64), X[5]))
        assert abs(lse[0, h] - (s + math.log(40))) < 1e-12
        assert np.allclose(out[0, h], X[5, :512], atol=1e-13, rtol=0)


def test_attention_fp8_dequant_closed_form(orc):
    L = 70
    codes = np.zeros((L, 512), np.uint8)
    scales = np.zeros((L, 4), np.float32)
    rope = np.zeros((L, 64), np.float32)
    codes[9, 0] = 0x38      # 1.0 in block 0
    codes[9, 130] = 0x3C    # 1.5 in block 1
    codes[9, 511] = 0x01    # 2^-9 in block 3 (subnormal)
    scales[9] = [3.0, 0.25, 7.0, 1024.0]
    rope[9, 2] = -2.0
    pool, bt = place_fp8(codes, scales, rope, 2, 1)
    q = np.zeros((1, 1, 576), np.float32)
    q[0, 0, 0] = 1.0
    q[0, 0, 130] = 2.0
    q[0, 0, 511] = 1.0
    q[0, 0, 514] = 0.5
    out, lse = run_attn(orc, q, pool, bt, 2, 1, 1, 1.0, topk=[[9]])
    # 1.0*3 + 2*(1.5*0.25) + 1*(2^-9*1024) + 0.5*(-2) = 3 + 0.75 + 2 - 1
    assert lse[0, 0] == 4.75
    assert out[0, 0, 0] == 3.0 and out[0, 0, 130] == 0.375 and out[0, 0, 511] == 2.0
    assert np.count_nonzero(out[0, 0]) == 3


def test_attention_sparse_all_tokens_equals_dense(orc):
    rng = np.random.default_rng(3)
    X = (rng.standard_normal((150, 576)) * 8).round() / 8
    pool, bt = place_bf16([X], 4, 1, rng=rng)
    q = (rng.standard_normal((1, 4, 576)) * 8).round() / 8
    o1, l1 = run_attn(orc, q, pool, bt, 4, 1, 0, SM, row_len=[150])
    o2, l2 = run_attn(orc, q, pool, bt, 4, 1, 0, SM, topk=[list(rng.permutation(150))])
    assert np.allclose(o1, o2, atol=1e-12, rtol=0) and np.allclose(l1, l2, atol=1e-12, rtol=0)


@pytest.mark.parametrize("dcp,interleave", [(2, 1), (4, 1), (3, 64)])
def test_shard_partials_merge_to_unsharded(orc, dcp, interleave):
    rng = np.random.default_rng(4 + dcp)
    seqs = [(rng.standard_normal((L, 576)) * 8).round() / 8 for L in (333, 100)]
    pool, bt = place_bf16(seqs, dcp, interleave, rng=rng)
    q = (rng.standard_normal((3, 8, 576)) * 8).round() / 8
    rs = [0, 1, 0]
    topk = [list(rng.choice(333, 90, replace=False)), list(rng.choice(100, 40, replace=False)) + [-1] * 50,
            [7] + [-1] * 89]
    for mode in ("sparse", "dense"):
        kw = dict(topk=topk) if mode == "sparse" else dict(row_len=[333, 100, 5])
        ou, lu = run_attn(orc, q, pool, bt, dcp, interleave, 0, SM, row_seq=rs, **kw)
        parts = [run_attn(orc, q, pool, bt, dcp, interleave, 0, SM, row_seq=rs, shard=s, **kw)
                 for s in range(dcp)]
        po = np.stack([p[0] for p in parts])
        pl = np.stack([p[1] for p in parts])
        mo, ml = orc.merge(po, pl)
        assert np.allclose(mo, ou, atol=1e-12, rtol=0)
        assert np.allclose(ml, lu, atol=1e-12, rtol=0)
        if mode == "sparse":
            # a shard that owns nothing of a row gives o = 0, lse = -inf (single-slot row)
            empty = [s for s in range(dcp) if np.isneginf(pl[s, 2, 0])]
            assert len(empty) == dcp - 1
            for s in empty:
                assert np.all(po[s, 2] == 0.0)


def test_shard_partial_counts_dense(orc):
    # q = 0: a shard's dense partial has lse = ln(number of slots it owns)
    for dcp, I in [(2, 1), (4, 1), (2, 64), (4, 64)]:
        L = 1000
        X = np.zeros((L, 576), np.float32)
        pool, bt = place_bf16([X], dcp, I)
        q = np.zeros((1, 1, 576), np.float32)
        for s in range(dcp):
            _, lse = run_attn(orc, q, pool, bt, dcp, I, 0, SM, row_len=[L], shard=s)
            n = sum(1 for t in range(L) if (t // I) % dcp == s)
            assert abs(lse[0, 0] - math.log(n)) < 1e-12


# ----------------------------------------------------------------------------- merge
def _read_merge_golden():
    cases = []
    for line in open(os.path.join(GOLDEN, "merge_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b, c = [p.strip() for p in line.split("|")]
        lse = [float(x) for x in a.split()]
        outs = [float(x) for x in b.split()]
        mo, ml = [float(x) for x in c.split(";")]
        cases.append((lse, outs, mo, ml))
    return cases


@pytest.mark.parametrize("case", _read_merge_golden())
def test_merge_golden(orc, case):
    lse, outs, mo, ml = case
    D = len(lse)
    po = np.array(outs, np.float64).reshape(D, 1, 1, 1)
    pl = np.array(lse, np.float64).reshape(D, 1, 1)
    o, l = orc.merge(po, pl)
    assert abs(o[0, 0, 0] - mo) < 1e-13
    if math.isinf(ml):
        assert np.isneginf(l[0, 0])
    else:
        assert abs(l[0, 0] - ml) < 1e-13


def test_merge_invariants(orc):
    rng = np.random.default_rng(9)
    D, R, H, dv = 5, 7, 3, 16
    po = rng.standard_normal((D, R, H, dv))
    pl = 5 + 3 * rng.standard_normal((D, R, H))
    pl[1, 2] = -np.inf
    po[1, 2] = 0
    pl[:, 4] = -np.inf
    po[:, 4] = 0
    o, l = orc.merge(po, pl)
    # D = 1 is the identity
    o1, l1 = orc.merge(po[:1], pl[:1])
    assert np.array_equal(o1, po[0]) and np.array_equal(l1, pl[0])
    # all-empty row -> zero output, -inf lse, no NaN
    assert np.all(o[4] == 0) and np.all(np.isneginf(l[4])) and not np.isnan(o).any()
    # shard order does not matter
    perm = rng.permutation(D)
    op, lp = orc.merge(po[perm], pl[perm])
    assert np.allclose(op, o, atol=1e-13, rtol=0) and np.allclose(lp, l, atol=1e-13, rtol=0)
    # adding an empty shard changes nothing
    oe, le = orc.merge(np.concatenate([po, np.zeros((1, R, H, dv))]),
                       np.concatenate([pl, np.full((1, R, H), -np.inf)]))
    assert np.allclose(oe, o, atol=1e-15, rtol=0) and np.array_equal(le, l)
    # merged lse is log-sum-exp over shards (scipy as an independent routine)
    from scipy.special import logsumexp
    assert np.allclose(l[:4], logsumexp(pl[:, :4], axis=0), atol=1e-12, rtol=0)
