"""GPU parity: the CUDA path through the C ABI against the oracle, element by element on
small and ragged cases and on every row of the full-size workloads."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_lse, check_out, run_fused, run_unfused

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def dcp():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from decode_context_sparse_gb300 import build
    build.build()
    import decode_context_sparse_gb300 as m
    m.load()
    return m


# ----------------------------------------------------------------------------- remap
@pytest.mark.parametrize("D", [2, 4, 8])
def test_remap_stress_full_size(dcp, D):
    prob = synth.cfg4_remap_merge(D, device=DEV, with_partials=False)
    loc, cnt = dcp.dcp_remap_topk(prob.topk, D, prob.interleave)
    rloc, rcnt = oracle.remap(prob.topk, D, prob.interleave)
    assert np.array_equal(cnt.cpu().numpy(), rcnt)
    assert np.array_equal(loc.cpu().numpy(), rloc)
    for s in (0, D - 1):
        l1, c1 = dcp.dcp_remap_topk(prob.topk, D, prob.interleave, shard=s)
        assert np.array_equal(l1[0].cpu().numpy(), rloc[s])
        assert np.array_equal(c1[0].cpu().numpy(), rcnt[s])


@pytest.mark.parametrize("k", [1, 7, 33, 255, 2048, 5000, 16384])
@pytest.mark.parametrize("D,I", [(1, 1), (3, 1), (8, 1), (5, 64), (64, 1)])
def test_remap_random(dcp, k, D, I):
    g = torch.Generator().manual_seed(k * 131 + D * 7 + I)
    rows = 37
    ids = torch.randint(-3, 500000, (rows, k), generator=g, dtype=torch.int32)
    ids[3] = -1
    loc, cnt = dcp.dcp_remap_topk(ids.to(DEV), D, I)
    rloc, rcnt = oracle.remap(ids, D, I)
    assert np.array_equal(cnt.cpu().numpy(), rcnt) and np.array_equal(loc.cpu().numpy(), rloc)


def test_local_lengths(dcp):
    g = torch.Generator().manual_seed(5)
    L = torch.randint(0, 200000, (300,), generator=g, dtype=torch.int32)
    L[:6] = torch.tensor([0, 1, 63, 64, 65, 4096], dtype=torch.int32)
    for D, I in [(1, 1), (2, 1), (3, 1), (4, 64), (8, 1), (8, 64)]:
        ll = dcp.dcp_local_lengths(L.to(DEV), D, I).cpu().numpy()
        for r in list(range(6)) + [50, 299]:
            for s in range(D):
                assert ll[s, r] == oracle.count_owned(int(L[r]), D, I, s)


# ----------------------------------------------------------------------------- merge
@pytest.mark.parametrize("D", [2, 4, 8])
def test_merge_stress_full_size(dcp, D):
    """Every row of the remap + merge stress workload (256 rows x 128 heads x 512)."""
    prob = synth.cfg4_remap_merge(D, device=DEV)
    out, lse = dcp.dcp_lse_merge(prob.part_out, prob.part_lse)
    torch.cuda.synchronize()
    R = prob.part_out.shape[1]
    ro, rl = oracle.merge(prob.part_out.cpu().numpy(), prob.part_lse.cpu().numpy())
    check_out(out, ro, "merge out")
    check_lse(lse, rl, "merge lse")
    assert torch.all(out[R // 2] == 0) and torch.all(torch.isneginf(lse[R // 2]))


@pytest.mark.parametrize("dv", [512, 4, 132])
def test_merge_shapes(dcp, dv):
    g = torch.Generator().manual_seed(dv)
    D, R, H = 3, 5, 6
    po = torch.randn((D, R, H, dv), generator=g)
    pl = 5 + 3 * torch.randn((D, R, H), generator=g)
    pl[0, 1] = -math.inf
    po[0, 1] = 0
    pl[:, 2] = -math.inf
    po[:, 2] = 0
    out, lse = dcp.dcp_lse_merge(po.to(DEV), pl.to(DEV))
    ro, rl = oracle.merge(po.numpy(), pl.numpy())
    check_out(out, ro)
    check_lse(lse, rl)


def test_merge_golden(dcp):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "merge_hand.txt")
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b, c = [x.strip() for x in line.split("|")]
        lse = torch.tensor([float(x) for x in a.split()])
        outs = torch.tensor([float(x) for x in b.split()])
        mo, ml = [float(x) for x in c.split(";")]
        D = lse.numel()
        po = outs.view(D, 1, 1, 1).repeat(1, 1, 1, 4).contiguous()
        o, l = dcp.dcp_lse_merge(po.to(DEV), lse.view(D, 1, 1).to(DEV))
        assert abs(o[0, 0, 0].item() - mo) <= 1e-2 * max(1.0, abs(mo))
        if math.isinf(ml):
            assert math.isinf(l.item()) and l.item() < 0
        else:
            assert abs(l.item() - ml) <= 1e-5


# ----------------------------------------------------------------------------- decode
def _check_problem(dcp, prob, rows=None, num_splits=0, check_partials=True):
    """Unfused and fused GPU paths vs the oracle (unsharded and per shard)."""
    g = prob.to(DEV)
    po, pl, mo, ml = run_unfused(dcp, g, num_splits=num_splits)
    fo, fl = run_fused(dcp, g, num_splits=num_splits)
    torch.cuda.synchronize()
    sel = slice(None) if rows is None else rows
    ro, rl = oracle.attention_problem(prob, rows=rows)
    check_out(mo[sel], ro, "merged out")
    check_lse(ml[sel], rl, "merged lse")
    check_out(fo[sel], ro, "fused out")
    check_lse(fl[sel], rl, "fused lse")
    if check_partials:
        for s in range(prob.dcp):
            so, sl = oracle.attention_problem(prob, rows=rows, shard=s)
            check_out(po[s][sel], so, "partial out shard %d" % s)
            check_lse(pl[s][sel], sl, "partial lse shard %d" % s)
    return mo, ml, fo, fl


def test_cfg1_tiny_dense_bf16(dcp):
    _check_problem(dcp, synth.cfg1_tiny_dense())


def test_cfg2_sparse_topk512_bf16(dcp):
    _check_problem(dcp, synth.cfg2_sparse_topk512())


def test_cfg3_scaled_sparse_fp8(dcp):
    prob = synth.make_decode_problem("cfg3s", [4100, 2500, 3333], 128, 2048, synth.KV_FP8, 8, 1,
                                     mtp=6, seed=21)
    _check_problem(dcp, prob)


def test_cfg5_scaled_dense_bf16(dcp):
    prob = synth.make_decode_problem("cfg5s", [1000, 3000, 4097], 128, None, synth.KV_BF16, 4, 1,
                                     seed=24)
    _check_problem(dcp, prob)


@pytest.mark.parametrize("heads", [16, 32, 64, 128])
@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8])
def test_heads_and_dtypes_ragged(dcp, heads, kv):
    prob = synth.make_decode_problem("ragged", [777, 130, 64], heads, 37, kv, 3, 1, mtp=2, seed=heads + kv)
    _check_problem(dcp, prob)


@pytest.mark.parametrize("heads", [48, 80, 96, 112])
@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8])
def test_padded_head_counts_tensor_core(dcp, heads, kv):
    """Head counts the tensor-core path pads to its 128-row tiles (48..112): the padded rows
    stay out of the outputs, LSEs and split merges.  Rows long enough to be cut between CTA
    pairs (1000 slots each over a few pairs) exercise the split merge too."""
    prob = synth.make_decode_problem("padh", [3000, 2200, 130], heads, 1000, kv, 4, 1, mtp=2,
                                     seed=heads * 3 + kv)
    _check_problem(dcp, prob)


@pytest.mark.parametrize("D,I,heads,kv", [(16, 1, 128, synth.KV_FP8), (64, 1, 64, synth.KV_BF16),
                                           (16, 64, 128, synth.KV_BF16)])
def test_many_shards(dcp, D, I, heads, kv):
    """Up to DCP_MAX_SHARDS shards: many shards hold few or no slots of a row (empty
    partials, -inf LSEs) and the fused path resolves owners across all their tables."""
    prob = synth.make_decode_problem("manyD", [2500, 700], heads, 300, kv, D, I, mtp=2,
                                     seed=D * 7 + I + heads)
    _check_problem(dcp, prob, check_partials=D <= 16)


@pytest.mark.parametrize("splits", [1, 3, 64])
def test_split_counts(dcp, splits):
    prob = synth.make_decode_problem("splits", [3000, 900], 64, 1000, synth.KV_FP8, 4, 1, mtp=3, seed=31)
    _check_problem(dcp, prob, num_splits=splits)
    dense = synth.make_decode_problem("splitsd", [3000, 900], 32, None, synth.KV_BF16, 2, 1, seed=32)
    _check_problem(dcp, dense, num_splits=splits)


def test_page_interleaved_and_single_shard(dcp):
    prob = synth.make_decode_problem("pagei", [5000, 700], 64, 512, synth.KV_BF16, 4, 64, mtp=2, seed=41)
    _check_problem(dcp, prob)
    dense = synth.make_decode_problem("pagei_d", [5000, 700], 64, None, synth.KV_FP8, 2, 64, seed=42)
    _check_problem(dcp, dense)
    one = synth.make_decode_problem("d1", [900], 128, 300, synth.KV_FP8, 1, 1, mtp=2, seed=43)
    _check_problem(dcp, one)


def test_empty_and_short_rows_fp8_many_heads(dcp):
    # rows with no slot at all, and FP8 rows whose shards hold one to three slots with
    # 128 heads (the short-KV FP8 case with > 32 heads that gave wrong LSE in a
    # third-party kernel, SGLang PR #42536 "FlashInfer workaround")
    prob = synth.make_decode_problem("short", [40, 40, 40, 40], 128, 24, synth.KV_FP8, 8, 1, seed=51)
    tk = prob.topk.clone()
    tk[0] = -1                       # empty row: every shard empty
    tk[1, 1:] = -1                   # a single slot
    tk[2, 3:] = -1                   # three slots
    tk[3, ::2] = -1                  # padding interleaved with ids
    prob.topk = tk
    mo, ml, fo, fl = _check_problem(dcp, prob)
    assert torch.all(fo[0] == 0) and torch.all(torch.isneginf(fl[0]))
    assert torch.all(mo[0] == 0) and torch.all(torch.isneginf(ml[0]))


def test_dense_zero_length_rows(dcp):
    prob = synth.make_decode_problem("zero", [200, 5, 1], 16, None, synth.KV_BF16, 4, 1, seed=52)
    prob.row_len = torch.tensor([200, 0, 1], dtype=torch.int32)
    _check_problem(dcp, prob)


def test_checked_mode_reports_bad_pages(dcp):
    prob = synth.make_decode_problem("bad", [300], 16, 64, synth.KV_BF16, 2, 1, seed=61).to(DEV)
    bt = prob.block_table.clone()
    bt[1, 0, 0] = prob.pool.shape[0] + 7     # out of range page
    prob.block_table = bt
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    fo, fl = run_fused(dcp, prob, checked=True, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & dcp.DCP_ERRBIT_PAGE_RANGE
    assert torch.isfinite(fo.float()).all() and not torch.isnan(fl).any()


# ----------------------------------------------------------------------------- full size
def _full_size(dcp, prob):
    """Every row of a full-size workload: fused and merged outputs against unsharded
    attention, and every shard's partials against the oracle restricted to that shard."""
    g = prob.to(DEV) if not prob.q.is_cuda else prob
    fo, fl = run_fused(dcp, g)
    po, pl, mo, ml = run_unfused(dcp, g)
    torch.cuda.synchronize()
    host = g.to("cpu")
    ro, rl = oracle.attention_problem(host)
    check_out(fo, ro, "fused out")
    check_lse(fl, rl, "fused lse")
    check_out(mo, ro, "merged out")
    check_lse(ml, rl, "merged lse")
    del ro, rl, fo, fl, mo, ml
    for s in range(prob.dcp):
        so, sl = oracle.attention_problem(host, shard=s)
        check_out(po[s], so, "partial out shard %d" % s)
        check_lse(pl[s], sl, "partial lse shard %d" % s)


def test_cfg3_full_size_all_rows(dcp):
    _full_size(dcp, synth.cfg3_sparse_topk2048_fp8(device=DEV))


def test_cfg5_full_size_all_rows(dcp):
    _full_size(dcp, synth.cfg5_dense_long(device=DEV))


@pytest.mark.parametrize("D,I", [(3, 1), (7, 5), (63, 1), (5, 1000), (64, 64), (2, 65536)])
def test_remap_large_ids_odd_rules(dcp, D, I):
    """Global slot ids up to 2^31 - 1 and divisors that are not powers of two: the owner rule
    (shard and local slot) must be bit-exact against the oracle everywhere in the id range."""
    g = torch.Generator().manual_seed(D * 1009 + I)
    rows, k = 19, 3000
    ids = torch.randint(0, 2**31 - 1, (rows, k), generator=g, dtype=torch.int64)
    ids[0, :8] = torch.tensor([0, 1, I - 1, I, I * D - 1, I * D, 2**31 - 2, 2**31 - 1])
    ids[1] = torch.arange(k, dtype=torch.int64) * 977 + (2**31 - 1 - 977 * k)
    ids = ids.to(torch.int32)
    loc, cnt = dcp.dcp_remap_topk(ids.to(DEV), D, I)
    rloc, rcnt = oracle.remap(ids, D, I)
    assert np.array_equal(cnt.cpu().numpy(), rcnt) and np.array_equal(loc.cpu().numpy(), rloc)
