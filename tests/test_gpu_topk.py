"""Parity of the DSA top-k producer kernels (dcp_topk_local, dcp_topk_merge) with the
oracle (oracle/topk.py): bit-exact candidate ids and scores, and bit-exact global top-k,
through the C ABI.  Covers ties, NaN / -inf / padding, empty and short lists, lists longer
than the shared-memory staging (the L2 re-read path), k up to DCP_MAX_TOPK, and the full
top-k 2048 decode batch (8 shards x 384 rows x 16384 local slots)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import topk as otk
import synth

pytestmark = pytest.mark.gpu
dev = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def dcp():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import decode_context_sparse_gb300 as m
    from decode_context_sparse_gb300 import build
    build.build()
    m.load()
    return m


def _local_lens(row_len, D, I):
    return np.array([[oracle.count_owned(int(L), D, I, s) for L in row_len] for s in range(D)],
                    dtype=np.int32)


def _scores(D, R, stride, seed, ties=False, masked=0.0, nan=0.0):
    g = torch.Generator().manual_seed(seed)
    s = synth.index_scores(D, R, stride, g, ties=ties, masked=masked)
    if nan > 0:
        s = torch.where(torch.rand(s.shape, generator=g) < nan, torch.full_like(s, float("nan")), s)
    return s


def _check_local(dcp, sc, ll, k, D, I, shard=-1):
    cs, ci = dcp.dcp_topk_local(sc.to(dev), torch.from_numpy(ll).to(dev), k, D, I, shard=shard)
    torch.cuda.synchronize()
    ws, wi = otk.local_topk(sc.numpy(), ll, k, D, I, shard=shard)
    assert np.array_equal(ci.cpu().numpy(), wi)
    assert np.array_equal(cs.cpu().numpy().view(np.int32), ws.view(np.int32))
    return cs, ci


@pytest.mark.parametrize("D,I,k,stride,ties", [
    (2, 1, 16, 300, False), (3, 1, 40, 257, True), (8, 1, 64, 1000, False),
    (4, 64, 100, 700, True), (1, 1, 1, 50, False), (2, 4, 2048, 5000, False),
    (8, 1, 300, 16384, True), (8, 1, 2048, 16384, True), (2, 1, 2048, 16384, False)])
def test_local_candidates_match_oracle(dcp, D, I, k, stride, ties):
    R = 7
    sc = _scores(D, R, stride, seed=D * 7 + k, ties=ties, masked=0.02, nan=0.01)
    rng = np.random.default_rng(k)
    ll = rng.integers(0, stride + 1, size=(D, R)).astype(np.int32)
    ll[:, 0] = 0                       # empty list
    ll[:, 1] = stride                  # the whole row
    ll[:, 2] = min(k, stride) // 2     # fewer slots than k
    ll[:, 3] = stride + 5              # clamped to the stride
    _check_local(dcp, sc, ll, k, D, I)


def test_local_single_shard_argument(dcp):
    D, R, stride, k = 4, 5, 900, 33
    sc = _scores(D, R, stride, seed=5)
    ll = np.full((D, R), 850, dtype=np.int32)
    for s in (0, 3):
        _check_local(dcp, sc[s:s + 1].contiguous(), ll[s:s + 1], k, D, 1, shard=s)


def test_local_lists_longer_than_the_staging(dcp):
    D, R, stride, k = 2, 3, 40000, 777
    sc = _scores(D, R, stride, seed=9, ties=True)
    ll = np.array([[40000, 16385, 30000], [16384, 39999, 0]], dtype=np.int32)
    _check_local(dcp, sc, ll, k, D, 1)


def test_all_equal_scores_keep_the_smallest_slots(dcp):
    D, R, stride, k = 4, 2, 3000, 500
    sc = torch.zeros((D, R, stride))
    sc[:, 1, ::2] = -0.0  # -0 ranks as +0
    ll = np.full((D, R), 2900, dtype=np.int32)
    cs, ci = _check_local(dcp, sc, ll, k, D, 1)
    top, cnt = dcp.dcp_topk_merge(cs, ci, k)
    torch.cuda.synchronize()
    assert np.array_equal(top.cpu().numpy(), np.tile(np.arange(k, dtype=np.int32), (R, 1)))
    assert list(cnt.cpu().numpy()) == [k, k]


def _random_candidates(D, R, kin, seed, pad=0.1):
    """Candidate lists with distinct ids per row (drawn without replacement), scores with
    ties, -inf and NaN, and -1 padding."""
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(D * kin * 3)[:D * kin].reshape(D, kin) for _ in range(R)], 1)
    sc = np.round(rng.standard_normal((D, R, kin)) * 3) / 3
    sc = sc.astype(np.float32)
    sc[rng.random(sc.shape) < 0.03] = -np.inf
    sc[rng.random(sc.shape) < 0.02] = np.nan
    ids[rng.random(ids.shape) < pad] = -1
    return torch.from_numpy(sc), torch.from_numpy(ids.astype(np.int32))


@pytest.mark.parametrize("D,kin,k", [(2, 50, 64), (3, 128, 128), (8, 2048, 2048), (5, 100, 1),
                                     (8, 4096, 4096), (1, 300, 299)])
def test_merge_matches_oracle(dcp, D, kin, k):
    R = 6
    cs, ci = _random_candidates(D, R, kin, seed=D * 31 + k)
    top, cnt = dcp.dcp_topk_merge(cs.to(dev), ci.to(dev), k)
    torch.cuda.synchronize()
    wt, wc = otk.merge_topk(cs.numpy(), ci.numpy(), k)
    assert np.array_equal(top.cpu().numpy(), wt)
    assert np.array_equal(cnt.cpu().numpy(), wc)


@pytest.mark.parametrize("D,kin,k", [(2, 50, 64), (8, 2048, 2048), (64, 20, 300), (1, 300, 100),
                                     (5, 100, 7), (8, 4096, 4096)])
def test_merge_of_ascending_lists_matches_oracle(dcp, D, kin, k):
    """Lists in increasing id order, as dcp_topk_local writes them (the merge then places
    every id by rank; other lists are sorted)."""
    R = 6
    cs, ci = _random_candidates(D, R, kin, seed=D * 17 + k)
    order = np.argsort(ci.numpy(), axis=2, kind="stable")
    ci = torch.from_numpy(np.take_along_axis(ci.numpy(), order, 2).copy())
    cs = torch.from_numpy(np.take_along_axis(cs.numpy(), order, 2).copy())
    top, cnt = dcp.dcp_topk_merge(cs.to(dev), ci.to(dev), k)
    torch.cuda.synchronize()
    wt, wc = otk.merge_topk(cs.numpy(), ci.numpy(), k)
    assert np.array_equal(top.cpu().numpy(), wt)
    assert np.array_equal(cnt.cpu().numpy(), wc)


def test_merge_max_topk(dcp):
    k = 16384
    cs, ci = _random_candidates(2, 2, k, seed=77, pad=0.3)
    top, cnt = dcp.dcp_topk_merge(cs.to(dev), ci.to(dev), k)
    torch.cuda.synchronize()
    wt, wc = otk.merge_topk(cs.numpy(), ci.numpy(), k)
    assert np.array_equal(top.cpu().numpy(), wt) and np.array_equal(cnt.cpu().numpy(), wc)


def _scatter_global(scores, row_len, D, I):
    """Global score array [R, Lmax] of the shards' local scores (oracle enumeration)."""
    Dn, R, stride = scores.shape
    L = int(max(row_len))
    glob = np.full((R, L), np.nan, dtype=np.float32)
    for s in range(D):
        g = otk.shard_slots(min(stride, oracle.count_owned(L, D, I, s)), D, I, s)
        for r in range(R):
            n = oracle.count_owned(int(row_len[r]), D, I, s)
            glob[r, g[:n]] = scores[s, r, :n]
    return glob


@pytest.mark.parametrize("D,I,k", [(2, 1, 256), (4, 64, 512), (8, 1, 2048)])
def test_local_then_merge_is_the_unsharded_topk(dcp, D, I, k):
    R = 5
    row_len = np.array([20000, 19999, 3000, 1, 0])
    stride = synth.local_len_bound(int(row_len.max()), D, I)
    sc = _scores(D, R, stride, seed=k + D, ties=(D == 4))
    ll = _local_lens(row_len, D, I)
    cs, ci = dcp.dcp_topk_local(sc.to(dev), torch.from_numpy(ll).to(dev), k, D, I)
    top, cnt = dcp.dcp_topk_merge(cs, ci, k)
    torch.cuda.synchronize()
    glob = _scatter_global(sc.numpy(), row_len, D, I)
    wt, wc = otk.global_topk(glob, row_len, k)
    assert np.array_equal(top.cpu().numpy(), wt) and np.array_equal(cnt.cpu().numpy(), wc)


def test_merge_padding_with_the_highest_scores(dcp):
    """Padding entries (id -1) carrying the largest scores: a selection by score alone would
    take them, so the merge must select again with the ids; rows without such padding keep
    the score-only selection.  Both against the oracle."""
    D, R, kin, k = 8, 4, 2048, 2048
    rng = np.random.default_rng(11)
    ids = np.stack([rng.permutation(D * kin * 2)[:D * kin].reshape(D, kin) for _ in range(R)], 1)
    ids = np.sort(ids, axis=2).astype(np.int32)
    sc = rng.standard_normal((D, R, kin)).astype(np.float32)
    pad = rng.random(ids.shape) < 0.05
    pad[:, 1, :] = False  # row 1: no padding
    ids[pad] = -1
    sc[pad] = 50.0        # above every real score
    sc[:, 2, :][pad[:, 2, :]] = -np.inf  # row 2: padding as the local lists write it
    top, cnt = dcp.dcp_topk_merge(torch.from_numpy(sc).to(dev), torch.from_numpy(ids).to(dev), k)
    torch.cuda.synchronize()
    wt, wc = otk.merge_topk(sc, ids, k)
    assert np.array_equal(top.cpu().numpy(), wt) and np.array_equal(cnt.cpu().numpy(), wc)


def test_infinities_and_signed_zeros(dcp):
    """+inf ranks above every finite score, -inf and NaN are never candidates, -0 ranks as
    +0 (ties by slot), through both kernels; aligned rows of 6000 and unaligned ones of
    1001 take the two staging paths."""
    for stride in (6000, 1001):
        D, R, k = 4, 4, 700
        rng = np.random.default_rng(stride)
        sc = rng.standard_normal((D, R, stride)).astype(np.float32)
        u = rng.random(sc.shape)
        sc[u < 0.01] = np.inf
        sc[(u >= 0.01) & (u < 0.02)] = -np.inf
        sc[(u >= 0.02) & (u < 0.03)] = np.nan
        sc[(u >= 0.03) & (u < 0.06)] = 0.0
        sc[(u >= 0.06) & (u < 0.09)] = -0.0
        sc[:, 3, :] = np.where(rng.random((D, stride)) < 0.5, np.float32(-0.0), np.float32(0.0))
        ll = np.full((D, R), stride, dtype=np.int32)
        ll[:, 1] = stride - 3
        cs, ci = _check_local(dcp, torch.from_numpy(sc), ll, k, D, 1)
        top, cnt = dcp.dcp_topk_merge(cs, ci, k)
        torch.cuda.synchronize()
        wt, wc = otk.merge_topk(cs.cpu().numpy(), ci.cpu().numpy(), k)
        assert np.array_equal(top.cpu().numpy(), wt) and np.array_equal(cnt.cpu().numpy(), wc)


def test_full_size_topk2048_batch(dcp):
    """The top-k 2048 decode batch: 8 shards x 384 rows x 16384 local slots, k = 2048, in the
    launch configuration the bench times.  Every row's global top-k is compared with the
    oracle's unsharded top-k; the candidate lists of a sample of (shard, row) pairs with the
    oracle's lists."""
    p = synth.topk_producer_topk2048(device="cpu")
    D, I, k = p.dcp, p.interleave, p.k
    row_len = p.row_len.numpy()
    ll = _local_lens(row_len, D, I)
    cs, ci = dcp.dcp_topk_local(p.scores.to(dev), torch.from_numpy(ll).to(dev), k, D, I)
    top, cnt = dcp.dcp_topk_merge(cs, ci, k)
    torch.cuda.synchronize()
    sc = p.scores.numpy()
    glob = _scatter_global(sc, row_len, D, I)
    wt, wc = otk.global_topk(glob, row_len, k)
    assert np.array_equal(top.cpu().numpy(), wt) and np.array_equal(cnt.cpu().numpy(), wc)
    rng = np.random.default_rng(0)
    csh, cih = cs.cpu().numpy(), ci.cpu().numpy()
    for _ in range(12):
        s, r = int(rng.integers(D)), int(rng.integers(p.scores.shape[1]))
        ws, wi = otk.local_topk(sc[s:s + 1, r:r + 1], ll[s:s + 1, r:r + 1], k, D, I, shard=s)
        assert np.array_equal(cih[s, r], wi[0, 0])
        assert np.array_equal(csh[s, r].view(np.int32), ws[0, 0].view(np.int32))

