"""Pins of the top-k producer oracle (oracle/topk.py) against things other than itself:
a brute-force search over subsets on tiny inputs, a hand-worked example with ties, padding
and NaN, the owner rule's enumeration against the pinned remap oracle, and the property the
DCP top-k merge rests on: merging every shard's own top-k gives the top-k of the unsharded
scores (LMDeploy PR #4952, Summary: DSA merges local candidates into the global top-k)."""
import itertools

import numpy as np
import pytest

import oracle
from oracle import topk as otk


def _dominates(sa, ta, sb, tb):
    """a ranks before b: higher score, or equal score and smaller id."""
    return sa > sb or (sa == sb and ta < tb)


def _brute(scores, ids, k):
    """The unique subset of min(k, valid) valid entries in which every member ranks before
    every valid non-member, found by trying all subsets."""
    valid = [i for i in range(len(ids))
             if ids[i] >= 0 and not np.isnan(scores[i]) and scores[i] != -np.inf]
    m = min(k, len(valid))
    found = []
    for sub in itertools.combinations(valid, m):
        rest = [j for j in valid if j not in sub]
        if all(_dominates(scores[a], ids[a], scores[b], ids[b]) for a in sub for b in rest):
            found.append(sorted(int(ids[a]) for a in sub))
    assert len(found) == 1
    return found[0]


def test_select_matches_brute_force_on_tiny_inputs():
    rng = np.random.default_rng(11)
    for trial in range(300):
        n = int(rng.integers(0, 8))
        scores = rng.choice(np.array([-1.0, 0.0, -0.0, 0.5, 2.0, np.nan, -np.inf, np.inf],
                                     dtype=np.float32), size=n)
        ids = rng.permutation(40)[:n] - (rng.random(n) < 0.15) * 100  # some padding ids
        k = int(rng.integers(1, 9))
        got, c = otk.select(scores, ids, k)
        want = _brute(scores, ids, k)
        assert c == len(want)
        assert list(got[:c]) == want and all(got[c:] == -1)


def test_select_hand_worked_example():
    # slots 0..7 with scores; 3 and 6 are not candidates (NaN, -inf), 7 is padding
    scores = np.array([3.0, 1.0, 3.0, np.nan, 2.0, 3.0, -np.inf, 9.0], dtype=np.float32)
    ids = np.array([0, 1, 2, 3, 4, 5, 6, -1])
    # three slots share the best score 3: all of them for k = 3
    assert list(otk.select(scores, ids, 3)[0]) == [0, 2, 5]
    # k = 2 keeps the two smaller ids of the tied three
    assert list(otk.select(scores, ids, 2)[0]) == [0, 2]
    # k = 4 adds the next score (2, slot 4); k = 8 takes every candidate and pads
    assert list(otk.select(scores, ids, 4)[0]) == [0, 2, 4, 5]
    got, c = otk.select(scores, ids, 8)
    assert c == 5 and list(got) == [0, 1, 2, 4, 5, -1, -1, -1]
    # -0 and +0 are the same score: the smaller id wins
    assert list(otk.select(np.array([-0.0, 0.0], np.float32), [7, 3], 1)[0]) == [3]
    assert list(otk.select(np.array([0.0, -0.0], np.float32), [7, 3], 1)[0]) == [3]
    # no candidate at all
    got, c = otk.select(np.array([np.nan, -np.inf], np.float32), [0, 1], 2)
    assert c == 0 and list(got) == [-1, -1]


@pytest.mark.parametrize("D,I", [(1, 1), (2, 1), (3, 1), (8, 1), (2, 64), (4, 4)])
def test_shard_slots_inverts_the_pinned_remap(D, I):
    """Local slot l of shard s is the l-th owned slot: the remap oracle (pinned by hand
    examples) sends each global slot t to exactly that local id."""
    L = 700
    g = np.arange(L, dtype=np.int32)[None, :]
    loc, cnt = oracle.remap(g, D, I)
    for s in range(D):
        slots = otk.shard_slots(int(cnt[s, 0]), D, I, s)
        owned = [t for t in range(L) if (t // I) % D == s]
        assert list(slots) == owned
        assert list(loc[s, 0, :cnt[s, 0]]) == list(range(cnt[s, 0]))


@pytest.mark.parametrize("D,I,k,ties", [(2, 1, 16, False), (3, 1, 40, True), (8, 1, 64, False),
                                        (4, 64, 100, True), (2, 4, 500, False), (1, 1, 32, True)])
def test_merge_of_shard_candidates_is_the_unsharded_topk(D, I, k, ties):
    rng = np.random.default_rng(D * 100 + k)
    rows, L = 6, 1200
    glob = rng.standard_normal((rows, L)).astype(np.float32)
    if ties:
        glob = (np.round(glob * 2) / 2).astype(np.float32)
    glob[rng.random((rows, L)) < 0.03] = -np.inf
    lengths = np.array([L, L - 1, 0, 5, 600, L - 333])
    # each shard's view of its own slots, as its index cache holds them
    stride = L // D + I + 1
    sc = np.full((D, rows, stride), np.nan, dtype=np.float32)
    ll = np.zeros((D, rows), dtype=np.int64)
    for s in range(D):
        for r in range(rows):
            n = oracle.count_owned(int(lengths[r]), D, I, s)
            g = otk.shard_slots(n, D, I, s)
            sc[s, r, :n] = glob[r, g]
            ll[s, r] = n
    cs, ci = otk.local_topk(sc, ll, k, D, I)
    top, cnt = otk.merge_topk(cs, ci, k)
    want, wcnt = otk.global_topk(glob, lengths, k)
    assert np.array_equal(top, want) and np.array_equal(cnt, wcnt)
    # every shard list holds its own slots only, ascending, with their scores
    for s in range(D):
        for r in range(rows):
            ids = ci[s, r][ci[s, r] >= 0]
            assert all((ids // I) % D == s) and np.all(np.diff(ids) > 0)
            assert np.array_equal(cs[s, r, :ids.size], glob[r, ids])


def test_local_topk_single_shard_argument():
    rng = np.random.default_rng(3)
    sc = rng.standard_normal((4, 3, 50)).astype(np.float32)
    ll = np.array([[50, 10, 0]] * 4)
    cs_all, ci_all = otk.local_topk(sc, ll, 8, 4, 1)
    cs2, ci2 = otk.local_topk(sc[2:3], ll[2:3], 8, 4, 1, shard=2)
    assert np.array_equal(ci_all[2:3], ci2) and np.array_equal(cs_all[2:3], cs2)
