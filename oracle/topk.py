"""The oracle of the DSA top-k producer under DCP -- TEST INFRASTRUCTURE ONLY.

Plain numpy statement of how the sparse-attention (DSA) top-k slot set of a decode row is
produced when the index cache is split across D context-parallel shards: every shard keeps
its own best k candidates among its local slots, and the D candidate lists are merged into
the row's global top-k.

Passages:
  * LMDeploy PR #4952 "support decode context parallelism for PyTorch MLA", Summary: for
    decode, DSA merges the local candidates into the global top-k; file list: the DCP top-k
    kernel packs the distributed candidates and merges them;
  * SGLang PR #36990, item 2 (split index cache): each indexer layer then merges the local
    top-k candidates of the ranks.

Readings where the pages are silent (each is also stated in the C header of the library):
  * a slot is a candidate unless its score is NaN or -inf, or its id is negative (padding);
  * candidates are ranked by score, higher first (-0 and +0 are equal), equal scores by
    the smaller global slot id; the first k are selected;
  * a selected set is reported as its global slot ids in increasing order, then -1; a
    shard's candidate list carries each selected slot's score beside its id (tail -inf);
  * a shard's local slot l is the l-th slot, in increasing global order, that the owner
    rule gives the shard (the layout of the shard's KV and index caches).

Only a library sort (numpy lexsort / sort) serves as a step; nothing is blocked or fused.
Pinned by tests/test_oracle_topk_pins.py (brute-force subset search on tiny inputs, a
hand-worked example, and sharded == unsharded selection).
"""
from __future__ import annotations

import numpy as np


def select(scores, ids, k: int):
    """Top-k of one candidate set: (selected ids ascending then -1 [k] int64, count).

    scores: fp32 values; ids: int global slot ids (negative = padding)."""
    s = np.asarray(scores, dtype=np.float32).astype(np.float64).reshape(-1)
    t = np.asarray(ids, dtype=np.int64).reshape(-1)
    valid = (t >= 0) & ~np.isnan(s) & (s != -np.inf)
    s, t = s[valid], t[valid]
    # primary key: the score, descending (negated; -(-0.0) == -(0.0) compare equal);
    # secondary key: the slot id, ascending
    order = np.lexsort((t, -s))
    chosen = np.sort(t[order[:k]])
    out = np.full(k, -1, dtype=np.int64)
    out[:chosen.size] = chosen
    return out, int(chosen.size)


def shard_slots(n: int, dcp: int, interleave: int, shard: int) -> np.ndarray:
    """Global slot ids of local slots 0..n-1 of a shard: the first n slots t = 0, 1, 2, ...
    whose owner (t // I) % D is the shard, in increasing order (enumerated, not inverted)."""
    if n <= 0:
        return np.zeros(0, dtype=np.int64)
    span = (n // interleave + 2) * interleave * dcp
    t = np.arange(span, dtype=np.int64)
    owned = t[(t // interleave) % dcp == shard]
    assert owned.size >= n
    return owned[:n]


def local_topk(scores, local_len, k: int, dcp: int, interleave: int, shard: int = -1):
    """Each shard's candidate list.

    scores [n_in, rows, stride] fp32 (n_in = dcp for shard = -1, else 1), local_len
    [n_in, rows] int -> (cand_score [n_in, rows, k] fp32, cand_idx [n_in, rows, k] int32)."""
    sc = np.asarray(scores, dtype=np.float32)
    ll = np.asarray(local_len, dtype=np.int64)
    n_in, rows, stride = sc.shape
    cs = np.full((n_in, rows, k), -np.inf, dtype=np.float32)
    ci = np.full((n_in, rows, k), -1, dtype=np.int32)
    for o in range(n_in):
        s = o if shard < 0 else shard
        for r in range(rows):
            n = int(min(max(ll[o, r], 0), stride))
            g = shard_slots(n, dcp, interleave, s)
            sel, c = select(sc[o, r, :n], g, k)
            pos = np.searchsorted(g, sel[:c])  # local slot of each selected global slot
            ci[o, r, :c] = sel[:c]
            cs[o, r, :c] = sc[o, r, pos]
    return cs, ci


def merge_topk(cand_score, cand_idx, k: int):
    """Global top-k of the D shards' candidates [D, rows, k_in] ->
    (topk [rows, k] int32 ascending then -1, count [rows] int32)."""
    cs = np.asarray(cand_score, dtype=np.float32)
    ci = np.asarray(cand_idx, dtype=np.int64)
    D, rows, _ = cs.shape
    top = np.full((rows, k), -1, dtype=np.int32)
    cnt = np.zeros(rows, dtype=np.int32)
    for r in range(rows):
        sel, c = select(cs[:, r, :].reshape(-1), ci[:, r, :].reshape(-1), k)
        top[r] = sel
        cnt[r] = c
    return top, cnt


def global_topk(scores, lengths, k: int):
    """Unsharded top-k: scores [rows, L] over global slots 0..L-1, row r sees slots
    t < lengths[r] -> (topk [rows, k] int32, count [rows] int32)."""
    sc = np.asarray(scores, dtype=np.float32)
    rows, L = sc.shape
    top = np.full((rows, k), -1, dtype=np.int32)
    cnt = np.zeros(rows, dtype=np.int32)
    for r in range(rows):
        n = int(min(max(int(lengths[r]), 0), L))
        sel, c = select(sc[r, :n], np.arange(n), k)
        top[r] = sel
        cnt[r] = c
    return top, cnt
