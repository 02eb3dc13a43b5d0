"""Shared helpers of the GPU parity tests: tolerances, comparisons against the oracle and
the two GPU pipelines (unfused remap -> partial -> merge, and the fused launch).

Tolerance (floating point), both bounds at once:
  * max abs error <= 1e-2 over every output element, and
  * max rel error <= 2e-2 over the elements whose reference has |ref| >= 0.5 (below that
    a relative error says nothing; the abs bound covers them);
  * an output stored in BF16 (merged, fused and prefill outputs) may exceed the abs bound
    by half a BF16 ulp of the reference where |ref| >= 4: rounding a value in [4, 8) to
    BF16 alone moves it by up to 2^-6 = 0.0156 > 1e-2.  Outputs kept in fp32 (per-shard
    partials) get no such allowance.
  * LSE: max abs error <= 1e-3 over finite entries; -inf must match exactly.
Remap, counts and every integer result are compared bit for bit.

Every check records the errors it reached (max abs, max abs where |ref| < 0.5, max rel
where |ref| >= 0.5, LSE error); tests/conftest.py prints them at the end of the run.
"""
import os

import numpy as np
import torch

OUT_ATOL = 1e-2
OUT_RTOL = 2e-2
REL_FLOOR = 0.5
BF16_ALLOWANCE_FLOOR = 4.0
LSE_ATOL = 1e-3

# (test id, what, stored, max abs, max abs |ref|<0.5, max rel |ref|>=0.5, lse err or None)
RECORD = []


def _test_id():
    t = os.environ.get("PYTEST_CURRENT_TEST", "")
    return t.split(" (")[0]


def to_np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def bf16_half_ulp(ref):
    """Half a BF16 ulp of |ref| (BF16 keeps 8 significant bits): 2^(floor(log2|ref|) - 8)."""
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def out_errors(got, ref, stored):
    """(err array, allowed abs array, max abs, max abs |ref|<0.5, max rel |ref|>=0.5)."""
    g, r = to_np(got), np.asarray(ref, np.float64)
    err = np.abs(g - r)
    allowed = np.full(r.shape, OUT_ATOL)
    if stored == "bf16":
        big = np.abs(r) >= BF16_ALLOWANCE_FLOOR
        allowed = np.where(big, OUT_ATOL + bf16_half_ulp(r), allowed)
    small = np.abs(r) < REL_FLOOR
    rel = np.where(small, 0.0, err / np.where(small, 1.0, np.abs(r)))
    return (err, allowed, float(err.max(initial=0.0)), float(err[small].max(initial=0.0)),
            float(rel.max(initial=0.0)))


def check_out(got, ref, what="", stored=None):
    """Output element check; stored = 'bf16' or 'fp32' (default: the dtype of `got`)."""
    if stored is None:
        stored = "bf16" if isinstance(got, torch.Tensor) and got.dtype == torch.bfloat16 else "fp32"
    g = to_np(got)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.isfinite(g).all(), "%s: non-finite output" % what
    err, allowed, mabs, msmall, mrel = out_errors(got, ref, stored)
    RECORD.append((_test_id(), what, stored, mabs, msmall, mrel, None))
    over = (err - allowed).max(initial=-1.0)
    assert over <= 0.0, "%s (%s): abs error %.4g exceeds its bound by %.3g" % (what, stored, mabs, over)
    assert mrel <= OUT_RTOL, "%s (%s): rel error %.4g on |ref| >= 0.5" % (what, stored, mrel)
    return mabs, mrel


def check_lse(got, ref, what=""):
    g, r = to_np(got), np.asarray(ref, np.float64)
    assert g.shape == r.shape
    ninf = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), ninf), "%s: -inf pattern differs" % what
    assert not np.isnan(g).any(), "%s: NaN lse" % what
    fin = ~ninf
    err = float(np.abs(g[fin] - r[fin]).max(initial=0.0))
    RECORD.append((_test_id(), what, "lse", None, None, None, err))
    assert err <= LSE_ATOL, "%s: max lse err %.3g" % (what, err)
    return err


def summary_lines():
    """One line per test: its worst output errors and LSE error over all its checks."""
    per = {}
    for tid, what, stored, mabs, msmall, mrel, lerr in RECORD:
        d = per.setdefault(tid, {"abs_bf16": 0.0, "abs_fp32": 0.0, "small": 0.0, "rel": 0.0,
                                 "lse": 0.0, "n": 0})
        d["n"] += 1
        if lerr is not None:
            d["lse"] = max(d["lse"], lerr)
            continue
        d["abs_" + stored] = max(d["abs_" + stored], mabs)
        d["small"] = max(d["small"], msmall)
        d["rel"] = max(d["rel"], mrel)
    out = ["%-80s %6s %10s %10s %10s %10s %10s" % ("test", "checks", "abs bf16", "abs fp32",
                                                   "abs<0.5", "rel>=0.5", "lse")]
    for tid, d in per.items():
        out.append("%-80s %6d %10.3g %10.3g %10.3g %10.3g %10.3g" % (
            tid[-80:], d["n"], d["abs_bf16"], d["abs_fp32"], d["small"], d["rel"], d["lse"]))
    return out


def run_unfused(dcp, g, num_splits=0, checked=False, err_flag=None):
    """remap (sparse) or local lengths (dense) -> per-shard partials -> LSE merge."""
    D, I = g.dcp, g.interleave
    common = dict(num_shards=D, num_splits=num_splits, checked=checked, err_flag=err_flag)
    if g.topk is not None:
        loc, cnt = dcp.dcp_remap_topk(g.topk, D, I)
        po, pl = dcp.mla_decode_partial_lse(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                            g.sm_scale, idx=loc, count=cnt, **common)
    else:
        ll = dcp.dcp_local_lengths(g.row_len, D, I)
        po, pl = dcp.mla_decode_partial_lse(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                            g.sm_scale, kv_len=ll,
                                            max_kv_len=int(g.row_len.max().item()), **common)
    mo, ml = dcp.dcp_lse_merge(po, pl)
    return po, pl, mo, ml


def run_fused(dcp, g, num_splits=0, checked=False, err_flag=None):
    if g.topk is not None:
        kw = dict(idx=g.topk)
    else:
        kw = dict(kv_len=g.row_len, max_kv_len=int(g.row_len.max().item()))
    return dcp.mla_decode_dcp_fused(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                    g.sm_scale, g.dcp, g.interleave, num_splits=num_splits,
                                    checked=checked, err_flag=err_flag, **kw)
