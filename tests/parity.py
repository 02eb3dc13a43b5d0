"""Shared helpers of the GPU parity tests: tolerances, comparisons against the oracle and
the two GPU pipelines (unfused remap -> partial -> merge, and the fused launch)."""
import numpy as np
import torch

# Tolerances of the path (floating point): an output element passes when its error is
# within 1e-2 absolute or 2e-2 relative to the reference, i.e. err <= max(1e-2, 2e-2*|ref|)
# (abs bound for small values, rel bound for large ones: BF16 storage alone rounds a value
# in [4, 8) by up to 0.0156).  LSE max abs error <= 1e-3 on finite entries, -inf must match
# exactly.  Remap is bit-exact.
OUT_ATOL = 1e-2
OUT_RTOL = 2e-2
REL_FLOOR = 0.5
LSE_ATOL = 1e-3


def to_np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def check_out(got, ref, what=""):
    g, r = to_np(got), np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.isfinite(g).all(), "%s: non-finite output" % what
    err = np.abs(g - r)
    allowed = np.maximum(OUT_ATOL, OUT_RTOL * np.abs(r))
    worst = (err / allowed).max(initial=0.0)
    small = np.abs(r) < REL_FLOOR
    assert worst <= 1.0, "%s: error %.3g of allowed (max abs err %.3g on |ref|<0.5: %.3g)" % (
        what, worst, err.max(), err[small].max(initial=0.0))
    return float(err.max(initial=0.0))


def check_lse(got, ref, what=""):
    g, r = to_np(got), np.asarray(ref, np.float64)
    assert g.shape == r.shape
    ninf = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), ninf), "%s: -inf pattern differs" % what
    assert not np.isnan(g).any(), "%s: NaN lse" % what
    fin = ~ninf
    err = np.abs(g[fin] - r[fin]).max(initial=0.0)
    assert err <= LSE_ATOL, "%s: max lse err %.3g" % (what, err)
    return float(err)


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
                                            g.sm_scale, kv_len=ll, **common)
    mo, ml = dcp.dcp_lse_merge(po, pl)
    return po, pl, mo, ml


def run_fused(dcp, g, num_splits=0, checked=False, err_flag=None):
    kw = dict(idx=g.topk) if g.topk is not None else dict(kv_len=g.row_len)
    return dcp.mla_decode_dcp_fused(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                    g.sm_scale, g.dcp, g.interleave, num_splits=num_splits,
                                    checked=checked, err_flag=err_flag, **kw)
