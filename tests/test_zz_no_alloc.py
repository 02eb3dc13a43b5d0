"""The no-allocation fused decode entry point, through the C ABI.

mla_decode_dcp_fused_noalloc serves callers that cannot allocate device memory (a
plugin inside another engine that owns the memory pool, a serving loop with memory
reserved at start-up, a step recorded into a CUDA graph): its split-KV scratch is a
static array inside the library instead of a caller workspace.  Its results must match
the regular mla_decode_dcp_fused within the parity tolerances, on two calls in a row
(the second call sees the first call's leftovers in the shared array).  This file is
collected last so that a run stopping at the first failure has run everything else.
"""
import pytest
import torch

import synth
from parity import check_lse, check_out, to_np

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


def _compare_two_calls(dcp, g, **kw):
    ref_o, ref_l = dcp.mla_decode_dcp_fused(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                            g.sm_scale, g.dcp, g.interleave, **kw)
    torch.cuda.synchronize()
    ro, rl = to_np(ref_o), to_np(ref_l)
    out = torch.empty_like(ref_o)
    lse = torch.empty_like(ref_l)
    for _ in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        before = torch.cuda.memory_allocated()
        dcp.mla_decode_dcp_fused_noalloc(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                         g.sm_scale, g.dcp, g.interleave, out=out, lse=lse, **kw)
        assert torch.cuda.memory_allocated() == before
        torch.cuda.synchronize()
        check_out(out, ro, "noalloc out")
        check_lse(lse, rl, "noalloc lse")


def test_noalloc_sparse_fp8_split_kv_matches_fused(dcp):
    prob = synth.make_decode_problem("noalloc_sparse", [3000, 1800], 128, 1500, synth.KV_FP8, 8,
                                     1, mtp=3, seed=71).to(DEV)
    _compare_two_calls(dcp, prob, idx=prob.topk, num_splits=4)


def test_noalloc_dense_bf16_auto_splits_matches_fused(dcp):
    prob = synth.make_decode_problem("noalloc_dense", [5000, 700, 2100], 64, None, synth.KV_BF16,
                                     4, 1, seed=72).to(DEV)
    _compare_two_calls(dcp, prob, kv_len=prob.row_len, max_kv_len=5000)


def test_noalloc_rejects_scratch_beyond_the_limit(dcp):
    prob = synth.make_decode_problem("noalloc_big", [300] * 64, 128, 256, synth.KV_BF16, 2, 1,
                                     seed=73).to(DEV)
    out = torch.empty((prob.rows, 128, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((prob.rows, 128), dtype=torch.float32, device=DEV)
    with pytest.raises(dcp.DcpError) as e:   # 64 rows x 64 splits x 128 heads x 2 KB >> 16 MiB
        dcp.mla_decode_dcp_fused_noalloc(prob.q, prob.pool, prob.kv_dtype, prob.block_table,
                                         prob.row_seq, prob.sm_scale, prob.dcp, prob.interleave,
                                         out=out, lse=lse, idx=prob.topk, num_splits=64)
    assert e.value.status == dcp.DCP_ERR_WORKSPACE


def test_noalloc_auto_splits_fit_the_static_scratch(dcp):
    """A short dense call with long contexts: the library's own split choice would need more
    than the static scratch; with num_splits = 0 it lowers the split count instead of
    refusing the call."""
    prob = synth.make_decode_problem("noalloc_long", [65536, 60000], 128, None, synth.KV_BF16, 2,
                                     1, seed=74).to(DEV)
    _compare_two_calls(dcp, prob, kv_len=prob.row_len, max_kv_len=65536)
