"""Parity of the chunked-prefill composition (mla_prefill_chunk_dcp: per-shard dense
partials over the cached prefix, per-shard sparse partials over the chunk slots each row
sees, LSE merge) with the oracle's dense attention over each row's visible range, through
the C ABI; and of the single-launch alternative (fused dense decode with the same lengths).
Covers the tensor-core path (128 and 64 heads) and the CUDA-core path (32 heads), BF16 and
FP8 pools, both owner rules, an empty prefix, and the bench's prefill chunk on every row."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_lse, check_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dcp():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import decode_context_sparse_gb300 as m
    from decode_context_sparse_gb300 import build
    build.build()
    m.load()
    return m


def _run(dcp, g, chunk):
    prefix, ids = synth.prefill_chunk_inputs(g, chunk)
    return dcp.mla_prefill_chunk_dcp(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq, g.sm_scale,
                                     g.dcp, g.interleave, prefix_len=prefix, chunk_idx=ids,
                                     max_prefix_len=int(prefix.max().item()))


@pytest.mark.parametrize("heads,kvt,D,I,prefixes,chunk", [
    (128, synth.KV_FP8, 8, 1, [3000, 1000], 48),
    (128, synth.KV_BF16, 4, 64, [2500, 700, 0], 40),
    (64, synth.KV_FP8, 2, 1, [0, 500], 33),
    (32, synth.KV_BF16, 4, 64, [2500, 700], 40),
])
def test_prefill_chunk_matches_oracle(dcp, heads, kvt, D, I, prefixes, chunk):
    prob = synth.prefill_chunk_problem("t", prefixes, chunk, heads, kvt, D, I, seed=heads + D)
    g = prob.to("cuda")
    out, lse = _run(dcp, g, chunk)
    fo, fl = dcp.mla_decode_dcp_fused(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq, g.sm_scale,
                                      D, I, kv_len=g.row_len, max_kv_len=int(prob.row_len.max()))
    torch.cuda.synchronize()
    ro, rl = oracle.attention_problem(prob)
    check_out(out, ro, "prefill chunk")
    check_lse(lse, rl, "prefill chunk")
    check_out(fo, ro, "fused dense")
    check_lse(fl, rl, "fused dense")


def test_bench_prefill_chunk_all_rows(dcp):
    """The bench's chunk (2 sequences x 64 chunk tokens after a 16384-token prefix, 128 heads,
    FP8, D = 8), in the launch configuration the bench times; every row checked."""
    prob = synth.prefill_chunk_fp8(device="cpu")
    g = prob.to("cuda")
    out, lse = _run(dcp, g, 64)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_problem(prob)
    check_out(out, ro, "bench prefill chunk")
    check_lse(lse, rl, "bench prefill chunk")
