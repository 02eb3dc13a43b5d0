"""CUDA-graph capture of the decode step (the pages' graph-mode decode; SGLang PR #42536,
Follow-ups; LMDeploy PR #4952 graph inputs): every entry point is asynchronous on its stream
and allocation-free (the workspace is sized and allocated before capture), so a whole step
records into one graph.  The remap of a row's top-k is
computed once per step and reused by every layer (the indices are the same for all layers
of a step).  Replays must reproduce eager execution bit for bit (the kernels are
deterministic for a fixed launch shape), and the replayed results must match the oracle
within the parity tolerances (top-k bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_lse, check_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dcp():
    import decode_context_sparse_gb300 as d
    from decode_context_sparse_gb300 import build
    build.build()
    d.load()
    return d


def _ws(dcp, g, idx, count, out, lse, n, fused):
    """The call's workspace, sized by mla_decode_workspace_size and allocated before capture."""
    a = dcp._decode_args(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq, g.sm_scale, idx, count,
                         None, None, out, lse, 0, False, None)
    return torch.zeros(dcp.mla_decode_workspace_size(a, n, fused) + 256, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("kind", ["fp8", "bf16"])
def test_fused_decode_graph_replay_matches_eager(dcp, kind):
    if kind == "fp8":
        g = synth.make_decode_problem("g", [5000, 3000], 128, 512, synth.KV_FP8, 4, 1, mtp=2, seed=31, device="cuda")
    else:
        g = synth.make_decode_problem("g", [6000, 2500, 900], 64, 512, synth.KV_BF16, 4, 64, seed=32, device="cuda")
    out = torch.empty((g.rows, g.heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((g.rows, g.heads), dtype=torch.float32, device="cuda")
    ws = _ws(dcp, g, g.topk, None, out, lse, g.dcp, True)

    def step():
        dcp.mla_decode_dcp_fused(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq, g.sm_scale,
                                 g.dcp, g.interleave, idx=g.topk, out=out, lse=lse, workspace=ws)

    step()  # eager first: one-time set-up stays out of the capture
    torch.cuda.synchronize()
    ref_o, ref_l = out.clone(), lse.clone()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        out.zero_()
        lse.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    ro, rl = oracle.attention_problem(g)
    check_out(out, ro, "graph replay out")
    check_lse(lse, rl, "graph replay lse")


def test_multi_layer_step_graph_with_shared_remap(dcp):
    """One step of L layers on the unfused path: remap once, then per layer the per-shard
    partials and the LSE merge, all in one graph; per-layer queries and caches differ."""
    L = 3
    probs = [synth.make_decode_problem("l%d" % i, [4000, 2000], 64, 256, synth.KV_BF16, 4, 1, seed=40 + i,
                                       device="cuda") for i in range(L)]
    g0 = probs[0]
    D, R, K, H = g0.dcp, g0.rows, g0.k, g0.heads
    topk = g0.topk  # the step's indices, shared by every layer
    loc = torch.empty((D, R, K), dtype=torch.int32, device="cuda")
    cnt = torch.empty((D, R), dtype=torch.int32, device="cuda")
    po = torch.empty((D, R, H, 512), dtype=torch.float32, device="cuda")
    pl = torch.empty((D, R, H), dtype=torch.float32, device="cuda")
    outs = [torch.empty((R, H, 512), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    lses = [torch.empty((R, H), dtype=torch.float32, device="cuda") for _ in range(L)]
    wss = [_ws(dcp, p, loc, cnt, po, pl, D, False) for p in probs]

    def step():
        dcp.dcp_remap_topk(topk, D, g0.interleave, local_idx=loc, count=cnt)
        for p, o, l, w in zip(probs, outs, lses, wss):
            # each layer keeps its own cache and tables; the sequence layout (and so the
            # remapped slots) is the same for every layer of the step
            dcp.mla_decode_partial_lse(p.q, p.pool, p.kv_dtype, p.block_table, p.row_seq, p.sm_scale,
                                       idx=loc, count=cnt, num_shards=D, out=po, lse=pl, workspace=w)
            dcp.dcp_lse_merge(po, pl, out=o, lse=l)

    step()
    torch.cuda.synchronize()
    ref = [(o.clone(), l.clone()) for o, l in zip(outs, lses)]
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for o, l in zip(outs, lses):
        o.zero_()
        l.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for (ro, rl), o, l in zip(ref, outs, lses):
        assert torch.equal(o, ro) and torch.equal(l, rl)
    for i, (p, o, l) in enumerate(zip(probs, outs, lses)):
        # layer i attends over its own cache with the step's shared top-k
        p.topk = topk
        wo, wl = oracle.attention_problem(p)
        check_out(o, wo, "graph replay layer %d out" % i)
        check_lse(l, wl, "graph replay layer %d lse" % i)


def test_topk_producer_and_decode_graph_replay(dcp):
    """A DSA decode step as one graph: every shard's top-k candidates from the indexer
    scores, their merge into the rows' global top-k, and the fused decode over that top-k.
    Replays reproduce eager execution bit for bit; the top-k holds k valid, increasing slot
    ids below each row's visible length."""
    g = synth.make_decode_problem("g", [5000, 3000], 128, 512, synth.KV_FP8, 4, 1, mtp=2, seed=33,
                                  device="cuda")
    D, R, k = g.dcp, g.rows, 512
    gen = torch.Generator(device="cuda").manual_seed(5)
    stride = synth.local_len_bound(int(g.row_len.max().item()), D, 1)
    sc = synth.index_scores(D, R, stride, gen)
    ll = dcp.dcp_local_lengths(g.row_len, D, 1)
    cs = torch.empty((D, R, k), dtype=torch.float32, device="cuda")
    ci = torch.empty((D, R, k), dtype=torch.int32, device="cuda")
    top = torch.empty((R, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((R,), dtype=torch.int32, device="cuda")
    out = torch.empty((R, g.heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((R, g.heads), dtype=torch.float32, device="cuda")
    ws = _ws(dcp, g, top, None, out, lse, D, True)

    def step():
        dcp.dcp_topk_local(sc, ll, k, D, 1, cand_score=cs, cand_idx=ci)
        dcp.dcp_topk_merge(cs, ci, k, topk=top, count=cnt)
        dcp.mla_decode_dcp_fused(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq, g.sm_scale,
                                 D, 1, idx=top, out=out, lse=lse, workspace=ws)

    step()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (top, cnt, out, lse)]
    t_h = top.cpu()
    assert bool((cnt.cpu() == k).all())
    assert bool((t_h[:, 1:] > t_h[:, :-1]).all()) and bool((t_h >= 0).all())
    assert bool((t_h < g.row_len.cpu().unsqueeze(1)).all())
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        for t in (top, cnt, out, lse):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for t, r in zip((top, cnt, out, lse), ref):
            assert torch.equal(t, r)
    from oracle import topk as otk
    ws_, wi_ = otk.local_topk(sc.cpu().numpy(), ll.cpu().numpy(), k, D, 1)
    wt, wc = otk.merge_topk(ws_, wi_, k)
    assert np.array_equal(top.cpu().numpy(), wt) and np.array_equal(cnt.cpu().numpy(), wc)
    g.topk = torch.from_numpy(wt).cuda()
    ro, rl = oracle.attention_problem(g)
    check_out(out, ro, "graph replay dsa step out")
    check_lse(lse, rl, "graph replay dsa step lse")
