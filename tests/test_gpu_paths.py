"""Both decode kernels through the C ABI: the tensor-core kernel (taken for 48..128 heads)
and the CUDA-core kernel (taken for fewer heads, or for any head count when a call sets
kernel_path = DCP_PATH_CUDA_CORES) agree with the oracle on the same inputs, including rows
cut across CTA pairs."""
import pytest
import torch

import oracle
import synth
from parity import check_lse, check_out, run_fused

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


@pytest.mark.parametrize("path", ["cuda_cores", "auto"])
@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8])
def test_both_paths_match_oracle(dcp, path, kv):
    kp = dcp.DCP_PATH_CUDA_CORES if path == "cuda_cores" else dcp.DCP_PATH_AUTO
    prob = synth.make_decode_problem("paths", [3100, 1700], 128, 1000, kv, 4, 1, mtp=3, seed=81)
    g = prob.to(DEV)
    D = g.dcp
    loc, cnt = dcp.dcp_remap_topk(g.topk, D, g.interleave)
    po, pl = dcp.mla_decode_partial_lse(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                        g.sm_scale, idx=loc, count=cnt, num_shards=D,
                                        kernel_path=kp)
    mo, ml = dcp.dcp_lse_merge(po, pl)
    fo, fl = dcp.mla_decode_dcp_fused(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                      g.sm_scale, D, g.interleave, idx=g.topk, kernel_path=kp)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_problem(prob)
    check_out(fo, ro, path + " fused out")
    check_lse(fl, rl, path + " fused lse")
    check_out(mo, ro, path + " merged out")
    check_lse(ml, rl, path + " merged lse")
    so, sl = oracle.attention_problem(prob, shard=2)
    check_out(po[2], so, path + " partial out")
    check_lse(pl[2], sl, path + " partial lse")


@pytest.mark.parametrize("heads", [128, 48])
def test_partial_every_shard_and_output_alignment(dcp, heads):
    """The tensor-core partial decode writes a finished unit's rows by tiled stores: every
    shard's output and LSE match the oracle, also with 48 heads (a head group's box partly
    outside the tensor).  An output that is not 16-B aligned is refused."""
    prob = synth.make_decode_problem("align", [2600, 900], heads, 700, synth.KV_FP8, 4, 1, mtp=2,
                                     seed=83)
    g = prob.to(DEV)
    D = g.dcp
    R = g.q.shape[0]
    loc, cnt = dcp.dcp_remap_topk(g.topk, D, g.interleave)
    args = (g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq, g.sm_scale)
    po, pl = dcp.mla_decode_partial_lse(*args, idx=loc, count=cnt, num_shards=D)
    torch.cuda.synchronize()
    for s in range(D):
        so, sl = oracle.attention_problem(prob, shard=s)
        check_out(po[s], so, "partial out shard %d" % s)
        check_lse(pl[s], sl, "partial lse shard %d" % s)
    buf = torch.zeros(D * R * heads * 512 + 1, dtype=torch.float32, device=DEV)
    off = buf[1:].view(D, R, heads, 512)
    with pytest.raises(dcp.DcpError):
        dcp.mla_decode_partial_lse(*args, idx=loc, count=cnt, num_shards=D, out=off)


def test_tc_timeout_flag_stays_clear(dcp):
    prob = synth.make_decode_problem("flag", [5000], 128, 2048, synth.KV_FP8, 8, 1, mtp=2, seed=82).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_fused(dcp, prob, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == 0


@pytest.mark.parametrize("path", ["cuda_cores", "auto"])
def test_second_device_after_first(dcp, path):
    """Per-device launch set-up: a decode on cuda:1 after one on cuda:0 in the same process
    (the shared-memory limit of each kernel and the SM count are per device).  Needs two
    visible GPUs."""
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    kp = dcp.DCP_PATH_CUDA_CORES if path == "cuda_cores" else dcp.DCP_PATH_AUTO
    prob = synth.make_decode_problem("dev2", [2000, 900], 128, 512, synth.KV_FP8, 4, 1, mtp=2, seed=83)
    ro, rl = oracle.attention_problem(prob)
    for dev in ("cuda:0", "cuda:1"):
        with torch.cuda.device(dev):
            g = prob.to(dev)
            fo, fl = dcp.mla_decode_dcp_fused(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                              g.sm_scale, g.dcp, g.interleave, idx=g.topk,
                                              kernel_path=kp)
            torch.cuda.synchronize()
        check_out(fo, ro, "%s %s fused out" % (dev, path))
        check_lse(fl, rl, "%s %s fused lse" % (dev, path))
