"""Both decode paths through the C ABI: the tensor-core path (taken for 48..128 heads) and
the CUDA-core path (taken for fewer heads, or for any head count with DCPMLA_PATH=simt)
agree with the oracle on the same inputs, including rows cut across CTA pairs."""
import os

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


@pytest.mark.parametrize("path", ["simt", "tc"])
@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8])
def test_both_paths_match_oracle(dcp, path, kv):
    prob = synth.make_decode_problem("paths", [3100, 1700], 128, 1000, kv, 4, 1, mtp=3, seed=81)
    old = os.environ.get("DCPMLA_PATH")
    os.environ["DCPMLA_PATH"] = path
    try:
        g = prob.to(DEV)
        po, pl, mo, ml = run_unfused(dcp, g)
        fo, fl = run_fused(dcp, g)
        torch.cuda.synchronize()
    finally:
        if old is None:
            del os.environ["DCPMLA_PATH"]
        else:
            os.environ["DCPMLA_PATH"] = old
    ro, rl = oracle.attention_problem(prob)
    check_out(fo, ro, path + " fused out")
    check_lse(fl, rl, path + " fused lse")
    check_out(mo, ro, path + " merged out")
    check_lse(ml, rl, path + " merged lse")
    so, sl = oracle.attention_problem(prob, shard=2)
    check_out(po[2], so, path + " partial out")
    check_lse(pl[2], sl, path + " partial lse")


def test_tc_timeout_flag_stays_clear(dcp):
    prob = synth.make_decode_problem("flag", [5000], 128, 2048, synth.KV_FP8, 8, 1, mtp=2, seed=82).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_fused(dcp, prob, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == 0
