"""Pin of the chunked-prefill decomposition in the oracle: for every row of a prefill
chunk, the LSE merge of the D per-shard dense partials over the cached prefix and the D
per-shard sparse partials over the chunk slots the row sees equals dense attention over
the row's whole visible range (LMDeploy PR #4952, Summary: prefill gathers the cached-prefix
KV in bounded chunks, and partial attention results merge with LSE weights).  Each oracle
function used here is pinned on its own in test_oracle_pins.py; this checks their
composition against the unsharded definition to ~1e-12."""
import numpy as np
import pytest

import oracle
import synth


@pytest.mark.parametrize("D,I,kvt", [(2, 1, synth.KV_BF16), (3, 64, synth.KV_FP8), (4, 1, synth.KV_FP8)])
def test_prefix_and_chunk_partials_merge_to_dense(orc, D, I, kvt):
    chunk = 5
    prob = synth.prefill_chunk_problem("pin", [130, 0, 67], chunk, 16, kvt, D, I, seed=3)
    prefix, ids = synth.prefill_chunk_inputs(prob, chunk)
    parts_o, parts_l = [], []
    for s in range(D):
        p = synth.DecodeProblem(**{**prob.__dict__, "row_len": prefix, "topk": None})
        o, l = oracle.attention_problem(p, shard=s)
        parts_o.append(o)
        parts_l.append(l)
    for s in range(D):
        p = synth.DecodeProblem(**{**prob.__dict__, "topk": ids})
        o, l = oracle.attention_problem(p, shard=s)
        parts_o.append(o)
        parts_l.append(l)
    mo, ml = oracle.merge(np.stack(parts_o), np.stack(parts_l))
    ro, rl = oracle.attention_problem(prob)
    assert np.abs(mo - ro).max() < 1e-12
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(ml), fin) and np.abs(ml[fin] - rl[fin]).max() < 1e-12
