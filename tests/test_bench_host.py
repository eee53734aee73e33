"""Host-side logic of bench.py for the shared-index-set mode (no GPU): which tokens run the
indexer and top-k, the algorithmic work counted for each call, and the oracle's sample run."""
import numpy as np

import bench
from dsa_sparse_mla_gb300 import inputs


def _w():
    return inputs.config2(seed=5, B=3, lo=300, hi=900, Hi=8, Di=64, H=4, topk=64)


def test_final_tokens_are_each_requests_last_position():
    w = _w()
    fin = bench.final_tokens(w)
    assert list(fin) == [3, 7, 11]
    for r, t in enumerate(fin):
        assert w.token_req[t] == r and w.token_kvlen[t] == w.token_kvlen[w.token_req == r].max()


def test_shared_sets_count_indexer_and_topk_for_final_tokens_only():
    w = _w()
    per, sh = bench.work_of(w), bench.work_of(w, shared=True)
    fin = bench.final_tokens(w)
    assert sh["indexer"].flops == 2 * w.Hi * w.Di * int(w.token_kvlen[fin].sum())
    assert per["indexer"].flops == 2 * w.Hi * w.Di * int(w.token_kvlen.sum())
    assert sh["topk"].bytes == 4 * int(w.token_kvlen[fin].sum()) + 4 * len(fin) * w.topk
    assert sh["mla"] == per["mla"]


def test_oracle_sample_runs_in_both_modes():
    w = _w()
    assert bench.oracle_sample(w, list(range(w.T)), threads=1) > 0
    assert bench.oracle_sample(w, list(range(w.T)), threads=1, shared=True) > 0


def test_long_prefill_cpu_sample_is_stratified_over_the_pass():
    """The CPU baseline of the long-prefill line samples 16 evenly spaced tokens in each of chunks
    3, 11, ..., 59: positions spread over the whole sequence, mean position that of the pass."""
    ws = inputs.config4_pass(total=64 * 64, chunk_len=64, Hi=8, Di=64, H=4, topk=16)
    assert len(ws) == 64
    calls = []
    orig = bench.oracle_sample
    try:
        bench.oracle_sample = lambda w, toks, threads=0, shared=False: calls.append((w, list(toks))) or 0.5
        ntok, wall = bench.long_prefill_cpu_sample(ws)
    finally:
        bench.oracle_sample = orig
    assert ntok == 128 and wall == 0.5 * 8
    pos = [int(w.token_kvlen[t]) - 1 for w, toks in calls for t in toks]
    assert [int(w.token_kvlen[0]) // 64 for w, _ in calls] == list(range(3, 64, 8))
    assert abs(np.mean(pos) - (64 * 64 - 1) / 2) < 64 * 64 * 0.02
