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
