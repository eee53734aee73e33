"""GPU parity of hs_indexer_scores against the oracle (tolerance from fp32 accumulation)."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_mla_gb300 import HSError, hs_check_flag, hs_indexer_scores, inputs
from dsa_sparse_mla_gb300.pipeline import DeviceWorkload, HotPath

from parity import SCORE_RTOL, abs_codes

pytestmark = pytest.mark.gpu


def _compare(w, scores_gpu, rows=None):
    rows = np.arange(w.T) if rows is None else np.asarray(rows)
    sl = lambda a: np.ascontiguousarray(a[rows])
    ref = oracle.indexer_scores(sl(w.q_idx), sl(w.q_scale), sl(w.weights), w.k_cache, w.k_scale, w.block_table,
                                sl(w.token_req), sl(w.token_kvlen), ld=w.ld)
    sabs = oracle.indexer_scores(abs_codes(sl(w.q_idx)), sl(w.q_scale), np.abs(sl(w.weights)), abs_codes(w.k_cache),
                                 w.k_scale, w.block_table, sl(w.token_req), sl(w.token_kvlen), ld=w.ld)
    g = scores_gpu[rows].astype(np.float64)
    worst = 0.0
    for i, t in enumerate(rows):
        n = int(w.token_kvlen[t])
        d = np.abs(g[i, :n] - ref[i, :n])
        tol = SCORE_RTOL * sabs[i, :n] + 1e-30
        assert np.all(d <= tol), (t, int(np.argmax(d - tol)), float(d.max()))
        if n:
            worst = max(worst, float((d / np.maximum(sabs[i, :n], 1e-30)).max()))
    return worst


@pytest.mark.parametrize("Hi,Di", [(64, 128), (32, 128), (16, 64), (8, 64)])
def test_decode_shapes(Hi, Di):
    w = inputs.config2(seed=21, B=5, lo=200, hi=1500, Hi=Hi, Di=Di, H=4, topk=64)
    hp = HotPath(DeviceWorkload.from_host(w))
    hp.scores.fill_(float("nan"))
    hp.indexer()
    assert hs_check_flag(hp.err) == 0
    _compare(w, hp.scores.cpu().numpy())


def test_prefill_ragged_groups_and_mixed_requests():
    """T not a multiple of the token group; groups that span two requests; tiny and empty rows."""
    ctx = np.array([130, 70, 257], np.int32)
    queries = [np.array([0, 1, 2, 63, 64, 127, 128, 129]), np.array([5, 69]), np.arange(200, 257)]
    w = inputs.make_workload("ragged", 3, ctx, queries, Hi=64, Di=128, H=4, topk=32, seed=22)
    hp = HotPath(DeviceWorkload.from_host(w))
    hp.indexer()
    assert hs_check_flag(hp.err) == 0
    _compare(w, hp.scores.cpu().numpy())


def test_tiny_prefill_config_full():
    w = inputs.config1()
    hp = HotPath(DeviceWorkload.from_host(w))
    hp.indexer()
    assert hs_check_flag(hp.err) == 0
    _compare(w, hp.scores.cpu().numpy())


def test_bad_length_is_flagged_not_fatal():
    w = inputs.config2(seed=23, B=2, lo=100, hi=200, Hi=64, Di=128, H=4, topk=16)
    dw = DeviceWorkload.from_host(w)
    hp = HotPath(dw)
    bad = dw.token_kvlen.clone()
    bad[1] = w.ld + 5
    hs_indexer_scores(dw.q_idx, dw.q_scale, dw.weights, dw.k_cache, dw.k_scale, dw.block_table, dw.token_req, bad,
                      hp.scores, hp.err, num_requests=w.B)
    assert hs_check_flag(hp.err) & 0x02
    with pytest.raises(HSError):
        hs_indexer_scores(dw.q_idx[:, :3], dw.q_scale, dw.weights, dw.k_cache, dw.k_scale, dw.block_table,
                          dw.token_req, bad, hp.scores, hp.err)
