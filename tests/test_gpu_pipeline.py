"""End-to-end parity of one hot-path step (indexer -> top-k -> sparse MLA) on the benchmark's
workloads: the tiny prefill in full, and the MTP-decode, chunked-prefill and long-prefill
workloads at full size on sampled query tokens (the oracle computes those tokens one by one)."""
import numpy as np
import pytest

import oracle
from dsa_sparse_mla_gb300 import hs_check_flag, inputs
from dsa_sparse_mla_gb300.pipeline import DeviceWorkload, HotPath, SharedSetHotPath

from parity import check_mla, check_topk_sets

pytestmark = pytest.mark.gpu


def _check_tokens(w, hp, rows):
    rows = np.asarray(rows)
    sl = lambda a: np.ascontiguousarray(a[rows])
    idx_gpu = hp.idx.cpu().numpy()[rows]
    # the oracle's own scores and top-k for these tokens
    ref_scores = oracle.indexer_scores(sl(w.q_idx), sl(w.q_scale), sl(w.weights), w.k_cache, w.k_scale, w.block_table,
                                       sl(w.token_req), sl(w.token_kvlen), ld=w.ld)
    ref_idx = oracle.topk(ref_scores, sl(w.token_kvlen), w.topk)
    ndiff = check_topk_sets(idx_gpu, ref_scores, sl(w.token_kvlen), w.topk, ref_idx)
    # attention checked on the GPU's index set
    out_ref, lse_ref = oracle.sparse_mla(sl(w.q_mla), w.kv_pool, idx_gpu, w.softmax_scale, w.block_table,
                                         sl(w.token_req))
    check_mla(hp.out[rows], hp.lse[rows], out_ref, lse_ref)
    return ndiff


def test_tiny_prefill_full():
    w = inputs.config1()
    hp = HotPath(DeviceWorkload.from_host(w))
    hp.step()
    assert hs_check_flag(hp.err) == 0
    _check_tokens(w, hp, np.arange(w.T))


def test_mtp_decode_full_size_sampled():
    w = inputs.config2()
    hp = HotPath(DeviceWorkload.from_host(w))
    hp.step()
    assert hs_check_flag(hp.err) == 0
    rows = [0, 1, 2, 3, 101, 254, 255]
    _check_tokens(w, hp, rows)


def test_chunked_prefill_full_size_sampled():
    """The 2048-token chunk after 65,536 cached tokens: 16 tokens spread over the chunk, so that
    the persistent indexer's and the MLA's per-position work splits are sampled throughout."""
    w = inputs.config3()
    hp = HotPath(DeviceWorkload.from_host(w))
    hp.step()
    assert hs_check_flag(hp.err) == 0
    rows = np.unique(np.concatenate([np.linspace(0, w.T - 1, 14).round().astype(int), [1, 1000]]))
    assert len(rows) == 16
    _check_tokens(w, hp, rows)


@pytest.mark.parametrize("chunk", [31, 63])
def test_long_prefill_full_size_sampled(chunk):
    """Long prefill of one 131,072-token sequence in 64 chunks of 2048: a middle chunk and the
    last one (each query sees up to 131,072 keys), whole-chunk launches, sampled tokens."""
    w = inputs.config4(chunk)
    hp = HotPath(DeviceWorkload.from_host(w))
    hp.step()
    assert hs_check_flag(hp.err) == 0
    assert int(w.token_kvlen.max()) == (chunk + 1) * 2048
    _check_tokens(w, hp, [0, 1023, 2047])


def test_repeat_is_deterministic():
    w = inputs.config2(seed=41, B=8, lo=3000, hi=9000)
    hp = HotPath(DeviceWorkload.from_host(w))
    hp.step()
    a = (hp.idx.clone(), hp.out.clone(), hp.lse.clone())
    hp.step()
    assert hp.idx.equal(a[0]) and hp.out.equal(a[1]) and hp.lse.equal(a[2])


def test_mtp_decode_shared_sets_full_size_sampled():
    """Shared index sets on the full MTP-decode batch: the indexer and top-k of each request's
    final token against the oracle's, and every token of the sampled requests attending that set
    (limited to what it can see) against the oracle on the expanded sets."""
    w = inputs.config2()
    hp = SharedSetHotPath(DeviceWorkload.from_host(w))
    hp.step()
    assert hs_check_flag(hp.err) == 0
    reqs = np.array([0, 17, 63])
    final = np.array([np.flatnonzero(w.token_req == r)[-1] for r in reqs])   # the last token of each request
    sl = lambda a: np.ascontiguousarray(a[final])
    idx_gpu = hp.idx.cpu().numpy()[reqs]
    ref_scores = oracle.indexer_scores(sl(w.q_idx), sl(w.q_scale), sl(w.weights), w.k_cache, w.k_scale, w.block_table,
                                       sl(w.token_req), sl(w.token_kvlen), ld=w.ld)
    ref_idx = oracle.topk(ref_scores, sl(w.token_kvlen), w.topk)
    check_topk_sets(idx_gpu, ref_scores, sl(w.token_kvlen), w.topk, ref_idx)
    rows = np.flatnonzero(np.isin(w.token_req, reqs))
    sets = oracle.shared_index_sets(idx_gpu, np.searchsorted(reqs, w.token_req[rows]), w.token_kvlen[rows])
    out_ref, lse_ref = oracle.sparse_mla(np.ascontiguousarray(w.q_mla[rows]), w.kv_pool, sets, w.softmax_scale,
                                         w.block_table, np.ascontiguousarray(w.token_req[rows]))
    check_mla(hp.out[rows], hp.lse[rows], out_ref, lse_ref)
