"""The one-call decode path hs_indexer_topk: the same indices as hs_indexer_scores followed by
hs_topk (bit for bit), with the scores kept in L2 between the two kernels and dropped from it
afterwards. Rows whose score lines are shared with a neighbouring row (a row stride that is not a
multiple of 32 floats) must not lose a neighbour's scores; the oracle checks sampled tokens."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_mla_gb300 import hs_check_flag, hs_indexer_scores, hs_indexer_topk, hs_topk, inputs
from dsa_sparse_mla_gb300.pipeline import DeviceWorkload, HotPath, SharedSetHotPath

from parity import check_topk_sets

pytestmark = pytest.mark.gpu


def _both(dw, ld):
    """idx from the two calls and from the one call, each on its own [T, ld] scores buffer."""
    d, w = dw, dw.w
    dev = d.q_idx.device
    args = (d.q_idx, d.q_scale, d.weights, d.k_cache, d.k_scale, d.block_table, d.token_req, d.token_kvlen)
    s1 = torch.full((w.T, ld), float("nan"), dtype=torch.float32, device=dev)
    s2 = torch.full((w.T, ld), float("nan"), dtype=torch.float32, device=dev)
    i1 = torch.full((w.T, w.topk), -7, dtype=torch.int32, device=dev)
    i2 = torch.full((w.T, w.topk), -7, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    hs_indexer_scores(*args, s1, err, num_requests=w.B)
    hs_topk(s1, d.token_kvlen, w.topk, i1, err)
    hs_indexer_topk(*args, s2, w.topk, i2, err, num_requests=w.B)
    assert hs_check_flag(err) == 0
    return i1.cpu().numpy(), i2.cpu().numpy()


def _oracle_rows(w, idx_gpu, rows):
    rows = np.asarray(rows)
    sl = lambda a: np.ascontiguousarray(a[rows])
    ref_scores = oracle.indexer_scores(sl(w.q_idx), sl(w.q_scale), sl(w.weights), w.k_cache, w.k_scale, w.block_table,
                                       sl(w.token_req), sl(w.token_kvlen), ld=w.ld)
    ref_idx = oracle.topk(ref_scores, sl(w.token_kvlen), w.topk)
    check_topk_sets(idx_gpu[rows], ref_scores, sl(w.token_kvlen), w.topk, ref_idx)


@pytest.mark.parametrize("pad", [0, 5])
def test_one_call_equals_two_calls_small(pad):
    """8 requests x 4 MTP tokens, contexts 3,000-9,000; a row stride of ld + 5 floats makes
    neighbouring rows share 128-byte lines."""
    w = inputs.config2(seed=11, B=8, lo=3000, hi=9000)
    dw = DeviceWorkload.from_host(w)
    i1, i2 = _both(dw, w.ld + pad)
    assert np.array_equal(i1, i2)
    _oracle_rows(w, i2, [0, 1, 2, 3, 13, 31])


def test_one_call_short_rows():
    """Contexts below k (every visible token is selected, -1 padded) and just above it."""
    w = inputs.config2(seed=12, B=6, lo=100, hi=2100)
    dw = DeviceWorkload.from_host(w)
    i1, i2 = _both(dw, w.ld + 3)
    assert np.array_equal(i1, i2)
    _oracle_rows(w, i2, np.arange(w.T))


def test_one_call_full_size_mtp_decode():
    """The full MTP-decode batch (64 requests x 4 tokens, contexts 16K-64K): bit-identical to the
    two calls, and the pipeline's fused step gives the same indices; sampled tokens against the
    oracle."""
    w = inputs.config2()
    dw = DeviceWorkload.from_host(w)
    i1, i2 = _both(dw, w.ld)
    assert np.array_equal(i1, i2)
    hp = HotPath(dw, fused=True)
    hp.step()
    assert hs_check_flag(hp.err) == 0
    assert np.array_equal(hp.idx.cpu().numpy(), i1)
    _oracle_rows(w, i2, [0, 3, 130, 255])


def test_shared_sets_fused_step():
    """Shared index sets with the one call: the final tokens' sets equal the two-call path's."""
    w = inputs.config2(seed=13, B=8, lo=5000, hi=12000)
    dw = DeviceWorkload.from_host(w)
    a, b = SharedSetHotPath(dw), SharedSetHotPath(dw, fused=True)
    a.step()
    b.step()
    assert hs_check_flag(a.err) == 0 and hs_check_flag(b.err) == 0
    assert torch.equal(a.idx, b.idx)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_one_call_chunked_prefill():
    """A prefill chunk through the one call (2,048 tokens after 65,536 cached, 553 MB of scores, far
    more than L2 holds): still the two calls' indices, bit for bit."""
    w = inputs.config3()
    dw = DeviceWorkload.from_host(w)
    i1, i2 = _both(dw, w.ld)
    assert np.array_equal(i1, i2)
