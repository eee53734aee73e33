"""Pins of the oracle's lightning-indexer scores: a hand-worked case, and invariants that a
dropped term, a wrong index or a wrong scale placement would break."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from dsa_sparse_mla_gb300 import inputs

CODE = {1.0: 0x38, 2.0: 0x40, 0.5: 0x30, -1.0: 0xB8, -2.0: 0xC0, 0.0: 0x00}


def _hand(golden_dir):
    with open(os.path.join(golden_dir, "indexer_hand.json")) as f:
        g = json.load(f)
    Hi, Di = g["Hi"], g["Di"]
    keys = np.array([[CODE[v] for v in row] for row in g["keys"]], np.uint8)
    k_cache = np.zeros((1, 64, Di), np.uint8)
    k_cache[0, :3] = keys
    k_scale = np.ones((1, 64), np.float32)
    k_scale[0, :3] = g["k_scale"]
    q = np.array([[[CODE[v] for v in h] for h in t] for t in g["q"]], np.uint8)
    return g, q, np.array(g["q_scale"], np.float32), np.array(g["weights"], np.float32), k_cache, k_scale


def test_hand_worked_scores_and_topk(golden_dir):
    g, q, qs, w, kc, ks = _hand(golden_dir)
    bt = np.zeros((1, 1), np.int32)
    s = oracle.indexer_scores(q, qs, w, kc, ks, bt, np.zeros(2, np.int32), np.array(g["token_kvlen"], np.int32), ld=3)
    want = np.array([[float(x) for x in row] for row in g["scores"]])
    assert np.array_equal(s, want)
    assert np.array_equal(oracle.topk(s, np.array(g["token_kvlen"], np.int32), 2), np.array(g["topk2"]))


def _random_case(seed, T=6, Hi=4, Di=16, ctx=(150, 70)):
    st = inputs.Stream(seed)
    ctx = np.array(ctx, np.int32)
    bt, nblk = inputs.paged_block_tables(ctx, st.sub("bt"))
    q, qs = inputs.quantize_rows(st.sub("q").normal((T, Hi, Di)))
    w = st.sub("w").uniform((T, Hi))
    kc, ks = inputs.quantize_rows(st.sub("k").normal((int(ctx.sum()), Di)))
    k_cache = inputs.scatter_paged(kc, ctx, bt, nblk).reshape(nblk, 64, Di)
    k_scale = inputs.scatter_paged(ks, ctx, bt, nblk).reshape(nblk, 64)
    k_scale[k_scale == 0] = 1
    req = np.array([0, 0, 0, 1, 1, 1], np.int32)[:T]
    kvlen = np.array([1, 77, 150, 5, 64, 70], np.int32)[:T]
    return q, qs, w, k_cache, k_scale, bt, req, kvlen, ctx, kc, ks


def test_masked_columns_are_minus_inf_and_ignore_later_keys():
    q, qs, w, kc, ks, bt, req, kvlen, *_ = _random_case(1)
    s = oracle.indexer_scores(q, qs, w, kc, ks, bt, req, kvlen, ld=160)
    for t in range(len(req)):
        assert np.all(np.isneginf(s[t, kvlen[t]:]))
        assert np.all(np.isfinite(s[t, :kvlen[t]]))
    # scribbling over keys no query sees changes nothing
    kc2 = kc.copy()
    r, j = 0, 149
    row = bt[r, j // 64] * 64 + j % 64
    kc2.reshape(-1, kc.shape[-1])[row] = 0x40
    s2 = oracle.indexer_scores(q, qs, w, kc2, ks, bt, req, np.minimum(kvlen, 149), ld=160)
    s1 = oracle.indexer_scores(q, qs, w, kc, ks, bt, req, np.minimum(kvlen, 149), ld=160)
    assert np.array_equal(s1, s2)


def test_paging_invariance():
    """The same logical keys behind two different page permutations score identically."""
    q, qs, w, kc, ks, bt, req, kvlen, ctx, kflat, sflat = _random_case(2)
    bt2, nblk2 = inputs.paged_block_tables(ctx, inputs.Stream(99).sub("other"))
    assert not np.array_equal(bt, bt2)
    kc2 = inputs.scatter_paged(kflat, ctx, bt2, nblk2).reshape(nblk2, 64, -1)
    ks2 = inputs.scatter_paged(sflat, ctx, bt2, nblk2).reshape(nblk2, 64)
    ks2[ks2 == 0] = 1
    a = oracle.indexer_scores(q, qs, w, kc, ks, bt, req, kvlen, ld=150)
    b = oracle.indexer_scores(q, qs, w, kc2, ks2, bt2, req, kvlen, ld=150)
    assert np.array_equal(a, b)


def test_scale_folding_and_linearity():
    """Doubling a positive scale doubles the score (the ReLU commutes with positive factors);
    the score is linear in the head weights; head order is irrelevant."""
    q, qs, w, kc, ks, bt, req, kvlen, *_ = _random_case(3)
    base = oracle.indexer_scores(q, qs, w, kc, ks, bt, req, kvlen, ld=150)
    fin = np.isfinite(base)
    s_q = oracle.indexer_scores(q, qs * 2, w, kc, ks, bt, req, kvlen, ld=150)
    s_k = oracle.indexer_scores(q, qs, w, kc, ks * 2, bt, req, kvlen, ld=150)
    s_w = oracle.indexer_scores(q, qs, w * 2, kc, ks, bt, req, kvlen, ld=150)
    for s in (s_q, s_k, s_w):
        assert np.array_equal(s[fin], 2 * base[fin])
    perm = np.array([2, 0, 3, 1])
    s_p = oracle.indexer_scores(q[:, perm], qs[:, perm], w[:, perm], kc, ks, bt, req, kvlen, ld=150)
    assert np.allclose(s_p[fin], base[fin], rtol=1e-14, atol=0)


def test_relu_drops_negative_heads():
    """Negating one head's query only changes the score by that head's (ReLU-ed) terms: the sum
    of the two scores equals sum_h w|v| over both signs of that head."""
    q, qs, w, kc, ks, bt, req, kvlen, *_ = _random_case(4)
    w1 = np.zeros_like(w)
    w1[:, 1] = w[:, 1]
    a = oracle.indexer_scores(q, qs, w1, kc, ks, bt, req, kvlen, ld=150)
    qn = q.copy()
    qn[:, 1] ^= 0x80  # flip the sign bit of every code of head 1
    b = oracle.indexer_scores(qn, qs, w1, kc, ks, bt, req, kvlen, ld=150)
    fin = np.isfinite(a)
    # for each pair exactly one of relu(v), relu(-v) is non-zero (or both zero)
    assert np.all((a[fin] == 0) | (b[fin] == 0))
    assert np.all(a[fin] >= 0) and np.all(b[fin] >= 0)
    assert (a[fin] > 0).any() and (b[fin] > 0).any()


def test_bad_lengths_rejected():
    q, qs, w, kc, ks, bt, req, kvlen, *_ = _random_case(5)
    with pytest.raises(oracle.OracleError):
        oracle.indexer_scores(q, qs, w, kc, ks, bt, req, kvlen, ld=100)
