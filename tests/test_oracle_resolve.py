"""Pins of the oracle's HiSparse resolve: a four-step case worked by hand, and the LRU
invariants over long random replays."""
import json
import os

import numpy as np
import pytest

import oracle
from dsa_sparse_mla_gb300 import inputs


def _state(B, S, R, ld):
    return (np.zeros((R, 656), np.uint8), np.full((B, S), -1, np.int32), np.full((B, S), -1, np.int32),
            np.full((B, ld), -1, np.int32))


def test_hand_worked_four_steps(golden_dir):
    with open(os.path.join(golden_dir, "resolve_hand.json")) as f:
        g = json.load(f)
    S, k, n = g["S"], g["k"], g["seq_len"]
    host = (np.arange(n)[:, None] * 7 + np.arange(656)[None, :]).astype(np.uint8)
    bt = np.full((1, 1), g["page0_block"], np.int32)
    slot_row = np.array([g["slot_row"]], np.int32)
    pool, stok, sstamp, t2s = _state(1, S, 400, n)
    for st in g["steps"]:
        out, cnt = oracle.hisparse_resolve(st["step"], np.array([st["idx"]], np.int32), [n], [g["resident_start"]],
                                           bt, [host], pool, slot_row, stok, sstamp, t2s)
        assert out[0].tolist() == st["out_rows"], st["why"]
        assert cnt[0].tolist() == st["counters"]
        assert stok[0].tolist() == st["slot_token"]
        assert sstamp[0].tolist() == st["slot_stamp"]
        want = np.full(n, -1); [want.__setitem__(int(j), s) for j, s in st["tok2slot"].items()]
        assert t2s[0].tolist() == want.tolist()
        for s in range(S):
            if stok[0, s] >= 0:
                assert np.array_equal(pool[slot_row[0, s]], host[stok[0, s]])


def _check_invariants(prev_stamp, prev_tok, step, idx, rs, host, pool, slot_row, stok, sstamp, t2s, out, cnt):
    S = stok.shape[0]
    k = idx.shape[0]
    valid = idx[idx >= 0]
    hot = stok[stok >= 0]
    assert len(hot) <= S and len(set(hot.tolist())) == len(hot)          # hot size <= S, no duplicates
    for s in range(S):                                                   # maps are mutual inverses
        if stok[s] >= 0:
            assert t2s[stok[s]] == s
            assert np.array_equal(pool[slot_row[s]], host[stok[s]])       # slot bytes = host row
    assert np.count_nonzero(t2s >= 0) == len(hot)
    nonres = valid[valid < rs]
    for j in nonres:                                                     # every selected old token is hot now
        assert t2s[j] >= 0 and sstamp[t2s[j]] == step
    misses = [j for j in nonres if j not in set(prev_tok[prev_tok >= 0].tolist())]
    assert cnt.tolist() == [int((valid >= rs).sum()), len(nonres) - len(misses), len(misses)]
    # each miss filled exactly once: the slots stamped `step` are exactly the selected old tokens
    assert sorted(stok[sstamp == step].tolist()) == sorted(nonres.tolist())
    # LRU: every evicted slot was, before the step, no more recent than any surviving untouched slot
    touched_prev = set(int(t2s[j]) for j in nonres if j not in misses)
    evicted = [s for s in range(S) if sstamp[s] == step and s not in touched_prev]
    kept_untouched = [s for s in range(S) if sstamp[s] != step]
    if evicted and kept_untouched:
        assert max((prev_stamp[s], s) for s in evicted) < min((prev_stamp[s], s) for s in kept_untouched)
    for i in range(k):
        j = idx[i]
        if j < 0:
            assert out[i] == -1
        elif j < rs:
            assert out[i] == slot_row[t2s[j]]


@pytest.mark.parametrize("seed", [0, 1])
def test_random_replay_invariants(seed):
    g = np.random.default_rng(seed)
    B, k, S, n, res = 3, 24, 48, 600, 64
    rs = n - res
    bt = np.full((B, (n + 63) // 64), -1, np.int32)
    for r in range(B):
        bt[r, rs // 64:] = np.arange((n + 63) // 64 - rs // 64) + 100 * r
    slot_row = (5000 + np.arange(B * S)).reshape(B, S).astype(np.int32)
    hosts = [g.integers(0, 256, size=(n, 656), dtype=np.uint8) for _ in range(B)]
    pool, stok, sstamp, t2s = _state(B, S, 5000 + B * S, n)
    stream = inputs.hisparse_index_stream(np.full(B, n), res, k - 4, 40, 0.7, inputs.Stream(seed))
    for step in range(40):
        idx = np.full((B, k), -1, np.int32)
        for r in range(B):
            sel = stream[step, r].tolist()
            if step % 3 == 0:   # add a few resident tokens
                sel = sorted(sel + [rs + 3, rs + 10 + r])
            idx[r, :len(sel)] = sel
        prev_stamp, prev_tok = sstamp.copy(), stok.copy()
        out, cnt = oracle.hisparse_resolve(step, idx, [n] * B, [rs] * B, bt, hosts, pool, slot_row, stok, sstamp, t2s)
        for r in range(B):
            _check_invariants(prev_stamp[r], prev_tok[r], step, idx[r], rs, hosts[r], pool, slot_row[r],
                              stok[r], sstamp[r], t2s[r], out[r], cnt[r])


def test_contract_violations_rejected_and_leave_state():
    n, S = 100, 4
    host = np.zeros((n, 656), np.uint8)
    bt = np.zeros((1, 2), np.int32)
    pool, stok, sstamp, t2s = _state(1, S, 200, n)
    for bad in ([5, 3, -1], [5, -1, 7], [5, 5, -1], [5, 100, -1]):
        with pytest.raises(oracle.OracleError):
            oracle.hisparse_resolve(0, np.array([bad], np.int32), [n], [90], bt, [host], pool,
                                    np.array([[190, 191, 192, 193]], np.int32), stok, sstamp, t2s)
        assert (stok == -1).all() and (t2s == -1).all()
