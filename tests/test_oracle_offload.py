"""Oracle KV offload (HiSparse write side): complete pages copied from each layer's pool to its host
rows, nothing else touched, incomplete or out-of-range entries refused."""
import numpy as np
import pytest

import oracle


def _setup(L=2, B=2, pages=3, seed=0):
    g = np.random.default_rng(seed)
    nblk = B * pages + 2
    bt = g.permutation(nblk)[:B * pages].reshape(B, pages).astype(np.int32)
    pools = [g.integers(0, 256, (nblk * 64, 656), dtype=np.uint8) for _ in range(L)]
    seq = np.array([pages * 64, 2 * 64 + 10], np.int32)[:B]
    hosts = [np.zeros((int(seq[r]), 656), np.uint8) for l in range(L) for r in range(B)]
    return pools, hosts, bt, seq


def test_pages_land_at_their_rows_and_nothing_else_changes():
    pools, hosts, bt, seq = _setup()
    layer, req, page = np.array([1, 0, 0]), np.array([0, 1, 0]), np.array([2, 1, 0])
    oracle.kv_offload(pools, hosts, layer, req, page, bt, seq)
    for l, r, p in zip(layer, req, page):
        blk = bt[r, p]
        assert np.array_equal(hosts[l * 2 + r][64 * p:64 * p + 64], pools[l][64 * blk:64 * blk + 64])
        hosts[l * 2 + r][64 * p:64 * p + 64] = 0
    assert not any(h.any() for h in hosts)


def test_incomplete_and_out_of_range_entries_are_refused():
    pools, hosts, bt, seq = _setup()
    # request 1 has 138 tokens: page 2 (tokens 128..191) is incomplete
    for l, r, p in ((0, 1, 2), (2, 0, 0), (0, 2, 0), (0, 0, 3), (0, 0, -1)):
        with pytest.raises(oracle.OracleError):
            oracle.kv_offload(pools, hosts, np.array([l]), np.array([r]), np.array([p]), bt, seq)
    bt[0, 1] = -1
    with pytest.raises(oracle.OracleError):
        oracle.kv_offload(pools, hosts, np.array([0]), np.array([0]), np.array([1]), bt, seq)
    assert not any(h.any() for h in hosts)
