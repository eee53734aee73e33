"""GPU KV offload (HiSparse write side) is bit-exact against the oracle: every complete page lands
in its layer's host rows, nothing else changes, bad entries are flagged and copy nothing."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_mla_gb300 import hs_check_flag, hs_kv_offload
from dsa_sparse_mla_gb300.pipeline import pinned_uint8

pytestmark = pytest.mark.gpu


def _setup(L, B, pages, seq, seed):
    g = np.random.default_rng(seed)
    nblk = B * pages + 3
    bt = g.permutation(nblk)[:B * pages].reshape(B, pages).astype(np.int32)
    pools_h = [g.integers(0, 256, (nblk * 64, 656), dtype=np.uint8) for _ in range(L)]
    pools = [torch.from_numpy(p).cuda() for p in pools_h]
    hosts = []
    for l in range(L):
        for r in range(B):
            h = pinned_uint8(int(seq[r]) * 656).reshape(int(seq[r]), 656)
            h[:] = (l * 7 + r) & 0xFF  # a pattern the copies overwrite
            hosts.append(h)
    return g, bt, pools_h, pools, hosts, nblk * 64


def _run(L, B, pages, seq, entries, seed, expect_flag=0):
    g, bt, pools_h, pools, hosts, R = _setup(L, B, pages, seq, seed)
    ref = [h.copy() for h in hosts]
    layer, req, page = (np.array([e[i] for e in entries], np.int32) for i in range(3))
    if expect_flag == 0:
        oracle.kv_offload(pools_h, ref, layer, req, page, bt, seq)
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs_kv_offload(torch.tensor([p.data_ptr() for p in pools], dtype=torch.int64, device="cuda"),
                  torch.tensor([h.ctypes.data for h in hosts], dtype=torch.int64, device="cuda"),
                  c(layer), c(req), c(page), c(bt), c(seq), err, R=R)
    assert hs_check_flag(err) == expect_flag
    return hosts, ref


def test_all_complete_pages_of_every_layer():
    L, B, pages = 3, 4, 6
    seq = np.array([6 * 64, 5 * 64 + 3, 64, 2 * 64 + 63], np.int32)
    entries = [(l, r, p) for l in range(L) for r in range(B) for p in range(int(seq[r]) // 64)]
    np.random.default_rng(1).shuffle(entries)
    hosts, ref = _run(L, B, pages, seq, entries, seed=2)
    for h, e in zip(hosts, ref):
        assert np.array_equal(h, e)


def test_many_pages_grid_stride():
    # more entries than CTAs of the launch (8 per SM)
    L, B, pages = 8, 2, 128
    seq = np.array([pages * 64, pages * 64 - 1], np.int32)
    entries = [(l, r, p) for l in range(L) for r in range(B) for p in range(int(seq[r]) // 64)]
    hosts, ref = _run(L, B, pages, seq, entries, seed=3)
    for h, e in zip(hosts, ref):
        assert np.array_equal(h, e)


def test_bad_entries_flagged_and_copy_nothing():
    L, B, pages = 2, 2, 3
    seq = np.array([3 * 64, 2 * 64 + 10], np.int32)
    # incomplete page, layer out of range, request out of range, page past bt_stride
    hosts, ref = _run(L, B, pages, seq, [(0, 1, 2), (2, 0, 0), (0, 2, 0), (1, 0, 3)], seed=4, expect_flag=0x01)
    for h, e in zip(hosts, ref):
        assert np.array_equal(h, e)  # ref: untouched copies
