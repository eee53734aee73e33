"""GPU HiSparse resolve is bit-exact against the oracle: rows, counters, LRU state, pool bytes."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_mla_gb300 import hs_check_flag, hs_hisparse_resolve, hs_hisparse_touch_host, inputs
from dsa_sparse_mla_gb300.pipeline import pinned_uint8

pytestmark = pytest.mark.gpu


class _State:
    def __init__(self, B, S, R, ld):
        self.pool = np.zeros((R, 656), np.uint8)
        self.stok = np.full((B, S), -1, np.int32)
        self.sstamp = np.full((B, S), -1, np.int32)
        self.t2s = np.full((B, ld), -1, np.int32)

    def to_dev(self):
        return [torch.from_numpy(a.copy()).cuda() for a in (self.pool, self.stok, self.sstamp, self.t2s)]


def _replay(B, k, S, n, res, steps, overlap, seed, resident_every=3, step_numbers=None, touch=False):
    """Replays `steps` resolve steps on the GPU and in the oracle and compares everything after each.
    step_numbers: the (increasing) step value passed at each step; 0, 1, 2, ... by default."""
    rs = n - res
    pages = (n + 63) // 64
    bt = np.full((B, pages), -1, np.int32)
    nres_pages = pages - rs // 64
    for r in range(B):
        bt[r, rs // 64:] = np.arange(nres_pages) + r * nres_pages
    R0 = B * nres_pages * 64
    slot_row = (R0 + np.random.default_rng(seed).permutation(B * S)).reshape(B, S).astype(np.int32)
    R = R0 + B * S
    g = np.random.default_rng(seed + 1)
    hosts = []
    for r in range(B):
        h = pinned_uint8(n * 656).reshape(n, 656)
        h[:] = g.integers(0, 256, size=(n, 656), dtype=np.uint8)
        hosts.append(h)
    stream = inputs.hisparse_index_stream(np.full(B, n), res, k - 4, steps, overlap, inputs.Stream(seed))
    ref = _State(B, S, R, n)
    dev = ref.to_dev()
    host_ptrs = torch.tensor([h.ctypes.data for h in hosts], dtype=torch.int64, device="cuda")
    btd = torch.from_numpy(bt).cuda()
    srd = torch.from_numpy(slot_row).cuda()
    seq = torch.full((B,), n, dtype=torch.int32, device="cuda")
    rsd = torch.full((B,), rs, dtype=torch.int32, device="cuda")
    out = torch.empty((B, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, 3), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if touch:
        hs_hisparse_touch_host(host_ptrs, seq, rsd, err)
        assert hs_check_flag(err) == 0
    for step in range(steps):
        snum = step if step_numbers is None else step_numbers[step]
        idx = np.full((B, k), -1, np.int32)
        for r in range(B):
            sel = stream[step, r].tolist()
            if step % resident_every == 0:
                sel = sorted(sel + [rs + 1, rs + 5 + r])
            idx[r, :len(sel)] = sel
        o_ref, c_ref = oracle.hisparse_resolve(snum, idx, [n] * B, [rs] * B, bt, hosts, ref.pool, slot_row, ref.stok,
                                               ref.sstamp, ref.t2s)
        hs_hisparse_resolve(snum, torch.from_numpy(idx).cuda(), seq, rsd, btd, host_ptrs, dev[0], srd, dev[1], dev[2],
                            dev[3], out, cnt, err)
        assert hs_check_flag(err) == 0
        assert np.array_equal(out.cpu().numpy(), o_ref), step
        assert np.array_equal(cnt.cpu().numpy(), c_ref), step
        assert np.array_equal(dev[1].cpu().numpy(), ref.stok), step
        assert np.array_equal(dev[2].cpu().numpy(), ref.sstamp), step
        assert np.array_equal(dev[3].cpu().numpy(), ref.t2s), step
        assert np.array_equal(dev[0].cpu().numpy(), ref.pool), step


@pytest.mark.parametrize("B,k,S,n,res,steps,overlap", [(3, 64, 128, 5000, 256, 12, 0.8), (2, 256, 512, 20000, 1024, 6, 0.5),
                                                      (4, 100, 100, 3000, 128, 8, 0.9), (1, 2048, 4096, 70000, 4096, 4, 0.8)])
def test_replay_matches_oracle(B, k, S, n, res, steps, overlap):
    _replay(B, k, S, n, res, steps, overlap, seed=B * 7 + k)


def test_replay_in_the_benchmark_launch_shape():
    """32 requests, k = 2048, S = 4096 (one CTA per request, 4096-slot sort, as the mixed-residency
    benchmark launches it); shorter contexts than the benchmark's so the oracle replays every step."""
    _replay(32, 2048, 4096, 20000, 4096, 3, 0.8, seed=32)


def test_replay_wide_stamp_spread():
    """Step numbers far apart (spreads of up to 2**30 between stamps): the victim order then needs
    every 4-bit digit of the stamp, not just the lowest ones."""
    nums = [0, 1, 17, 4099, 70001, 1 << 20, (1 << 24) + 3, (1 << 30) + 5, (1 << 30) + 6, 2**31 - 2]
    _replay(3, 64, 128, 5000, 256, len(nums), 0.6, seed=11, step_numbers=nums)


@pytest.mark.parametrize("B,k,S,n,res,steps,overlap", [(2, 4096, 8192, 60000, 2048, 4, 0.7),
                                                      (2, 700, 1500, 9000, 512, 5, 0.6)])
def test_replay_large_and_ragged_slot_counts(B, k, S, n, res, steps, overlap):
    """S = 8192 (the largest, 8 slots per thread in the sort) and S = 1500 (not a multiple of the
    block), after a host-tier touch."""
    _replay(B, k, S, n, res, steps, overlap, seed=B * 5 + S, touch=True)


def test_touch_host_changes_nothing_and_flags_misaligned_rows():
    n = 3000
    host = pinned_uint8(n * 656).reshape(n, 656)
    host[:] = (np.arange(n)[:, None] + np.arange(656)[None, :]).astype(np.uint8)
    before = host.copy()
    seq = torch.tensor([n, n, n], dtype=torch.int32, device="cuda")
    rs = torch.tensor([n - 64, 0, n + 50], dtype=torch.int32, device="cuda")  # a normal tier, none, clamped
    ptrs = torch.tensor([host.ctypes.data] * 3, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs_hisparse_touch_host(ptrs, seq, rs, err)
    assert hs_check_flag(err) == 0
    assert np.array_equal(host, before)
    bad = torch.tensor([host.ctypes.data + 8], dtype=torch.int64, device="cuda")
    hs_hisparse_touch_host(bad, seq[:1], rs[:1], err)
    assert hs_check_flag(err) & 0x01


def test_hand_worked_case(golden_dir):
    with open(os.path.join(golden_dir, "resolve_hand.json")) as f:
        g = json.load(f)
    n, S, k = g["seq_len"], g["S"], g["k"]
    host = pinned_uint8(n * 656).reshape(n, 656)
    host[:] = (np.arange(n)[:, None] * 7 + np.arange(656)[None, :]).astype(np.uint8)
    pool = torch.zeros((400, 656), dtype=torch.uint8, device="cuda")
    stok = torch.full((1, S), -1, dtype=torch.int32, device="cuda")
    sst = torch.full((1, S), -1, dtype=torch.int32, device="cuda")
    t2s = torch.full((1, n), -1, dtype=torch.int32, device="cuda")
    out = torch.empty((1, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((1, 3), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for st in g["steps"]:
        hs_hisparse_resolve(st["step"], torch.tensor([st["idx"]], dtype=torch.int32, device="cuda"),
                            torch.tensor([n], dtype=torch.int32, device="cuda"),
                            torch.tensor([g["resident_start"]], dtype=torch.int32, device="cuda"),
                            torch.tensor([[g["page0_block"]]], dtype=torch.int32, device="cuda"),
                            torch.tensor([host.ctypes.data], dtype=torch.int64, device="cuda"), pool,
                            torch.tensor([g["slot_row"]], dtype=torch.int32, device="cuda"), stok, sst, t2s, out, cnt, err)
        assert hs_check_flag(err) == 0
        assert out.cpu().tolist()[0] == st["out_rows"], st["why"]
        assert cnt.cpu().tolist()[0] == st["counters"]
        assert stok.cpu().tolist()[0] == st["slot_token"]
        assert sst.cpu().tolist()[0] == st["slot_stamp"]


def test_contract_violation_flagged_and_state_untouched():
    n, S = 100, 4
    host = pinned_uint8(n * 656).reshape(n, 656)
    pool = torch.zeros((300, 656), dtype=torch.uint8, device="cuda")
    stok = torch.full((1, S), -1, dtype=torch.int32, device="cuda")
    sst = torch.full((1, S), -1, dtype=torch.int32, device="cuda")
    t2s = torch.full((1, n), -1, dtype=torch.int32, device="cuda")
    out = torch.empty((1, 3), dtype=torch.int32, device="cuda")
    cnt = torch.empty((1, 3), dtype=torch.int32, device="cuda")
    for bad, bit in (([5, 3, -1], 0x08), ([5, -1, 7], 0x08), ([5, 100, -1], 0x01)):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        hs_hisparse_resolve(0, torch.tensor([bad], dtype=torch.int32, device="cuda"),
                            torch.tensor([n], dtype=torch.int32, device="cuda"),
                            torch.tensor([90], dtype=torch.int32, device="cuda"),
                            torch.zeros((1, 2), dtype=torch.int32, device="cuda"),
                            torch.tensor([host.ctypes.data], dtype=torch.int64, device="cuda"), pool,
                            torch.tensor([[200, 201, 202, 203]], dtype=torch.int32, device="cuda"), stok, sst, t2s,
                            out, cnt, err)
        assert hs_check_flag(err) & bit
        assert (stok == -1).all() and (t2s == -1).all()
