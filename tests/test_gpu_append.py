"""GPU FP8 KV append is bit-exact against the oracle: codes, scales, RoPE bytes and placement."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_mla_gb300 import hs_check_flag, hs_kv_append

pytestmark = pytest.mark.gpu


def _inputs(T, Di, B=3, pages=None, seed=0):
    g = np.random.default_rng(seed)
    pages = pages or max(40, -(-T // (B * 64)) + 8)
    # magnitudes from tiny (scale floor) to large, zero rows, exact ties at multiples of 2^-10
    mag = g.choice([1e-6, 1e-3, 0.05, 1.0, 7.0, 200.0], size=(T, 1))
    lat = (g.normal(0, 1, (T, 512)) * mag).astype(np.float32)
    lat[0] = 0.0
    if T > 1:
        lat[1, :128] = np.arange(128) * 2.0 ** -10
    key = (g.normal(0, 1, (T, Di)) * g.choice([1e-5, 0.3, 4.0], size=(T, 1))).astype(np.float32)
    rope = g.normal(0, 1, (T, 64)).astype(np.float32)
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    nblk = B * pages + 5
    bt = g.permutation(nblk)[:B * pages].reshape(B, pages).astype(np.int32)
    # distinct (request, position) pairs: every token its own row
    pairs = g.choice(B * pages * 64, size=T, replace=False)
    req, pos = (pairs // (pages * 64)).astype(np.int32), (pairs % (pages * 64)).astype(np.int32)
    return bf(lat), bf(rope), bf(key), req, pos, bt, nblk


def _run(T, Di, latent=True, key=True, seed=0):
    lat, rope, kk, req, pos, bt, nblk = _inputs(T, Di, seed=seed)
    R = nblk * 64
    kv_ref = np.zeros((R, 656), np.uint8)
    kc_ref = np.zeros((nblk, 64, Di), np.uint8)
    ks_ref = np.zeros((nblk, 64), np.float32)
    u16 = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    oracle.kv_append(u16(lat) if latent else None, u16(rope) if latent else None, u16(kk) if key else None, req, pos,
                     bt, kv_ref, kc_ref.reshape(-1, Di), ks_ref.reshape(-1), B=bt.shape[0])
    kv = torch.zeros((R, 656), dtype=torch.uint8, device="cuda")
    kc = torch.zeros((nblk, 64, Di), dtype=torch.uint8, device="cuda")
    ks = torch.zeros((nblk, 64), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = lambda a: torch.from_numpy(a).cuda()
    hs_kv_append(c(req), c(pos), c(bt), err, latent=lat.cuda() if latent else None, rope=rope.cuda() if latent else None,
                 kv_pool=kv if latent else None, index_key=kk.cuda() if key else None, k_cache=kc if key else None,
                 k_scale=ks if key else None)
    assert hs_check_flag(err) == 0
    assert np.array_equal(kv.cpu().numpy(), kv_ref)
    assert np.array_equal(kc.cpu().numpy(), kc_ref)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), ks_ref.view(np.uint32))


@pytest.mark.parametrize("T,Di", [(1, 128), (37, 128), (300, 64), (2000, 128)])
def test_matches_oracle_bit_for_bit(T, Di):
    _run(T, Di, seed=T)


def test_latent_only_and_key_only():
    _run(50, 128, key=False, seed=5)
    _run(50, 64, latent=False, seed=6)


def test_prefill_sized_launch():
    # grid-stride: more tokens than the launch has warps
    _run(20000, 128, seed=7)


def test_bad_tokens_flagged_and_skipped():
    lat, rope, kk, _, _, bt, nblk = _inputs(4, 128, seed=9)
    # token 0 valid; 1: request out of range (B = 3); 2: page past bt_stride; 3: negative block
    req = np.array([0, 3, 1, 2], np.int32)
    pos = np.array([5, 10, 40 * 64, 130], np.int32)
    bt[2, 2] = -1
    kv = torch.zeros((nblk * 64, 656), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = lambda a: torch.from_numpy(a).cuda()
    hs_kv_append(c(req), c(pos), c(bt), err, latent=lat.cuda(), rope=rope.cuda(), kv_pool=kv)
    assert hs_check_flag(err) == 0x01 | 0x04
    # only token 0 was written
    row0 = int(bt[req[0], pos[0] // 64]) * 64 + pos[0] % 64
    out = kv.cpu().numpy()
    assert out[row0].any()
    out[row0] = 0
    assert not out.any()
