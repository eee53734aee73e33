"""Oracle KV append (FP8 quantiser of new tokens) against the OCP e4m3 rules and hand-worked values.

The pages give the row sizes (656-byte MLA row, 132-byte indexer key: 128 FP8 values + 4-byte
scale); the quantiser is the plain reading scale = max(amax / 448, 2^-14), code = e4m3(x / scale)
in binary32, rounding to nearest even and saturating at +-448.
"""
import math

import numpy as np
import pytest
import torch

import oracle

FINITE = [c for c in range(256) if c not in (0x7F, 0xFF)]


def test_every_finite_code_round_trips():
    for c in FINITE:
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_midpoints_go_to_the_even_code_and_neighbours_to_the_nearer_one():
    for c in range(0x00, 0x7E):  # positive codes c, c + 1 (0x7E is the largest finite)
        a, b = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = np.float32((a + b) / 2)
        assert float(mid) == (a + b) / 2  # exactly representable
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even, hex(c)
        assert oracle.e4m3_encode(-mid) == 0x80 | even
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(1000))
        assert oracle.e4m3_encode(below) == c
        assert oracle.e4m3_encode(above) == c + 1


def test_saturation_and_nan():
    for x, code in ((448.0, 0x7E), (463.9, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (math.inf, 0x7E),
                    (-500.0, 0xFE), (-math.inf, 0xFE), (0.0, 0x00), (-0.0, 0x80)):
        assert oracle.e4m3_encode(x) == code, x
    assert oracle.e4m3_encode(math.nan) & 0x7F == 0x7F


def test_matches_torch_float8_cast_in_range():
    g = np.random.default_rng(0)
    x = np.concatenate([g.normal(0, s, 20000) for s in (1e-3, 0.05, 1.0, 30.0, 150.0)]).astype(np.float32)
    x = np.clip(x, -448.0, 448.0)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _layout(B=2, pages=4, R_extra=64, Di=128, seed=1):
    g = np.random.default_rng(seed)
    nblk = B * pages + 3
    perm = g.permutation(nblk).astype(np.int32)
    bt = perm[:B * pages].reshape(B, pages)
    kv = np.zeros((nblk * 64 + R_extra, 656), np.uint8)
    kc = np.zeros((nblk, 64, Di), np.uint8)
    ks = np.zeros((nblk, 64), np.float32)
    return bt, kv, kc, ks


def test_hand_worked_token():
    # group 0 amax 3.5: scale = 3.5 / 448 = 2^-7 exactly, so the codes are those of 128 x
    lat = np.zeros((1, 512), np.float32)
    lat[0, :5] = [1.0, 3.5, -0.5, 0.01, -3.5]
    lat[0, 128] = 0.75  # group 1: amax 0.75 -> scale 0.75 / 448
    rope = np.arange(64, dtype=np.float32)[None] / 8
    key = np.zeros((1, 128), np.float32)
    key[0, 0], key[0, 1] = -7.0, 1.75  # amax 7: scale 2^-6, codes of 64 x
    bt, kv, kc, ks = _layout()
    oracle.kv_append(_bf16(lat), _bf16(rope), _bf16(key), np.array([1], np.int32), np.array([70], np.int32), bt,
                     kv, kc.reshape(-1, 128), ks.reshape(-1), B=2)
    row = int(bt[1, 1]) * 64 + 6
    r = kv[row]
    # 128 -> 2^7: exponent 7 + 7 = 14, mantissa 0; 448 -> 0x7E; -64 -> 0x80 | (6 + 7) << 3;
    # 0.01 (bf16 0.010009765625) x 128 = 1.28125 -> 1.25 = 0x3A; -448 -> 0xFE
    assert list(r[:5]) == [0x70, 0x7E, 0xE8, 0x3A, 0xFE]
    assert not r[5:128].any() and r[128] == 0x7E
    scales = r[512:528].view(np.float32)
    assert scales[0] == np.float32(2.0 ** -7)
    assert scales[1] == np.float32(np.float32(0.75) / np.float32(448.0))
    assert scales[2] == scales[3] == np.float32(2.0 ** -14)  # all-zero groups: the floor
    assert np.array_equal(r[528:656].view(np.uint16), _bf16(rope)[0])
    krow = kc.reshape(-1, 128)[row]
    # -7 x 64 = -448 -> 0xFE; 1.75 x 64 = 112 -> 2^6 x 1.75: exponent 13, mantissa 6 -> 0x6E
    assert krow[0] == 0xFE and krow[1] == 0x6E and not krow[2:].any()
    assert ks.reshape(-1)[row] == np.float32(2.0 ** -6)
    # nothing else was written
    kv[row] = 0
    assert not kv.any()


def test_dequantised_rows_approximate_the_inputs():
    g = np.random.default_rng(3)
    T, Di = 40, 128
    lat = g.normal(0, 1, (T, 512)).astype(np.float32) * g.uniform(0.01, 20, (T, 1)).astype(np.float32)
    rope = g.normal(0, 1, (T, 64)).astype(np.float32)
    key = g.normal(0, 2, (T, Di)).astype(np.float32)
    bt, kv, kc, ks = _layout(B=2, pages=4, Di=Di, seed=4)
    req = g.integers(0, 2, T).astype(np.int32)
    # distinct positions per request so that no row is written twice
    pos = np.array([i * 6 + (1 if req[i] else 0) for i in range(T)], np.int32)
    lb, kb = _bf16(lat), _bf16(key)
    oracle.kv_append(lb, _bf16(rope), kb, req, pos, bt, kv, kc.reshape(-1, Di), ks.reshape(-1), B=2)
    dec = np.array([oracle.e4m3_decode(c) for c in range(256)])
    xl = torch.from_numpy(lb.view(np.int16)).view(torch.bfloat16).float().numpy()
    xk = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).float().numpy()
    for t in range(T):
        row = int(bt[req[t], pos[t] // 64]) * 64 + pos[t] % 64
        r = kv[row]
        sc = r[512:528].view(np.float32)
        for gi in range(4):
            x = xl[t, 128 * gi:128 * (gi + 1)]
            y = dec[r[128 * gi:128 * (gi + 1)]] * sc[gi]
            assert sc[gi] >= 2.0 ** -14
            assert np.abs(y).max() == pytest.approx(np.abs(x).max(), rel=2 ** -4)  # the amax maps to +-448
            # e4m3 keeps 3 mantissa bits: error <= 2^-4 relative (normal codes) or 2^-10 * scale
            assert np.all(np.abs(y - x) <= np.maximum(np.abs(x) * 2 ** -4, sc[gi] * 2 ** -10) * 1.0001)
        yk = dec[kc.reshape(-1, Di)[row]] * ks.reshape(-1)[row]
        assert np.all(np.abs(yk - xk[t]) <= np.maximum(np.abs(xk[t]) * 2 ** -4, ks.reshape(-1)[row] * 2 ** -10) * 1.0001)


def test_optional_parts_and_contract_violations():
    bt, kv, kc, ks = _layout()
    lat, rope, key = np.ones((1, 512), np.float32), np.ones((1, 64), np.float32), np.ones((1, 128), np.float32)
    oracle.kv_append(None, None, _bf16(key), np.array([0], np.int32), np.array([3], np.int32), bt, kv,
                     kc.reshape(-1, 128), ks.reshape(-1), B=2)
    assert not kv.any() and kc.any()
    for req, pos in ((2, 0), (-1, 0), (0, -1), (0, 4 * 64)):
        with pytest.raises(oracle.OracleError):
            oracle.kv_append(_bf16(lat), _bf16(rope), _bf16(key), np.array([req], np.int32), np.array([pos], np.int32),
                             bt, kv, kc.reshape(-1, 128), ks.reshape(-1), B=2)
