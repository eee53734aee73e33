"""Pins the oracle's FP8 / bf16 decoders to library conversions (torch)."""
import math

import numpy as np
import torch

import oracle


def test_e4m3_all_256_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])


def test_e4m3_landmarks():
    # OCP e4m3: max normal 448, min normal 2^-6, min subnormal 2^-9, NaN at S.1111.111
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x80) == 0.0 and math.copysign(1, oracle.e4m3_decode(0x80)) < 0
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4096).astype(np.uint16)
    bits[:4] = [0x3F80, 0xBF80, 0x7F80, 0x0001]
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b, r in zip(bits, ref):
        got = oracle.bf16_decode(int(b))
        assert (math.isnan(got) and math.isnan(r)) or got == r
