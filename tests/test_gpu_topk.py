"""GPU top-k is bit-exact against the oracle when both rank the same fp32 scores."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_mla_gb300 import hs_check_flag, hs_topk

pytestmark = pytest.mark.gpu


def _run(scores: np.ndarray, kvlen: np.ndarray, k: int) -> np.ndarray:
    s = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float32)).cuda()
    kl = torch.from_numpy(np.ascontiguousarray(kvlen, dtype=np.int32)).cuda()
    idx = torch.full((scores.shape[0], k), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs_topk(s, kl, k, idx, err)
    assert hs_check_flag(err) == 0
    return idx.cpu().numpy()


@pytest.mark.parametrize("ld,k", [(700, 64), (5000, 256), (70000, 2048)])
def test_random_with_ties_and_short_rows(ld, k):
    rng = np.random.default_rng(ld)
    T = 24
    s = rng.standard_normal((T, ld)).astype(np.float32)
    s[::2] = np.round(s[::2] * 8) / 8          # heavy ties
    s[3, :] = 1.0                              # all equal
    s[5, ::7] = 0.0
    s[5, 1::7] = -0.0                          # signed zeros tie
    kvlen = rng.integers(0, ld + 1, size=T).astype(np.int32)
    kvlen[:5] = [0, 1, k, k + 1, ld]
    got = _run(s, kvlen, k)
    ref = oracle.topk(s.astype(np.float64), kvlen, k)
    assert np.array_equal(got, ref)


def test_long_rows_like_long_prefill():
    rng = np.random.default_rng(7)
    T, ld, k = 6, 131072, 2048
    s = (rng.random((T, ld), dtype=np.float32) * 40).astype(np.float32)   # positive, like ReLU sums
    s[1] = np.float32(3.0)                                                 # one giant tie
    kvlen = np.array([ld, ld, ld - 1, 65537, 2049, 4096], np.int32)
    got = _run(s, kvlen, k)
    ref = oracle.topk(s.astype(np.float64), kvlen, k)
    assert np.array_equal(got, ref)


def test_specials_nan_and_infinities():
    s = np.array([[np.nan, -np.inf, 3.0, np.nan, np.inf, -0.0, 0.0, 2.0] * 40], np.float32)
    kvlen = np.array([320], np.int32)
    for k in (1, 7, 100, 300):
        assert np.array_equal(_run(s, kvlen, k), oracle.topk(s.astype(np.float64), kvlen, k))


def test_bad_length_flagged():
    s = torch.zeros((2, 100), dtype=torch.float32, device="cuda")
    kl = torch.tensor([50, 101], dtype=torch.int32, device="cuda")
    idx = torch.empty((2, 8), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs_topk(s, kl, 8, idx, err)
    assert hs_check_flag(err) & 0x02


@pytest.mark.parametrize("k", [256, 2048])
def test_sampled_threshold_rows(k):
    """Rows shaped for the sampled-threshold path (and its fall-backs): indexer-like positive scores,
    sorted ramps (all winners at one end), heavy upper tails, a few huge outliers, rows barely
    longer than k, and rows whose whole length fits the sample."""
    rng = np.random.default_rng(11 + k)
    ld = 70000
    rows = []
    rows.append((rng.random(ld) * 40).astype(np.float32))                      # positive, like ReLU sums
    rows.append(np.arange(ld, dtype=np.float32))                               # ascending ramp
    rows.append(np.arange(ld, 0, -1).astype(np.float32))                       # descending ramp
    rows.append(rng.exponential(1.0, ld).astype(np.float32) ** 3)             # heavy upper tail
    r = rng.standard_normal(ld).astype(np.float32)
    r[rng.choice(ld, 50, replace=False)] = 1e30                                # a few huge outliers
    rows.append(r)
    rows.append(np.round(rng.standard_normal(ld) * 2).astype(np.float32))      # few distinct values
    s = np.stack(rows + [rng.standard_normal(ld).astype(np.float32) for _ in range(6)])
    T = s.shape[0]
    kvlen = rng.integers(16384, ld + 1, size=T).astype(np.int32)
    kvlen[-4:] = [k + 1, k + 37, 4096, 4097]
    got = _run(s, kvlen, k)
    ref = oracle.topk(s.astype(np.float64), kvlen, k)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("c", [1, 20, 31, 33, 500, 1000])
def test_tie_group_at_the_threshold(c):
    """A group of c equal scores straddles the k-th place (the rest distinct): the threshold bin of
    the candidate histogram holds about c entries, so small groups take the one-warp ranking, larger
    ones the block-wide sort, and the lowest indices of the group win."""
    rng = np.random.default_rng(c)
    ld, k = 40000, 2048
    rows = []
    for r in range(4):
        s = (rng.permutation(ld) + 1).astype(np.float32)       # distinct, exactly representable
        v = np.float32(ld - k + 1 + c // 2)                      # the group's value: c // 2 of it above place k
        s[(s <= v) & (s > v - c)] = v
        rows.append(s)
    s = np.stack(rows)
    kvlen = np.array([ld, ld, ld - 5, 30000], np.int32)
    got = _run(s, kvlen, k)
    ref = oracle.topk(s.astype(np.float64), kvlen, k)
    assert np.array_equal(got, ref)
