"""GPU parity of hs_sparse_mla_fwd against the oracle run on the same index set."""
import math

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_mla_gb300 import HSError, hs_check_flag, hs_sparse_mla_fwd, hs_sparse_mla_workspace_size, inputs

from parity import check_mla

pytestmark = pytest.mark.gpu


def _rows(n, seed, group_scales=False):
    st = inputs.Stream(seed)
    lat = st.sub("l").normal((n, 512))
    rope = st.sub("r").normal((n, 64))
    gs = None
    if group_scales:
        gs = (np.abs(lat).reshape(n, 4, 128).max(-1) / 448 * np.array([1.25, 3.0, 1.5, 7.0])).astype(np.float32)
    return inputs.pack_kv_rows(lat, rope, gs)


def _workspace(H):
    return torch.empty(hs_sparse_mla_workspace_size(H), dtype=torch.uint8, device="cuda")


def _run(q_bits, kv, idx, scale, bt=None, req=None, split=False, idx_row=None, kvlen=None):
    T, H, _ = q_bits.shape
    q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(torch.bfloat16)
    kvt = torch.from_numpy(kv).cuda()
    it = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda()
    out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    btt = None if bt is None else torch.from_numpy(bt).cuda()
    rt = None if req is None else torch.from_numpy(req).cuda()
    ws = _workspace(H) if split else None
    if ws is not None:
        ws.fill_(0xFF)   # the workspace needs no initialisation: stale contents must not matter
    ir = None if idx_row is None else torch.from_numpy(np.ascontiguousarray(idx_row, np.int32)).cuda()
    kl = None if kvlen is None else torch.from_numpy(np.ascontiguousarray(kvlen, np.int32)).cuda()
    hs_sparse_mla_fwd(q, kvt, it, scale, out, err, lse=lse, block_table=btt, token_req=rt, workspace=ws,
                      idx_row=ir, token_kvlen=kl)
    flag = hs_check_flag(err)
    return out, lse, flag


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("H,k,n", [(64, 2048, 5000), (64, 130, 300), (16, 256, 1024), (64, 64, 64), (1, 1, 1),
                                   (40, 200, 777)])
def test_random_index_sets(H, k, n, split):
    rng = np.random.default_rng(H * 1000 + k)
    T = 7
    kv = _rows(n, seed=k + n)
    q = inputs.bf16_bits(inputs.Stream(n).sub("q").normal((T, H, 576)))
    idx = np.stack([rng.permutation(n)[:k] if k <= n else rng.integers(0, n, k) for _ in range(T)]).astype(np.int32)
    idx[1, k // 3:] = -1                       # ragged valid count
    if k > 4:
        idx[2, 3] = idx[2, 0]                  # duplicate entry
    idx[4, :] = -1                             # empty query
    scale = 1 / math.sqrt(576)
    out, lse, flag = _run(q, kv, idx, scale, split=split)
    assert flag == 0
    ref, lref = oracle.sparse_mla(q, kv, idx, scale)
    check_mla(out, lse, ref, lref)


@pytest.mark.parametrize("T,k", [(1, 2048), (3, 2048), (157, 512), (40, 256), (64, 1984)])
def test_work_split_across_sms(T, k):
    """Equal shares per SM: queries split between SMs (partials merged by log-sum-exp), fewer
    queries than SMs, batches that are not a multiple of the SM count, a ragged last tile;
    the result equals the oracle and the one-CTA-per-query path."""
    n, H = 3000, 64
    rng = np.random.default_rng(T * 7 + k)
    kv = _rows(n, seed=T + k)
    q = inputs.bf16_bits(inputs.Stream(T + 11).sub("q").normal((T, H, 576)))
    idx = np.stack([rng.integers(0, n, k) for _ in range(T)]).astype(np.int32)
    idx[0, k // 2:] = -1                       # a query whose second half is padding
    if T > 2:
        idx[2, :] = -1                         # an empty query
    scale = 1 / math.sqrt(576)
    out, lse, flag = _run(q, kv, idx, scale, split=True)
    assert flag == 0
    ref, lref = oracle.sparse_mla(q, kv, idx, scale)
    check_mla(out, lse, ref, lref)
    out1, lse1, flag1 = _run(q, kv, idx, scale, split=False)
    assert flag1 == 0
    d = (out.float() - out1.float()).abs().max().item()
    assert d <= 2e-2 * max(1.0, out1.float().abs().max().item())


def test_workspace_too_small_rejected():
    H = 64
    q = torch.zeros((2, H, 576), dtype=torch.bfloat16, device="cuda")
    kvt = torch.zeros((8, 656), dtype=torch.uint8, device="cuda")
    it = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    out = torch.empty((2, H, 512), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(hs_sparse_mla_workspace_size(H) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(HSError, match="workspace"):
        hs_sparse_mla_fwd(q, kvt, it, 0.1, out, err, workspace=ws)


@pytest.mark.parametrize("sigma", [1.5, 3.0, 4.0])
def test_distinct_group_scales_and_large_logits(sigma):
    """Four different group scales per row (up to 7x the row's amax / 448) and a peaky softmax:
    with q ~ N(0, 3^2) the logits' spread is a few tens, so a few rows carry the weight and any
    bias in a row's dequantised values moves the output."""
    n, T, H, k = 600, 5, 64, 512
    kv = _rows(n, seed=3, group_scales=True)
    q = inputs.bf16_bits(inputs.Stream(4).sub("q").normal((T, H, 576), sigma=sigma))
    rng = np.random.default_rng(0)
    idx = np.stack([rng.permutation(n)[:k] for _ in range(T)]).astype(np.int32)
    out, lse, flag = _run(q, kv, idx, 0.125)
    assert flag == 0
    ref, lref = oracle.sparse_mla(q, kv, idx, 0.125)
    check_mla(out, lse, ref, lref)


@pytest.mark.parametrize("sigma", [1e-5, 1e-30, 3e4, 1e12])
def test_query_magnitudes_outside_fp16(sigma):
    """Queries far below fp16's normal range (|q| < 2^-14) or far above its largest value: every
    head's row is brought into fp16's range by an exact power of two, so the result matches the
    oracle as for ordinary magnitudes and no range flag is raised. The softmax scale keeps the
    logits of order one; one head is scaled 2^20 above the others."""
    n, T, H, k = 700, 4, 64, 600
    kv = _rows(n, seed=8)
    x = inputs.Stream(9).sub("q").normal((T, H, 576))
    x[:, 5] *= 2.0 ** 20
    q = inputs.bf16_bits(x * sigma)
    rng = np.random.default_rng(2)
    idx = np.stack([rng.permutation(n)[:k] for _ in range(T)]).astype(np.int32)
    scale = 0.3 / sigma
    out, lse, flag = _run(q, kv, idx, scale)
    assert flag == 0
    ref, lref = oracle.sparse_mla(q, kv, idx, scale)
    check_mla(out, lse, ref, lref)


def test_non_finite_query_is_flagged():
    kv = _rows(64, seed=6)
    x = inputs.Stream(6).sub("q").normal((2, 8, 576))
    x[1, 3, 100] = np.inf
    q = inputs.bf16_bits(x)
    _, _, flag = _run(q, kv, np.arange(64, dtype=np.int32)[None].repeat(2, 0), 0.05)
    assert flag & 0x40


def test_paged_logical_indices():
    w = inputs.config2(seed=31, B=3, lo=300, hi=3000, Hi=8, Di=64, H=64, topk=256)
    rng = np.random.default_rng(1)
    idx = np.full((w.T, w.topk), -1, np.int32)
    for t in range(w.T):
        n = int(w.token_kvlen[t])
        sel = np.sort(rng.choice(n, size=min(n, w.topk), replace=False))
        idx[t, :len(sel)] = sel
    out, lse, flag = _run(w.q_mla, w.kv_pool, idx, w.softmax_scale, w.block_table, w.token_req)
    assert flag == 0
    ref, lref = oracle.sparse_mla(w.q_mla, w.kv_pool, idx, w.softmax_scale, w.block_table, w.token_req)
    check_mla(out, lse, ref, lref)


def test_out_of_range_rows_flagged_and_skipped():
    kv = _rows(100, seed=5)
    q = inputs.bf16_bits(inputs.Stream(5).sub("q").normal((2, 8, 576)))
    idx = np.array([[1, 2, 100, 3], [5, 6, 7, 8]], np.int32)
    out, lse, flag = _run(q, kv, idx, 0.05)
    assert flag & 0x01
    ref, lref = oracle.sparse_mla(q, kv, np.array([[1, 2, -1, 3], [5, 6, 7, 8]], np.int32), 0.05)
    check_mla(out, lse, ref, lref)


def test_host_side_validation():
    kv = torch.zeros((10, 656), dtype=torch.uint8, device="cuda")
    q = torch.zeros((1, 65, 576), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    out = torch.empty((1, 65, 512), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(HSError):
        hs_sparse_mla_fwd(q, kv, idx, 1.0, out, err)   # H = 65 > 64


def test_out_of_fp16_range_scale_is_flagged():
    """A group scale too large for the fp16 compute path sets HS_FLAG_RANGE (0x40)."""
    n = 64
    lat = np.zeros((n, 512), np.float32)
    gs = np.full((n, 4), 0.01, np.float32)
    gs[7, 2] = 1000.0
    kv = inputs.pack_kv_rows(lat, np.zeros((n, 64), np.float32), gs)
    q = inputs.bf16_bits(np.ones((1, 4, 576), np.float32))
    _, _, flag = _run(q, kv, np.arange(n, dtype=np.int32)[None], 0.05)
    assert flag & 0x40
    _, _, flag = _run(q, kv, np.array([[0, 1, 2, 3]], np.int32), 0.05)
    assert flag == 0


def _final_token_sets(w, rng):
    """Per request, a top-k-sized set for its final query token that always holds the three
    latest positions (the ones the earlier MTP tokens may not see), in random order."""
    B = w.block_table.shape[0]
    final = np.full((B, w.topk), -1, np.int32)
    for r in range(B):
        n = int(w.token_kvlen[w.token_req == r].max())
        m = min(n - 3, w.topk - 3)
        sel = np.concatenate([np.arange(n - 3, n), rng.choice(n - 3, size=m, replace=False)])
        final[r, :len(sel)] = rng.permutation(sel)
    return final


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("topk", [256, 2048])
def test_shared_index_sets_across_mtp_tokens(topk, split):
    """The four MTP tokens of a request attend its final token's set (idx_row), each limited to
    the tokens it can see (token_kvlen): parity with the oracle on the expanded sets, and the same
    bits as a call on those expanded sets."""
    w = inputs.config2(seed=37, B=5, lo=300, hi=3000, Hi=8, Di=64, H=64, topk=topk)
    final = _final_token_sets(w, np.random.default_rng(topk))
    sets = oracle.shared_index_sets(final, w.token_req, w.token_kvlen)
    assert (sets >= 0).sum() < 4 * (final >= 0).sum()   # the earlier tokens lost entries
    out, lse, flag = _run(w.q_mla, w.kv_pool, final, w.softmax_scale, w.block_table, w.token_req, split=split,
                          idx_row=w.token_req, kvlen=w.token_kvlen)
    assert flag == 0
    ref, lref = oracle.sparse_mla(w.q_mla, w.kv_pool, sets, w.softmax_scale, w.block_table, w.token_req)
    check_mla(out, lse, ref, lref)
    out2, lse2, flag2 = _run(w.q_mla, w.kv_pool, sets, w.softmax_scale, w.block_table, w.token_req, split=split)
    assert flag2 == 0
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_shared_index_row_out_of_range_flagged():
    """A query naming an idx row that does not exist gets no rows (out 0, lse -inf) and sets
    HS_FLAG_BAD_INDEX; the other queries are unaffected."""
    w = inputs.config2(seed=38, B=2, lo=300, hi=900, Hi=8, Di=64, H=16, topk=128)
    final = _final_token_sets(w, np.random.default_rng(5))
    rows = w.token_req.copy()
    rows[2] = 2                                          # only rows 0 and 1 exist
    out, lse, flag = _run(w.q_mla, w.kv_pool, final, w.softmax_scale, w.block_table, w.token_req,
                          idx_row=rows, kvlen=w.token_kvlen)
    assert flag & 0x01
    sets = oracle.shared_index_sets(final, w.token_req, w.token_kvlen)
    sets[2] = -1
    ref, lref = oracle.sparse_mla(w.q_mla, w.kv_pool, sets, w.softmax_scale, w.block_table, w.token_req)
    check_mla(out, lse, ref, lref)
