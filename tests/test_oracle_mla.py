"""Pins of the oracle's sparse MLA: dense attention through torch's scaled_dot_product_attention
when the index set is every visible row, closed forms on hand-built rows, and invariances."""
import math

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_mla_gb300 import inputs


def _decode_rows(rows):
    """Library decode of 656-byte rows: (latent*scale [N,512], rope [N,64]) in float64."""
    codes = torch.from_numpy(np.ascontiguousarray(rows[:, :512])).view(torch.float8_e4m3fn).double()
    scales = torch.from_numpy(np.ascontiguousarray(rows[:, 512:528]).view(np.float32).copy()).double()
    lat = codes * scales.repeat_interleave(128, dim=1)
    rope = torch.from_numpy(np.ascontiguousarray(rows[:, 528:]).view(np.int16).copy()).view(torch.bfloat16).double()
    return lat, rope


def _q64(qbits):
    return torch.from_numpy(qbits.view(np.int16)).view(torch.bfloat16).double()


@pytest.mark.parametrize("H,n", [(1, 1), (4, 7), (16, 130)])
def test_full_index_set_equals_dense_attention(H, n):
    st = inputs.Stream(10 + n)
    rows = inputs.pack_kv_rows(st.sub("l").normal((n, 512)), st.sub("r").normal((n, 64)))
    qbits = inputs.bf16_bits(st.sub("q").normal((1, H, 576), sigma=0.5))
    idx = np.arange(n, dtype=np.int32)[None, ::-1].copy()  # any order
    scale = 1 / math.sqrt(576)
    out, lse = oracle.sparse_mla(qbits, rows, idx, scale)
    lat, rope = _decode_rows(rows)
    K = torch.cat([lat, rope], dim=1)[None, None]       # [1,1,n,576]
    V = lat[None, None]                                 # [1,1,n,512]
    Q = _q64(qbits)[:, :, None, :].permute(0, 1, 2, 3)  # [1,H,1,576]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K.expand(1, H, n, 576), V.expand(1, H, n, 512), scale=scale)
    assert np.allclose(out[0], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12)
    logits = (Q[0, :, 0] @ K[0, 0].T) * scale
    assert np.allclose(lse[0], torch.logsumexp(logits, dim=1).numpy(), rtol=1e-12, atol=1e-12)


def _rows(latent, rope, group_scales=None):
    return inputs.pack_kv_rows(np.asarray(latent, np.float32), np.asarray(rope, np.float32),
                               None if group_scales is None else np.asarray(group_scales, np.float32))


def test_two_rows_closed_form():
    """logits +1 and -1 -> out[0] = 2 tanh(1), lse = ln(2 cosh 1)."""
    lat = np.zeros((2, 512)); lat[0, 0], lat[1, 0] = 2.0, -2.0
    rows = _rows(lat, np.zeros((2, 64)), np.ones((2, 4)))
    q = np.zeros((1, 1, 576), np.float32); q[0, 0, 0] = 0.5
    out, lse = oracle.sparse_mla(inputs.bf16_bits(q), rows, np.array([[0, 1]], np.int32), 1.0)
    assert out[0, 0, 0] == pytest.approx(2 * math.tanh(1), rel=1e-15)
    assert np.all(out[0, 0, 1:] == 0)
    assert lse[0, 0] == pytest.approx(math.log(2 * math.cosh(1)), rel=1e-15)


def test_rope_part_enters_logits_only():
    """q on a RoPE dim: logits (1, 0); outputs mix latents only."""
    lat = np.zeros((2, 512)); lat[0, 3], lat[1, 3] = 1.0, 2.0
    rope = np.zeros((2, 64)); rope[0, 0] = 1.0; rope[1, 5] = 100.0
    rows = _rows(lat, rope, np.ones((2, 4)))
    q = np.zeros((1, 1, 576), np.float32); q[0, 0, 512] = 1.0
    out, lse = oracle.sparse_mla(inputs.bf16_bits(q), rows, np.array([[1, 0]], np.int32), 1.0)
    p0 = math.e / (1 + math.e)
    assert out[0, 0, 3] == pytest.approx(p0 * 1 + (1 - p0) * 2, rel=1e-15)
    assert lse[0, 0] == pytest.approx(math.log(1 + math.e), rel=1e-15)


def test_uniform_logits_mean_and_group_scales():
    """q = 0: out = mean of the (group-scaled) latents, lse = ln n."""
    n = 5
    lat = np.ones((n, 512))
    gs = np.array([[1, 2, 3, 4]] * n, np.float32)
    rows = _rows(lat * np.repeat(gs, 128, axis=1), np.zeros((n, 64)), gs)
    q = np.zeros((1, 2, 576), np.float32)
    out, lse = oracle.sparse_mla(inputs.bf16_bits(q), rows, np.arange(n, dtype=np.int32)[None], 0.3)
    want = np.repeat(np.array([1.0, 2.0, 3.0, 4.0]), 128)
    assert np.array_equal(out[0, 0], want) and np.array_equal(out[0, 1], want)
    assert lse[0, 0] == pytest.approx(math.log(n), rel=1e-15)


def test_padding_duplicates_empty_and_paging():
    st = inputs.Stream(7)
    n = 200
    ctx = np.array([n], np.int32)
    bt, nblk = inputs.paged_block_tables(ctx, st.sub("bt"))
    tok_rows = inputs.pack_kv_rows(st.sub("l").normal((n, 512)), st.sub("r").normal((n, 64)))
    pool = inputs.scatter_paged(tok_rows, ctx, bt, nblk)
    q = inputs.bf16_bits(st.sub("q").normal((3, 2, 576)))
    idx = np.array([[5, 17, 199, -1, -1], [-1, -1, -1, -1, -1], [199, 5, -1, 17, -1]], np.int32)
    out, lse = oracle.sparse_mla(q, pool, idx, 0.05, block_table=bt, token_req=np.zeros(3, np.int32))
    # logical indices through the block table == physical indices into token-ordered rows
    out_p, lse_p = oracle.sparse_mla(q, tok_rows, idx, 0.05)
    assert np.array_equal(out, out_p) and np.array_equal(lse, lse_p)
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    # order and padding position do not matter
    q2 = q.copy(); q2[2] = q[0]
    out2, _ = oracle.sparse_mla(q2, tok_rows, idx, 0.05)
    assert np.allclose(out2[2], out2[0], rtol=1e-14, atol=1e-14)
    # a duplicated row counts twice: equivalent to doubling its weight -> shifts the mean toward it
    dup = np.array([[5, 5, 17]], np.int32)
    o_dup, l_dup = oracle.sparse_mla(q[:1], tok_rows, dup, 0.0)
    lat, _ = _decode_rows(tok_rows)
    assert np.allclose(o_dup[0, 0], ((2 * lat[5] + lat[17]) / 3).numpy(), rtol=1e-13, atol=1e-13)
    assert l_dup[0, 0] == pytest.approx(math.log(3))


def test_out_of_range_row_rejected():
    rows = _rows(np.zeros((2, 512)), np.zeros((2, 64)), np.ones((2, 4)))
    with pytest.raises(oracle.OracleError):
        oracle.sparse_mla(np.zeros((1, 1, 576), np.uint16), rows, np.array([[0, 2]], np.int32), 1.0)


def test_shared_index_sets_hand_case():
    """One request's set [0, 5, 9, -1] shared by three tokens that see 3, 6 and 10 tokens: each
    keeps the entries it can see (worked by hand)."""
    idx = np.array([[0, 5, 9, -1], [7, 7, 1, 2]], np.int32)
    got = oracle.shared_index_sets(idx, np.array([0, 0, 0, 1]), np.array([3, 6, 10, 2]))
    want = np.array([[0, -1, -1, -1], [0, 5, -1, -1], [0, 5, 9, -1], [-1, -1, 1, -1]], np.int32)
    assert np.array_equal(got, want)
    # without a limit the rows are copied as they are
    assert np.array_equal(oracle.shared_index_sets(idx, np.array([1, 0])), idx[::-1])
    with pytest.raises(oracle.OracleError):
        oracle.shared_index_sets(idx, np.array([0, 2]))


def test_shared_sets_give_causal_attention_for_every_mtp_token():
    """Two requests decode 1 + 3 MTP tokens each; all four share the set of the final token.
    When that set holds every token of the request (in any order, padded), token i at position
    p must attend exactly the tokens at positions <= p: dense causal attention, here torch's
    scaled_dot_product_attention with a position mask."""
    st = inputs.Stream(41)
    ctx = np.array([150, 97], np.int32)
    bt, nblk = inputs.paged_block_tables(ctx, st.sub("bt"))
    tok_rows = inputs.pack_kv_rows(st.sub("l").normal((int(ctx.sum()), 512)), st.sub("r").normal((int(ctx.sum()), 64)))
    pool = inputs.scatter_paged(tok_rows, ctx, bt, nblk)
    H, k = 3, 160
    token_req = np.repeat(np.arange(2, dtype=np.int32), 4)
    pos = np.concatenate([c - 4 + np.arange(4) for c in ctx]).astype(np.int32)
    g = st.sub("perm").gen()
    final = np.full((2, k), -1, np.int32)
    for r, c in enumerate(ctx):
        final[r, :c] = g.permutation(int(c))
        final[r] = final[r][g.permutation(k)]  # padding anywhere
    sets = oracle.shared_index_sets(final, token_req, pos + 1)
    q = inputs.bf16_bits(st.sub("q").normal((8, H, 576), sigma=0.5))
    scale = 1 / math.sqrt(576)
    out, lse = oracle.sparse_mla(q, pool, sets, scale, block_table=bt, token_req=token_req)
    lat, rope = _decode_rows(tok_rows)
    Q = _q64(q)
    off = np.concatenate([[0], np.cumsum(ctx)[:-1]])
    for t in range(8):
        r = token_req[t]
        K = torch.cat([lat, rope], dim=1)[off[r]:off[r] + ctx[r]]
        V = lat[off[r]:off[r] + ctx[r]]
        mask = (torch.arange(int(ctx[r])) <= int(pos[t]))[None, None, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q[t][None, :, None, :], K[None, None].expand(1, H, -1, 576), V[None, None].expand(1, H, -1, 512),
            attn_mask=mask, scale=scale)
        assert np.allclose(out[t], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12), t
        logits = (Q[t] @ K.T) * scale
        logits[:, int(pos[t]) + 1:] = -math.inf
        assert np.allclose(lse[t], torch.logsumexp(logits, dim=1).numpy(), rtol=1e-12, atol=1e-12), t
    # the final token of each request sees its whole set
    assert np.array_equal(sets[3], final[0]) and np.array_equal(sets[7], final[1])
