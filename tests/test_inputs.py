"""The seeded generator is deterministic and produces the documented layouts."""
import numpy as np

from dsa_sparse_mla_gb300 import inputs


def test_streams_are_reproducible_and_independent():
    a = inputs.Stream(3).sub("x").normal((1000,))
    b = inputs.Stream(3).sub("x").normal((1000,))
    c = inputs.Stream(3).sub("y").normal((1000,))
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    big = inputs.Stream(1).sub("z").normal((3 * (1 << 22) + 5,))   # several chunks, threaded
    assert np.array_equal(big, inputs.Stream(1).sub("z").normal((3 * (1 << 22) + 5,)))


def test_small_decode_workload_layout():
    w = inputs.config2(seed=11, B=3, lo=100, hi=300, Hi=8, Di=64, H=4, topk=32)
    assert w.T == 12 and w.q_idx.shape == (12, 8, 64) and w.q_mla.shape == (12, 4, 576)
    for r in range(3):
        n = int(w.ctx[r])
        assert w.token_kvlen[4 * r:4 * r + 4].tolist() == [n - 3, n - 2, n - 1, n]
        pages = w.block_table[r][w.block_table[r] >= 0]
        assert len(pages) == (n + 63) // 64
    used = w.block_table[w.block_table >= 0]
    assert sorted(used.tolist()) == list(range(w.nblk))       # one permutation of all pages
    assert w.kv_pool.shape == (w.nblk * 64, 656) and w.ld % 4 == 0 and w.ld >= w.token_kvlen.max()
    # per-row scale replicated into the four group slots, all positive
    sc = w.kv_pool[:, 512:528].copy().view(np.float32)
    live = sc[:, 0] > 0
    assert np.all(sc[live] == sc[live, :1])


def test_hisparse_stream_overlap_and_order():
    seq = np.array([20000, 30000])
    s = inputs.hisparse_index_stream(seq, 4096, 256, 5, 0.8, inputs.Stream(2))
    for r in range(2):
        for st in range(5):
            row = s[st, r]
            assert np.all(np.diff(row) > 0) and row[0] >= 0 and row[-1] < seq[r] - 4096
        for st in range(1, 5):
            assert len(np.intersect1d(s[st, r], s[st - 1, r])) == round(0.8 * 256)


def test_long_prefill_pass_chunks_equal_single_chunk_builds():
    """config4_pass builds the cache once and each chunk's queries from the chunk's own stream:
    every chunk is byte for byte the workload config4 builds for that chunk alone, and different
    chunks have different query values."""
    kw = dict(total=4096, chunk_len=512, Hi=8, Di=64, H=4, topk=64)
    ws = inputs.config4_pass(chunks=[0, 3, 7], **kw)
    for c, w in zip([0, 3, 7], ws):
        one = inputs.config4(c, **kw)
        for f in ("q_idx", "q_scale", "weights", "q_mla", "token_kvlen", "token_req", "k_cache", "k_scale",
                  "block_table", "kv_pool"):
            assert np.array_equal(getattr(w, f), getattr(one, f)), (c, f)
        assert w.token_kvlen.tolist() == list(range(512 * c + 1, 512 * c + 513))
    assert not np.array_equal(ws[0].q_mla, ws[1].q_mla)
    assert ws[1].kv_pool is ws[0].kv_pool          # the cache is shared, not copied
