"""Seeded synthetic inputs shaped like the pages' workloads.

This module is shared by the CUDA path's tests and benchmark and by the CPU oracle. It only
draws random numbers and lays them out (paged KV, block tables, FP8 encoding of the drawn
values); it contains none of the method's arithmetic (no scoring, selection, attention or
LRU logic).

All draws come from numpy's PCG64, split into fixed-size chunks with spawned seed sequences,
so the bytes are identical on every machine and for any thread count.

Workloads (sizes from the configuration list this library is measured on):
  1  tiny prefill: one sequence of 1024 tokens, all of them queries; index heads 8 x 64-d,
     top-k 256, 16 MLA heads, q ~ N(0, 0.5^2), softmax scale 1/sqrt(576)
  2  MTP decode: 64 requests x (1+3) query tokens, contexts ~ U{16384..65536}; 64 x 128-d index
     heads, top-k 2048, 64 MLA heads
  3  chunked prefill: one 2048-token chunk after 65536 cached tokens
  4  long prefill: one 131072-token sequence as 64 chunks of 2048 tokens (``chunk`` selects one)
  5  HiSparse mixed residency: 32 requests, contexts ~ U{262144..1048576}, last 4096 tokens
     resident, 4096 hot slots per request, Zipf(1.1) index stream with 80 % step-to-step overlap
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

PAGE = 64
ROW_BYTES = 656
D_LATENT = 512
D_ROPE = 64
D_QK = 576
E4M3_MAX = 448.0
_CHUNK = 1 << 22


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


class Stream:
    """Named, reproducible random streams: ``Stream(seed).sub("kv")`` is independent of
    every other name and of the order in which streams are used."""

    def __init__(self, seed: int, path: tuple = ()):
        self.seed = int(seed)
        self.path = tuple(path)

    def sub(self, name: str) -> "Stream":
        return Stream(self.seed, self.path + (name,))

    def _seq(self) -> np.random.SeedSequence:
        words = [self.seed] + [int.from_bytes(n.encode()[:8].ljust(8, b"\0"), "little") for n in self.path]
        return np.random.SeedSequence(words)

    def gen(self) -> np.random.Generator:
        return np.random.Generator(np.random.PCG64(self._seq()))

    def _fill(self, n: int, draw) -> np.ndarray:
        nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
        seqs = self._seq().spawn(nchunks)
        out = np.empty(n, dtype=np.float32)

        def work(i):
            lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
            draw(np.random.Generator(np.random.PCG64(seqs[i])), out[lo:hi])

        if nchunks == 1:
            work(0)
        else:
            with ThreadPoolExecutor(_threads()) as ex:
                list(ex.map(work, range(nchunks)))
        return out

    def normal(self, shape, sigma: float = 1.0) -> np.ndarray:
        n = int(np.prod(shape))
        out = self._fill(n, lambda g, o: g.standard_normal(o.shape[0], dtype=np.float32, out=o))
        if sigma != 1.0:
            out *= np.float32(sigma)
        return out.reshape(shape)

    def uniform(self, shape) -> np.ndarray:
        n = int(np.prod(shape))
        return self._fill(n, lambda g, o: g.random(o.shape[0], dtype=np.float32, out=o)).reshape(shape)


# ----------------------------------------------------------------------- encodings -----------

def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """uint8 OCP e4m3 codes of float32 values already within [-448, 448] (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values rounded to bfloat16 (nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def quantize_rows(x: np.ndarray):
    """Per-row FP8 encoding: scale = max|row| / 448, codes = e4m3(row / scale).

    Returns (codes uint8 with x's shape, scale float32 with x.shape[:-1])."""
    amax = np.abs(x).max(axis=-1)
    scale = (np.maximum(amax, np.float32(1e-30)) / np.float32(E4M3_MAX)).astype(np.float32)
    codes = e4m3_encode(x / scale[..., None])
    return codes, scale


def pack_kv_rows(latent: np.ndarray, rope: np.ndarray, group_scales: np.ndarray | None = None) -> np.ndarray:
    """Pack float32 latent [N, 512] and rope [N, 64] into 656-byte rows.

    With ``group_scales`` None, one per-row scale (max|row| / 448) is stored in all four
    128-element group slots. Otherwise ``group_scales`` float32 [N, 4] are used as given and
    the codes are e4m3(latent / scale_of_group).
    """
    n = latent.shape[0]
    rows = np.empty((n, ROW_BYTES), dtype=np.uint8)
    if group_scales is None:
        codes, scale = quantize_rows(latent)
        gs = np.repeat(scale[:, None], 4, axis=1).astype(np.float32)
    else:
        gs = np.ascontiguousarray(group_scales, dtype=np.float32)
        scaled = latent / np.repeat(gs, 128, axis=1)
        if np.abs(scaled).max() > E4M3_MAX:
            raise ValueError("group scales too small: |latent / scale| exceeds the e4m3 range (448)")
        codes = e4m3_encode(scaled)
    rows[:, :D_LATENT] = codes
    rows[:, D_LATENT:D_LATENT + 16] = gs.view(np.uint8).reshape(n, 16)
    rows[:, D_LATENT + 16:] = bf16_bits(rope).view(np.uint8).reshape(n, 2 * D_ROPE)
    return rows


# ----------------------------------------------------------------------- layouts -------------

def paged_block_tables(ctx: np.ndarray, stream: Stream):
    """One global random permutation of all sum(ceil(ctx/64)) pages.

    Returns (block_table int32 [B, max_pages] padded with -1, nblk)."""
    pages = [(int(c) + PAGE - 1) // PAGE for c in ctx]
    nblk = int(sum(pages))
    perm = stream.gen().permutation(nblk).astype(np.int32)
    bt = np.full((len(pages), max(pages) if pages else 1), -1, dtype=np.int32)
    off = 0
    for r, p in enumerate(pages):
        bt[r, :p] = perm[off:off + p]
        off += p
    return bt, nblk


def scatter_paged(per_token: np.ndarray, ctx: np.ndarray, block_table: np.ndarray, nblk: int) -> np.ndarray:
    """Place request-ordered token rows (concatenated over requests) into the paged pool
    [nblk * 64, ...]. Pool rows of unused page tails are zero."""
    pool = np.zeros((nblk * PAGE,) + per_token.shape[1:], dtype=per_token.dtype)
    off = 0
    for r, c in enumerate(ctx):
        c = int(c)
        j = np.arange(c)
        rows = block_table[r, j // PAGE].astype(np.int64) * PAGE + j % PAGE
        pool[rows] = per_token[off:off + c]
        off += c
    return pool


# ----------------------------------------------------------------------- workloads -----------

@dataclasses.dataclass
class Workload:
    """Inputs of one step of the hot path (indexer -> top-k -> sparse MLA)."""
    name: str
    B: int
    T: int
    Hi: int
    Di: int
    H: int
    topk: int
    softmax_scale: float
    ctx: np.ndarray            # int32 [B] tokens in each request's cache
    token_req: np.ndarray      # int32 [T]
    token_kvlen: np.ndarray    # int32 [T] visible keys (absolute position + 1)
    block_table: np.ndarray    # int32 [B, bt_stride]
    nblk: int
    q_idx: np.ndarray          # uint8 e4m3 [T, Hi, Di]
    q_scale: np.ndarray        # float32 [T, Hi]
    weights: np.ndarray        # float32 [T, Hi]
    k_cache: np.ndarray        # uint8 e4m3 [nblk, 64, Di]
    k_scale: np.ndarray        # float32 [nblk, 64]
    q_mla: np.ndarray          # uint16 bf16 bits [T, H, 576]
    kv_pool: np.ndarray        # uint8 [nblk * 64, 656]

    @property
    def ld(self) -> int:
        """Leading dimension of the score matrix: max visible keys, rounded up to 4."""
        return int(-(-int(self.token_kvlen.max()) // 4) * 4)

    @property
    def R(self) -> int:
        return int(self.kv_pool.shape[0])


def draw_queries(qs: Stream, T: int, Hi: int, Di: int, H: int, q_sigma: float = 1.0):
    """Query-side inputs of T tokens from stream ``qs``: (q_idx e4m3 codes [T, Hi, Di], q_scale
    [T, Hi], weights [T, Hi], q_mla bf16 bits [T, H, 576])."""
    q_idx, q_scale = quantize_rows(qs.sub("q_idx").normal((T, Hi, Di)))
    weights = qs.sub("weights").uniform((T, Hi))
    q_mla = bf16_bits(qs.sub("q_mla").normal((T, H, D_QK), sigma=q_sigma))
    return q_idx, q_scale, weights, q_mla


def make_workload(name: str, B: int, ctx, queries, Hi: int, Di: int, H: int, topk: int,
                  seed: int, q_sigma: float = 1.0, softmax_scale: float = 1.0 / math.sqrt(576.0),
                  query_stream: Stream | None = None) -> Workload:
    """Generic builder. ``queries[r]`` lists the absolute positions of request r's query tokens
    (their token_kvlen is position + 1, so a query sees itself and everything before it).
    The query-side values are drawn from ``query_stream`` (default: the workload's own stream)."""
    s = Stream(seed)
    ctx = np.asarray(ctx, dtype=np.int32)
    token_req = np.concatenate([np.full(len(q), r, np.int32) for r, q in enumerate(queries)])
    token_kvlen = np.concatenate([np.asarray(q, np.int32) + 1 for q in queries]).astype(np.int32)
    T = int(token_req.shape[0])
    bt, nblk = paged_block_tables(ctx, s.sub("pages"))
    ntok = int(ctx.sum())
    q_idx, q_scale, weights, q_mla = draw_queries(query_stream or s, T, Hi, Di, H, q_sigma)
    # indexer keys
    kk = s.sub("k").normal((ntok, Di))
    kc, ks = quantize_rows(kk)
    del kk
    k_cache = scatter_paged(kc, ctx, bt, nblk).reshape(nblk, PAGE, Di)
    k_scale = scatter_paged(ks, ctx, bt, nblk).reshape(nblk, PAGE)
    k_scale[k_scale == 0] = 1.0  # page tails: any positive scale
    # sparse MLA rows
    lat = s.sub("latent").normal((ntok, D_LATENT))
    rope = s.sub("rope").normal((ntok, D_ROPE))
    rows = pack_kv_rows(lat, rope)
    del lat, rope
    kv_pool = scatter_paged(rows, ctx, bt, nblk)
    return Workload(name, int(B), T, Hi, Di, H, topk, float(softmax_scale), ctx, token_req,
                    token_kvlen, bt, nblk, q_idx, q_scale, weights, k_cache, k_scale, q_mla, kv_pool)


def config1(seed: int = 1) -> Workload:
    """Tiny prefill: L = 1024, every token a query."""
    L = 1024
    return make_workload("tiny-prefill-L1024", 1, [L], [np.arange(L)], Hi=8, Di=64, H=16, topk=256,
                         seed=seed, q_sigma=0.5)


def config2(seed: int = 2, B: int = 64, lo: int = 16384, hi: int = 65536, mtp: int = 3,
            Hi: int = 64, Di: int = 128, H: int = 64, topk: int = 2048) -> Workload:
    """MTP decode: B requests x (1 + mtp) query tokens, the last 1 + mtp positions of each cache."""
    ctx = Stream(seed).sub("ctx").gen().integers(lo, hi + 1, size=B).astype(np.int32)
    queries = [np.arange(int(c) - (mtp + 1), int(c)) for c in ctx]
    return make_workload("mtp-decode-B%d" % B, B, ctx, queries, Hi, Di, H, topk, seed)


def config3(seed: int = 3, cached: int = 65536, chunk: int = 2048, Hi: int = 64, Di: int = 128,
            H: int = 64, topk: int = 2048) -> Workload:
    """Chunked prefill: one chunk of `chunk` tokens after `cached` cached tokens."""
    ctx = np.array([cached + chunk], np.int32)
    return make_workload("chunked-prefill-%dK+%d" % (cached // 1024, chunk), 1, ctx,
                         [np.arange(cached, cached + chunk)], Hi, Di, H, topk, seed)


def config4(chunk: int, seed: int = 4, total: int = 131072, chunk_len: int = 2048, Hi: int = 64,
            Di: int = 128, H: int = 64, topk: int = 2048) -> Workload:
    """Long prefill from scratch: chunk `chunk` of total/chunk_len sequential chunks.

    The cache holds the whole sequence (same bytes for every chunk); the chunk's queries see
    everything up to themselves. Each chunk's query values are its own draws."""
    ctx = np.array([total], np.int32)
    q = np.arange(chunk * chunk_len, (chunk + 1) * chunk_len)
    return make_workload("long-prefill-chunk%d" % chunk, 1, ctx, [q], Hi, Di, H, topk, seed,
                         query_stream=Stream(seed).sub("chunk%d" % chunk))


def config4_pass(seed: int = 4, total: int = 131072, chunk_len: int = 2048, Hi: int = 64, Di: int = 128,
                 H: int = 64, topk: int = 2048, chunks=None) -> list:
    """The chunks of one long-prefill pass (all total/chunk_len of them, or those listed), each
    the Workload config4 would build for it; the cache arrays are built once and shared."""
    n = total // chunk_len
    chunks = list(range(n)) if chunks is None else list(chunks)
    first = config4(chunks[0], seed, total, chunk_len, Hi, Di, H, topk)
    out = [first]
    for c in chunks[1:]:
        qs = Stream(seed).sub("chunk%d" % c)
        q_idx, q_scale, weights, q_mla = draw_queries(qs, chunk_len, Hi, Di, H)
        kvlen = (np.arange(c * chunk_len, (c + 1) * chunk_len) + 1).astype(np.int32)
        out.append(dataclasses.replace(first, name="long-prefill-chunk%d" % c, token_kvlen=kvlen, q_idx=q_idx,
                                       q_scale=q_scale, weights=weights, q_mla=q_mla))
    return out


# ----------------------------------------------------------------------- HiSparse ------------

@dataclasses.dataclass
class HiSparseWorkload:
    """Inputs of the mixed-residency decode (resolve + sparse MLA), one query token per request."""
    name: str
    B: int
    k: int
    S: int
    H: int
    softmax_scale: float
    seq_len: np.ndarray         # int32 [B]
    resident_start: np.ndarray  # int32 [B]
    block_table: np.ndarray     # int32 [B, ceil(max seq_len / 64)]; only resident pages mapped
    slot_row: np.ndarray        # int32 [B, S] pool rows of the hot slots
    R: int                      # pool rows (resident pages + hot slots)
    kv_pool: np.ndarray         # uint8 [R, 656]: resident rows filled, slot rows zero
    host_rows: list             # B x uint8 [seq_len_r, 656]
    q_mla: np.ndarray           # uint16 bf16 bits [steps, B, H, 576]
    idx: np.ndarray             # int32 [steps, B, k], ascending, logical token indices


def _zipf_distinct(g: np.random.Generator, n_old: int, count: int, exclude: set, a: float) -> list:
    """`count` distinct recency ranks in [1, n_old] drawn Zipf(a) (rank 1 = most recent old
    token), skipping ranks in `exclude`."""
    out = []
    seen = set(exclude)
    while len(out) < count:
        z = g.zipf(a, size=max(4 * (count - len(out)), 1024))
        for v in z:
            v = int(v)
            if v <= n_old and v not in seen:
                seen.add(v)
                out.append(v)
                if len(out) == count:
                    break
    return out


def hisparse_index_stream(seq_len: np.ndarray, resident: int, k: int, steps: int, overlap: float,
                          stream: Stream, a: float = 1.1) -> np.ndarray:
    """int32 [steps, B, k] ascending indices of older (non-resident) tokens.

    Step 0 draws k distinct indices Zipf(a) by recency rank over the older tokens (rank 1 =
    seq_len - resident - 1); each later step keeps a uniformly random round(overlap * k) of
    the previous set and draws the rest fresh, distinct and outside the whole previous set, so
    consecutive steps share exactly round(overlap * k) indices."""
    B = len(seq_len)
    out = np.empty((steps, B, k), dtype=np.int32)
    keep = int(round(overlap * k))
    for r in range(B):
        g = stream.sub("req%d" % r).gen()
        n_old = int(seq_len[r]) - resident
        newest_old = n_old - 1
        ranks = _zipf_distinct(g, n_old, k, set(), a)
        for st in range(steps):
            if st > 0:
                kept = list(g.choice(np.array(ranks), size=keep, replace=False))
                ranks = kept + _zipf_distinct(g, n_old, k - keep, set(ranks), a)
            out[st, r] = np.sort(newest_old - (np.array(ranks, dtype=np.int64) - 1)).astype(np.int32)
    return out


def config5(seed: int = 5, B: int = 32, lo: int = 262144, hi: int = 1048576, resident: int = 4096,
            k: int = 2048, S: int = 4096, H: int = 64, steps: int = 50, overlap: float = 0.8,
            pool_rows: int = 65536, host_alloc=None) -> HiSparseWorkload:
    """HiSparse mixed residency. Host rows are drawn from a bank of `pool_rows` distinct
    random rows (each host row picks one bank row at random), so that ~13 GB of host rows can
    be produced quickly. ``host_alloc(nbytes) -> uint8 numpy array`` allocates each request's
    host rows (e.g. pinned memory); numpy memory by default."""
    s = Stream(seed)
    seq_len = s.sub("ctx").gen().integers(lo, hi + 1, size=B).astype(np.int32)
    resident_start = (seq_len - resident).astype(np.int32)
    max_pages = (int(seq_len.max()) + PAGE - 1) // PAGE
    # pool: resident pages of every request, then the hot slots, in one random order
    res_pages = [(int(seq_len[r]) + PAGE - 1) // PAGE - int(resident_start[r]) // PAGE for r in range(B)]
    n_res_pages = int(sum(res_pages))
    slot_pages = (B * S + PAGE - 1) // PAGE
    R = (n_res_pages + slot_pages) * PAGE
    page_perm = s.sub("pages").gen().permutation(n_res_pages + slot_pages).astype(np.int32)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for r in range(B):
        first = int(resident_start[r]) // PAGE
        for p in range(res_pages[r]):
            bt[r, first + p] = page_perm[off]
            off += 1
    slot_page_ids = page_perm[off:]
    slot_rows_all = (slot_page_ids[:, None].astype(np.int64) * PAGE + np.arange(PAGE)).reshape(-1)[:B * S]
    slot_row = s.sub("slots").gen().permutation(slot_rows_all).astype(np.int32).reshape(B, S)
    # bank of distinct rows
    bank = pack_kv_rows(s.sub("bank_lat").normal((pool_rows, D_LATENT)),
                        s.sub("bank_rope").normal((pool_rows, D_ROPE)))
    kv_pool = np.zeros((R, ROW_BYTES), dtype=np.uint8)
    host_rows = []
    for r in range(B):
        n = int(seq_len[r])
        pick = s.sub("pick%d" % r).gen().integers(0, pool_rows, size=n)
        buf = host_alloc(n * ROW_BYTES) if host_alloc is not None else np.empty(n * ROW_BYTES, np.uint8)
        buf = buf.reshape(n, ROW_BYTES)
        np.take(bank, pick, axis=0, out=buf)
        host_rows.append(buf)
        j = np.arange(int(resident_start[r]), n)
        kv_pool[bt[r, j // PAGE].astype(np.int64) * PAGE + j % PAGE] = buf[j]
    idx = hisparse_index_stream(seq_len, resident, k, steps, overlap, s.sub("stream"))
    q_mla = bf16_bits(s.sub("q_mla").normal((steps, B, H, D_QK)))
    return HiSparseWorkload("hisparse-B%d" % B, B, k, S, H, 1.0 / math.sqrt(576.0), seq_len,
                            resident_start, bt, slot_row, R, kv_pool, host_rows, q_mla, idx)
