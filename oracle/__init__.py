"""CPU oracle of the sparse-MLA (DSA) hot path: numpy front end of ``oracle.c``.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package. The product path (``dsa_sparse_mla_gb300``) never
imports it, and the two share no code: the only common module is the seeded input generator,
which holds none of the method's arithmetic.

Each function takes numpy arrays laid out exactly as the C ABI of the CUDA library (see
``include/hs.h``) and returns float64 results computed by the plain definitions in
``oracle.c``. ``threads=0`` uses every online core.

Pages cited here besides those listed in ``oracle.c``:
  [P4] "vLLMによるNVIDIA B300 GPU上でのGLM-5.2のサービング"
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/liboracle.so with the host C compiler (gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_decode.restype = f64
        lib.orc_bf16_decode.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_decode.restype = f64
        lib.orc_num_threads.argtypes = [ctypes.c_int]
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_indexer_scores.argtypes = [i32, i32, i32, P, P, P, P, P, i64, P, i32, P, P, P, i64,
                                           ctypes.c_int]
        lib.orc_indexer_scores.restype = ctypes.c_int
        lib.orc_topk.argtypes = [P, i64, P, i32, i32, P, ctypes.c_int]
        lib.orc_topk.restype = ctypes.c_int
        lib.orc_sparse_mla.argtypes = [i32, i32, i32, P, P, i64, P, P, i32, P, f64, P, P,
                                       ctypes.c_int]
        lib.orc_sparse_mla.restype = ctypes.c_int
        lib.orc_hisparse_resolve.argtypes = [i32, i32, i32, i32, P, P, P, P, i32, P, P, i64, P, P,
                                             P, P, i64, P, P, ctypes.c_int]
        lib.orc_hisparse_resolve.restype = ctypes.c_int
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_kv_append.argtypes = [i32, i32, P, P, P, i32, P, P, P, i32, P, i64, P, P, i64]
        lib.orc_kv_append.restype = ctypes.c_int
        lib.orc_kv_offload.argtypes = [i32, i32, i32, P, i64, P, P, P, P, P, i32, P]
        lib.orc_kv_offload.restype = ctypes.c_int
        _lib = lib
    return _lib


class OracleError(ValueError):
    """An input broke the contract of the operation (bad length, index or ordering)."""


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a) -> int | None:
    return None if a is None else a.ctypes.data


def num_threads(threads: int = 0) -> int:
    return int(_load().orc_num_threads(threads))


def e4m3_decode(code: int) -> float:
    return float(_load().orc_e4m3_decode(int(code)))


def bf16_decode(bits: int) -> float:
    return float(_load().orc_bf16_decode(int(bits)))


def indexer_scores(q, q_scale, weights, k_cache, k_scale, block_table, token_req, token_kvlen,
                   ld: int, threads: int = 0) -> np.ndarray:
    """float64 [T, ld] lightning-indexer scores; -inf at j >= token_kvlen[t]."""
    q = _c(q, np.uint8)
    T, Hi, Di = q.shape
    q_scale, weights = _c(q_scale, np.float32), _c(weights, np.float32)
    k_cache, k_scale = _c(k_cache, np.uint8), _c(k_scale, np.float32)
    block_table = _c(block_table, np.int32)
    token_req, token_kvlen = _c(token_req, np.int32), _c(token_kvlen, np.int32)
    out = np.empty((T, ld), dtype=np.float64)
    st = _load().orc_indexer_scores(T, Hi, Di, _p(q), _p(q_scale), _p(weights), _p(k_cache),
                                    _p(k_scale), k_cache.shape[0], _p(block_table),
                                    block_table.shape[1], _p(token_req), _p(token_kvlen), _p(out),
                                    ld, threads)
    if st:
        raise OracleError("indexer: token_kvlen or block table out of range")
    return out


def topk(scores, token_kvlen, k: int, threads: int = 0) -> np.ndarray:
    """int32 [T, k]: top-k indices per row, ascending, padded with -1."""
    scores = _c(scores, np.float64)
    token_kvlen = _c(token_kvlen, np.int32)
    T, ld = scores.shape
    out = np.empty((T, k), dtype=np.int32)
    if _load().orc_topk(_p(scores), ld, _p(token_kvlen), T, k, _p(out), threads):
        raise OracleError("topk: token_kvlen out of [0, ld]")
    return out


def sparse_mla(q_bits, kv_pool, idx, softmax_scale: float, block_table=None, token_req=None,
               threads: int = 0):
    """(out float64 [T, H, 512], lse float64 [T, H]) of sparse MLA over the given rows.

    ``q_bits`` holds the bf16 bit patterns (uint16 [T, H, 576]).
    """
    q_bits = _c(q_bits, np.uint16)
    T, H, D = q_bits.shape
    assert D == 576
    kv_pool = _c(kv_pool, np.uint8)
    idx = _c(idx, np.int32)
    k = idx.shape[1]
    bt = None if block_table is None else _c(block_table, np.int32)
    tr = None if token_req is None else _c(token_req, np.int32)
    out = np.empty((T, H, 512), dtype=np.float64)
    lse = np.empty((T, H), dtype=np.float64)
    st = _load().orc_sparse_mla(T, H, k, _p(q_bits), _p(kv_pool), kv_pool.shape[0], _p(idx), _p(bt),
                                0 if bt is None else bt.shape[1], _p(tr), float(softmax_scale),
                                _p(out), _p(lse), threads)
    if st:
        raise OracleError("sparse_mla: row out of range")
    return out, lse


def shared_index_sets(idx, idx_row, token_kvlen=None) -> np.ndarray:
    """int32 [T, k]: the index set each query token attends when the query tokens of a request
    share one set.

    [P4] section 「MTP受理率の安定化」: the indexer's top-k indices are reused rather than re-running
    the indexer for every MTP token, and the shared index buffer of a batch keeps only each
    request's final query token's indices. Query t takes row ``idx_row[t]`` of ``idx`` [rows, k];
    with ``token_kvlen`` (logical indices), an entry j >= token_kvlen[t] is a token that query t
    may not see (a later draft position) and becomes -1 padding. Raises OracleError for a row
    outside idx.
    """
    idx = np.asarray(idx, dtype=np.int32)
    idx_row = np.asarray(idx_row, dtype=np.int64)
    if idx_row.size and (idx_row.min() < 0 or idx_row.max() >= idx.shape[0]):
        raise OracleError("shared_index_sets: idx_row outside idx")
    out = idx[idx_row].copy()
    if token_kvlen is not None:
        n = np.asarray(token_kvlen, dtype=np.int64)[:, None]
        out[out >= n] = -1
    return out


def hisparse_resolve(step: int, idx, seq_len, resident_start, block_table, host_rows, kv_pool,
                     slot_row, slot_token, slot_stamp, tok2slot, threads: int = 0):
    """One resolve step. Mutates kv_pool, slot_token, slot_stamp and tok2slot in place.

    ``host_rows`` is a list of B uint8 arrays [seq_len_r, 656]. Returns (out_rows, counters).
    The state arrays must already be C-contiguous of the right dtype, since they are updated in
    place.
    """
    idx = _c(idx, np.int32)
    B, k = idx.shape
    for a, dt in ((kv_pool, np.uint8), (slot_token, np.int32), (slot_stamp, np.int32),
                  (tok2slot, np.int32)):
        if a.dtype != dt or not a.flags.c_contiguous:
            raise TypeError("state arrays must be C-contiguous %s" % np.dtype(dt))
    slot_row = _c(slot_row, np.int32)
    S = slot_row.shape[1]
    seq_len, resident_start = _c(seq_len, np.int32), _c(resident_start, np.int32)
    block_table = _c(block_table, np.int32)
    rows = [np.ascontiguousarray(h, dtype=np.uint8) for h in host_rows]
    ptrs = (ctypes.c_void_p * B)(*[h.ctypes.data for h in rows])
    out_rows = np.empty((B, k), dtype=np.int32)
    counters = np.empty((B, 3), dtype=np.int32)
    st = _load().orc_hisparse_resolve(B, k, S, int(step), _p(idx), _p(seq_len), _p(resident_start),
                                      _p(block_table), block_table.shape[1],
                                      ctypes.cast(ptrs, ctypes.c_void_p), _p(kv_pool),
                                      kv_pool.shape[0], _p(slot_row), _p(slot_token),
                                      _p(slot_stamp), _p(tok2slot), tok2slot.shape[1], _p(out_rows),
                                      _p(counters), threads)
    if st:
        raise OracleError("resolve: idx not strictly ascending / out of range, or k > S")
    return out_rows, counters


def e4m3_encode(x: float) -> int:
    """OCP e4m3 code of a binary32 value (round to nearest even, saturating at +-448)."""
    return int(_load().orc_e4m3_encode(float(np.float32(x))))


def kv_append(latent_bits, rope_bits, index_key_bits, token_req, token_pos, block_table, kv_pool, k_cache,
              k_scale, B: int) -> None:
    """Quantises new tokens into ``kv_pool`` (uint8 [R, 656]) and ``k_cache`` / ``k_scale``
    (uint8 [nblk, 64, Di], float32 [nblk, 64]) in place. ``*_bits`` are uint16 bf16 bit patterns
    ([T, 512], [T, 64], [T, Di]); pass ``latent_bits=None`` or ``index_key_bits=None`` to skip that
    part. Raises OracleError if a token's request, position or block is out of range."""
    T = int(token_req.shape[0])
    lat = None if latent_bits is None else _c(latent_bits, np.uint16)
    rope = None if latent_bits is None else _c(rope_bits, np.uint16)
    key = None if index_key_bits is None else _c(index_key_bits, np.uint16)
    Di = 0 if key is None else int(key.shape[1])
    for a, dt in ((kv_pool, np.uint8), (k_cache, np.uint8), (k_scale, np.float32)):
        if a is not None and not (a.dtype == dt and a.flags.c_contiguous):
            raise OracleError("kv_pool / k_cache / k_scale must be C-contiguous of their dtype (updated in place)")
    bt = _c(block_table, np.int32)
    treq, tpos = _c(token_req, np.int32), _c(token_pos, np.int32)  # kept alive across the call
    st = _load().orc_kv_append(T, int(B), _p(lat), _p(rope), _p(key), Di, _p(treq), _p(tpos), _p(bt), bt.shape[1],
                               _p(kv_pool),
                               0 if kv_pool is None else kv_pool.shape[0], _p(k_cache), _p(k_scale),
                               0 if k_cache is None else k_cache.shape[0])
    if st:
        raise OracleError("a token's request, position or block is out of range")


def kv_offload(pools, host_rows, layer, req, page, block_table, seq_len) -> None:
    """Copies complete pages from the per-layer pools (uint8 [R, 656] each) into the per-(layer,
    request) host rows (uint8 [seq_len_r, 656]; list indexed layer * B + r), in place. Raises
    OracleError if an entry is out of range."""
    L, B = len(pools), int(np.asarray(block_table).shape[0])
    R = int(pools[0].shape[0])
    for a in list(pools) + list(host_rows):
        if not (a.dtype == np.uint8 and a.flags.c_contiguous):
            raise OracleError("pools and host rows must be C-contiguous uint8")
    pp = (ctypes.c_void_p * L)(*[a.ctypes.data for a in pools])
    hp = (ctypes.c_void_p * len(host_rows))(*[a.ctypes.data for a in host_rows])
    bt = _c(block_table, np.int32)
    lay, rq, pg, sl = _c(layer, np.int32), _c(req, np.int32), _c(page, np.int32), _c(seq_len, np.int32)  # kept alive
    st = _load().orc_kv_offload(int(lay.shape[0]), L, B, ctypes.addressof(pp), R, ctypes.addressof(hp), _p(lay), _p(rq),
                                _p(pg), _p(bt), bt.shape[1], _p(sl))
    if st:
        raise OracleError("an offload entry is out of range")
