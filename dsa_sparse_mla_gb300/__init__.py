"""GB300-native sparse MLA (DeepSeek sparse attention) hot path.

Thin Python binding of ``libhs.so`` (C ABI in ``include/hs.h``): the functions below have the
C names, take torch CUDA tensors, marshal pointers and sizes, and call the library on the
current (or given) CUDA stream. Every step of the computation runs in the library's sm_103a
kernels; there is no fallback. If the library is missing, import succeeds but every call raises
``HSError`` telling how to build it (``python -m dsa_sparse_mla_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["HSError", "lib_path", "load", "hs_abi_version", "hs_check_flag", "hs_indexer_scores", "hs_topk",
           "hs_indexer_topk",
           "hs_sparse_mla_fwd", "hs_sparse_mla_workspace_size", "hs_sparse_mla_fwd_static", "hs_hisparse_resolve",
           "hs_hisparse_touch_host", "hs_kv_append", "hs_kv_offload", "FLAGS"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libhs.so")
_lib = None

FLAGS = {"BAD_INDEX": 0x01, "BAD_LENGTH": 0x02, "BAD_BLOCK": 0x04, "NOT_ASCENDING": 0x08, "BAD_STATE": 0x10,
         "TIMEOUT": 0x20}
_STATUS = {0: "HS_OK", 1: "HS_ERR_INVALID", 2: "HS_ERR_UNSUPPORTED", 3: "HS_ERR_CUDA", 4: "HS_ERR_DEVICE_FLAG",
           5: "HS_ERR_TIMEOUT"}


class HSError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS.get(status, status), message))
        self.status = status


_P = ctypes.c_void_p
_i32, _i64, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float


class _IndexerArgs(ctypes.Structure):
    _fields_ = [("T", _i32), ("B", _i32), ("Hi", _i32), ("Di", _i32), ("q", _P), ("q_scale", _P), ("weights", _P),
                ("k_cache", _P), ("k_scale", _P), ("nblk", _i64), ("block_table", _P), ("bt_stride", _i32),
                ("token_req", _P), ("token_kvlen", _P), ("scores", _P), ("ld", _i64), ("err_flag", _P)]


class _MlaArgs(ctypes.Structure):
    _fields_ = [("T", _i32), ("H", _i32), ("k", _i32), ("q", _P), ("kv_pool", _P), ("R", _i64), ("idx", _P),
                ("block_table", _P), ("bt_stride", _i32), ("token_req", _P), ("softmax_scale", _f32),
                ("out", _P), ("lse", _P), ("err_flag", _P), ("workspace", _P), ("workspace_bytes", ctypes.c_uint64),
                ("idx_row", _P), ("idx_rows", _i32), ("token_kvlen", _P)]


class _ResolveArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("k", _i32), ("S", _i32), ("step", _i32), ("idx", _P), ("seq_len", _P),
                ("resident_start", _P), ("block_table", _P), ("bt_stride", _i32), ("host_rows", _P),
                ("kv_pool", _P), ("R", _i64), ("slot_row", _P), ("slot_token", _P), ("slot_stamp", _P),
                ("tok2slot", _P), ("ld_t2s", _i64), ("out_rows", _P), ("counters", _P), ("err_flag", _P)]


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libhs.so once. Raises HSError if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise HSError(2, "libhs.so not found at %s; build it with `python -m dsa_sparse_mla_gb300.build`"
                          % _LIB_PATH)
        lib = ctypes.CDLL(_LIB_PATH)
        lib.hs_abi_version.restype = ctypes.c_int
        lib.hs_status_str.argtypes = [ctypes.c_int]
        lib.hs_status_str.restype = ctypes.c_char_p
        lib.hs_last_error.restype = ctypes.c_char_p
        lib.hs_check_flag.argtypes = [_P, _P, _P]
        lib.hs_indexer_scores.argtypes = [ctypes.POINTER(_IndexerArgs), _P]
        lib.hs_topk.argtypes = [_P, _i64, _P, _i32, _i32, _P, _P, _P]
        lib.hs_indexer_topk.argtypes = [ctypes.POINTER(_IndexerArgs), _i32, _P, _P]
        lib.hs_sparse_mla_fwd.argtypes = [ctypes.POINTER(_MlaArgs), _P]
        lib.hs_sparse_mla_workspace_size.argtypes = [_i32, ctypes.POINTER(ctypes.c_uint64)]
        lib.hs_sparse_mla_fwd_static.argtypes = [ctypes.POINTER(_MlaArgs), _P]
        lib.hs_hisparse_resolve.argtypes = [ctypes.POINTER(_ResolveArgs), _P]
        lib.hs_hisparse_touch_host.argtypes = [_i32, _P, _P, _P, _P, _P]
        lib.hs_kv_append.argtypes = [ctypes.POINTER(_AppendArgs), _P]
        lib.hs_kv_offload.argtypes = [ctypes.POINTER(_OffloadArgs), _P]
        for f in ("hs_check_flag", "hs_indexer_scores", "hs_topk", "hs_indexer_topk", "hs_sparse_mla_fwd", "hs_sparse_mla_workspace_size",
                  "hs_sparse_mla_fwd_static", "hs_hisparse_resolve", "hs_hisparse_touch_host", "hs_kv_append", "hs_kv_offload"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _check(status: int):
    if status != 0:
        raise HSError(status, load().hs_last_error().decode(errors="replace"))


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise HSError(1, "%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise HSError(1, "%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise HSError(1, "%s must be %s (got %s)" % (name, dtype, t.dtype))
    return t


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def hs_abi_version() -> int:
    return int(load().hs_abi_version())


def hs_check_flag(err_flag: torch.Tensor, stream=None) -> int:
    """Synchronise `stream` and return the raw device error bits (0 = none)."""
    out = ctypes.c_int32(0)
    st = load().hs_check_flag(_ptr(_dev(err_flag, "err_flag", torch.int32)), ctypes.addressof(out), _stream(stream))
    if st not in (0, 4, 5):
        _check(st)
    return int(out.value)


def _indexer_args(q, q_scale, weights, k_cache, k_scale, block_table, token_req, token_kvlen, scores, err_flag,
                  num_requests):
    _dev(q, "q", torch.uint8), _dev(q_scale, "q_scale", torch.float32), _dev(weights, "weights", torch.float32)
    _dev(k_cache, "k_cache", torch.uint8), _dev(k_scale, "k_scale", torch.float32)
    _dev(block_table, "block_table", torch.int32), _dev(token_req, "token_req", torch.int32)
    _dev(token_kvlen, "token_kvlen", torch.int32), _dev(scores, "scores", torch.float32)
    _dev(err_flag, "err_flag", torch.int32)
    T, Hi, Di = q.shape
    return _IndexerArgs(T, num_requests if num_requests is not None else block_table.shape[0], Hi, Di, _ptr(q),
                        _ptr(q_scale), _ptr(weights), _ptr(k_cache), _ptr(k_scale), k_cache.shape[0],
                        _ptr(block_table), block_table.shape[1], _ptr(token_req), _ptr(token_kvlen), _ptr(scores),
                        scores.shape[1], _ptr(err_flag))


def hs_indexer_scores(q, q_scale, weights, k_cache, k_scale, block_table, token_req, token_kvlen, scores, err_flag,
                      num_requests: int | None = None, stream=None):
    """Lightning-indexer scores into ``scores`` (float32 [T, ld]); see include/hs.h."""
    a = _indexer_args(q, q_scale, weights, k_cache, k_scale, block_table, token_req, token_kvlen, scores, err_flag,
                      num_requests)
    _check(load().hs_indexer_scores(ctypes.byref(a), _stream(stream)))


def hs_indexer_topk(q, q_scale, weights, k_cache, k_scale, block_table, token_req, token_kvlen, scores, k: int, idx,
                    err_flag, num_requests: int | None = None, stream=None):
    """Indexer scores and their top-k in one call (``scores`` is scratch, undefined afterwards);
    the indices go to ``idx`` (int32 [T, k]), as hs_indexer_scores + hs_topk would write them."""
    a = _indexer_args(q, q_scale, weights, k_cache, k_scale, block_table, token_req, token_kvlen, scores, err_flag,
                      num_requests)
    _dev(idx, "idx", torch.int32)
    if tuple(idx.shape) != (q.shape[0], k):
        raise HSError(1, "idx must have shape [T, k]")
    _check(load().hs_indexer_topk(ctypes.byref(a), k, _ptr(idx), _stream(stream)))


def hs_topk(scores, token_kvlen, k: int, idx, err_flag, stream=None):
    """Top-k indices (ascending, -1 padded) into ``idx`` (int32 [T, k])."""
    _dev(scores, "scores", torch.float32), _dev(token_kvlen, "token_kvlen", torch.int32)
    _dev(idx, "idx", torch.int32), _dev(err_flag, "err_flag", torch.int32)
    T, ld = scores.shape
    if idx.shape != (T, k):
        raise HSError(1, "idx must have shape [T, k]")
    _check(load().hs_topk(_ptr(scores), ld, _ptr(token_kvlen), T, k, _ptr(idx), _ptr(err_flag), _stream(stream)))


def hs_sparse_mla_workspace_size(H: int) -> int:
    """Bytes of workspace hs_sparse_mla_fwd needs for H heads on the current device."""
    n = ctypes.c_uint64(0)
    _check(load().hs_sparse_mla_workspace_size(int(H), ctypes.byref(n)))
    return int(n.value)


def _mla_args(q, kv_pool, idx, softmax_scale, out, err_flag, lse, block_table, token_req, workspace, idx_row,
              token_kvlen):
    _dev(q, "q", torch.bfloat16), _dev(kv_pool, "kv_pool", torch.uint8), _dev(idx, "idx", torch.int32)
    _dev(workspace, "workspace", torch.uint8)
    _dev(out, "out", torch.bfloat16), _dev(err_flag, "err_flag", torch.int32), _dev(lse, "lse", torch.float32)
    _dev(block_table, "block_table", torch.int32), _dev(token_req, "token_req", torch.int32)
    _dev(idx_row, "idx_row", torch.int32), _dev(token_kvlen, "token_kvlen", torch.int32)
    T, H, D = q.shape
    if D != 576 or kv_pool.shape[-1] != 656 or out.shape != (T, H, 512) or (idx_row is None and idx.shape[0] != T):
        raise HSError(1, "shape mismatch: q [T,H,576], kv_pool [R,656], idx [T,k] (or [rows,k] with idx_row), "
                         "out [T,H,512]")
    for t, n in ((idx_row, "idx_row"), (token_kvlen, "token_kvlen")):
        if t is not None and t.shape != (T,):
            raise HSError(1, "%s must be int32 [T]" % n)
    return _MlaArgs(T, H, idx.shape[1], _ptr(q), _ptr(kv_pool), kv_pool.shape[0], _ptr(idx), _ptr(block_table),
                    0 if block_table is None else block_table.shape[1], _ptr(token_req), float(softmax_scale),
                    _ptr(out), _ptr(lse), _ptr(err_flag), _ptr(workspace),
                    0 if workspace is None else workspace.numel(), _ptr(idx_row), idx.shape[0], _ptr(token_kvlen))


def hs_sparse_mla_fwd(q, kv_pool, idx, softmax_scale: float, out, err_flag, lse=None, block_table=None,
                      token_req=None, workspace=None, stream=None, idx_row=None, token_kvlen=None):
    """Sparse MLA forward: ``out`` bf16 [T, H, 512] (and ``lse`` float32 [T, H] if given). With a
    ``workspace`` (uint8 CUDA tensor of at least hs_sparse_mla_workspace_size(H) bytes) every SM
    gets an equal share of the work and split queries are merged by log-sum-exp. Shared index sets:
    ``idx_row`` (int32 [T]) names the row of ``idx`` each query reads, and ``token_kvlen`` (int32
    [T], with a block table) skips the entries a query may not see."""
    a = _mla_args(q, kv_pool, idx, softmax_scale, out, err_flag, lse, block_table, token_req, workspace, idx_row,
                  token_kvlen)
    _check(load().hs_sparse_mla_fwd(ctypes.byref(a), _stream(stream)))


def hs_sparse_mla_fwd_static(q, kv_pool, idx, softmax_scale: float, out, err_flag, lse=None, block_table=None,
                             token_req=None, stream=None, idx_row=None, token_kvlen=None):
    """hs_sparse_mla_fwd for callers that cannot allocate device memory: the split-work scratch is
    the library's own fixed device array (see include/hs.h), so no workspace is passed."""
    a = _mla_args(q, kv_pool, idx, softmax_scale, out, err_flag, lse, block_table, token_req, None, idx_row,
                  token_kvlen)
    _check(load().hs_sparse_mla_fwd_static(ctypes.byref(a), _stream(stream)))


def hs_hisparse_resolve(step: int, idx, seq_len, resident_start, block_table, host_rows, kv_pool, slot_row,
                        slot_token, slot_stamp, tok2slot, out_rows, counters, err_flag, stream=None):
    """One HiSparse resolve step. ``host_rows`` is an int64 CUDA tensor [B] of device-accessible
    pointers to each request's pinned host rows [seq_len, 656]."""
    for t, n, dt in ((idx, "idx", torch.int32), (seq_len, "seq_len", torch.int32),
                     (resident_start, "resident_start", torch.int32), (block_table, "block_table", torch.int32),
                     (host_rows, "host_rows", torch.int64), (kv_pool, "kv_pool", torch.uint8),
                     (slot_row, "slot_row", torch.int32), (slot_token, "slot_token", torch.int32),
                     (slot_stamp, "slot_stamp", torch.int32), (tok2slot, "tok2slot", torch.int32),
                     (out_rows, "out_rows", torch.int32), (counters, "counters", torch.int32),
                     (err_flag, "err_flag", torch.int32)):
        _dev(t, n, dt)
    B, k = idx.shape
    a = _ResolveArgs(B, k, slot_row.shape[1], int(step), _ptr(idx), _ptr(seq_len), _ptr(resident_start),
                     _ptr(block_table), block_table.shape[1], _ptr(host_rows), _ptr(kv_pool), kv_pool.shape[0],
                     _ptr(slot_row), _ptr(slot_token), _ptr(slot_stamp), _ptr(tok2slot), tok2slot.shape[1],
                     _ptr(out_rows), _ptr(counters), _ptr(err_flag))
    _check(load().hs_hisparse_resolve(ctypes.byref(a), _stream(stream)))


def hs_hisparse_touch_host(host_rows, seq_len, resident_start, err_flag, stream=None):
    """Read one word of every host page of each request's offloaded rows, so that the GPU's
    first-access cost for the host tier is paid here rather than inside a resolve.
    ``host_rows`` is the int64 CUDA tensor [B] of pointers that hs_hisparse_resolve takes."""
    for t, n, dt in ((host_rows, "host_rows", torch.int64), (seq_len, "seq_len", torch.int32),
                     (resident_start, "resident_start", torch.int32), (err_flag, "err_flag", torch.int32)):
        _dev(t, n, dt)
    B = host_rows.shape[0]
    if seq_len.shape[0] != B or resident_start.shape[0] != B:
        raise HSError(1, "host_rows, seq_len and resident_start must have the same length")
    _check(load().hs_hisparse_touch_host(B, _ptr(host_rows), _ptr(seq_len), _ptr(resident_start), _ptr(err_flag),
                                         _stream(stream)))


class _AppendArgs(ctypes.Structure):
    _fields_ = [("T", _i32), ("B", _i32), ("latent", _P), ("rope", _P), ("index_key", _P), ("Di", _i32),
                ("token_req", _P), ("token_pos", _P), ("block_table", _P), ("bt_stride", _i32),
                ("kv_pool", _P), ("R", _i64), ("k_cache", _P), ("k_scale", _P), ("nblk", _i64), ("err_flag", _P)]


def hs_kv_append(token_req, token_pos, block_table, err_flag, latent=None, rope=None, kv_pool=None,
                 index_key=None, k_cache=None, k_scale=None, stream=None):
    """Quantise new tokens into the paged FP8 layouts (see include/hs.h). ``latent`` / ``rope`` are
    bf16 [T, 512] / [T, 64] written into ``kv_pool`` (uint8 [R, 656]); ``index_key`` is bf16 [T, Di]
    written into ``k_cache`` (uint8 [nblk, 64, Di]) and ``k_scale`` (float32 [nblk, 64])."""
    _dev(token_req, "token_req", torch.int32), _dev(token_pos, "token_pos", torch.int32)
    _dev(block_table, "block_table", torch.int32), _dev(err_flag, "err_flag", torch.int32)
    a = _AppendArgs()
    a.T, a.B = token_req.shape[0], block_table.shape[0]
    if latent is not None:
        _dev(latent, "latent", torch.bfloat16), _dev(rope, "rope", torch.bfloat16), _dev(kv_pool, "kv_pool", torch.uint8)
        a.latent, a.rope, a.kv_pool, a.R = _ptr(latent), _ptr(rope), _ptr(kv_pool), kv_pool.shape[0]
    if index_key is not None:
        _dev(index_key, "index_key", torch.bfloat16), _dev(k_cache, "k_cache", torch.uint8)
        _dev(k_scale, "k_scale", torch.float32)
        a.index_key, a.Di, a.k_cache, a.k_scale, a.nblk = _ptr(index_key), index_key.shape[1], _ptr(k_cache), \
            _ptr(k_scale), k_cache.shape[0]
    a.token_req, a.token_pos, a.block_table, a.bt_stride = _ptr(token_req), _ptr(token_pos), _ptr(block_table), \
        block_table.shape[1]
    a.err_flag = _ptr(err_flag)
    _check(load().hs_kv_append(ctypes.byref(a), _stream(stream)))


class _OffloadArgs(ctypes.Structure):
    _fields_ = [("n", _i32), ("L", _i32), ("B", _i32), ("pools", _P), ("R", _i64), ("host_rows", _P), ("layer", _P),
                ("req", _P), ("page", _P), ("block_table", _P), ("bt_stride", _i32), ("seq_len", _P), ("err_flag", _P)]


def hs_kv_offload(pools, host_rows, layer, req, page, block_table, seq_len, err_flag, R: int, stream=None):
    """Copy complete KV pages to the host tier (see include/hs.h). ``pools`` is an int64 CUDA tensor
    [L] of device pointers to each layer's pool (uint8 [R, 656]); ``host_rows`` an int64 CUDA tensor
    [L * B] of device-accessible pointers to pinned host rows, indexed layer * B + request."""
    for t, nm, dt in ((pools, "pools", torch.int64), (host_rows, "host_rows", torch.int64), (layer, "layer", torch.int32),
                      (req, "req", torch.int32), (page, "page", torch.int32), (block_table, "block_table", torch.int32),
                      (seq_len, "seq_len", torch.int32), (err_flag, "err_flag", torch.int32)):
        _dev(t, nm, dt)
    a = _OffloadArgs()
    a.n, a.L, a.B = layer.shape[0], pools.shape[0], block_table.shape[0]
    if host_rows.shape[0] != a.L * a.B:
        raise HSError(1, "host_rows must hold L * B pointers")
    a.pools, a.R, a.host_rows = _ptr(pools), int(R), _ptr(host_rows)
    a.layer, a.req, a.page = _ptr(layer), _ptr(req), _ptr(page)
    a.block_table, a.bt_stride, a.seq_len, a.err_flag = _ptr(block_table), block_table.shape[1], _ptr(seq_len), _ptr(err_flag)
    _check(load().hs_kv_offload(ctypes.byref(a), _stream(stream)))
