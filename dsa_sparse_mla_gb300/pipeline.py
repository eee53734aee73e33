"""Device-side driver of the hot path.

``DeviceWorkload`` moves a seeded ``inputs.Workload`` into GPU memory; ``HotPath`` owns the
intermediate and output buffers and runs one step: hs_indexer_scores -> hs_topk ->
hs_sparse_mla_fwd (logical indices through the paged block table), or for decode batches
hs_indexer_topk -> hs_sparse_mla_fwd; ``SharedSetHotPath`` runs the
indexer and top-k for each request's final query token only and lets the request's other query
tokens reuse that set in hs_sparse_mla_fwd (shared index sets); ``LongPrefillPass`` runs every
chunk of a long prefill through the same three calls. ``DeviceHiSparse`` does the
same for the mixed-residency decode (hs_hisparse_resolve -> hs_sparse_mla_fwd on physical rows),
with the older rows in pinned host memory.

Only buffer management lives here; all arithmetic runs in libhs.so.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import (hs_hisparse_resolve, hs_hisparse_touch_host, hs_indexer_scores, hs_indexer_topk, hs_sparse_mla_fwd,
               hs_sparse_mla_workspace_size, hs_topk)
from .inputs import HiSparseWorkload, Workload


def _t(a: np.ndarray, device, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


@dataclasses.dataclass
class DeviceWorkload:
    w: Workload
    q_idx: torch.Tensor
    q_scale: torch.Tensor
    weights: torch.Tensor
    k_cache: torch.Tensor
    k_scale: torch.Tensor
    block_table: torch.Tensor
    token_req: torch.Tensor
    token_kvlen: torch.Tensor
    q_mla: torch.Tensor
    kv_pool: torch.Tensor

    @classmethod
    def from_host(cls, w: Workload, device="cuda") -> "DeviceWorkload":
        return cls(w, _t(w.q_idx, device), _t(w.q_scale, device), _t(w.weights, device), _t(w.k_cache, device),
                   _t(w.k_scale, device), _t(w.block_table, device), _t(w.token_req, device),
                   _t(w.token_kvlen, device), _t(w.q_mla.view(np.int16), device).view(torch.bfloat16),
                   _t(w.kv_pool, device))


class HotPath:
    """Buffers and launches for one step of indexer -> top-k -> sparse MLA. With ``fused`` (decode
    batches) the step runs indexer and top-k as the one call hs_indexer_topk, whose scores stay in
    L2 between the two kernels."""

    def __init__(self, dw: DeviceWorkload, fused: bool = False):
        w = dw.w
        dev = dw.q_idx.device
        self.dw = dw
        self.fused = fused
        self.scores = torch.empty((w.T, w.ld), dtype=torch.float32, device=dev)
        self.idx = torch.empty((w.T, w.topk), dtype=torch.int32, device=dev)
        self.out = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        # sparse-MLA scratch: every SM gets an equal share of the (query, tile) work
        self.workspace = torch.empty(hs_sparse_mla_workspace_size(w.H), dtype=torch.uint8, device=dev)

    def step_inputs(self) -> list:
        """The device tensors a step reads that change from step to step (a serving loop copies
        them in); everything else (caches, block tables, pools) stays resident."""
        d = self.dw
        return [d.q_idx, d.q_scale, d.weights, d.q_mla, d.token_req, d.token_kvlen]

    def indexer(self, stream=None):
        d = self.dw
        hs_indexer_scores(d.q_idx, d.q_scale, d.weights, d.k_cache, d.k_scale, d.block_table, d.token_req,
                          d.token_kvlen, self.scores, self.err, num_requests=d.w.B, stream=stream)

    def topk(self, stream=None):
        hs_topk(self.scores, self.dw.token_kvlen, self.dw.w.topk, self.idx, self.err, stream=stream)

    def indexer_topk(self, stream=None):
        d = self.dw
        hs_indexer_topk(d.q_idx, d.q_scale, d.weights, d.k_cache, d.k_scale, d.block_table, d.token_req,
                        d.token_kvlen, self.scores, d.w.topk, self.idx, self.err, num_requests=d.w.B, stream=stream)

    def mla(self, stream=None):
        d = self.dw
        hs_sparse_mla_fwd(d.q_mla, d.kv_pool, self.idx, d.w.softmax_scale, self.out, self.err, lse=self.lse,
                          block_table=d.block_table, token_req=d.token_req, workspace=self.workspace, stream=stream)

    def step(self, stream=None):
        if self.fused:
            self.indexer_topk(stream)
        else:
            self.indexer(stream)
            self.topk(stream)
        self.mla(stream)


class LongPrefillPass:
    """One long-prefill pass: every chunk of one sequence through indexer -> top-k -> sparse MLA,
    chunk after chunk. The sequence's K cache and KV pool and every chunk's query inputs stay
    resident; the scores and top-k buffers are reused by each chunk, and the output holds the
    whole sequence ([chunks, chunk_len, H, 512] bf16 and its LSE)."""

    def __init__(self, chunks: list, device="cuda"):
        w0 = chunks[0]
        self.chunks = chunks
        self.n = len(chunks)
        self.T = w0.T
        self.k_cache = _t(w0.k_cache, device)
        self.k_scale = _t(w0.k_scale, device)
        self.block_table = _t(w0.block_table, device)
        self.token_req = _t(w0.token_req, device)
        self.kv_pool = _t(w0.kv_pool, device)
        self.q_idx = [_t(w.q_idx, device) for w in chunks]
        self.q_scale = [_t(w.q_scale, device) for w in chunks]
        self.weights = [_t(w.weights, device) for w in chunks]
        self.q_mla = [_t(w.q_mla.view(np.int16), device).view(torch.bfloat16) for w in chunks]
        self.token_kvlen = [_t(w.token_kvlen, device) for w in chunks]
        ld = max(w.ld for w in chunks)
        self.scores = torch.empty((w0.T, ld), dtype=torch.float32, device=device)
        self.idx = torch.empty((w0.T, w0.topk), dtype=torch.int32, device=device)
        self.out = torch.empty((self.n, w0.T, w0.H, 512), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((self.n, w0.T, w0.H), dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.workspace = torch.empty(hs_sparse_mla_workspace_size(w0.H), dtype=torch.uint8, device=device)

    def step_inputs(self, c: int) -> list:
        """The device tensors of chunk c that a serving loop would copy in for it."""
        return [self.q_idx[c], self.q_scale[c], self.weights[c], self.q_mla[c], self.token_kvlen[c]]

    def indexer(self, c: int, stream=None, q_idx=None, q_scale=None, weights=None, token_kvlen=None):
        hs_indexer_scores(self.q_idx[c] if q_idx is None else q_idx, self.q_scale[c] if q_scale is None else q_scale,
                          self.weights[c] if weights is None else weights, self.k_cache, self.k_scale,
                          self.block_table, self.token_req,
                          self.token_kvlen[c] if token_kvlen is None else token_kvlen, self.scores, self.err,
                          num_requests=1, stream=stream)

    def topk(self, c: int, stream=None, token_kvlen=None):
        hs_topk(self.scores, self.token_kvlen[c] if token_kvlen is None else token_kvlen, self.chunks[c].topk,
                self.idx, self.err, stream=stream)

    def mla(self, c: int, stream=None, q_mla=None, out=None, lse=None):
        hs_sparse_mla_fwd(self.q_mla[c] if q_mla is None else q_mla, self.kv_pool, self.idx,
                          self.chunks[c].softmax_scale, self.out[c] if out is None else out, self.err,
                          lse=self.lse[c] if lse is None else lse, block_table=self.block_table,
                          token_req=self.token_req, workspace=self.workspace, stream=stream)

    def step(self, stream=None):
        for c in range(self.n):
            self.indexer(c, stream)
            self.topk(c, stream)
            self.mla(c, stream)


class SharedSetHotPath(HotPath):
    """One step with shared index sets: hs_indexer_scores and hs_topk run for the final query token
    of each request only, and hs_sparse_mla_fwd gives every query token its request's set
    (idx_row), limited to the tokens it can see (token_kvlen), so MTP tokens do not re-run the
    indexer."""

    def __init__(self, dw: DeviceWorkload, fused: bool = False):
        super().__init__(dw, fused)
        w = dw.w
        dev = dw.q_idx.device
        req = np.asarray(w.token_req)
        last = np.array([np.flatnonzero(req == r)[np.argmax(w.token_kvlen[req == r])] for r in np.unique(req)])
        row_of_req = np.full(int(req.max()) + 1, -1, np.int32)
        row_of_req[req[last]] = np.arange(len(last), dtype=np.int32)
        li = torch.from_numpy(last).to(dev)
        self.f_q_idx, self.f_q_scale, self.f_weights = (dw.q_idx[li].contiguous(), dw.q_scale[li].contiguous(),
                                                        dw.weights[li].contiguous())
        self.f_req, self.f_kvlen = dw.token_req[li].contiguous(), dw.token_kvlen[li].contiguous()
        self.idx_row = _t(row_of_req[req], dev)
        self.scores = torch.empty((len(last), w.ld), dtype=torch.float32, device=dev)
        self.idx = torch.empty((len(last), w.topk), dtype=torch.int32, device=dev)

    def step_inputs(self) -> list:
        """Only the final tokens' indexer inputs change per step here, with every token's MLA query
        and the token-to-request, visible-length and index-row maps."""
        d = self.dw
        return [self.f_q_idx, self.f_q_scale, self.f_weights, self.f_req, self.f_kvlen, self.idx_row, d.q_mla,
                d.token_req, d.token_kvlen]

    def indexer(self, stream=None):
        d = self.dw
        hs_indexer_scores(self.f_q_idx, self.f_q_scale, self.f_weights, d.k_cache, d.k_scale, d.block_table,
                          self.f_req, self.f_kvlen, self.scores, self.err, num_requests=d.w.B, stream=stream)

    def topk(self, stream=None):
        hs_topk(self.scores, self.f_kvlen, self.dw.w.topk, self.idx, self.err, stream=stream)

    def indexer_topk(self, stream=None):
        d = self.dw
        hs_indexer_topk(self.f_q_idx, self.f_q_scale, self.f_weights, d.k_cache, d.k_scale, d.block_table,
                        self.f_req, self.f_kvlen, self.scores, d.w.topk, self.idx, self.err, num_requests=d.w.B,
                        stream=stream)

    def mla(self, stream=None):
        d = self.dw
        hs_sparse_mla_fwd(d.q_mla, d.kv_pool, self.idx, d.w.softmax_scale, self.out, self.err, lse=self.lse,
                          block_table=d.block_table, token_req=d.token_req, workspace=self.workspace, stream=stream,
                          idx_row=self.idx_row, token_kvlen=d.token_kvlen)


def pinned_uint8(nbytes: int) -> np.ndarray:
    """Page-locked host buffer (device-accessible through unified addressing) as a numpy view.
    The torch tensor owning the memory is kept alive by the returned array's base chain."""
    t = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    a = t.numpy()
    _PINNED_KEEPALIVE.append(t)
    return a


_PINNED_KEEPALIVE: list = []


class DeviceHiSparse:
    """Device state of the mixed-residency decode: pool, block table, LRU state, index stream.
    ``touch_host()`` maps the host tier for the GPU once (hs_hisparse_touch_host); a serving
    system does this when it sets the tier up."""

    def __init__(self, hw: HiSparseWorkload, device="cuda"):
        self.hw = hw
        B, S, k = hw.B, hw.S, hw.k
        self.kv_pool = _t(hw.kv_pool, device)
        self.block_table = _t(hw.block_table, device)
        self.seq_len = _t(hw.seq_len, device)
        self.resident_start = _t(hw.resident_start, device)
        self.slot_row = _t(hw.slot_row, device)
        self.slot_token = torch.full((B, S), -1, dtype=torch.int32, device=device)
        self.slot_stamp = torch.full((B, S), -1, dtype=torch.int32, device=device)
        self.ld_t2s = int(hw.seq_len.max())
        self.tok2slot = torch.full((B, self.ld_t2s), -1, dtype=torch.int32, device=device)
        self.host_rows = torch.tensor([int(h.ctypes.data) for h in hw.host_rows], dtype=torch.int64, device=device)
        self.idx = _t(hw.idx, device)                                     # [steps, B, k]
        self.q = _t(hw.q_mla.view(np.int16), device).view(torch.bfloat16)  # [steps, B, H, 576]
        self.rows = torch.empty((B, k), dtype=torch.int32, device=device)
        self.counters = torch.zeros((B, 3), dtype=torch.int32, device=device)
        self.out = torch.empty((B, hw.H, 512), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((B, hw.H), dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.workspace = torch.empty(hs_sparse_mla_workspace_size(hw.H), dtype=torch.uint8, device=device)

    def touch_host(self, stream=None):
        hs_hisparse_touch_host(self.host_rows, self.seq_len, self.resident_start, self.err, stream=stream)

    def resolve(self, step: int, stream=None):
        hs_hisparse_resolve(step, self.idx[step], self.seq_len, self.resident_start, self.block_table,
                            self.host_rows, self.kv_pool, self.slot_row, self.slot_token, self.slot_stamp,
                            self.tok2slot, self.rows, self.counters, self.err, stream=stream)

    def mla(self, step: int, stream=None):
        hs_sparse_mla_fwd(self.q[step], self.kv_pool, self.rows, self.hw.softmax_scale, self.out, self.err,
                          lse=self.lse, workspace=self.workspace, stream=stream)

    def step(self, step: int, stream=None):
        self.resolve(step, stream)
        self.mla(step, stream)
