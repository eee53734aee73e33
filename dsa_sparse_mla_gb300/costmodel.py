"""Algorithmic bytes and FLOPs of the hot path, used for roofline fractions.

Accounting follows the per-query arithmetic of the GLM-5.3 Part-2 article ([P1]
"vLLM v0.32.0 GLM-5.3 サービング: 16基のH200上でのPCP、DCP、およびハイブリッドHiSparse",
section 「数字がうまくいく理由」; [P2] "Optimizaciones de GLM-5.3, Parte 2", footnotes 1-3):

* sparse MLA reads each selected 656-byte FP8 latent row plus its 4-byte index (660 B);
* each head adds 2,176 B (its bf16 query of 576 and output of 512 values) and does
  2,176 FLOPs per row (QK over 576 dims plus PV over 512 dims, 2 FLOPs per multiply-add);
* per token the FP8 KV of GLM-5.3 is 78 x 656 B (MLA) + 21 x 132 B (indexer keys:
  128 FP8 values and a 4-byte scale) + 788 B (MTP layer).
"""
from __future__ import annotations

from dataclasses import dataclass

KV_ROW_BYTES = 656
INDEX_BYTES = 4
D_QK = 576
D_V = 512
BF16 = 2


def mla_row_bytes() -> int:
    """Bytes read per gathered row: FP8 KV row plus its index."""
    return KV_ROW_BYTES + INDEX_BYTES


def mla_flops_per_row_head() -> int:
    """QK (576) and PV (512) multiply-adds, 2 FLOPs each."""
    return 2 * (D_QK + D_V)


def mla_head_bytes() -> int:
    """bf16 query (576) and output (512) per head."""
    return BF16 * (D_QK + D_V)


def mla_query_flops(heads: int, rows: int) -> int:
    return heads * rows * mla_flops_per_row_head()


def mla_query_bytes(heads: int, rows: int) -> int:
    return rows * mla_row_bytes() + heads * mla_head_bytes()


def mla_intensity(heads: int, rows: int = 2048) -> float:
    return mla_query_flops(heads, rows) / mla_query_bytes(heads, rows)


def kv_bytes_per_token(mla_layers: int = 78, indexer_layers: int = 21, index_dim: int = 128,
                       mtp_bytes: int = 788) -> int:
    return mla_layers * KV_ROW_BYTES + indexer_layers * (index_dim + 4) + mtp_bytes


def kv_gib_per_request(tokens: int, **kw) -> float:
    return tokens * kv_bytes_per_token(**kw) / 2**30


def ridge(flops_per_s: float, bytes_per_s: float) -> float:
    return flops_per_s / bytes_per_s


def indexer_crossover_tokens(gpus: int = 8, shard_indexer: bool = False, heads: int = 64,
                             rows: int = 2048, mla_layers: int = 78, indexer_layers: int = 21,
                             index_heads: int = 64, index_dim: int = 128) -> float:
    """Prompt length at which the indexer's prefill-from-scratch work overtakes sparse MLA's.

    Sparse MLA: every query attends `rows` rows with all heads -> linear in L. Under tensor
    parallelism each GPU serves heads/gpus heads; under prompt (context) parallelism each GPU
    serves L/gpus queries. Indexer: index_heads x index_dim multiply-adds per (query, key) pair
    over L^2/2 causal pairs, counted as multiply-adds (FP8 runs at twice the BF16 rate, so one
    FP8 multiply-add costs what one BF16 FLOP does); replicated on every GPU unless sharded.
    Crossover where indexer_layers * index_heads * index_dim * L^2 / 2 / s_i equals
    mla_layers * L * mla_query_flops / s_m (s = the per-GPU share)."""
    mla_per_query = mla_query_flops(heads, rows)
    idx_per_pair = index_heads * index_dim / 2.0
    if shard_indexer:
        # each GPU: 1/gpus of the queries for both kernels
        return mla_layers * mla_per_query / (indexer_layers * idx_per_pair)
    return mla_layers * (mla_per_query / gpus) / (indexer_layers * idx_per_pair)


# --------------------------------------------------------------------- per-call work --------

@dataclass
class Work:
    flops: float
    bytes: float


def indexer_work(Hi: int, Di: int, kvlen_sum: int, ctx_sum: int, T: int) -> Work:
    """FP8 dot products over every visible (query, key) pair; bytes = keys read once per
    request (Di codes + 4-byte scale), queries (Di per head + 8 B of scale and weight), and the
    fp32 scores written."""
    flops = 2.0 * Hi * Di * kvlen_sum
    byts = ctx_sum * (Di + 4) + T * Hi * (Di + 8) + kvlen_sum * 4
    return Work(flops, byts)


def topk_work(kvlen_sum: int, T: int, k: int) -> Work:
    return Work(0.0, kvlen_sum * 4.0 + T * k * 4.0)


def mla_work(H: int, valid_rows: int, T: int) -> Work:
    """[P1]-style accounting: selected rows x 660 B plus per-head query/output bytes."""
    return Work(float(H) * valid_rows * mla_flops_per_row_head(),
                float(valid_rows) * mla_row_bytes() + float(T) * H * mla_head_bytes())


def resolve_work(misses: int, B: int, k: int) -> Work:
    """Host rows read and pool rows written for misses; index and row lists."""
    return Work(0.0, 2.0 * misses * KV_ROW_BYTES + 8.0 * B * k)
