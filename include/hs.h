/*
 * hs.h — C ABI of the GB300 (sm_103a) sparse-MLA (DeepSeek sparse attention, "DSA") hot path.
 *
 * Four calls make one attention layer's data-parallel hot path:
 *
 *   hs_indexer_scores   lightning-indexer scores of every visible prior token  (FP8 tcgen05 GEMM)
 *   hs_topk             per-query top-k of those scores, lowest index wins ties
 *   hs_indexer_topk     the two in one call, the scores kept in L2 between them (decode)
 *   hs_sparse_mla_fwd   softmax attention of all heads over the selected latent-KV rows
 *   hs_hisparse_resolve serve each selected token from resident KV, the hot buffer (LRU),
 *                       or a copy from pinned host memory into an LRU slot
 *
 * and around them:
 *
 *   hs_sparse_mla_workspace_size, hs_sparse_mla_fwd_static
 *                       the MLA's optional split-work scratch (caller-provided, or a fixed array
 *                       inside the library)
 *   hs_hisparse_touch_host  map the host tier for the GPU once, before the first resolve
 *   hs_kv_append        quantise new tokens into the paged FP8 rows and indexer keys
 *   hs_kv_offload       copy complete KV pages of every layer to the pinned host tier
 *
 * Sources (web pages describing GLM-5.x serving with DSA in vLLM):
 *   [P1] "vLLM v0.32.0 GLM-5.3 サービング: 16基のH200上でのPCP、DCP、およびハイブリッドHiSparse"
 *   [P2] "Optimizaciones de GLM-5.3, Parte 2: PCP, DCP e Hybrid HiSparse en 16 H200"
 *   [P3] "vLLM GLM 5.3 最適化: ハイブリッド HiSparse オフロード"
 *   [P4] "vLLMによるNVIDIA B300 GPU上でのGLM-5.2のサービング"
 *
 * Conventions shared by every call
 *  - All buffers are caller-owned device memory unless stated; the library allocates nothing
 *    and keeps no state between calls (hs_last_error's thread-local string aside; the fixed
 *    scratch array of hs_sparse_mla_fwd_static is the one stated exception).
 *  - Every call only enqueues work on `stream` (NULL = legacy default stream); none waits on
 *    the host for the GPU.
 *  - Arguments are checked on the host first. A bad argument returns HS_ERR_INVALID and
 *    launches nothing; hs_last_error() then names the argument.
 *  - Data that only the GPU sees (indices, lengths, block-table entries) is checked in the
 *    kernels. A bad value sets a bit of *err_flag (an int32 in device memory that the caller
 *    zeroes and reads whenever it likes) and the offending element is skipped. Kernels never
 *    trap. Every wait inside a kernel is bounded; running out sets HS_FLAG_TIMEOUT.
 *  - Requires a device of compute capability 10.3 (sm_103a); otherwise HS_ERR_UNSUPPORTED.
 *
 * Layouts
 *  - FP8 is OCP e4m3 ("e4m3fn": bias 7, no infinities, 0x7F/0xFF are NaN).
 *  - Paged KV: pages of HS_PAGE = 64 tokens. A request's token j lives in physical page
 *    block_table[r * bt_stride + j / 64], at row (page * 64 + j % 64) of the pool.
 *  - Latent-KV row ("fp8_ds_mla", 656 bytes, [P1] section 「数字がうまくいく理由」: 656 B of FP8 KV
 *    plus a 4 B index per gathered row):
 *        bytes   0..511  512 x e4m3 latent codes
 *        bytes 512..527  4 x fp32 dequantisation scales, one per 128-element group
 *        bytes 528..655  64 x bf16 RoPE part, used as stored
 *    latent[c] = e4m3(code[c]) * scale[c / 128].
 *  - Indexer key row: Di e4m3 codes in k_cache plus one fp32 scale in k_scale
 *    ([P1] same section: 128 FP8 values and a 4-byte scale).
 */
#ifndef HS_H_
#define HS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as CUDA's cudaStream_t, declared here so the header needs no CUDA headers. */
typedef struct CUstream_st* hs_stream_t;

typedef enum {
  HS_OK = 0,
  HS_ERR_INVALID = 1,      /* an argument failed the host-side checks; nothing was launched */
  HS_ERR_UNSUPPORTED = 2,  /* valid request that the library cannot serve (device, size limit) */
  HS_ERR_CUDA = 3,         /* a CUDA runtime call or a launch failed; see hs_last_error() */
  HS_ERR_DEVICE_FLAG = 4,  /* returned by hs_check_flag when the device error flag is non-zero */
  HS_ERR_TIMEOUT = 5       /* returned by hs_check_flag when HS_FLAG_TIMEOUT is set */
} hs_status;

/* Bits a kernel may OR into *err_flag. */
#define HS_FLAG_BAD_INDEX      0x01  /* an index or physical row outside its valid range */
#define HS_FLAG_BAD_LENGTH     0x02  /* a token_kvlen / seq_len outside [0, limit] */
#define HS_FLAG_BAD_BLOCK      0x04  /* a block-table entry outside [0, nblk) */
#define HS_FLAG_NOT_ASCENDING  0x08  /* resolve: a request's indices are not strictly ascending */
#define HS_FLAG_BAD_STATE      0x10  /* resolve: inconsistent LRU state (slot/token maps disagree) */
#define HS_FLAG_TIMEOUT        0x20  /* a bounded in-kernel wait ran out */
#define HS_FLAG_RANGE          0x40  /* sparse MLA: a value outside the 16-bit compute range (see below) */

#define HS_PAGE 64               /* tokens per KV page */
#define HS_KV_ROW_BYTES 656      /* latent-KV row size */
#define HS_D_LATENT 512          /* latent (value) width */
#define HS_D_ROPE 64             /* RoPE width */
#define HS_D_QK 576              /* query / key width = HS_D_LATENT + HS_D_ROPE */
#define HS_ABI_VERSION 7

int hs_abi_version(void);
const char* hs_status_str(hs_status s);
/* Text of the last error on the calling host thread ("" if none). Valid until the next call. */
const char* hs_last_error(void);

/* Copies *err_flag to the host (synchronising `stream`) and maps it to a status:
 * 0 -> HS_OK, HS_FLAG_TIMEOUT set -> HS_ERR_TIMEOUT, other bits -> HS_ERR_DEVICE_FLAG.
 * *flag_out (may be NULL) receives the raw bits. Convenience for tests; never used inside
 * the other calls. */
hs_status hs_check_flag(const int32_t* err_flag, int32_t* flag_out, hs_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * hs_indexer_scores — lightning-indexer scores.
 *
 * [P1] section 「DP8とTP8が不十分な理由」 and [P2] "¿Por qué no TP o DP?": the indexer scores
 * every prior token to choose the 2,048 that sparse MLA attends; its cost is quadratic in the
 * prompt length ([P1] 「PCP: ヘッドではなくトークンを分割」). Keys are 128-d FP8 with a 4-byte
 * scale ([P1] 「数字がうまくいく理由」). The pages do not print the score formula; this library
 * uses the DSA lightning-indexer form (ReLU of the FP8 dot product, weighted sum over index heads):
 *
 *   s[t, j] = sum_h  w[t,h] * max(0, q_scale[t,h] * k_scale[row(j)] * <q[t,h,:], k[row(j),:]>)
 *
 * for 0 <= j < token_kvlen[t] ("prior" includes the token itself), row(j) as in the paged layout
 * of request token_req[t]. Columns j >= token_kvlen[t] are masked (-inf by definition) and are
 * NOT written: callers read only j < token_kvlen[t].
 *
 * Requirements: q_scale > 0 and k_scale > 0 (the kernel folds them out of the ReLU).
 * Tokens are processed in groups of 256/Hi consecutive tokens; a group may mix requests.
 *
 * Arguments (device pointers unless noted):
 *   T, B          query tokens, requests (B >= 1)
 *   Hi, Di        index heads in {8, 16, 32, 64}; head dim in {64, 128}
 *   q             e4m3 [T, Hi, Di]
 *   q_scale       fp32 [T, Hi]
 *   weights       fp32 [T, Hi]
 *   k_cache       e4m3 [nblk, 64, Di] (16-byte aligned)
 *   k_scale       fp32 [nblk, 64]
 *   block_table   int32 [B, bt_stride]
 *   token_req     int32 [T], in [0, B)
 *   token_kvlen   int32 [T], in [0, min(ld, bt_stride * 64)]
 *   scores        fp32 [T, ld] (output)
 *   err_flag      int32 (device)
 * ---------------------------------------------------------------------------------------- */
typedef struct {
  int32_t T, B, Hi, Di;
  const uint8_t* q;
  const float* q_scale;
  const float* weights;
  const uint8_t* k_cache;
  const float* k_scale;
  int64_t nblk;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* token_req;
  const int32_t* token_kvlen;
  float* scores;
  int64_t ld;
  int32_t* err_flag;
} hs_indexer_args;

hs_status hs_indexer_scores(const hs_indexer_args* a, hs_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * hs_topk — per-query top-k selection.
 *
 * [P1] 「PCP: ヘッドではなくトークンを分割」: each query attends a fixed 2,048 tokens, chosen from
 * the indexer scores. For query t with n = token_kvlen[t] visible scores, writes the
 * min(k, n) indices j < n with the largest scores[t, j], in ascending index order, followed by
 * -1 up to k. Order: larger score first; equal scores -> the lower index wins; -0.0 equals +0.0;
 * NaN ranks below every number (-inf included).
 *
 *   scores       fp32 [T, ld] (device)       token_kvlen int32 [T], in [0, ld]
 *   T, k         1 <= k <= 65536             idx int32 [T, k] (output)
 * ---------------------------------------------------------------------------------------- */
hs_status hs_topk(const float* scores, int64_t ld, const int32_t* token_kvlen, int32_t T, int32_t k,
                  int32_t* idx, int32_t* err_flag, hs_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * hs_indexer_topk — indexer scores and their top-k in one call, the scores kept on chip.
 *
 * [P1] 「DP8とTP8が不十分な理由」: the indexer scores every prior token only so that top-k can
 * pick 2,048 of them; the scores themselves are not needed afterwards. Same result as
 * hs_indexer_scores(a) followed by hs_topk(a->scores, a->ld, a->token_kvlen, a->T, k, idx,
 * a->err_flag): bit-identical idx. The difference is where the scores live between the two
 * kernels: the indexer reads the keys and key scales under an L2 evict-first policy and stores
 * the scores under evict-last, so that (when they fit beside the other live data of the L2,
 * e.g. 256 MTP tokens x 64K keys = 64 MB of 129 MB) top-k reads them from L2, and top-k then
 * drops each row's scores from L2 without writing them back. The scores do not go to HBM and
 * back. Meant for decode batches, whose keys are read once per step; a prefill chunk reads its
 * keys many times and should use the two calls.
 *
 *   a            as hs_indexer_scores; a->scores is scratch of the same shape [T, a->ld], whose
 *                contents are undefined after the call
 *   k, idx       as hs_topk: 1 <= k <= 65536; idx int32 [T, k] (output)
 * Errors: as the two calls.
 * ---------------------------------------------------------------------------------------- */
hs_status hs_indexer_topk(const hs_indexer_args* a, int32_t k, int32_t* idx, hs_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * hs_sparse_mla_fwd — sparse MLA forward, MQA form (every KV row serves all heads).
 *
 * [P1] 「再現方法と必要なフラグ」 (sparse_mla_force_mqa) and 「数字がうまくいく理由」: each query
 * reads its selected 656-byte FP8 latent rows once for all heads; QK runs over 576 dims, PV over
 * 512. For query token t and head h, over the valid entries i of idx[t, :]:
 *
 *   logit_i = softmax_scale * ( sum_{c<512} q[t,h,c] * latent_i[c]  +  sum_{c<64} q[t,h,512+c] * rope_i[c] )
 *   out[t,h,:] = sum_i softmax(logit)_i * latent_i[:]          (bf16, fp32 accumulation)
 *   lse[t,h]   = ln sum_i exp(logit_i)                          (natural log; -inf if no row)
 *
 * Compute precision: the latent part of q and the dequantised latent rows enter the tensor cores as
 * IEEE half (fp16, 10-bit mantissa), the RoPE part as bf16, P as fp16, all accumulated in fp32.
 * Each dequantised value code * scale is rounded once to fp16. A head's q row whose largest |q|
 * lies outside [2^-6, 2^15) is scaled by an exact power of two that puts that value in
 * [2^14, 2^15) before the fp16 conversion (its logits are scaled back in fp32), so any finite bf16
 * q is accepted at full fp16 precision. fp16 bounds the group scales to [2^-14, 146] (so
 * |code * scale| < 65504). A scale outside these bounds, or a latent q value that is not finite,
 * sets HS_FLAG_RANGE; the result is then not reliable.
 *
 * idx entries < 0 are padding and skipped. With block_table == NULL they are physical pool rows
 * (< R); otherwise logical token indices of request token_req[t] mapped through the paged layout.
 * A query with no valid entry gets out = 0 and lse = -inf. Each occurrence of a duplicated entry counts.
 *
 * Shared index sets ([P4] 「MTP受理率の安定化」: the indexer's top-k indices are reused instead of
 * re-running the indexer for every MTP token, and the shared index buffer of a batch keeps only
 * each request's final query token's indices): with idx_row != NULL, query t reads index row
 * idx_row[t] of idx [idx_rows, k] instead of row t, so the query tokens of a request can share the
 * set selected for its final token. token_kvlen (with a block table only) is each query's count of
 * visible tokens: entries j >= token_kvlen[t] are skipped, which keeps a shared set causal for the
 * earlier tokens (they do not see the later draft positions the final token selected). An
 * idx_row[t] outside [0, idx_rows) sets HS_FLAG_BAD_INDEX and the query gets no rows.
 *
 *   T, H          query tokens; heads, 1 <= H <= 64
 *   k             entries per idx row
 *   q             bf16 [T, H, 576] (16-byte aligned)
 *   kv_pool       uint8 [R, 656] (16-byte aligned), 1 <= R <= 2^31 - 1 rows
 *   idx           int32 [T, k], or [idx_rows, k] with idx_row
 *   block_table   int32 [B, bt_stride] or NULL; token_req int32 [T] (required with block_table)
 *   idx_row       int32 [T] or NULL; idx_rows >= 1 rows of idx when given
 *   token_kvlen   int32 [T] or NULL (needs block_table)
 *   out           bf16 [T, H, 512]
 *   lse           fp32 [T, H] or NULL
 *   workspace     NULL: one CTA per query token. Otherwise at least hs_sparse_mla_workspace_size()
 *                 bytes of 16-byte aligned device memory (contents need no initialisation, and are
 *                 scratch after the call): when one CTA per query would leave more than a quarter
 *                 of the SMs' time idle (fewer queries than SMs, or a mostly empty last wave), the
 *                 call gives every SM an equal share of the (query, 64-row tile) work instead. A query split between SMs leaves per-SM
 *                 partial results (softmax-normalised bf16 output and log-sum-exp) in the workspace,
 *                 which a second kernel on the same stream merges by log-sum-exp, as in [P1]
 *                 「DCP: KVキャッシュもシャーディング」 (partial attention merged across shards). Calls that
 *                 share a workspace must not overlap on the GPU.
 * ---------------------------------------------------------------------------------------- */
typedef struct {
  int32_t T, H, k;
  const uint16_t* q;
  const uint8_t* kv_pool;
  int64_t R;
  const int32_t* idx;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* token_req;
  float softmax_scale;
  uint16_t* out;
  float* lse;
  int32_t* err_flag;
  void* workspace;           /* NULL, or caller-owned device scratch (see below) */
  uint64_t workspace_bytes;  /* its size in bytes */
  const int32_t* idx_row;    /* NULL, or the idx row of each query (shared index sets) */
  int32_t idx_rows;          /* rows of idx when idx_row is given */
  const int32_t* token_kvlen;  /* NULL, or each query's visible tokens (entries >= it skipped) */
} hs_mla_args;

hs_status hs_sparse_mla_fwd(const hs_mla_args* a, hs_stream_t stream);

/* Bytes of workspace hs_sparse_mla_fwd needs for H heads on the current device (it depends on the
 * device's SM count): 2 * SMs * H * 1028. */
hs_status hs_sparse_mla_workspace_size(int32_t H, uint64_t* bytes);

/* hs_sparse_mla_fwd_static — hs_sparse_mla_fwd for callers that cannot allocate device memory.
 *
 * The pages describe no such call; it exists for callers whose device memory belongs to another
 * allocator (a serving engine's pooled allocator, a runtime with a fixed budget), or that run
 * where an allocation, which may synchronise the device, is not allowed, and so cannot supply the
 * workspace. Same arguments and results as hs_sparse_mla_fwd; a->workspace and
 * a->workspace_bytes are ignored. The scratch is a 24 MiB array inside the library, present on
 * every GPU that loads it until the process exits; the call allocates nothing.
 *  - HS_ERR_UNSUPPORTED when the split path would need more than those 24 MiB (H heads on a
 *    device with so many SMs that 2 * SMs * H * 1028 bytes exceed them).
 *  - The first call on each device looks up the array's device address (cudaGetSymbolAddress)
 *    with that device current; make it before capturing a stream. The address is cached per
 *    device ordinal for the life of the process, so the call must not be used after
 *    cudaDeviceReset or from a second driver context on the same device.
 *  - All calls share the array and it keeps the last call's contents; nothing in it needs to
 *    start at zero. Calls that overlap on the GPU race on it and must be ordered by the caller. */
hs_status hs_sparse_mla_fwd_static(const hs_mla_args* a, hs_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * hs_hisparse_resolve — Hybrid HiSparse top-k resolve ("mixed residency").
 *
 * [P3] section 「ハイブリッド HiSparse の技術的実装」, item 2: one kernel resolves the top-k of a
 * request whose tail is GPU-resident and whose older pages live in host memory: resident tokens
 * are read as they are, hot tokens are read while their LRU entry is refreshed, and a miss copies
 * one row from pinned host memory into an LRU slot. [P3] 「主要なアーキテクチャ的詳細」: hot
 * buffers are ordinary KV blocks borrowed from the shared pool, 2 x top-k rows per request by
 * default. For each request r (one step):
 *   1. Classify each valid idx[r, i] (i in list order): j >= resident_start[r] -> resident, row =
 *      paged row of j; else tok2slot[r, j] >= 0 -> hit, row = slot_row[r, slot]; else miss.
 *   2. Every hit slot gets slot_stamp = step.
 *   3. The m misses take the m slots not hit this step with the smallest (slot_stamp, slot)
 *      pairs (an empty slot has stamp -1 and token -1, so empty slots go first).
 *   4. The i-th miss in ascending token order takes the i-th such slot: the evicted token's
 *      tok2slot entry becomes -1, the slot gets the new token, tok2slot maps it, its stamp
 *      becomes step, and the 656-byte row j of host_rows[r] is copied to pool row slot_row[slot].
 *   5. out_rows[r, i] = the physical row of entry i (-1 for padding); counters[r] =
 *      {resident, hit, miss}.
 *
 * Requirements: valid entries of each idx row are strictly ascending, followed only by -1;
 * k <= S <= 8192; step is larger than every stamp already in the state; slot_row entries are
 * distinct pool rows that no resident page uses.
 *
 *   B, k, S, step  requests, idx columns, hot slots per request, step number (>= 0)
 *   idx            int32 [B, k]           seq_len int32 [B]     resident_start int32 [B]
 *   block_table    int32 [B, bt_stride]   (pages of resident tokens, indexed by absolute page)
 *   host_rows      device array of B device-accessible pointers, each to pinned uint8 [seq_len, 656]
 *   kv_pool        uint8 [R, 656]
 *   slot_row       int32 [B, S]   slot_token int32 [B, S]   slot_stamp int32 [B, S]  (in/out)
 *   tok2slot       int32 [B, ld_t2s], ld_t2s >= max seq_len (in/out)
 *   out_rows       int32 [B, k]   counters int32 [B, 3] (outputs)
 * ---------------------------------------------------------------------------------------- */
typedef struct {
  int32_t B, k, S, step;
  const int32_t* idx;
  const int32_t* seq_len;
  const int32_t* resident_start;
  const int32_t* block_table;
  int32_t bt_stride;
  const uint8_t* const* host_rows;
  uint8_t* kv_pool;
  int64_t R;
  const int32_t* slot_row;
  int32_t* slot_token;
  int32_t* slot_stamp;
  int32_t* tok2slot;
  int64_t ld_t2s;
  int32_t* out_rows;
  int32_t* counters;
  int32_t* err_flag;
} hs_resolve_args;

hs_status hs_hisparse_resolve(const hs_resolve_args* a, hs_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * hs_hisparse_touch_host — map the host tier for the GPU before the first resolve.
 *
 * [P3] 「ハイブリッド HiSparse の技術的実装」 item 2 has the resolve copy missed rows straight from
 * pinned host memory. The GPU's first read of a host page costs far more than the read itself
 * (about 0.5 us per 64 KB page on a GB300 with its Grace host, where a 13.6 GB tier took 102 ms
 * and a second pass 1.4 ms): a resolve whose misses land on pages the GPU has never read waits on
 * those first reads, and the wait grows with the tier, not with the misses. This call reads one
 * 4-byte word of every host page holding rows [0, min(resident_start[r], seq_len[r])) of each
 * request (the rows a resolve may copy), so that this cost is paid once, when the tier is set up.
 * It changes no memory and nothing a resolve computes.
 *
 *   B               requests
 *   host_rows       device array of B device-accessible pointers (as in hs_resolve_args),
 *                   each 16-byte aligned, to pinned uint8 [seq_len[r], 656]
 *   seq_len, resident_start   int32 [B], device
 *   err_flag        device int32; a misaligned host pointer sets HS_FLAG_BAD_INDEX and its
 *                   request is skipped
 * The page size is the host's (sysconf). Asynchronous on `stream`; allocates nothing.
 * ---------------------------------------------------------------------------------------- */
hs_status hs_hisparse_touch_host(int32_t B, const uint8_t* const* host_rows, const int32_t* seq_len,
                                 const int32_t* resident_start, int32_t* err_flag, hs_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * hs_kv_append — quantise new tokens into the paged FP8 layouts the other calls read.
 *
 * [P1] 「数字がうまくいく理由」: a token's MLA KV is a 656-byte FP8 row and its indexer key is 128
 * FP8 values with a 4-byte scale. For each new token t of request token_req[t] at absolute
 * position token_pos[t], row = block_table[r][pos / 64] * 64 + pos % 64 receives
 *   kv_pool[row]  = [512 x e4m3 latent][4 x fp32 scales, one per 128-dim group][64 x bf16 RoPE]
 *   k_cache[row]  = Di x e4m3,  k_scale[row] = fp32
 * with, per latent group and per key, in IEEE binary32:
 *   scale = max(amax / 448, 2^-14),  code = e4m3(x / scale) (nearest even, saturating at +-448).
 * Inputs must be finite.
 *
 *   T, B            new tokens, requests (token_req[t] in [0, B))
 *   latent, rope    bf16 [T, 512] and [T, 64] (16-byte aligned), or latent = NULL: no MLA rows
 *   index_key       bf16 [T, Di] (16-byte aligned), Di in {64, 128}, or NULL: no indexer keys
 *   token_req, token_pos   int32 [T]
 *   block_table     int32 [B, bt_stride]
 *   kv_pool, R      uint8 [R, 656] (16-byte aligned), needed with latent
 *   k_cache, k_scale, nblk   uint8 [nblk, 64, Di] (16-byte aligned), fp32 [nblk, 64], needed with
 *                   index_key
 *   err_flag        a token with a request or position out of range sets HS_FLAG_BAD_INDEX, one
 *                   whose block is negative or past the pool/cache sets HS_FLAG_BAD_BLOCK; such a
 *                   token writes nothing. Two tokens mapping to one row race (caller error).
 * Asynchronous on `stream`; allocates nothing.
 * ---------------------------------------------------------------------------------------- */
typedef struct {
  int32_t T, B;
  const void* latent;
  const void* rope;
  const void* index_key;
  int32_t Di;
  const int32_t* token_req;
  const int32_t* token_pos;
  const int32_t* block_table;
  int32_t bt_stride;
  uint8_t* kv_pool;
  int64_t R;
  uint8_t* k_cache;
  float* k_scale;
  int64_t nblk;
  int32_t* err_flag;
} hs_kv_append_args;

hs_status hs_kv_append(const hs_kv_append_args* a, hs_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * hs_kv_offload — HiSparse write side: copy complete KV pages to the host tier.
 *
 * [P3] 「主要なアーキテクチャ的詳細」: completed prefix pages are copied to host memory ahead of
 * memory pressure, while the GPU still serves them, and after the forward pass all sparse-MLA
 * layers are copied in one launch ordered on the model's stream. Entry i copies page p = page[i]
 * (tokens 64 p .. 64 p + 63) of request r = req[i] in layer l = layer[i]: the 64 rows of block
 * block_table[r][p] of pools[l] go to rows 64 p .. 64 p + 63 of host_rows[l * B + r]. Block ids
 * are shared by all layers (one block table).
 *
 *   n, L, B         entries, layers, requests
 *   pools           device array of L device pointers, each to uint8 [R, 656] (16-byte aligned)
 *   host_rows       device array of L * B device-accessible pointers, each to pinned uint8
 *                   [seq_len[r], 656] (16-byte aligned)
 *   layer, req, page   int32 [n]
 *   block_table     int32 [B, bt_stride];  seq_len int32 [B]
 *   err_flag        an entry out of range, or a page not complete (64 (p + 1) > seq_len[r]), or a
 *                   misaligned pointer sets HS_FLAG_BAD_INDEX; a negative block or one past R sets
 *                   HS_FLAG_BAD_BLOCK; such an entry copies nothing.
 * Asynchronous on `stream`; allocates nothing. Entries writing the same host rows race (caller
 * error).
 * ---------------------------------------------------------------------------------------- */
typedef struct {
  int32_t n, L, B;
  const uint8_t* const* pools;
  int64_t R;
  uint8_t* const* host_rows;
  const int32_t* layer;
  const int32_t* req;
  const int32_t* page;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_len;
  int32_t* err_flag;
} hs_kv_offload_args;

hs_status hs_kv_offload(const hs_kv_offload_args* a, hs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HS_H_ */
