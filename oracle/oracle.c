/*
 * oracle.c — plain, slow CPU oracle of the sparse-MLA (DSA) hot path.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the benchmark's CPU
 * baseline may load this library. The product (the CUDA library and its Python binding) never
 * calls it and shares no code, header, table or constant with it.
 *
 * Every function computes the plain definition in double precision, one element at a time,
 * with no blocking, fusion or reordering beyond what the definition states. Threads only split
 * independent outputs (query tokens or requests) between cores.
 *
 * Sources (web pages describing GLM-5.x serving with DeepSeek sparse attention in vLLM):
 *   [P1] "vLLM v0.32.0 GLM-5.3 サービング: 16基のH200上でのPCP、DCP、およびハイブリッドHiSparse"
 *   [P3] "vLLM GLM 5.3 最適化: ハイブリッド HiSparse オフロード"
 *   OCP 8-bit floating point specification (e4m3) and IEEE 754 binary16/bfloat16 bit layouts.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_PAGE 64
#define ORC_ROW 656
#define ORC_DL 512
#define ORC_DR 64

/* ---------------------------------------------------------------- codecs -------------- */

/* OCP e4m3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal
 * (m * 2^-9); S.1111.111 is NaN; there are no infinities. */
double orc_e4m3_decode(uint8_t b) {
  int sign = b >> 7;
  int e = (b >> 3) & 0xF;
  int m = b & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double orc_bf16_decode(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double e4m3_table[256];
static pthread_once_t table_once = PTHREAD_ONCE_INIT;
static void build_table(void) {
  for (int i = 0; i < 256; ++i) e4m3_table[i] = orc_e4m3_decode((uint8_t)i);
}

/* ---------------------------------------------------------------- threads ------------- */

typedef void (*orc_body)(void* ctx, int64_t i);
typedef struct {
  orc_body body;
  void* ctx;
  int64_t n;
  int64_t next;
  pthread_mutex_t mu;
} orc_pool;

static void* orc_worker(void* arg) {
  orc_pool* p = (orc_pool*)arg;
  for (;;) {
    pthread_mutex_lock(&p->mu);
    int64_t i = p->next++;
    pthread_mutex_unlock(&p->mu);
    if (i >= p->n) break;
    p->body(p->ctx, i);
  }
  return NULL;
}

/* Runs body(ctx, i) for i in [0, n) on `threads` threads (0 = all online cores). */
static void orc_parallel_for(int64_t n, int threads, orc_body body, void* ctx) {
  if (threads <= 0) threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if (threads > n) threads = (int)(n > 0 ? n : 1);
  orc_pool p = {body, ctx, n, 0, PTHREAD_MUTEX_INITIALIZER};
  if (threads == 1) {
    orc_worker(&p);
    return;
  }
  pthread_t tid[256];
  for (int i = 0; i < threads; ++i) pthread_create(&tid[i], NULL, orc_worker, &p);
  for (int i = 0; i < threads; ++i) pthread_join(tid[i], NULL);
}

int orc_num_threads(int threads) {
  if (threads <= 0) threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  return threads < 1 ? 1 : threads;
}

/* Records a contract violation; several worker threads may report at once. */
static void orc_flag(int* status) { __atomic_store_n(status, 1, __ATOMIC_RELAXED); }

/* Physical pool row of logical token j of request r in the paged layout (pages of 64 tokens). */
static int64_t paged_row(const int32_t* block_table, int32_t bt_stride, int32_t r, int64_t j) {
  int64_t page = block_table[(int64_t)r * bt_stride + j / ORC_PAGE];
  return page * ORC_PAGE + j % ORC_PAGE;
}

/* ---------------------------------------------------------------- indexer ------------- */
/*
 * s[t, j] = sum_h w[t,h] * max(0, q_scale[t,h] * k_scale[row(j)] * sum_d q[t,h,d] * k[row(j),d])
 * for j < token_kvlen[t]; -inf for token_kvlen[t] <= j < ld.
 * [P1] 「DP8とTP8が不十分な理由」: the indexer scores every prior token; 「数字がうまくいく理由」:
 * keys are FP8 values with a 4-byte scale. The ReLU and the per-head weights are the DSA
 * lightning-indexer form, which the pages do not print.
 */
typedef struct {
  int32_t T, Hi, Di;
  const uint8_t* q;
  const float* q_scale;
  const float* w;
  const uint8_t* k_cache;
  const float* k_scale;
  int64_t nblk;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* token_req;
  const int32_t* token_kvlen;
  double* scores;
  int64_t ld;
  int status;
} idx_ctx;

static void indexer_token(void* vctx, int64_t t) {
  idx_ctx* c = (idx_ctx*)vctx;
  int32_t r = c->token_req[t];
  int64_t n = c->token_kvlen[t];
  double* out = c->scores + t * c->ld;
  if (n < 0 || n > c->ld || n > (int64_t)c->bt_stride * ORC_PAGE) {
    orc_flag(&c->status);
    return;
  }
  for (int64_t j = 0; j < c->ld; ++j) {
    if (j >= n) {
      out[j] = -INFINITY;
      continue;
    }
    int64_t row = paged_row(c->block_table, c->bt_stride, r, j);
    if (row < 0 || row >= c->nblk * ORC_PAGE) {
      orc_flag(&c->status);
      out[j] = NAN;
      continue;
    }
    double s = 0.0;
    for (int h = 0; h < c->Hi; ++h) {
      const uint8_t* qv = c->q + ((int64_t)t * c->Hi + h) * c->Di;
      const uint8_t* kv = c->k_cache + row * c->Di;
      double dot = 0.0;
      for (int d = 0; d < c->Di; ++d) dot += e4m3_table[qv[d]] * e4m3_table[kv[d]];
      double v = (double)c->q_scale[(int64_t)t * c->Hi + h] * (double)c->k_scale[row] * dot;
      s += (double)c->w[(int64_t)t * c->Hi + h] * (v > 0.0 ? v : 0.0);
    }
    out[j] = s;
  }
}

int orc_indexer_scores(int32_t T, int32_t Hi, int32_t Di, const uint8_t* q, const float* q_scale,
                       const float* w, const uint8_t* k_cache, const float* k_scale, int64_t nblk,
                       const int32_t* block_table, int32_t bt_stride, const int32_t* token_req,
                       const int32_t* token_kvlen, double* scores, int64_t ld, int threads) {
  pthread_once(&table_once, build_table);
  idx_ctx c = {T, Hi, Di, q, q_scale, w, k_cache, k_scale, nblk, block_table, bt_stride,
               token_req, token_kvlen, scores, ld, 0};
  orc_parallel_for(T, threads, indexer_token, &c);
  return c.status;
}

/* ---------------------------------------------------------------- top-k --------------- */
/*
 * For query t: the min(k, n) indices j < n = token_kvlen[t] with the largest scores, ties to
 * the lower index, NaN below everything; written in ascending index order, padded with -1.
 * [P1] 「PCP: ヘッドではなくトークンを分割」: each query attends a fixed set of 2,048 tokens.
 */
typedef struct {
  double s;
  int64_t j;
} orc_pair;

/* Larger score first; NaN last; equal scores (including -0 == +0) by ascending index. */
static int pair_cmp(const void* a, const void* b) {
  const orc_pair* x = (const orc_pair*)a;
  const orc_pair* y = (const orc_pair*)b;
  int xn = isnan(x->s), yn = isnan(y->s);
  if (xn != yn) return xn ? 1 : -1;
  if (!xn && x->s != y->s) return x->s > y->s ? -1 : 1;
  return x->j < y->j ? -1 : (x->j > y->j ? 1 : 0);
}

static int idx_cmp(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return x < y ? -1 : (x > y ? 1 : 0);
}

typedef struct {
  const double* scores;
  int64_t ld;
  const int32_t* token_kvlen;
  int32_t k;
  int32_t* idx;
  int status;
} topk_ctx;

static void topk_token(void* vctx, int64_t t) {
  topk_ctx* c = (topk_ctx*)vctx;
  int64_t n = c->token_kvlen[t];
  int32_t* out = c->idx + t * c->k;
  if (n < 0 || n > c->ld) {
    orc_flag(&c->status);
    for (int i = 0; i < c->k; ++i) out[i] = -1;
    return;
  }
  orc_pair* p = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)(n > 0 ? n : 1));
  for (int64_t j = 0; j < n; ++j) {
    p[j].s = c->scores[t * c->ld + j];
    p[j].j = j;
  }
  qsort(p, (size_t)n, sizeof(orc_pair), pair_cmp);
  int64_t m = n < c->k ? n : c->k;
  for (int64_t i = 0; i < m; ++i) out[i] = (int32_t)p[i].j;
  qsort(out, (size_t)m, sizeof(int32_t), idx_cmp);
  for (int64_t i = m; i < c->k; ++i) out[i] = -1;
  free(p);
}

int orc_topk(const double* scores, int64_t ld, const int32_t* token_kvlen, int32_t T, int32_t k,
             int32_t* idx, int threads) {
  topk_ctx c = {scores, ld, token_kvlen, k, idx, 0};
  orc_parallel_for(T, threads, topk_token, &c);
  return c.status;
}

/* ---------------------------------------------------------------- sparse MLA ---------- */
/*
 * For query t, head h, over valid entries i of idx[t, :] (row = physical, or paged if a block
 * table is given):
 *   latent_i[c] = e4m3(code[c]) * scale[c / 128],  rope_i[c] = bf16 value
 *   logit_i     = sm_scale * (sum_{c<512} q[c] latent_i[c] + sum_{c<64} q[512 + c] rope_i[c])
 *   out[c]      = sum_i exp(logit_i - m) latent_i[c] / Z,  Z = sum_i exp(logit_i - m),
 *   lse         = m + ln Z,  m = max_i logit_i;   no valid entry: out = 0, lse = -inf.
 * [P1] 「数字がうまくいく理由」: 656-byte fp8_ds_mla rows, QK over 576 dims, PV over 512;
 * 「再現方法と必要なフラグ」: every KV row serves all heads (MQA form).
 */
typedef struct {
  int32_t H, k;
  const uint16_t* q;
  const uint8_t* kv;
  int64_t R;
  const int32_t* idx;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* token_req;
  double sm_scale;
  double* out;
  double* lse;
  int status;
} mla_ctx;

static void mla_token(void* vctx, int64_t t) {
  mla_ctx* c = (mla_ctx*)vctx;
  double* lat = (double*)malloc(sizeof(double) * (size_t)(c->k > 0 ? c->k : 1) * (ORC_DL + ORC_DR));
  double* logit = (double*)malloc(sizeof(double) * (size_t)(c->k > 0 ? c->k : 1));
  int nv = 0;
  /* decode the selected rows once: latent (scaled) then rope */
  for (int i = 0; i < c->k; ++i) {
    int64_t j = c->idx[t * c->k + i];
    if (j < 0) continue;
    int64_t row = c->block_table ? paged_row(c->block_table, c->bt_stride, c->token_req[t], j) : j;
    if (row < 0 || row >= c->R) {
      orc_flag(&c->status);
      continue;
    }
    const uint8_t* src = c->kv + row * ORC_ROW;
    float scale[4];
    memcpy(scale, src + ORC_DL, sizeof scale);
    double* dst = lat + (int64_t)nv * (ORC_DL + ORC_DR);
    for (int d = 0; d < ORC_DL; ++d) dst[d] = e4m3_table[src[d]] * (double)scale[d / 128];
    for (int d = 0; d < ORC_DR; ++d) {
      uint16_t h;
      memcpy(&h, src + ORC_DL + 16 + 2 * d, 2);
      dst[ORC_DL + d] = orc_bf16_decode(h);
    }
    ++nv;
  }
  for (int h = 0; h < c->H; ++h) {
    const uint16_t* qh = c->q + ((int64_t)t * c->H + h) * (ORC_DL + ORC_DR);
    double* o = c->out + ((int64_t)t * c->H + h) * ORC_DL;
    double m = -INFINITY;
    for (int i = 0; i < nv; ++i) {
      const double* x = lat + (int64_t)i * (ORC_DL + ORC_DR);
      double acc = 0.0;
      for (int d = 0; d < ORC_DL + ORC_DR; ++d) acc += orc_bf16_decode(qh[d]) * x[d];
      logit[i] = c->sm_scale * acc;
      if (logit[i] > m) m = logit[i];
    }
    for (int d = 0; d < ORC_DL; ++d) o[d] = 0.0;
    if (nv == 0) {
      if (c->lse) c->lse[(int64_t)t * c->H + h] = -INFINITY;
      continue;
    }
    double Z = 0.0;
    for (int i = 0; i < nv; ++i) {
      double p = exp(logit[i] - m);
      Z += p;
      const double* x = lat + (int64_t)i * (ORC_DL + ORC_DR);
      for (int d = 0; d < ORC_DL; ++d) o[d] += p * x[d];
    }
    for (int d = 0; d < ORC_DL; ++d) o[d] /= Z;
    if (c->lse) c->lse[(int64_t)t * c->H + h] = m + log(Z);
  }
  free(lat);
  free(logit);
}

int orc_sparse_mla(int32_t T, int32_t H, int32_t k, const uint16_t* q, const uint8_t* kv_pool,
                   int64_t R, const int32_t* idx, const int32_t* block_table, int32_t bt_stride,
                   const int32_t* token_req, double sm_scale, double* out, double* lse,
                   int threads) {
  pthread_once(&table_once, build_table);
  mla_ctx c = {H, k, q, kv_pool, R, idx, block_table, bt_stride, token_req, sm_scale, out, lse, 0};
  orc_parallel_for(T, threads, mla_token, &c);
  return c.status;
}

/* ---------------------------------------------------------------- HiSparse resolve ---- */
/*
 * One step of the hybrid-HiSparse top-k resolve, request by request, in this order:
 *  (1) classify each valid idx in list order: resident (j >= resident_start), hit
 *      (tok2slot[j] >= 0), or miss;
 *  (2) each hit's slot gets stamp = step;
 *  (3) the m misses take the m slots not hit this step with the smallest (stamp, slot);
 *  (4) the i-th miss in ascending token order takes the i-th such slot: clear the evicted
 *      token's tok2slot, copy the 656-byte host row j into pool row slot_row[slot], set
 *      slot_token, tok2slot and stamp = step;
 *  (5) out_rows = resident paged row or slot_row[slot]; counters = {resident, hit, miss}.
 * [P3] 「ハイブリッド HiSparse の技術的実装」 item 2 (resident / hot + LRU update / miss copied from
 * pinned host memory into an LRU slot) and 「主要なアーキテクチャ的詳細」 (hot buffer borrowed from
 * the shared block pool, 2 x top-k rows by default). The pages say only "LRU slot"; the
 * (stamp, slot) batch order above is the reading this oracle fixes.
 * Returns 0, or 1 when an input breaks the contract (the request is then left as it was).
 */
typedef struct {
  int32_t stamp;
  int32_t slot;
} orc_victim;

static int victim_cmp(const void* a, const void* b) {
  const orc_victim* x = (const orc_victim*)a;
  const orc_victim* y = (const orc_victim*)b;
  if (x->stamp != y->stamp) return x->stamp < y->stamp ? -1 : 1;
  return x->slot < y->slot ? -1 : (x->slot > y->slot ? 1 : 0);
}

typedef struct {
  int32_t j;
  int32_t pos;
} orc_miss;

static int miss_cmp(const void* a, const void* b) {
  const orc_miss* x = (const orc_miss*)a;
  const orc_miss* y = (const orc_miss*)b;
  return x->j < y->j ? -1 : (x->j > y->j ? 1 : 0);
}

typedef struct {
  int32_t k, S, step;
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
  int status;
} res_ctx;

static void resolve_request(void* vctx, int64_t r) {
  res_ctx* c = (res_ctx*)vctx;
  const int32_t* ids = c->idx + r * c->k;
  int32_t* out = c->out_rows + r * c->k;
  int32_t* stoken = c->slot_token + r * c->S;
  int32_t* sstamp = c->slot_stamp + r * c->S;
  const int32_t* srow = c->slot_row + r * c->S;
  int32_t* t2s = c->tok2slot + r * c->ld_t2s;
  char* touched = (char*)calloc((size_t)c->S, 1);
  orc_miss* miss = (orc_miss*)malloc(sizeof(orc_miss) * (size_t)c->k);
  orc_victim* vic = (orc_victim*)malloc(sizeof(orc_victim) * (size_t)c->S);
  int32_t n_res = 0, n_hit = 0, n_miss = 0;
  int bad = 0;
  int32_t prev = -1;
  int ended = 0;
  /* contract checks first, so that a bad request is left untouched */
  for (int i = 0; i < c->k; ++i) {
    int32_t j = ids[i];
    if (j < 0) {
      ended = 1;
      continue;
    }
    if (ended || j <= prev || j >= c->seq_len[r] || j >= c->ld_t2s) bad = 1;
    prev = j;
  }
  if (bad) {
    orc_flag(&c->status);
    free(touched);
    free(miss);
    free(vic);
    return;
  }
  /* (1) classify */
  for (int i = 0; i < c->k; ++i) {
    int32_t j = ids[i];
    if (j < 0) {
      out[i] = -1;
      continue;
    }
    if (j >= c->resident_start[r]) {
      out[i] = (int32_t)paged_row(c->block_table, c->bt_stride, (int32_t)r, j);
      ++n_res;
    } else if (t2s[j] >= 0) {
      int32_t s = t2s[j];
      touched[s] = 1;
      out[i] = srow[s];
      ++n_hit;
    } else {
      miss[n_miss].j = j;
      miss[n_miss].pos = i;
      ++n_miss;
    }
  }
  /* (2) refresh hits */
  for (int s = 0; s < c->S; ++s)
    if (touched[s]) sstamp[s] = c->step;
  /* (3) victims: untouched slots by (stamp, slot) */
  int nv = 0;
  for (int s = 0; s < c->S; ++s)
    if (!touched[s]) {
      vic[nv].stamp = sstamp[s];
      vic[nv].slot = s;
      ++nv;
    }
  qsort(vic, (size_t)nv, sizeof(orc_victim), victim_cmp);
  /* (4) fill misses in ascending token order */
  qsort(miss, (size_t)n_miss, sizeof(orc_miss), miss_cmp);
  for (int i = 0; i < n_miss; ++i) {
    int32_t s = vic[i].slot;
    int32_t old = stoken[s];
    if (old >= 0) t2s[old] = -1;
    stoken[s] = miss[i].j;
    t2s[miss[i].j] = s;
    sstamp[s] = c->step;
    memcpy(c->kv_pool + (int64_t)srow[s] * ORC_ROW, c->host_rows[r] + (int64_t)miss[i].j * ORC_ROW,
           ORC_ROW);
    out[miss[i].pos] = srow[s];
  }
  /* (5) counters */
  c->counters[r * 3 + 0] = n_res;
  c->counters[r * 3 + 1] = n_hit;
  c->counters[r * 3 + 2] = n_miss;
  free(touched);
  free(miss);
  free(vic);
}

int orc_hisparse_resolve(int32_t B, int32_t k, int32_t S, int32_t step, const int32_t* idx,
                         const int32_t* seq_len, const int32_t* resident_start,
                         const int32_t* block_table, int32_t bt_stride,
                         const uint8_t* const* host_rows, uint8_t* kv_pool, int64_t R,
                         const int32_t* slot_row, int32_t* slot_token, int32_t* slot_stamp,
                         int32_t* tok2slot, int64_t ld_t2s, int32_t* out_rows, int32_t* counters,
                         int threads) {
  if (k > S) return 1;
  res_ctx c = {k, S, step, idx, seq_len, resident_start, block_table, bt_stride, host_rows, kv_pool,
               R, slot_row, slot_token, slot_stamp, tok2slot, ld_t2s, out_rows, counters, 0};
  orc_parallel_for(B, threads, resolve_request, &c);
  return c.status;
}

/* ---------------------------------------------------------------- KV append ----------- */
/*
 * Quantise new tokens into the paged FP8 layouts the other operations read.
 * [P1] 「数字がうまくいく理由」: a token's MLA KV is a 656-byte FP8 row (fp8_ds_mla format) and its
 * indexer key is 128 FP8 values with a 4-byte scale. The row is read as
 *   [512 x e4m3 latent codes][4 x fp32 scales, one per 128-dim group][64 x bf16 RoPE],
 * the key as e4m3 codes [Di] plus one fp32 scale. The pages do not print the quantiser; the
 * plain reading used here: per group (latent) or per key (indexer), in IEEE binary32,
 *   scale = max(amax / 448, 2^-14),   code = e4m3_rn_satfinite(x / scale),
 * with x the bf16 input value. These are integer decisions taken from binary32 arithmetic, so
 * this function computes in binary32 (float), not in double: the definition is the binary32 one.
 */

/* OCP e4m3 encoding of a binary32 value: round to nearest, ties to an even mantissa; finite values
 * beyond 448 (and infinities) saturate to +-448; NaN gives S.1111.111. */
uint8_t orc_e4m3_encode(float x) {
  if (isnan(x)) return signbit(x) ? 0xFF : 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  const double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: multiples of 2^-9; 8 * 2^-9 is the smallest normal (code 0x08) */
    const double q = nearbyint(ldexp(a, 9));
    return sign | (uint8_t)q;
  }
  int e;
  frexp(a, &e);                         /* a = f * 2^e, f in [0.5, 1): a in [2^(e-1), 2^e) */
  const int E = e - 1;                  /* a in [2^E, 2^(E+1)) */
  double q = nearbyint(ldexp(a, 3 - E));  /* 8 + mantissa, in [8, 16] */
  int EE = E;
  if (q >= 16.0) {
    q = 8.0;
    EE = E + 1;
  }
  const int code = ((EE + 7) << 3) | ((int)q - 8);
  return sign | (uint8_t)(code > 0x7E ? 0x7E : code);
}

static float bf16_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static float group_scale(const uint16_t* x, int n) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    const float v = fabsf(bf16_to_float(x[i]));
    if (v > amax) amax = v;
  }
  const float s = amax / 448.0f;
  const float floor_s = 6.103515625e-05f; /* 2^-14 */
  return s > floor_s ? s : floor_s;
}

/*
 * For each new token t (request token_req[t] < B, absolute position token_pos[t] >= 0): its row is
 * bt[r][pos / 64] * 64 + pos % 64. latent [T,512], rope [T,64], index_key [T,Di] are bf16 bit
 * patterns; any of latent (with rope) or index_key may be NULL (that part is not written).
 * Returns 1 (nothing written for that token) when a token's request, position or block is out of
 * range.
 */
int orc_kv_append(int32_t T, int32_t B, const uint16_t* latent, const uint16_t* rope, const uint16_t* index_key,
                  int32_t Di, const int32_t* token_req, const int32_t* token_pos, const int32_t* block_table,
                  int32_t bt_stride, uint8_t* kv_pool, int64_t R, uint8_t* k_cache, float* k_scale, int64_t nblk) {
  int status = 0;
  for (int32_t t = 0; t < T; ++t) {
    const int32_t r = token_req[t], pos = token_pos[t];
    if (r < 0 || r >= B || pos < 0 || pos / ORC_PAGE >= bt_stride) {
      status = 1;
      continue;
    }
    const int32_t blk = block_table[(int64_t)r * bt_stride + pos / ORC_PAGE];
    const int64_t row = (int64_t)blk * ORC_PAGE + pos % ORC_PAGE;
    if (blk < 0 || (latent && row >= R) || (index_key && blk >= nblk)) {
      status = 1;
      continue;
    }
    if (latent) {
      uint8_t* dst = kv_pool + row * ORC_ROW;
      for (int g = 0; g < ORC_DL / 128; ++g) {
        const uint16_t* x = latent + (int64_t)t * ORC_DL + 128 * g;
        const float s = group_scale(x, 128);
        for (int c = 0; c < 128; ++c) dst[128 * g + c] = orc_e4m3_encode(bf16_to_float(x[c]) / s);
        memcpy(dst + ORC_DL + 4 * g, &s, 4);
      }
      memcpy(dst + ORC_DL + 16, rope + (int64_t)t * ORC_DR, 2 * ORC_DR);
    }
    if (index_key) {
      const uint16_t* x = index_key + (int64_t)t * Di;
      const float s = group_scale(x, Di);
      for (int c = 0; c < Di; ++c) k_cache[row * Di + c] = orc_e4m3_encode(bf16_to_float(x[c]) / s);
      k_scale[row] = s;
    }
  }
  return status;
}

/* ---------------------------------------------------------------- KV offload ---------- */
/*
 * HiSparse write side: copy complete KV pages from the device pools to the host tier.
 * [P3] 「主要なアーキテクチャ的詳細」: completed prefix pages are copied to host memory ahead of
 * pressure, while the GPU still serves them, and all sparse-MLA layers are copied in one batch
 * after the forward pass. Entry i copies page page[i] (tokens 64 p .. 64 p + 63) of request req[i]
 * in layer layer[i]: the 64 rows of pool block block_table[r][p] of that layer's pool to rows
 * 64 p .. 64 p + 63 of host_rows[layer * B + r]. A page must be complete: 64 (p + 1) <= seq_len[r].
 * Returns 1 (that entry copies nothing) for an entry out of range.
 */
int orc_kv_offload(int32_t n, int32_t L, int32_t B, const uint8_t* const* pools, int64_t R,
                   uint8_t* const* host_rows, const int32_t* layer, const int32_t* req, const int32_t* page,
                   const int32_t* block_table, int32_t bt_stride, const int32_t* seq_len) {
  int status = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t l = layer[i], r = req[i], p = page[i];
    if (l < 0 || l >= L || r < 0 || r >= B || p < 0 || p >= bt_stride || (int64_t)ORC_PAGE * (p + 1) > seq_len[r]) {
      status = 1;
      continue;
    }
    const int32_t blk = block_table[(int64_t)r * bt_stride + p];
    if (blk < 0 || (int64_t)(blk + 1) * ORC_PAGE > R) {
      status = 1;
      continue;
    }
    memcpy(host_rows[(int64_t)l * B + r] + (int64_t)p * ORC_PAGE * ORC_ROW, pools[l] + (int64_t)blk * ORC_PAGE * ORC_ROW,
           (size_t)ORC_PAGE * ORC_ROW);
  }
  return status;
}
