// hs_api.cu — the C ABI declared in include/hs.h: host-side argument checks, then launches.
// Nothing here allocates device memory, synchronises the stream (hs_check_flag aside) or keeps
// state between calls except the calling thread's last error text.
#include <stdarg.h>
#include <stdio.h>
#include <unistd.h>

#include "common.cuh"

namespace hs {
cudaError_t launch_indexer(const hs_indexer_args* a, int num_sms, bool keep_scores, cudaStream_t stream,
                           const char** why);
cudaError_t launch_topk(const float* scores, int64_t ld, const int32_t* kvlen, int32_t T, int32_t k, int32_t* idx,
                        int32_t* err, bool discard, cudaStream_t stream);
cudaError_t launch_mla(const hs_mla_args* a, int sms, cudaStream_t stream, const char** why);
uint64_t mla_workspace_bytes(int32_t H, int sms);
cudaError_t launch_resolve(const hs_resolve_args* a, cudaStream_t stream);
cudaError_t launch_append(const hs_kv_append_args* a, int sms, cudaStream_t stream);
cudaError_t launch_offload(const hs_kv_offload_args* a, int sms, cudaStream_t stream);
cudaError_t launch_touch_host(int32_t B, const uint8_t* const* host_rows, const int32_t* seq_len,
                              const int32_t* resident_start, int64_t page, int32_t* err, cudaStream_t stream);
}  // namespace hs

namespace {

thread_local char g_last_error[512] = "";

hs_status fail(hs_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}

hs_status ok() {
  g_last_error[0] = '\0';
  return HS_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// The kernels use sm_103a instructions (tcgen05, TMA); other devices are refused up front.
hs_status check_device(int* num_sms) {
  int dev = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess && num_sms) e = cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(HS_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
  if (major != 10 || minor != 3)
    return fail(HS_ERR_UNSUPPORTED, "device %d has compute capability %d.%d; this library needs 10.3 (sm_103a)", dev,
                major, minor);
  return HS_OK;
}

hs_status launched(cudaError_t e, const char* what, const char* why) {
  if (e != cudaSuccess) {
    if (e == cudaErrorInvalidValue && why) return fail(HS_ERR_INVALID, "%s: %s", what, why);
    return fail(HS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  }
  return ok();
}

}  // namespace

namespace hs {
// Sets the calling thread's hs_last_error() text; returns s (for calls defined in other files).
hs_status set_last_error(hs_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}
}  // namespace hs

#define REQUIRE(cond, ...) \
  do {                     \
    if (!(cond)) return fail(HS_ERR_INVALID, __VA_ARGS__); \
  } while (0)

extern "C" {

int hs_abi_version(void) { return HS_ABI_VERSION; }

const char* hs_status_str(hs_status s) {
  switch (s) {
    case HS_OK: return "HS_OK";
    case HS_ERR_INVALID: return "HS_ERR_INVALID";
    case HS_ERR_UNSUPPORTED: return "HS_ERR_UNSUPPORTED";
    case HS_ERR_CUDA: return "HS_ERR_CUDA";
    case HS_ERR_DEVICE_FLAG: return "HS_ERR_DEVICE_FLAG";
    case HS_ERR_TIMEOUT: return "HS_ERR_TIMEOUT";
  }
  return "HS_(unknown status)";
}

const char* hs_last_error(void) { return g_last_error; }

hs_status hs_check_flag(const int32_t* err_flag, int32_t* flag_out, hs_stream_t stream) {
  REQUIRE(err_flag, "err_flag is NULL");
  int32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, err_flag, sizeof h, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fail(HS_ERR_CUDA, "reading err_flag: %s", cudaGetErrorString(e));
  if (flag_out) *flag_out = h;
  if (h == 0) return ok();
  if (h & HS_FLAG_TIMEOUT) return fail(HS_ERR_TIMEOUT, "device flag 0x%x (bounded wait ran out)", h);
  return fail(HS_ERR_DEVICE_FLAG, "device flag 0x%x", h);
}

hs_status hs_indexer_scores(const hs_indexer_args* a, hs_stream_t stream) {
  REQUIRE(a, "args is NULL");
  REQUIRE(a->T >= 0 && a->B >= 1, "need T >= 0 and B >= 1 (T=%d, B=%d)", a->T, a->B);
  REQUIRE(a->Hi == 8 || a->Hi == 16 || a->Hi == 32 || a->Hi == 64, "Hi must be 8, 16, 32 or 64 (got %d)", a->Hi);
  REQUIRE(a->Di == 64 || a->Di == 128, "Di must be 64 or 128 (got %d)", a->Di);
  REQUIRE(a->err_flag, "err_flag is NULL");
  if (a->T == 0) return ok();
  REQUIRE(a->q && a->q_scale && a->weights && a->k_cache && a->k_scale && a->block_table && a->token_req &&
              a->token_kvlen && a->scores,
          "a required pointer is NULL");
  REQUIRE(aligned16(a->q) && aligned16(a->k_cache), "q and k_cache must be 16-byte aligned");
  REQUIRE(a->nblk >= 1 && a->nblk * 64 <= INT32_MAX, "nblk out of range (%lld)", (long long)a->nblk);
  REQUIRE(a->bt_stride >= 1 && a->ld >= 1, "bt_stride and ld must be >= 1");
  REQUIRE((int64_t)a->T * a->Hi <= INT32_MAX, "T * Hi too large");
  int sms = 0;
  hs_status st = check_device(&sms);
  if (st != HS_OK) return st;
  const char* why = nullptr;
  return launched(hs::launch_indexer(a, sms, false, (cudaStream_t)stream, &why), "hs_indexer_scores", why);
}

hs_status hs_topk(const float* scores, int64_t ld, const int32_t* token_kvlen, int32_t T, int32_t k, int32_t* idx,
                  int32_t* err_flag, hs_stream_t stream) {
  REQUIRE(T >= 0, "T must be >= 0");
  REQUIRE(k >= 1 && k <= 65536, "k must be in [1, 65536] (got %d)", k);
  REQUIRE(ld >= 1, "ld must be >= 1");
  REQUIRE(err_flag, "err_flag is NULL");
  if (T == 0) return ok();
  REQUIRE(scores && token_kvlen && idx, "a required pointer is NULL");
  hs_status st = check_device(nullptr);
  if (st != HS_OK) return st;
  return launched(hs::launch_topk(scores, ld, token_kvlen, T, k, idx, err_flag, false, (cudaStream_t)stream), "hs_topk",
                  nullptr);
}

hs_status hs_indexer_topk(const hs_indexer_args* a, int32_t k, int32_t* idx, hs_stream_t stream) {
  REQUIRE(a, "args is NULL");
  REQUIRE(a->T >= 0 && a->B >= 1, "need T >= 0 and B >= 1 (T=%d, B=%d)", a->T, a->B);
  REQUIRE(a->Hi == 8 || a->Hi == 16 || a->Hi == 32 || a->Hi == 64, "Hi must be 8, 16, 32 or 64 (got %d)", a->Hi);
  REQUIRE(a->Di == 64 || a->Di == 128, "Di must be 64 or 128 (got %d)", a->Di);
  REQUIRE(k >= 1 && k <= 65536, "k must be in [1, 65536] (got %d)", k);
  REQUIRE(a->err_flag, "err_flag is NULL");
  if (a->T == 0) return ok();
  REQUIRE(a->q && a->q_scale && a->weights && a->k_cache && a->k_scale && a->block_table && a->token_req &&
              a->token_kvlen && a->scores && idx,
          "a required pointer is NULL");
  REQUIRE(aligned16(a->q) && aligned16(a->k_cache), "q and k_cache must be 16-byte aligned");
  REQUIRE(a->nblk >= 1 && a->nblk * 64 <= INT32_MAX, "nblk out of range (%lld)", (long long)a->nblk);
  REQUIRE(a->bt_stride >= 1 && a->ld >= 1, "bt_stride and ld must be >= 1");
  REQUIRE((int64_t)a->T * a->Hi <= INT32_MAX, "T * Hi too large");
  int sms = 0;
  hs_status st = check_device(&sms);
  if (st != HS_OK) return st;
  const char* why = nullptr;
  st = launched(hs::launch_indexer(a, sms, true, (cudaStream_t)stream, &why), "hs_indexer_topk (indexer)", why);
  if (st != HS_OK) return st;
  return launched(hs::launch_topk(a->scores, a->ld, a->token_kvlen, a->T, k, idx, a->err_flag, true,
                                  (cudaStream_t)stream),
                  "hs_indexer_topk (top-k)", nullptr);
}

hs_status hs_sparse_mla_fwd(const hs_mla_args* a, hs_stream_t stream) {
  REQUIRE(a, "args is NULL");
  REQUIRE(a->T >= 0, "T must be >= 0");
  REQUIRE(a->H >= 1 && a->H <= 64, "H must be in [1, 64] (got %d)", a->H);
  REQUIRE(a->k >= 1, "k must be >= 1");
  REQUIRE(a->err_flag, "err_flag is NULL");
  if (a->T == 0) return ok();
  REQUIRE(a->q && a->kv_pool && a->idx && a->out, "a required pointer is NULL");
  REQUIRE(aligned16(a->q) && aligned16(a->kv_pool), "q and kv_pool must be 16-byte aligned");
  REQUIRE(a->R >= 1 && a->R <= INT32_MAX, "R must be in [1, 2^31 - 1]");
  REQUIRE(!a->block_table || (a->token_req && a->bt_stride >= 1), "block_table needs token_req and bt_stride >= 1");
  REQUIRE(!a->idx_row || a->idx_rows >= 1, "idx_row needs idx_rows >= 1");
  REQUIRE(!a->token_kvlen || a->block_table, "token_kvlen needs block_table (it limits logical token indices)");
  REQUIRE((int64_t)a->T * a->H <= INT32_MAX && (int64_t)a->T * a->k <= ((int64_t)1 << 40), "T * H or T * k too large");
  REQUIRE(a->softmax_scale == a->softmax_scale, "softmax_scale is NaN");
  int sms = 0;
  hs_status st = check_device(&sms);
  if (st != HS_OK) return st;
  if (a->workspace) {
    REQUIRE(aligned16(a->workspace), "workspace must be 16-byte aligned");
    const uint64_t need = hs::mla_workspace_bytes(a->H, sms);
    REQUIRE(a->workspace_bytes >= need, "workspace holds %llu bytes; H = %d needs %llu on this device",
            (unsigned long long)a->workspace_bytes, a->H, (unsigned long long)need);
  }
  const char* why = nullptr;
  return launched(hs::launch_mla(a, sms, (cudaStream_t)stream, &why), "hs_sparse_mla_fwd", why);
}

hs_status hs_sparse_mla_workspace_size(int32_t H, uint64_t* bytes) {
  REQUIRE(bytes, "bytes is NULL");
  REQUIRE(H >= 1 && H <= 64, "H must be in [1, 64] (got %d)", H);
  int sms = 0;
  hs_status st = check_device(&sms);
  if (st != HS_OK) return st;
  *bytes = hs::mla_workspace_bytes(H, sms);
  return ok();
}

hs_status hs_hisparse_resolve(const hs_resolve_args* a, hs_stream_t stream) {
  REQUIRE(a, "args is NULL");
  REQUIRE(a->B >= 0, "B must be >= 0");
  REQUIRE(a->k >= 1 && a->k <= a->S, "need 1 <= k <= S (k=%d, S=%d)", a->k, a->S);
  REQUIRE(a->S <= 8192, "S must be <= 8192 (got %d)", a->S);
  REQUIRE(a->step >= 0, "step must be >= 0");
  REQUIRE(a->err_flag, "err_flag is NULL");
  if (a->B == 0) return ok();
  REQUIRE(a->idx && a->seq_len && a->resident_start && a->block_table && a->host_rows && a->kv_pool && a->slot_row &&
              a->slot_token && a->slot_stamp && a->tok2slot && a->out_rows && a->counters,
          "a required pointer is NULL");
  REQUIRE(aligned16(a->kv_pool), "kv_pool must be 16-byte aligned");
  REQUIRE(a->R >= 1 && a->ld_t2s >= 1 && a->bt_stride >= 1, "R, ld_t2s and bt_stride must be >= 1");
  hs_status st = check_device(nullptr);
  if (st != HS_OK) return st;
  return launched(hs::launch_resolve(a, (cudaStream_t)stream), "hs_hisparse_resolve", nullptr);
}

hs_status hs_kv_append(const hs_kv_append_args* a, hs_stream_t stream) {
  REQUIRE(a, "args is NULL");
  REQUIRE(a->T >= 0, "T must be >= 0");
  REQUIRE(a->err_flag, "err_flag is NULL");
  if (a->T == 0) return ok();
  REQUIRE(a->B >= 1, "B must be >= 1");
  REQUIRE(a->latent || a->index_key, "nothing to append: latent and index_key are both NULL");
  REQUIRE(a->token_req && a->token_pos && a->block_table && a->bt_stride >= 1,
          "token_req, token_pos and block_table are required (bt_stride >= 1)");
  if (a->latent) {
    REQUIRE(a->rope && a->kv_pool && a->R >= 1, "latent needs rope, kv_pool and R >= 1");
    REQUIRE(aligned16(a->latent) && aligned16(a->rope) && aligned16(a->kv_pool),
            "latent, rope and kv_pool must be 16-byte aligned");
  }
  if (a->index_key) {
    REQUIRE(a->Di == 64 || a->Di == 128, "Di must be 64 or 128 (got %d)", a->Di);
    REQUIRE(a->k_cache && a->k_scale && a->nblk >= 1, "index_key needs k_cache, k_scale and nblk >= 1");
    REQUIRE(aligned16(a->index_key) && aligned16(a->k_cache), "index_key and k_cache must be 16-byte aligned");
  }
  int sms = 0;
  hs_status st = check_device(&sms);
  if (st != HS_OK) return st;
  return launched(hs::launch_append(a, sms, (cudaStream_t)stream), "hs_kv_append", nullptr);
}

hs_status hs_kv_offload(const hs_kv_offload_args* a, hs_stream_t stream) {
  REQUIRE(a, "args is NULL");
  REQUIRE(a->n >= 0, "n must be >= 0");
  REQUIRE(a->err_flag, "err_flag is NULL");
  if (a->n == 0) return ok();
  REQUIRE(a->L >= 1 && a->B >= 1, "L and B must be >= 1");
  REQUIRE(a->pools && a->host_rows && a->layer && a->req && a->page && a->block_table && a->seq_len,
          "a required pointer is NULL");
  REQUIRE(a->bt_stride >= 1 && a->R >= 64, "bt_stride must be >= 1 and R >= 64");
  int sms = 0;
  hs_status st = check_device(&sms);
  if (st != HS_OK) return st;
  return launched(hs::launch_offload(a, sms, (cudaStream_t)stream), "hs_kv_offload", nullptr);
}

hs_status hs_hisparse_touch_host(int32_t B, const uint8_t* const* host_rows, const int32_t* seq_len,
                                 const int32_t* resident_start, int32_t* err_flag, hs_stream_t stream) {
  REQUIRE(B >= 0, "B must be >= 0");
  REQUIRE(err_flag, "err_flag is NULL");
  if (B == 0) return ok();
  REQUIRE(host_rows && seq_len && resident_start, "a required pointer is NULL");
  hs_status st = check_device(nullptr);
  if (st != HS_OK) return st;
  const long page = sysconf(_SC_PAGESIZE);
  return launched(hs::launch_touch_host(B, host_rows, seq_len, resident_start, page > 0 ? page : 4096, err_flag,
                                        (cudaStream_t)stream),
                  "hs_hisparse_touch_host", nullptr);
}

}  // extern "C"
