// offload.cu — HiSparse write side: complete KV pages from the device pools to the host tier.
//
// [P3] "vLLM GLM 5.3 最適化: ハイブリッド HiSparse オフロード", section 「主要なアーキテクチャ的詳細」:
// completed prefix pages are copied to host memory ahead of memory pressure, while the GPU still
// serves them, and after the forward pass all sparse-MLA layers are copied in one launch ordered
// on the model's stream. Entry i copies page page[i] of request req[i] in layer layer[i]: the 64 rows
// of pool block block_table[r][p] of that layer's pool to rows 64 p .. 64 p + 63 of the layer's host
// rows of the request. Only complete pages (64 (p + 1) <= seq_len[r]) are copied.
//
// One CTA per page (grid-stride over the entries): 256 threads move the page's 2,624 16-byte pieces,
// every thread issuing all of its loads before its stores; the stores go straight to pinned host
// memory. Bound by the host link.
#include "common.cuh"

namespace hs {
namespace offload {

constexpr int kThreads = 256;
constexpr int kPageBytes = 64 * HS_KV_ROW_BYTES;           // 41,984
constexpr int kVecs = kPageBytes / 16;                      // 2,624
constexpr int kPer = (kVecs + kThreads - 1) / kThreads;     // 11

struct Params {
  int32_t n, L, B, bt_stride;
  const uint8_t* const* pools;
  int64_t R;
  uint8_t* const* host_rows;
  const int32_t* layer;
  const int32_t* req;
  const int32_t* page;
  const int32_t* bt;
  const int32_t* seq_len;
  int32_t* err;
};

__global__ void __launch_bounds__(kThreads) offload_kernel(const Params p) {
  for (int64_t i = blockIdx.x; i < p.n; i += gridDim.x) {
    const int32_t l = p.layer[i], r = p.req[i], pg = p.page[i];
    // every thread evaluates the same conditions: the CTA stays uniform
    if (l < 0 || l >= p.L || r < 0 || r >= p.B || pg < 0 || pg >= p.bt_stride || 64LL * (pg + 1) > p.seq_len[r]) {
      if (threadIdx.x == 0) flag_error(p.err, HS_FLAG_BAD_INDEX);
      continue;
    }
    const int32_t blk = p.bt[(int64_t)r * p.bt_stride + pg];
    if (blk < 0 || (int64_t)(blk + 1) * 64 > p.R) {
      if (threadIdx.x == 0) flag_error(p.err, HS_FLAG_BAD_BLOCK);
      continue;
    }
    const uint8_t* pool = p.pools[l];
    uint8_t* host = p.host_rows[(int64_t)l * p.B + r];
    if ((((uintptr_t)pool) | ((uintptr_t)host)) & 15u) {
      if (threadIdx.x == 0) flag_error(p.err, HS_FLAG_BAD_INDEX);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(pool + (int64_t)blk * kPageBytes);
    uint4* dst = reinterpret_cast<uint4*>(host + (int64_t)pg * kPageBytes);
    uint4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int j = threadIdx.x + u * kThreads;
      if (j < kVecs) v[u] = ldg_nc_v4(src + j);
    }
    asm volatile("" ::: "memory");  // every load is issued before the first store
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int j = threadIdx.x + u * kThreads;
      if (j < kVecs) dst[j] = v[u];
    }
  }
}

}  // namespace offload

cudaError_t launch_offload(const hs_kv_offload_args* a, int sms, cudaStream_t stream) {
  using namespace offload;
  Params p;
  p.n = a->n;
  p.L = a->L;
  p.B = a->B;
  p.bt_stride = a->bt_stride;
  p.pools = a->pools;
  p.R = a->R;
  p.host_rows = a->host_rows;
  p.layer = a->layer;
  p.req = a->req;
  p.page = a->page;
  p.bt = a->block_table;
  p.seq_len = a->seq_len;
  p.err = a->err_flag;
  if (a->n == 0) return cudaSuccess;
  int64_t blocks = a->n;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  offload_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace hs
