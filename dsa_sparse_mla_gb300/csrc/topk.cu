// topk.cu — per-query top-k of the indexer scores by radix select.
//
// [P1] "vLLM v0.32.0 GLM-5.3 サービング ...", section 「PCP: ヘッドではなくトークンを分割」: every
// query attends a fixed number (2,048) of tokens chosen from the indexer scores. For query t with
// n = token_kvlen[t] scores: the min(k, n) indices with the largest scores; equal scores go to
// the lower index; -0.0 equals +0.0; NaN ranks below every number. Written ascending, -1 padded.
//
// One CTA of 1024 threads per query. Each score maps to an unsigned key whose order is the
// score order (sign flip trick), so selection is exact integer work:
//   passes 1-3: histograms of key bits [31:21], [20:10], [9:0] restricted to the keys that match
//               the prefix found so far -> the exact k-th largest key K and how many of the
//               keys equal to K are still needed;
//   pass 4:     one ordered sweep over the row; a block-wide scan of (above K, equal to K) counts
//               places each selected index at its rank, so the output is ascending and the
//               lowest-indexed ties are the ones kept.
// The row is re-read from L2 on every pass (a 2048-token-query row is at most a few hundred KB).
#include "common.cuh"

namespace hs {
namespace topk {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (x != x) return 0u;                 // NaN: below everything
  if (u == 0x80000000u) u = 0u;          // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive block scan of one uint32 per thread. `scratch` holds kWarps + 1 words.
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t* scratch, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? scratch[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) scratch[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? scratch[warp - 1] : 0u;
  *total = scratch[kWarps - 1];
  __syncthreads();
  return v + before;
}

__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ kvlen, int32_t k,
                int32_t* __restrict__ idx, int32_t* err) {
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t scratch[kWarps + 1];
  __shared__ uint32_t sel_bin, sel_above;
  const int tid = threadIdx.x;
  const int64_t t = blockIdx.x;
  int64_t n = kvlen[t];
  if (n < 0 || n > ld) {
    if (tid == 0) flag_error(err, HS_FLAG_BAD_LENGTH);
    n = n < 0 ? 0 : ld;
  }
  int32_t* out = idx + t * k;
  if (n <= k) {
    for (int i = tid; i < k; i += kThreads) out[i] = i < n ? i : -1;
    return;
  }
  const float* row = scores + t * ld;

  // ---- passes 1-3: find the k-th largest key --------------------------------------------
  uint32_t prefix = 0, mask = 0;
  uint32_t need = (uint32_t)k;  // how many keys >= the answer still to account for inside the prefix
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t nb = pass == 2 ? 1024u : 2048u;
    for (int i = tid; i < (int)nb; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int64_t j = tid; j < n; j += kThreads) {
      const uint32_t key = order_key(__ldg(row + j));
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    // scan bins from the top: thread i owns reversed bins [2i, 2i+1] (fewer when nb = 1024)
    const int per = (int)nb / kThreads;  // 2 or 1
    uint32_t c0 = 0, c1 = 0;
    if (per == 2) {
      c0 = hist[nb - 1 - 2 * tid];
      c1 = hist[nb - 2 - 2 * tid];
    } else {
      c0 = hist[nb - 1 - tid];
    }
    uint32_t total;
    const uint32_t incl = block_incl_scan(c0 + c1, scratch, &total);
    const uint32_t excl = incl - c0 - c1;
    // the bin where the running count (from the top) first reaches `need`
    if (excl < need && need <= excl + c0) {
      sel_bin = per == 2 ? nb - 1 - 2 * tid : nb - 1 - tid;
      sel_above = excl;
    } else if (per == 2 && excl + c0 < need && need <= excl + c0 + c1) {
      sel_bin = nb - 2 - 2 * tid;
      sel_above = excl + c0;
    }
    __syncthreads();
    prefix |= sel_bin << shift;
    mask |= (nb - 1) << shift;
    need -= sel_above;
    __syncthreads();
  }
  const uint32_t kth = prefix;  // exact k-th largest key; `need` of the keys equal to it are taken

  // ---- pass 4: ordered compaction ----------------------------------------------------------
  // Tiles of 4 * kThreads scores, thread i owning 4 consecutive indices. An index's output slot
  // is (#keys > kth before it) + min(#keys == kth before it, need).
  uint32_t gt_run = 0, eq_run = 0;  // counts over the previous tiles
#pragma unroll 1
  for (int64_t base = 0; base < n && gt_run + (eq_run < need ? eq_run : need) < (uint32_t)k;
       base += 4 * kThreads) {
    const int64_t j0 = base + 4 * tid;
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t j = j0 + u;
      if (j < n) {
        const uint32_t key = order_key(__ldg(row + j));
        gt |= key > kth ? (1u << u) : 0u;
        eq |= key == kth ? (1u << u) : 0u;
      }
    }
    const uint32_t packed = ((uint32_t)__popc(gt) << 16) | (uint32_t)__popc(eq);
    uint32_t total;
    const uint32_t excl = block_incl_scan(packed, scratch, &total) - packed;
    uint32_t eq_before = eq_run + (excl & 0xFFFFu);
    uint32_t o = gt_run + (excl >> 16) + (eq_before < need ? eq_before : need);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (gt & (1u << u)) {
        out[o++] = (int32_t)(j0 + u);
      } else if (eq & (1u << u)) {
        if (eq_before < need) out[o++] = (int32_t)(j0 + u);
        ++eq_before;
      }
    }
    gt_run += total >> 16;
    eq_run += total & 0xFFFFu;
  }
}

}  // namespace topk

cudaError_t launch_topk(const float* scores, int64_t ld, const int32_t* kvlen, int32_t T, int32_t k,
                        int32_t* idx, int32_t* err, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  topk::topk_kernel<<<T, topk::kThreads, 0, stream>>>(scores, ld, kvlen, k, idx, err);
  return cudaGetLastError();
}

}  // namespace hs
