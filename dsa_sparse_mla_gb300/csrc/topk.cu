// topk.cu — per-query top-k of the indexer scores.
//
// [P1] "vLLM v0.32.0 GLM-5.3 サービング ...", section 「PCP: ヘッドではなくトークンを分割」: every
// query attends a fixed number (2,048) of tokens chosen from the indexer scores. For query t with
// n = token_kvlen[t] scores: the min(k, n) indices with the largest scores; equal scores go to
// the lower index; -0.0 equals +0.0; NaN ranks below every number. Written ascending, -1 padded.
//
// One CTA of 512 threads per query (two CTAs share an SM). Each score maps to an unsigned key whose
// order is the score order (sign flip trick), so selection is exact integer work. Each warp owns a
// contiguous chunk of the row and streams it with the next step's loads issued before the current
// step is processed (every pass is a walk over L2-resident data, so latency, not bandwidth, rules).
//   pass 0: min and max key of the row;
//   pass 1: histograms of (key - lo) >> shift over 8192 bins, shift chosen so the live key range
//           [lo, hi] fills the bins, narrow [lo, hi] until its keys fit the candidate buffer.
//           Adapting the bins to the data matters: scores of similar magnitude share their top
//           key bits, so fixed top-bit digits would pile them into a handful of bins;
//   pass 2: per chunk, count the keys above hi; collect the keys in [lo, hi] (a few dozen) as
//           candidates, sort them by (key descending, index ascending) and keep the first `need`,
//           i.e. everything at or above one composite threshold (key, index);
//   pass 3: per chunk, in index order, write every key above hi and every kept candidate at
//           its rank: ascending output without a global sort.
#include "common.cuh"

namespace hs {
namespace topk {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 8192;
constexpr int kMaxCand = 4096;
constexpr int kSmem = kBins * 4 + kMaxCand * 8;

// Order-preserving key: x + 0 turns -0 into +0; negative numbers flip all bits, others the sign;
// NaN maps to 0 (below every number).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return x == x ? k : 0u;
}

// Walks this warp's chunk [c0, c1) of the row in index order, 4 keys per lane per step (lane l
// holds indices s + 4l .. s + 4l + 3). Loads are issued kDepth steps at a time (4 KB per warp in
// flight), then f(j0, keys[4], valid_mask) runs on each step; every lane of the warp calls it on
// every step.
constexpr int kDepth = 8;
template <typename F>
__device__ __forceinline__ void walk_chunk(const float* row, int c0, int c1, bool vec, F&& f) {
  const int lane = threadIdx.x & 31;
  for (int s0 = c0; s0 < c1; s0 += 128 * kDepth) {
    float4 v[kDepth];
#pragma unroll
    for (int d = 0; d < kDepth; ++d) {
      const int j0 = s0 + 128 * d + 4 * lane;
      if (vec && j0 + 4 <= c1) {
        v[d] = __ldg(reinterpret_cast<const float4*>(row + j0));
      } else {
        v[d].x = j0 < c1 ? __ldg(row + j0) : 0.f;
        v[d].y = j0 + 1 < c1 ? __ldg(row + j0 + 1) : 0.f;
        v[d].z = j0 + 2 < c1 ? __ldg(row + j0 + 2) : 0.f;
        v[d].w = j0 + 3 < c1 ? __ldg(row + j0 + 3) : 0.f;
      }
    }
#pragma unroll
    for (int d = 0; d < kDepth; ++d) {
      const int sd = s0 + 128 * d;
      if (sd >= c1) break;  // warp-uniform
      const int j0 = sd + 4 * lane;
      const uint32_t keys[4] = {order_key(v[d].x), order_key(v[d].y), order_key(v[d].z), order_key(v[d].w)};
      // all four valid except on the chunk's last (partial) step
      const uint32_t valid = sd + 128 <= c1 ? 0xFu : (uint32_t)((j0 < c1) | ((j0 + 1 < c1) << 1) |
                                                                ((j0 + 2 < c1) << 2) | ((j0 + 3 < c1) << 3));
      f(j0, keys, valid);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2)
    topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ kvlen, int32_t k,
                int32_t* __restrict__ idx, int32_t* err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem_raw);              // [kBins]
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem_raw + kBins * 4);  // [kMaxCand]
  __shared__ uint32_t red_min[kWarps], red_max[kWarps], warp_cnt[kWarps], warp_off[kWarps];
  __shared__ uint32_t scan_part[kWarps];
  __shared__ uint32_t sel_bin, sel_above, sel_count, n_cand;
  __shared__ uint64_t thr;  // composite (key << 32 | ~index) of the last kept candidate
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
  const bool vec = (((uintptr_t)row) & 15u) == 0;
  // warp chunks: multiples of 128 indices so every step but the last is a full float4 per lane
  const int ni = (int)n;  // n <= ld < 2^31 per row
  const int per = ((ni + kWarps - 1) / kWarps + 127) / 128 * 128;
  const int c0 = warp * per;
  const int c1 = c0 + per < ni ? c0 + per : ni;

  // ---- pass 0: key range --------------------------------------------------------------------
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  walk_chunk(row, c0, c1, vec, [&](int, const uint32_t (&key)[4], uint32_t valid) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (valid & (1u << e)) {
        kmin = min(kmin, key[e]);
        kmax = max(kmax, key[e]);
      }
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    red_min[warp] = kmin;
    red_max[warp] = kmax;
  }
  __syncthreads();
  uint32_t lo = red_min[0], hi = red_max[0];
  for (int w = 1; w < kWarps; ++w) {
    lo = min(lo, red_min[w]);
    hi = max(hi, red_max[w]);
  }

  // ---- pass 1: narrow [lo, hi] until it holds at most kMaxCand keys ---------------------------
  uint32_t need = (uint32_t)k;  // keys to take from [lo, hi]; the rest are above hi
  uint32_t in_range = (uint32_t)n;
#pragma unroll 1
  while (in_range > (uint32_t)kMaxCand && lo < hi) {
    const uint32_t range = hi - lo;
    const int bits = 32 - __clz(range);
    const int shift = bits > 13 ? bits - 13 : 0;
    const uint32_t nb = (range >> shift) + 1;  // <= kBins
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    walk_chunk(row, c0, c1, vec, [&](int, const uint32_t (&key)[4], uint32_t valid) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((valid & (1u << e)) && key[e] - lo <= range) atomicAdd(&hist[(key[e] - lo) >> shift], 1u);
    });
    __syncthreads();
    // from the top: thread i sums reversed bins [16i, 16i + 16)
    constexpr int kPerT = kBins / kThreads;
    uint32_t csum = 0;
#pragma unroll
    for (int u = 0; u < kPerT; ++u) {
      const uint32_t rb = kPerT * tid + u;
      csum += rb < nb ? hist[nb - 1 - rb] : 0u;
    }
    uint32_t v = csum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) scan_part[warp] = v;
    __syncthreads();
    uint32_t before = 0;
    for (int w = 0; w < warp; ++w) before += scan_part[w];
    uint32_t run = before + v - csum;
#pragma unroll 1
    for (int u = 0; u < kPerT; ++u) {
      const uint32_t rb = kPerT * tid + u;
      const uint32_t c = rb < nb ? hist[nb - 1 - rb] : 0u;
      if (run < need && need <= run + c) {
        sel_bin = nb - 1 - rb;
        sel_above = run;
        sel_count = c;
      }
      run += c;
    }
    __syncthreads();
    const uint32_t new_lo = lo + (sel_bin << shift);
    const uint32_t width = (1u << shift) - 1u;
    hi = (hi - new_lo) > width ? new_lo + width : hi;
    lo = new_lo;
    need -= sel_above;
    in_range = sel_count;
    __syncthreads();
  }
  // keys in [lo, hi]: in_range (<= kMaxCand, or one single key value repeated), need of them kept

  // ---- pass 2: count keys above hi per chunk; collect candidates ------------------------------
  if (tid == 0) n_cand = 0;
  __syncthreads();
  const bool one_key = lo == hi;  // then the kept candidates are simply the first `need` by index
  uint32_t above = 0;
  walk_chunk(row, c0, c1, vec, [&](int j0, const uint32_t (&key)[4], uint32_t valid) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (!(valid & (1u << e))) continue;
      if (key[e] > hi) {
        ++above;
      } else if (!one_key && key[e] >= lo) {
        const uint32_t slot = atomicAdd(&n_cand, 1u);
        if (slot < (uint32_t)kMaxCand)
          cand[slot] = ((uint64_t)key[e] << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)(j0 + e));
      }
    }
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
  if (lane == 0) warp_cnt[warp] = above;
  __syncthreads();
  if (!one_key) {
    // sort candidates ascending; the kept ones are the top `need`: composite >= cand[P - need]
    const int nc = (int)min(n_cand, (uint32_t)kMaxCand);
    int P = 2;
    while (P < nc) P <<= 1;
    for (int i = nc + tid; i < P; i += kThreads) cand[i] = 0;
    __syncthreads();
    for (int size = 2; size <= P; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < (P >> 1); i += kThreads) {
          const int a = 2 * stride * (i / stride) + (i % stride), b = a + stride;
          const bool asc = (a & size) == 0;
          const uint64_t x = cand[a], y = cand[b];
          if ((x > y) == asc) {
            cand[a] = y;
            cand[b] = x;
          }
        }
        __syncthreads();
      }
    }
    if (tid == 0) thr = cand[P - (int)need];
    __syncthreads();
  }

  // ---- pass 3: ordered write -------------------------------------------------------------------
  // kept(j, key): key > hi, or key in [lo, hi] and (one_key ? its rank among equal keys < need
  //               : composite(key, j) >= thr). For one_key the rank is the running count of
  //               equal keys in index order, so chunks also need their count of equal keys first.
  const uint64_t threshold = thr;
  uint32_t eq_cnt = 0;
  if (one_key) {
    walk_chunk(row, c0, c1, vec, [&](int, const uint32_t (&key)[4], uint32_t valid) {
#pragma unroll
      for (int e = 0; e < 4; ++e) eq_cnt += ((valid >> e) & 1u) && key[e] == lo;
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) eq_cnt += __shfl_xor_sync(0xffffffffu, eq_cnt, o);
  }
  if (lane == 0) scan_part[warp] = eq_cnt;
  __syncthreads();
  // chunk offsets: keys above hi before this chunk + kept candidates before this chunk
  uint32_t eq_before = 0;
  for (int w = 0; w < warp; ++w) eq_before += scan_part[w];
  if (tid == 0) {
    uint32_t off = 0, eq_seen = 0;
    for (int w = 0; w < kWarps; ++w) {
      warp_off[w] = off;
      off += warp_cnt[w];
      if (one_key) {
        const uint32_t take = eq_seen >= need ? 0u : min(need - eq_seen, scan_part[w]);
        off += take;
        eq_seen += scan_part[w];
      }
    }
  }
  __syncthreads();
  if (!one_key) {
    // kept candidates per chunk are counted from the sorted candidate list
    if (tid == 0) {
      for (int w = 0; w < kWarps; ++w) scan_part[w] = 0;
    }
    __syncthreads();
    const int nc = (int)min(n_cand, (uint32_t)kMaxCand);
    int P = 2;
    while (P < nc) P <<= 1;
    for (int i = tid; i < (int)need; i += kThreads) {
      const uint32_t j = 0xFFFFFFFFu - (uint32_t)(cand[P - 1 - i] & 0xFFFFFFFFu);
      atomicAdd(&scan_part[(int)(j / per)], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t extra = 0;
      for (int w = 0; w < kWarps; ++w) {
        warp_off[w] += extra;
        extra += scan_part[w];
      }
    }
    __syncthreads();
  }
  uint32_t pos = warp_off[warp];
  uint32_t eq_run = eq_before;
  walk_chunk(row, c0, c1, vec, [&](int j0, const uint32_t (&key)[4], uint32_t valid) {
    uint32_t keep = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (!(valid & (1u << e))) continue;
      bool kp = key[e] > hi;
      if (!kp && key[e] >= lo) {
        if (one_key) {
          // rank among equal keys = eq_run + equal keys before this one within the step
          kp = true;  // decided below with a warp scan
          keep |= 0x10u << e;
        } else {
          kp = (((uint64_t)key[e] << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)(j0 + e))) >= threshold;
        }
      }
      if (kp && !(keep & (0x10u << e))) keep |= 1u << e;
    }
    if (one_key) {
      const uint32_t ne = (uint32_t)__popc(keep >> 4);
      uint32_t incl = ne;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t r = eq_run + incl - ne;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (keep & (0x10u << e)) {
          if (r < need) keep |= 1u << e;
          ++r;
        }
      eq_run += __shfl_sync(0xffffffffu, incl, 31);
    }
    const uint32_t cnt = (uint32_t)__popc(keep & 0xFu);
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    uint32_t o = pos + incl - cnt;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (keep & (1u << e)) out[o++] = (int32_t)(j0 + e);
    pos += __shfl_sync(0xffffffffu, incl, 31);
  });
}

}  // namespace topk

cudaError_t launch_topk(const float* scores, int64_t ld, const int32_t* kvlen, int32_t T, int32_t k,
                        int32_t* idx, int32_t* err, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(topk::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, topk::kSmem);
  if (e != cudaSuccess) return e;
  topk::topk_kernel<<<T, topk::kThreads, topk::kSmem, stream>>>(scores, ld, kvlen, k, idx, err);
  return cudaGetLastError();
}

}  // namespace hs
