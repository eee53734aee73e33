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
// step is processed.
//
// Fast path (one full pass over the row):
//   sample: about 1/16 of the row (evenly spaced 128-score blocks) gives a key threshold tau that
//           roughly 1.5 k scores of the row reach (adaptive histogram of the sample);
//   filter: one pass appends the index and score of every score whose key is >= tau to its
//           warp's region of a shared candidate list (ballots give the positions);
//   select: an adaptive histogram of the candidates finds the bin holding the k-th largest; the
//           few candidates in it are sorted by (key descending, index ascending), which fixes the
//           exact composite threshold T; every candidate at or above T is kept;
//   write:  the candidate list is in index order already (warps own consecutive chunks and
//           append in index order), so a ballot of the kept flags per 32 slots and a block-wide
//           prefix sum of their popcounts give each kept index its output place.
// The fast path gives up (and the exact path below runs) when the row has more than 262,144
// scores, when the filter finds fewer than k candidates or more than 512 in one warp's chunk, or
// when more than 1,024 candidates share the threshold bin.
//
// Exact path (several passes, any data):
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
constexpr int kSelBins = 4096;         // fast path: sample and candidate histograms
constexpr int kFastCand = kMaxCand * 2;  // fast path: candidate indices (uint32, same memory as cand)
constexpr int kSample = 4096;          // fast path: sampled scores (at most)
constexpr int kSmallSort = 1024;       // fast path: candidates of the threshold bin (at most)
constexpr int kFastMaxN = 262144;      // fast path: rows of up to this many scores
constexpr int kOffCand = 0;                            // uint64 [kMaxCand] (fast path: candidate indices)
constexpr int kOffHist = kOffCand + kMaxCand * 8;      // uint32 [kBins]
constexpr int kOffCKey = kOffHist + kBins * 4;         // fast path: uint32 [kFastCand] candidate scores
constexpr int kSmem = kOffCKey + kFastCand * 4;         // (the fast path's small sort buffer sits in hist)

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

// As walk_chunk, handing the raw scores instead of keys: f(j0, x[4], valid_mask).
template <typename F>
__device__ __forceinline__ void walk_chunk_f(const float* row, int c0, int c1, bool vec, F&& f) {
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
      const float x[4] = {v[d].x, v[d].y, v[d].z, v[d].w};
      const uint32_t valid = sd + 128 <= c1 ? 0xFu : (uint32_t)((j0 < c1) | ((j0 + 1 < c1) << 1) |
                                                                ((j0 + 2 < c1) << 2) | ((j0 + 3 < c1) << 3));
      f(j0, x, valid);
    }
  }
}

// Block-wide exclusive prefix sum of one value per thread; also returns the total. Each warp scans
// its lanes, then every warp scans the sixteen warp totals itself (no second pass through shared
// memory).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* part, uint32_t& total) {
  static_assert(kWarps <= 32, "one lane per warp total");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) part[warp] = incl;
  __syncthreads();
  const uint32_t x = lane < kWarps ? part[lane] : 0u;
  uint32_t xs = x;
#pragma unroll
  for (int o = 1; o < kWarps; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, xs, o);
    if (lane >= o) xs += y;
  }
  const uint32_t before = __shfl_sync(0xffffffffu, xs - x, warp);
  total = __shfl_sync(0xffffffffu, xs, kWarps - 1);
  __syncthreads();  // part may be written again right after
  return before + incl - v;
}

// Over bins [0, nb) (nb <= kSelBins; every bin from nb up to kSelBins holds 0), finds the bin where
// the count accumulated from the top reaches `need`: returns it with the count strictly above it
// (in *above) and its own count. Thread t owns the eight bins NB - 8 - 8t .. NB - 1 - 8t (NB = nb
// rounded up to 8), read with two 16-byte loads and visited from the top.
__device__ __forceinline__ uint32_t bin_from_top(const uint32_t* hist, uint32_t nb, uint32_t need, uint32_t* part,
                                                 uint32_t* sh, uint32_t& above, uint32_t& count) {
  static_assert(kSelBins == 8 * kThreads, "eight bins per thread");
  const int tid = threadIdx.x;
  const int NB = (int)((nb + 7u) & ~7u);
  const int base = NB - 8 - 8 * tid;  // lowest bin of this thread's eight
  uint32_t c[8];
  if (base >= 0) {
    const uint4 a = *reinterpret_cast<const uint4*>(hist + base);
    const uint4 b = *reinterpret_cast<const uint4*>(hist + base + 4);
    c[0] = b.w, c[1] = b.z, c[2] = b.y, c[3] = b.x, c[4] = a.w, c[5] = a.z, c[6] = a.y, c[7] = a.x;
  } else {
#pragma unroll
    for (int u = 0; u < 8; ++u) c[u] = 0u;
  }
  uint32_t csum = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) csum += c[u];
  if (tid == 0) {  // ordered before the reads below by the scan's barriers
    sh[0] = 0xFFFFFFFFu;
    sh[1] = 0;
    sh[2] = 0;
  }
  uint32_t total;
  uint32_t run = block_excl_scan(csum, part, total);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    if (run < need && need <= run + c[u]) {
      sh[0] = (uint32_t)(base + 7 - u);
      sh[1] = run;
      sh[2] = c[u];
    }
    run += c[u];
  }
  __syncthreads();
  above = sh[1];
  count = sh[2];
  const uint32_t b = sh[0];
  __syncthreads();
  return b;
}

// Inverse of order_key for keys of real numbers: the float whose key is `key`.
__device__ __forceinline__ float key_to_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

// Fast path (see the file header). Returns true when it wrote the row's output; false (with the
// output untouched) when the exact path has to run. All decisions are block-uniform.
// Candidates are score indices in per-warp regions of kFastCand / kWarps slots (the memory of the
// exact path's candidate buffer), with their scores at the same slots of cscore.
__device__ bool fast_topk(const float* row, int n, int k, int c0, int c1, bool vec, uint32_t* hist, uint32_t* cidx,
                          uint32_t* cscore, int32_t* out) {
  constexpr int kRegion = kFastCand / kWarps;  // candidate slots per warp
  static_assert(kRegion == kThreads, "slot u * kRegion + t of the candidate list is thread t's u-th slot");
  __shared__ uint32_t part[kWarps], sh[4], f_min, f_max, f_small, f_valid, f_over, wcnt[kWarps];
  __shared__ uint32_t kflag[kFastCand / 32], kbase[kFastCand / 32];  // kept flags and their prefix, per 32 slots
  __shared__ uint64_t s_T;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (n > kFastMaxN || 3 * k > 2 * kFastCand / 2) return false;
  // ---- sample: evenly spaced 128-score blocks, two per warp, loads issued together; the
  // histogram is cleared while they are in flight, and each lane keeps its keys in registers ----
  const int nblk = (n + 127) / 128;
  const int sblk = nblk < kSample / 128 ? nblk : kSample / 128;
  float4 v[2];
  int jb[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = warp + kWarps * u;
    jb[u] = i < sblk ? 128 * (i * nblk / sblk) : n;  // i * nblk < 2^16: 32-bit math
    const int j0 = jb[u] + 4 * lane;
    if (vec && j0 + 4 <= n) {
      v[u] = __ldg(reinterpret_cast<const float4*>(row + j0));
    } else {
      v[u].x = j0 < n ? __ldg(row + j0) : 0.f;
      v[u].y = j0 + 1 < n ? __ldg(row + j0 + 1) : 0.f;
      v[u].z = j0 + 2 < n ? __ldg(row + j0 + 2) : 0.f;
      v[u].w = j0 + 3 < n ? __ldg(row + j0 + 3) : 0.f;
    }
  }
  if (tid == 0) {
    f_min = 0xFFFFFFFFu;
    f_max = 0u;
    f_valid = 0u;
    f_over = 0u;
  }
  for (int i = tid; i < kSelBins; i += kThreads) hist[i] = 0;
  __syncthreads();
  uint32_t skey[8];
  uint32_t sok = 0;  // bit 4 u + e: skey[4 u + e] is a sampled score of the row
  {
    uint32_t smin = 0xFFFFFFFFu, smax = 0u;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const bool blk = warp + kWarps * u < sblk;
      const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool ok = blk && jb[u] + 4 * lane + e < n;
        const uint32_t key = order_key(f[e]);
        skey[4 * u + e] = key;
        sok |= ok ? 1u << (4 * u + e) : 0u;
        if (ok) {
          smin = min(smin, key);
          smax = max(smax, key);
        }
      }
    }
    uint32_t svalid = (uint32_t)__popc(sok);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      smin = min(smin, __shfl_xor_sync(0xffffffffu, smin, o));
      smax = max(smax, __shfl_xor_sync(0xffffffffu, smax, o));
      svalid += __shfl_xor_sync(0xffffffffu, svalid, o);
    }
    if (lane == 0) {
      atomicMin(&f_min, smin);
      atomicMax(&f_max, smax);
      atomicAdd(&f_valid, svalid);
    }
  }
  __syncthreads();
  const uint32_t S = f_valid, lo_s = f_min, hi_s = f_max;
  // sample rank m whose key becomes tau: about 1.5 k of the row (k itself when the sample is the row)
  uint32_t m = (uint32_t)(S == (uint32_t)n ? k : ((3LL * k * S + 2LL * n - 1) / (2LL * n)));
  if (m < 1) m = 1;
  if (m > S) m = S;
  // ---- adaptive histogram of the sample -> tau ----
  {
    const uint32_t range = hi_s - lo_s;
    const int bits = 32 - __clz(range);
    const int shift = bits > 12 ? bits - 12 : 0;
    const uint32_t nb = (range >> shift) + 1;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if ((sok >> q) & 1u) atomicAdd(&hist[(skey[q] - lo_s) >> shift], 1u);
    __syncthreads();
    uint32_t above, count;
    const uint32_t b = bin_from_top(hist, nb, m, part, sh, above, count);
    if (b == 0xFFFFFFFFu) return false;
    if (tid == 0) sh[3] = lo_s + (b << shift);
  }
  __syncthreads();
  const uint32_t tau = sh[3];
  // key >= tau  <=>  score >= ftau for every number (NaN fails both, its key being 0 < tau unless
  // tau is 0; then ftau is NaN, no candidate is found and the exact path runs)
  const float ftau = key_to_float(tau);
  // ---- filter: the index of every score >= ftau goes to this warp's region ----
  uint32_t* region = cidx + kRegion * warp;
  uint32_t* rscore = cscore + kRegion * warp;  // the candidates' scores (float bits), beside their indices
  uint32_t cnt = 0;  // candidates of this warp so far (warp-uniform)
  const uint32_t lt = (1u << lane) - 1u;
  // Each lane counts its candidates of the step (0-4); three ballots of the count's bits give
  // every lane its offset (lanes in order, each lane's candidates in index order). A step that
  // would overflow the region stores nothing; the count still grows, and the overflow sends the
  // row to the exact path.
  walk_chunk_f(row, c0, c1, vec, [&](int j0, const float (&x)[4], uint32_t valid) {
    uint32_t cm = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) cm |= (x[e] >= ftau) ? (1u << e) : 0u;
    cm &= valid;
    const uint32_t c = (uint32_t)__popc(cm);
    const uint32_t b0 = __ballot_sync(0xffffffffu, c & 1u), b1 = __ballot_sync(0xffffffffu, c & 2u);
    const uint32_t b2 = __ballot_sync(0xffffffffu, c & 4u);
    const uint32_t tot = (uint32_t)__popc(b0) + 2u * (uint32_t)__popc(b1) + 4u * (uint32_t)__popc(b2);
    if (cnt + tot <= (uint32_t)kRegion) {  // warp-uniform
      uint32_t o = cnt + (uint32_t)__popc(b0 & lt) + 2u * (uint32_t)__popc(b1 & lt) + 4u * (uint32_t)__popc(b2 & lt);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (cm & (1u << e)) {
          region[o] = (uint32_t)j0 + e;
          rscore[o++] = __float_as_uint(x[e]);
        }
    }
    cnt += tot;
  });
  if (lane == 0) {
    wcnt[warp] = cnt;
    if (cnt > (uint32_t)kRegion) atomicOr(&f_over, 1u);
    atomicAdd(&f_valid, cnt);  // f_valid now counts S + candidates
  }
  __syncthreads();
  const uint32_t C = f_valid - S;
  if (f_over || C < (uint32_t)k) return false;
  // ---- select: the k-th largest composite (key, -index) among the candidates ----
  // Thread t owns slots t + 512 u (u < 16): their keys, from the scores the filter stored, are
  // kept in registers (0 marks an empty slot: no candidate has key 0, tau > 0).
  constexpr int kPer = kFastCand / kThreads;
  uint32_t ckey[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + kThreads * u;
    const bool used = (uint32_t)(i % kRegion) < wcnt[i / kRegion];
    ckey[u] = used ? order_key(__uint_as_float(cscore[i])) : 0u;
  }
  // Bins over [tau, sample max]; larger keys share the top bin (the map stays monotone, so the
  // selection stays exact: only the few candidates of the threshold bin are compared in full).
  uint64_t T;
  {
    const uint32_t lo = tau, hi = hi_s > tau ? hi_s : tau;
    const uint32_t range = hi - lo;
    const int bits = 32 - __clz(range);
    const int shift = bits > 12 ? bits - 12 : 0;
    const uint32_t nb = (range >> shift) + 1;
    auto bin_of = [&](uint32_t key) -> uint32_t {
      const uint32_t b = (key - lo) >> shift;
      return b < nb ? b : nb - 1;
    };
    for (int i = tid; i < kSelBins; i += kThreads) hist[i] = 0;
    if (tid == 0) f_small = 0;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kPer; ++u)
      if (ckey[u] != 0u) atomicAdd(&hist[bin_of(ckey[u])], 1u);
    __syncthreads();
    uint32_t above, count;
    const uint32_t b = bin_from_top(hist, nb, (uint32_t)k, part, sh, above, count);
    if (b == 0xFFFFFFFFu || count > (uint32_t)kSmallSort) return false;
    // gather the threshold bin's candidates (behind the first kSelBins bins of hist)
    uint64_t* small = reinterpret_cast<uint64_t*>(hist + kSelBins);
#pragma unroll
    for (int u = 0; u < kPer; ++u)
      if (ckey[u] != 0u && bin_of(ckey[u]) == b) {
        const uint32_t j = cidx[tid + kThreads * u];
        small[atomicAdd(&f_small, 1u)] = ((uint64_t)ckey[u] << 32) | (uint32_t)(0xFFFFFFFFu - j);
      }
    __syncthreads();
    const uint32_t want = (uint32_t)k - above - 1;  // rank of T within the bin, from the top
    if (count <= 32) {
      // one warp: each entry's rank is the number of larger entries (the composites are distinct)
      if (warp == 0) {
        const uint64_t v = lane < (int)count ? small[lane] : 0ull;
        uint32_t r = 0;
        for (int j = 0; j < (int)count; ++j) r += __shfl_sync(0xffffffffu, v, j) > v ? 1u : 0u;
        if (lane < (int)count && r == want) s_T = v;
      }
      __syncthreads();
      T = s_T;
    } else {
      int P = 2;
      while (P < (int)count) P <<= 1;
      for (int i = (int)count + tid; i < P; i += kThreads) small[i] = 0;
      __syncthreads();
      // bitonic sort, descending
      for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int i = tid; i < (P >> 1); i += kThreads) {
            const int a = 2 * stride * (i / stride) + (i % stride), c = a + stride;
            const bool desc = (a & size) == 0;
            const uint64_t x = small[a], y = small[c];
            if ((x < y) == desc) {
              small[a] = y;
              small[c] = x;
            }
          }
          __syncthreads();
        }
      }
      T = small[want];
    }
  }
  // ---- write: the kept candidates in index order ----
  // The candidate list is already in index order: region w before region w + 1 (the warps' chunks
  // are consecutive) and ascending within a region. Slot (region u, position t) is thread t's
  // u-th slot, so a ballot per region gives each warp's 32 kept flags as one word; an exclusive
  // prefix over the 256 words in (region, word) order gives every kept candidate its output place.
  uint32_t kept = 0;  // bit u: slot (u, tid) is kept
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const uint32_t j = cidx[tid + kThreads * u];
    const bool kp = ckey[u] != 0u && ((((uint64_t)ckey[u] << 32) | (uint32_t)(0xFFFFFFFFu - j)) >= T);
    kept |= kp ? 1u << u : 0u;
    const uint32_t f = __ballot_sync(0xffffffffu, kp);
    if (lane == 0) kflag[u * kWarps + warp] = f;
  }
  __syncthreads();
  {
    constexpr int kWords = kPer * kWarps;
    static_assert(kWords <= kThreads, "one flag word per thread");
    const uint32_t c = tid < kWords ? (uint32_t)__popc(kflag[tid]) : 0u;
    uint32_t total;
    const uint32_t before = block_excl_scan(c, part, total);
    if (tid < kWords) kbase[tid] = before;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kPer; ++u)
    if ((kept >> u) & 1u) {
      const uint32_t o = kbase[u * kWarps + warp] + (uint32_t)__popc(kflag[u * kWarps + warp] & lt);
      if (o < (uint32_t)k) out[o] = (int32_t)cidx[tid + kThreads * u];
    }
  return true;
}

__global__ void __launch_bounds__(kThreads, 2)
    topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ kvlen, int32_t k,
                int32_t* __restrict__ idx, int32_t* err, int32_t discard) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem_raw + kOffHist);   // [kBins]
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem_raw + kOffCand);   // [kMaxCand]
  uint32_t* cscore = reinterpret_cast<uint32_t*>(smem_raw + kOffCKey);  // [kFastCand]
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
  // the selection; every exit from it is taken by the whole block
  [&]() {
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

    if (fast_topk(row, ni, k, c0, c1, vec, hist, reinterpret_cast<uint32_t*>(cand), cscore, out)) return;

    // ================================ exact path ==================================================
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
  }();
  if (discard) {
    // the row has been read for the last time: its scores leave L2 without being written back to
    // HBM (whole 128-byte lines inside the row only; a line shared with a neighbouring row stays)
    __syncthreads();
    const uintptr_t b = (uintptr_t)(scores + t * ld), e = (uintptr_t)(scores + t * ld + n);
    const uintptr_t l0 = (b + 127) & ~(uintptr_t)127, l1 = e & ~(uintptr_t)127;
    for (uintptr_t a = l0 + (uintptr_t)tid * 128; a < l1; a += (uintptr_t)kThreads * 128)
      discard_l2_line(reinterpret_cast<const void*>(a));
  }
}

}  // namespace topk

cudaError_t launch_topk(const float* scores, int64_t ld, const int32_t* kvlen, int32_t T, int32_t k,
                        int32_t* idx, int32_t* err, bool discard, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(topk::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, topk::kSmem);
  if (e != cudaSuccess) return e;
  // the same shared-memory carve-out as the indexer and sparse-MLA kernels, so the SMs keep their
  // configuration between the three launches of a step
  e = cudaFuncSetAttribute(topk::topk_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  topk::topk_kernel<<<T, topk::kThreads, topk::kSmem, stream>>>(scores, ld, kvlen, k, idx, err, discard ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace hs
