// resolve.cu — Hybrid HiSparse top-k resolve (mixed residency), one step.
//
// [P3] "vLLM GLM 5.3 最適化: ハイブリッド HiSparse オフロード", section 「ハイブリッド HiSparse の技術的
// 実装」 item 2: a single kernel resolves a request's top-k: resident tokens are read as they are,
// hot tokens are read while their LRU entry is refreshed, and a miss copies one row from pinned
// host memory into an LRU slot. Section 「主要なアーキテクチャ的詳細」: the hot buffer is made of
// ordinary pool blocks, 2 x top-k rows per request by default.
//
// "LRU slot" is resolved in batch form so that the result does not depend on thread timing:
// hits of this step are refreshed first, then the m misses, in ascending token order, take the
// m slots not hit this step with the smallest (stamp, slot) pairs (empty slots: stamp -1).
//
// One CTA (1024 threads) per request:
//   1. load the idx row, check it (strictly ascending valid prefix, in range); a bad row is
//      flagged and the request is left untouched;
//   2. classify every entry (resident / hit / miss), mark hit slots, write resident and hit rows;
//   3. list the misses in index order with a block scan;
//   4. order the slots by (stamp, slot), untouched ones first: a stable LSD radix sort on
//      stamp - (smallest untouched stamp), 4 bits a pass, starting from slot order, so ties keep
//      slot order. Stamps are step numbers, so their spread is small in practice (one or two
//      passes; none on an all-empty buffer). The first m entries are the victims in order;
//   5. refresh hits, evict the victims' old tokens, insert the misses, write their rows;
//   6. copy each missed 656-byte row from pinned host memory, one warp per row, 16-byte loads,
//      four rows in flight per warp (host-link bound).
//
// touch_kernel reads one word of every host page holding rows a resolve may copy, so that the
// GPU's translation of those pages exists before the first resolve (see hs_hisparse_touch_host).
#include "common.cuh"

namespace hs {
namespace resolve {

constexpr int kThreads = 1024;
constexpr int kChunks = HS_KV_ROW_BYTES / 16;  // 41 x 16 bytes per row

constexpr int kMaxItems = 8;    // slots per thread in the radix sort: S <= 8192
constexpr int kBins = 16;       // 4-bit digits
constexpr int kSlotBits = 16;   // key = (stamp offset << 16) | slot

struct Params {
  int32_t B, k, S, step, items;  // items = ceil(S / kThreads)
  const int32_t* idx;
  const int32_t* seq_len;
  const int32_t* resident_start;
  const int32_t* bt;
  int32_t bt_stride;
  const uint8_t* const* host_rows;
  uint8_t* kv;
  int64_t R;
  const int32_t* slot_row;
  int32_t* slot_token;
  int32_t* slot_stamp;
  int32_t* t2s;
  int64_t ld_t2s;
  int32_t* out_rows;
  int32_t* counters;
  int32_t* err;
};

__global__ void __launch_bounds__(kThreads, 1) resolve_kernel(const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint64_t* sKeyBuf = (uint64_t*)smem_raw;                // [2][S] radix sort ping-pong
  int32_t* sIdx = (int32_t*)(sKeyBuf + 2 * p.S);          // [k]
  int32_t* sMiss = sIdx + p.k;                            // [k] positions of misses, ascending
  uint8_t* sTouched = (uint8_t*)(sMiss + p.k);            // [S]
  __shared__ int32_t sBad, sCnt[3], sMinU, sMaxU, sAnyHit;
  __shared__ uint32_t sScan[kThreads / 32];
  __shared__ uint32_t sTot[kBins * 32], sBinTot[kBins];

  const int tid = threadIdx.x;
  const int64_t r = blockIdx.x;
  const int k = p.k, S = p.S;
  const int32_t n = p.seq_len[r];
  const int32_t rs = p.resident_start[r];
  const int32_t* idx = p.idx + r * k;
  int32_t* out = p.out_rows + r * k;
  const int32_t* srow = p.slot_row + r * S;
  int32_t* stok = p.slot_token + r * S;
  int32_t* sstamp = p.slot_stamp + r * S;
  int32_t* t2s = p.t2s + r * p.ld_t2s;
  const uint8_t* host = p.host_rows[r];

  if (tid == 0) {
    sBad = 0;
    sCnt[0] = sCnt[1] = sCnt[2] = 0;
    sMinU = INT32_MAX;
    sMaxU = INT32_MIN;
    sAnyHit = 0;
  }
  __syncthreads();
  // ---- 1. load and check ----------------------------------------------------------------
  int bad = 0;
  for (int i = tid; i < k; i += kThreads) {
    const int32_t j = idx[i];
    sIdx[i] = j;
    if (j >= 0) {
      if (j >= n || (int64_t)j >= p.ld_t2s) bad |= HS_FLAG_BAD_INDEX;
      if (i > 0) {
        const int32_t prev = idx[i - 1];
        if (prev < 0 || prev >= j) bad |= HS_FLAG_NOT_ASCENDING;
      }
    }
  }
  if (tid == 0 && (((uintptr_t)host) & 15u)) bad |= HS_FLAG_BAD_INDEX;
  if (bad) atomicOr(&sBad, bad);
  for (int s = tid; s < S; s += kThreads) sTouched[s] = 0;
  __syncthreads();
  if (sBad) {
    if (tid == 0) flag_error(p.err, sBad);
    return;
  }
  // ---- 2. classify ---------------------------------------------------------------------------
  int c_res = 0, c_hit = 0;
  for (int i = tid; i < k; i += kThreads) {
    const int32_t j = sIdx[i];
    if (j < 0) {
      out[i] = -1;
    } else if (j >= rs) {
      const int32_t page = j >> 6;
      const int32_t blk = page < p.bt_stride ? p.bt[r * p.bt_stride + page] : -1;
      const int64_t row = (int64_t)blk * 64 + (j & 63);
      if (blk < 0 || row >= p.R) {
        flag_error(p.err, HS_FLAG_BAD_BLOCK);
        out[i] = -1;
      } else {
        out[i] = (int32_t)row;
      }
      ++c_res;
    } else {
      const int32_t sl = t2s[j];
      if (sl >= 0 && sl < S) {
        if (stok[sl] != j) flag_error(p.err, HS_FLAG_BAD_STATE);
        sTouched[sl] = 1;
        out[i] = srow[sl];
        ++c_hit;
      } else if (sl >= S) {
        flag_error(p.err, HS_FLAG_BAD_STATE);
      }
    }
  }
  if (c_res) atomicAdd(&sCnt[0], c_res);
  if (c_hit) atomicAdd(&sCnt[1], c_hit);
  __syncthreads();
  // ---- 3. misses in index order: thread owns a contiguous chunk of entries ----------------
  const int per = (k + kThreads - 1) / kThreads;
  const int i0 = tid * per;
  uint32_t mine = 0;
  for (int i = i0; i < i0 + per && i < k; ++i) {
    const int32_t j = sIdx[i];
    if (j >= 0 && j < rs && !(t2s[j] >= 0 && t2s[j] < S)) ++mine;
  }
  uint32_t v = mine;
  const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) sScan[wid] = v;
  __syncthreads();
  if (wid == 0) {
    uint32_t w = sScan[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sScan[lane] = w;
  }
  __syncthreads();
  uint32_t pos = v - mine + (wid > 0 ? sScan[wid - 1] : 0u);
  const int m = (int)sScan[kThreads / 32 - 1];
  for (int i = i0; i < i0 + per && i < k; ++i) {
    const int32_t j = sIdx[i];
    if (j >= 0 && j < rs && !(t2s[j] >= 0 && t2s[j] < S)) sMiss[pos++] = i;
  }
  // ---- 4. victims: slots ordered by (stamp, slot), untouched first ---------------------------
  const uint64_t* sKeys = sKeyBuf;
  if (m > 0) {
    const int items = p.items;
    // smallest and largest stamp among untouched slots
    int lo = INT32_MAX, hi = INT32_MIN, hit = 0;
    for (int s = tid; s < S; s += kThreads) {
      if (sTouched[s]) {
        hit = 1;
      } else {
        const int st = sstamp[s];
        lo = min(lo, st);
        hi = max(hi, st);
      }
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    hit = __reduce_or_sync(0xffffffffu, hit);
    if (lane == 0) {
      atomicMin(&sMinU, lo);
      atomicMax(&sMaxU, hi);
      if (hit) atomicOr(&sAnyHit, 1);
    }
    __syncthreads();
    // untouched: stamp - lo; touched: one past the largest, so they sort last
    const int32_t minU = sMinU;
    const uint32_t spread = (uint32_t)((int64_t)sMaxU - minU);
    const uint32_t vmax = sAnyHit ? spread + 1u : spread;
    const int passes = (32 - __clz(vmax) + 3) / 4;
    for (int u = 0; u < items; ++u) {
      const int s = tid * items + u;
      if (s < S) {
        const uint32_t v = sTouched[s] ? spread + 1u : (uint32_t)((int64_t)sstamp[s] - minU);
        sKeyBuf[s] = ((uint64_t)v << kSlotBits) | (uint32_t)s;
      }
    }
    __syncthreads();
    int cur = 0;
    for (int pass = 0; pass < passes; ++pass) {
      const uint64_t* in = sKeyBuf + cur * S;
      uint64_t* outk = sKeyBuf + (cur ^ 1) * S;
      const int shift = kSlotBits + 4 * pass;
      uint64_t key[kMaxItems];
      int dig[kMaxItems];
      // per-thread digit counts, 16 bits per bin, bins 4q..4q+3 in c[q]
      uint64_t c0 = 0, c1 = 0, c2 = 0, c3 = 0;
#pragma unroll
      for (int u = 0; u < kMaxItems; ++u) {
        const int pos = tid * items + u;
        dig[u] = -1;
        if (u < items && pos < S) {
          key[u] = in[pos];
          const int d = (int)((key[u] >> shift) & 15u);
          dig[u] = d;
          const uint64_t inc = 1ull << (16 * (d & 3));
          const int q = d >> 2;
          c0 += q == 0 ? inc : 0ull;
          c1 += q == 1 ? inc : 0ull;
          c2 += q == 2 ? inc : 0ull;
          c3 += q == 3 ? inc : 0ull;
        }
      }
      // warp-inclusive scan of the packed counts (a bin's warp total is at most 32 x 8)
      uint64_t i0 = c0, i1 = c1, i2 = c2, i3 = c3;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y0 = __shfl_up_sync(0xffffffffu, i0, o), y1 = __shfl_up_sync(0xffffffffu, i1, o);
        const uint64_t y2 = __shfl_up_sync(0xffffffffu, i2, o), y3 = __shfl_up_sync(0xffffffffu, i3, o);
        if (lane >= o) {
          i0 += y0;
          i1 += y1;
          i2 += y2;
          i3 += y3;
        }
      }
      if (lane == 31) {
#pragma unroll
        for (int d = 0; d < kBins; ++d) {
          const uint64_t w = d < 4 ? i0 : d < 8 ? i1 : d < 12 ? i2 : i3;
          sTot[d * 32 + wid] = (uint32_t)(w >> (16 * (d & 3))) & 0xffffu;
        }
      }
      __syncthreads();
      // exclusive scan of the (bin, warp) totals in bin-major order
      uint32_t incl = 0, mine_tot = 0;
      if (tid < kBins * 32) {
        mine_tot = sTot[tid];
        incl = mine_tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane == 31) sBinTot[wid] = incl;
      }
      __syncthreads();
      if (tid < kBins * 32) {
        uint32_t before = 0;
        for (int d = 0; d < wid; ++d) before += sBinTot[d];
        sTot[tid] = before + incl - mine_tot;
      }
      __syncthreads();
      // scatter, stable: a thread's items go in order after every earlier thread's of that bin
      const uint64_t e0 = i0 - c0, e1 = i1 - c1, e2 = i2 - c2, e3 = i3 - c3;
#pragma unroll
      for (int u = 0; u < kMaxItems; ++u) {
        const int d = dig[u];
        if (d >= 0) {
          const uint64_t e = d < 4 ? e0 : d < 8 ? e1 : d < 12 ? e2 : e3;
          uint32_t rank = sTot[d * 32 + wid] + ((uint32_t)(e >> (16 * (d & 3))) & 0xffffu);
#pragma unroll
          for (int v = 0; v < u; ++v) rank += dig[v] == d ? 1u : 0u;
          outk[rank] = key[u];
        }
      }
      __syncthreads();
      cur ^= 1;
    }
    sKeys = sKeyBuf + cur * S;
  }
  __syncthreads();
  // ---- 5. refresh hits, evict, insert ------------------------------------------------------
  for (int s = tid; s < S; s += kThreads)
    if (sTouched[s]) sstamp[s] = p.step;
  for (int i = tid; i < m; i += kThreads) {
    const int32_t vs = (int32_t)(sKeys[i] & 0xffffu);
    const int32_t old = stok[vs];
    if (old >= 0 && (int64_t)old < p.ld_t2s) t2s[old] = -1;
  }
  __syncthreads();
  for (int i = tid; i < m; i += kThreads) {
    const int32_t vs = (int32_t)(sKeys[i] & 0xffffu);
    const int ip = sMiss[i];
    const int32_t j = sIdx[ip];
    stok[vs] = j;
    t2s[j] = vs;
    sstamp[vs] = p.step;
    out[ip] = srow[vs];
  }
  // ---- 6. copy missed rows from host memory: warp per row, lanes over 16-byte pieces -------
  constexpr int kRowsInFlight = 4;
  for (int i0w = wid; i0w < m; i0w += kRowsInFlight * (kThreads / 32)) {
    uint4 v[kRowsInFlight][2];
    int64_t dst[kRowsInFlight];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int i = i0w + u * (kThreads / 32);
      dst[u] = -1;
      if (i < m) {
        const int32_t j = sIdx[sMiss[i]];
        const int64_t drow = srow[(int32_t)(sKeys[i] & 0xffffu)];
        if (drow >= 0 && drow < p.R) {
          const uint4* src = reinterpret_cast<const uint4*>(host + (int64_t)j * HS_KV_ROW_BYTES);
          v[u][0] = src[lane];
          if (lane + 32 < kChunks) v[u][1] = src[lane + 32];
          dst[u] = drow * HS_KV_ROW_BYTES;
        } else if (lane == 0) {
          flag_error(p.err, HS_FLAG_BAD_INDEX);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      if (dst[u] >= 0) {
        uint4* d = reinterpret_cast<uint4*>(p.kv + dst[u]);
        d[lane] = v[u][0];
        if (lane + 32 < kChunks) d[lane + 32] = v[u][1];
      }
    }
  }
  if (tid == 0) {
    p.counters[r * 3 + 0] = sCnt[0];
    p.counters[r * 3 + 1] = sCnt[1];
    p.counters[r * 3 + 2] = m;
  }
}

// One word of every host page that holds rows [0, min(resident_start, seq_len)) of a request.
__global__ void touch_kernel(const uint8_t* const* host_rows, const int32_t* seq_len, const int32_t* resident_start,
                             int32_t B, int64_t page, int32_t* err) {
  for (int32_t r = blockIdx.y; r < B; r += gridDim.y) {
    const int32_t rows = max(0, min(resident_start[r], seq_len[r]));
    const uint64_t base = (uint64_t)(uintptr_t)host_rows[r];
    if (rows == 0) continue;
    if (base & 15u) {
      if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(err, HS_FLAG_BAD_INDEX);
      continue;
    }
    const uint64_t end = base + (uint64_t)rows * HS_KV_ROW_BYTES;  // a multiple of 16
    const uint64_t first = base / (uint64_t)page, last = (end - 1) / (uint64_t)page;
    for (uint64_t pg = first + blockIdx.x * blockDim.x + threadIdx.x; pg <= last; pg += gridDim.x * blockDim.x) {
      // the page's first word inside the rows; 16-byte aligned, so the 4 bytes lie below end.
      // A volatile load: the value is unused, and a plain one could be dropped as dead code.
      const uint64_t addr = max(base, pg * (uint64_t)page);
      [[maybe_unused]] uint32_t v;
      asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
    }
  }
}

}  // namespace resolve

cudaError_t launch_touch_host(int32_t B, const uint8_t* const* host_rows, const int32_t* seq_len,
                              const int32_t* resident_start, int64_t page, int32_t* err, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const dim3 grid(16, (unsigned)min(B, 65535));
  resolve::touch_kernel<<<grid, 256, 0, stream>>>(host_rows, seq_len, resident_start, B, page, err);
  return cudaGetLastError();
}

cudaError_t launch_resolve(const hs_resolve_args* a, cudaStream_t stream) {
  using namespace resolve;
  Params p;
  p.B = a->B;
  p.k = a->k;
  p.S = a->S;
  p.step = a->step;
  p.items = (a->S + kThreads - 1) / kThreads;
  p.idx = a->idx;
  p.seq_len = a->seq_len;
  p.resident_start = a->resident_start;
  p.bt = a->block_table;
  p.bt_stride = a->bt_stride;
  p.host_rows = a->host_rows;
  p.kv = a->kv_pool;
  p.R = a->R;
  p.slot_row = a->slot_row;
  p.slot_token = a->slot_token;
  p.slot_stamp = a->slot_stamp;
  p.t2s = a->tok2slot;
  p.ld_t2s = a->ld_t2s;
  p.out_rows = a->out_rows;
  p.counters = a->counters;
  p.err = a->err_flag;
  if (a->B == 0) return cudaSuccess;
  const size_t smem = (size_t)a->S * 16 + (size_t)a->k * 8 + (size_t)a->S + 16;
  cudaError_t e = cudaFuncSetAttribute(resolve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  resolve_kernel<<<a->B, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace hs
