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
//   4. sort the 64-bit keys ((stamp + 1) << 32 | slot) of the untouched slots (bitonic, in shared
//      memory); the first m keys are the victims in order;
//   5. refresh hits, evict the victims' old tokens, insert the misses, write their rows;
//   6. copy each missed 656-byte row from pinned host memory with 16-byte loads (host-link bound).
#include "common.cuh"

namespace hs {
namespace resolve {

constexpr int kThreads = 1024;
constexpr int kChunks = HS_KV_ROW_BYTES / 16;  // 41 x 16 bytes per row

struct Params {
  int32_t B, k, S, step, P;  // P: power of two >= S
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
  uint64_t* sKeys = (uint64_t*)smem_raw;                  // [P]
  int32_t* sIdx = (int32_t*)(sKeys + p.P);                // [k]
  int32_t* sMiss = sIdx + p.k;                            // [k] positions of misses, ascending
  uint8_t* sTouched = (uint8_t*)(sMiss + p.k);            // [S]
  __shared__ int32_t sBad, sCnt[3];
  __shared__ uint32_t sScan[kThreads / 32];

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
  // ---- 4. victims: smallest (stamp, slot) among untouched slots ----------------------------
  if (m > 0) {
    for (int s = tid; s < p.P; s += kThreads) {
      uint64_t key = ~0ull;
      if (s < S && !sTouched[s]) key = ((uint64_t)((int64_t)sstamp[s] + 1) << 32) | (uint32_t)s;
      sKeys[s] = key;
    }
    __syncthreads();
    for (int size = 2; size <= p.P; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < (p.P >> 1); i += kThreads) {
          const int lo = 2 * stride * (i / stride) + (i % stride);
          const int hi = lo + stride;
          const bool asc = (lo & size) == 0;
          const uint64_t a = sKeys[lo], b = sKeys[hi];
          if ((a > b) == asc) {
            sKeys[lo] = b;
            sKeys[hi] = a;
          }
        }
        __syncthreads();
      }
    }
  }
  __syncthreads();
  // ---- 5. refresh hits, evict, insert ------------------------------------------------------
  for (int s = tid; s < S; s += kThreads)
    if (sTouched[s]) sstamp[s] = p.step;
  for (int i = tid; i < m; i += kThreads) {
    const int32_t vs = (int32_t)(uint32_t)sKeys[i];
    const int32_t old = stok[vs];
    if (old >= 0 && (int64_t)old < p.ld_t2s) t2s[old] = -1;
  }
  __syncthreads();
  for (int i = tid; i < m; i += kThreads) {
    const int32_t vs = (int32_t)(uint32_t)sKeys[i];
    const int ip = sMiss[i];
    const int32_t j = sIdx[ip];
    stok[vs] = j;
    t2s[j] = vs;
    sstamp[vs] = p.step;
    out[ip] = srow[vs];
  }
  // ---- 6. copy missed rows from host memory --------------------------------------------------
  const int total = m * kChunks;
  for (int c0 = tid; c0 < total; c0 += 4 * kThreads) {
    uint4 v4[4];
    int64_t dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * kThreads;
      dst[u] = -1;
      if (c < total) {
        const int i = c / kChunks, part = c - i * kChunks;
        const int32_t j = sIdx[sMiss[i]];
        const int64_t drow = srow[(int32_t)(uint32_t)sKeys[i]];
        if (drow >= 0 && drow < p.R) {
          v4[u] = __ldg(reinterpret_cast<const uint4*>(host + (int64_t)j * HS_KV_ROW_BYTES) + part);
          dst[u] = drow * HS_KV_ROW_BYTES + part * 16;
        } else if (part == 0) {
          flag_error(p.err, HS_FLAG_BAD_INDEX);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dst[u] >= 0) *reinterpret_cast<uint4*>(p.kv + dst[u]) = v4[u];
  }
  if (tid == 0) {
    p.counters[r * 3 + 0] = sCnt[0];
    p.counters[r * 3 + 1] = sCnt[1];
    p.counters[r * 3 + 2] = m;
  }
}

}  // namespace resolve

cudaError_t launch_resolve(const hs_resolve_args* a, cudaStream_t stream) {
  using namespace resolve;
  Params p;
  p.B = a->B;
  p.k = a->k;
  p.S = a->S;
  p.step = a->step;
  int P = 1;
  while (P < a->S) P <<= 1;
  if (P < 2) P = 2;
  p.P = P;
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
  const size_t smem = (size_t)P * 8 + (size_t)a->k * 8 + (size_t)a->S + 16;
  cudaError_t e = cudaFuncSetAttribute(resolve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  resolve_kernel<<<a->B, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace hs
