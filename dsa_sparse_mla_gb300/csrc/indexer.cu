// indexer.cu — lightning-indexer scores as an FP8 tcgen05 GEMM with a fused epilogue.
//
// [P1] "vLLM v0.32.0 GLM-5.3 サービング ...", section 「DP8とTP8が不十分な理由」: the indexer
// scores every prior token to pick the tokens sparse MLA attends; section 「数字がうまくいく理由」:
// keys are 128 FP8 values with a 4-byte scale. Score (DSA lightning-indexer form):
//   s[t, j] = sum_h w[t,h] * max(0, q_scale[t,h] * k_scale[j] * <q[t,h,:], k[j,:]>),  j < n_t.
// Since both scales are positive, s = k_scale[j] * sum_h (w*q_scale)[t,h] * max(0, <q, k>):
// the GEMM runs on raw e4m3 codes and the scales are applied in the epilogue.
//
// Work split: a CTA owns one group of 256/Hi consecutive query tokens (so the MMA's N is
// tokens x heads = 256) and a contiguous range of 128-key tiles of each request in the group.
// Keys sit on the MMA's M (TMEM lanes), so each epilogue thread owns one key and does the ReLU,
// the weighted head sum and the causal mask in registers, then writes one coalesced score.
//
// Roles (576 threads): warp 0 issues TMA loads (query tile once, two 64-key pages per stage, and
// the pages' key scales), warp 1 allocates TMEM and issues tcgen05.mma (e4m3 x e4m3 -> fp32,
// M=128, N=256, K=32), warps 2..17 drain the two TMEM accumulators: each warp owns its 32-lane
// quarter and a 64-column slice, reads the slice into registers, hands the accumulator back to
// the MMA at once, and only then does the arithmetic (so the tensor pipe never waits for the ALU
// work of the tile before). Four epilogue warps per scheduler keep its ALU work issuing.
#include "common.cuh"

namespace hs {
namespace indexer {

constexpr int kBlockM = 128;   // keys per tile (two pages)
constexpr int kN = 256;        // (token, head) columns per group
constexpr int kStages = 6;
constexpr int kEpiWarps = 16;   // four per TMEM lane quarter, each a 64-column slice
constexpr int kSlice = kN * 4 / kEpiWarps;  // accumulator columns per epilogue warp
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxG = 32;      // tokens per group when Hi = 8
constexpr int kMaxTpc = 64;    // tiles per CTA and segment
// Key scales of tile i sit in slot i % kScaleRing. The TMA warp refills a slot for tile i + 8 only
// after MMA of tile i + 2 released stage (i + 8) % kStages, and that MMA waited for every epilogue
// warp to have read tile i (scales included) from the accumulator it reuses: 8 slots never race.
constexpr int kScaleRing = kStages + 2;

struct Params {
  int32_t T, B, Hi, Di;
  const float* q_scale;
  const float* weights;
  const float* k_scale;
  int64_t nblk;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* token_req;
  const int32_t* token_kvlen;
  float* scores;
  int64_t ld;
  int32_t* err;
  int32_t tiles_per_cta;
  int32_t scale_tma;  // k_scale is 16-byte aligned: the TMA warp copies each page's 64 scales to smem
};

// Shared-memory load issued where it is written: the folded head weights are the same for every
// tile, and letting the compiler hoist them out of the tile loop makes it spill them to local
// memory and reload them from there on every tile.
__device__ __forceinline__ float4 lds_f4(const float* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

template <int DI, int HI>
struct Cfg {
  static constexpr int G = kN / HI;
  static constexpr int kTileBytes = kBlockM * DI;
  static constexpr int kQBytes = kN * DI;
  static constexpr uint32_t kSwizzle = DI == 128 ? 2u : 4u;  // 128-byte / 64-byte swizzle
  static constexpr uint32_t kSBO = 8 * DI;                    // one 8-row swizzle atom
  static constexpr int kKSteps = DI / 32;                     // K = 32 per e4m3 MMA
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQBytes;
  static constexpr int kOffW = kOffK + kStages * kTileBytes;
  static constexpr int kOffTok = kOffW + kN * 4;              // int32 x 4 x kMaxG
  static constexpr int kOffSeg = kOffTok + 4 * kMaxG * 4;     // int32 x 4 x kMaxG
  static constexpr int kOffBlk = kOffSeg + 4 * kMaxG * 4;   // int32 [kMaxG][2 * kMaxTpc]
  static constexpr int kOffLim = kOffBlk + kMaxG * 2 * kMaxTpc * 4;  // int32 [kMaxG][kMaxG]
  static constexpr int kOffScale = kOffLim + kMaxG * kMaxG * 4;  // float [kScaleRing][kBlockM]
  static constexpr int kOffBar = kOffScale + kScaleRing * kBlockM * 4;
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffMisc + 64 + 1024;          // + alignment slack
};

template <int DI, int HI>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const Params p) {
  using C = Cfg<DI, HI>;
  constexpr int G = C::G;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sK = smem + C::kOffK;
  float* sW = (float*)(smem + C::kOffW);                 // (w * q_scale) [G][HI]
  int32_t* sTokN = (int32_t*)(smem + C::kOffTok);        // visible keys per token (0 = skip)
  int32_t* sTokSeg = sTokN + kMaxG;                      // segment of each token (-1 = none)
  int32_t* sSegReq = (int32_t*)(smem + C::kOffSeg);      // request of each segment
  int32_t* sSegN = sSegReq + kMaxG;                      // max visible keys in the segment
  int32_t* sSegLo = sSegN + kMaxG;                       // first tile of this CTA
  int32_t* sSegHi = sSegLo + kMaxG;                      // one past the last tile
  int32_t* sBlk = (int32_t*)(smem + C::kOffBlk);         // physical page of each of the CTA's pages
  int32_t* sLim = (int32_t*)(smem + C::kOffLim);         // [segment][token]: visible keys, 0 = other request
  float* sScale = (float*)(smem + C::kOffScale);         // key scales of the tiles in flight
  uint64_t* bars = (uint64_t*)(smem + C::kOffBar);
  uint64_t* full = bars;                                 // [kStages]
  uint64_t* empty = bars + kStages;                      // [kStages]
  uint64_t* acc_full = bars + 2 * kStages;               // [2]
  uint64_t* acc_empty = acc_full + 2;                    // [2]
  uint64_t* q_full = acc_empty + 2;
  uint64_t* mma_done = q_full + 1;
  int32_t* misc = (int32_t*)(smem + C::kOffMisc);        // [0] nseg, [1] abort, [2] tmem base
  volatile int32_t* abort_flag = misc + 1;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int group = blockIdx.x, split = blockIdx.y;
  const int t0 = group * G;

  // ---------------- setup: token metadata, folded weights, segments, barriers, TMEM -------------
  if (tid < G) {
    const int t = t0 + tid;
    int32_t n = 0, r = -1;
    if (t < p.T) {
      r = p.token_req[t];
      n = p.token_kvlen[t];
      const int64_t nmax = p.ld < (int64_t)p.bt_stride * 64 ? p.ld : (int64_t)p.bt_stride * 64;
      if (r < 0 || r >= p.B) {
        flag_error(p.err, HS_FLAG_BAD_INDEX);
        n = 0;
      } else if (n < 0 || (int64_t)n > nmax) {
        flag_error(p.err, HS_FLAG_BAD_LENGTH);
        n = 0;
      }
    }
    sTokN[tid] = n;
    sTokSeg[tid] = (n > 0) ? r : -1;  // request for now; turned into a segment id below
  }
  if (tid < G * HI) {
    // folded weight w * q_scale; heads 4m+2, 4m+3 take their ReLU as x + |x| = 2 max(x, 0), so
    // their weight carries the factor 1/2 (exact)
    const int g = tid / HI, h = tid % HI, t = t0 + g;
    const float half = (h & 2) ? 0.5f : 1.f;
    sW[tid] = (t < p.T) ? half * (p.weights[(int64_t)t * HI + h] * p.q_scale[(int64_t)t * HI + h]) : 0.f;
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
    }
    mbar_init(q_full, 1);
    mbar_init(mma_done, 1);
    mbar_fence_init();
    misc[1] = 0;
  }
  if (warp == 1) tmem_alloc((uint32_t*)&misc[2], 512);
  __syncthreads();
  if (tid == 0) {
    int nseg = 0;
    for (int g = 0; g < G; ++g) {
      const int r = sTokSeg[g];
      if (r < 0) continue;
      int s = 0;
      while (s < nseg && sSegReq[s] != r) ++s;
      if (s == nseg) {
        sSegReq[s] = r;
        sSegN[s] = 0;
        ++nseg;
      }
      sTokSeg[g] = s;
      if (sTokN[g] > sSegN[s]) sSegN[s] = sTokN[g];
    }
    for (int s = 0; s < nseg; ++s) {
      const int tiles = (sSegN[s] + kBlockM - 1) / kBlockM;
      const int lo = split * p.tiles_per_cta;
      int hi = lo + p.tiles_per_cta;
      if (hi > tiles) hi = tiles;
      sSegLo[s] = lo;
      sSegHi[s] = hi > lo ? hi : lo;
    }
    misc[0] = nseg;
  }
  __syncthreads();
  // keys token g may see while the CTA scores segment s (0 when g belongs to another request)
  for (int i = tid; i < misc[0] * G; i += kThreads) {
    const int sg = i / G, g = i % G;
    sLim[sg * kMaxG + g] = sTokSeg[g] == sg ? sTokN[g] : 0;
  }
  // stage this CTA's block-table entries (2 pages per tile) so no warp waits on them later
  for (int s = 0; s < misc[0]; ++s) {
    const int r = sSegReq[s];
    const int npg = 2 * (sSegHi[s] - sSegLo[s]);
    for (int i = tid; i < npg; i += kThreads) {
      const int page = 2 * sSegLo[s] + i;
      int32_t b = -1;
      if (page * 64 < sSegN[s]) {
        b = p.block_table[(int64_t)r * p.bt_stride + page];
        if (b < 0 || (int64_t)b >= p.nblk) {
          flag_error(p.err, HS_FLAG_BAD_BLOCK);
          b = -1;
        }
      }
      sBlk[s * 2 * kMaxTpc + i] = b;
    }
  }
  __syncthreads();
  tc_fence_after();
  const int nseg = misc[0];
  const uint32_t tmem = (uint32_t)misc[2];
  int total = 0;
  for (int s = 0; s < nseg; ++s) total += sSegHi[s] - sSegLo[s];

  if (total > 0) {
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer ----------------
      if (lane == 0) {
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_k);
        mbar_arrive_expect_tx(q_full, C::kQBytes);
        tma_load_2d(sQ, &map_q, q_full, 0, t0 * HI);
        int it = 0;
        for (int s = 0; s < nseg && !*abort_flag; ++s) {
          for (int kt = sSegLo[s]; kt < sSegHi[s]; ++kt, ++it) {
            const int st = it % kStages;
            const uint32_t ph = (uint32_t)(it / kStages) & 1u;
            if (!mbar_wait(&empty[st], ph ^ 1u, p.err)) {
              *abort_flag = 1;
              break;
            }
            int32_t blk[2];
            uint32_t bytes = 0;
            for (int pg = 0; pg < 2; ++pg) {
              blk[pg] = sBlk[s * 2 * kMaxTpc + 2 * (kt - sSegLo[s]) + pg];
              if (blk[pg] >= 0) bytes += 64 * DI + (p.scale_tma ? 64 * 4 : 0);
            }
            mbar_arrive_expect_tx(&full[st], bytes);
            for (int pg = 0; pg < 2; ++pg)
              if (blk[pg] >= 0) {
                tma_load_2d(sK + st * C::kTileBytes + pg * 64 * DI, &map_k, &full[st], 0, blk[pg] * 64);
                if (p.scale_tma)
                  bulk_g2s(sScale + (it % kScaleRing) * kBlockM + pg * 64, p.k_scale + (int64_t)blk[pg] * 64, 64 * 4,
                           &full[st]);
              }
          }
        }
        // every issued copy must land before the CTA's shared memory is released
        mbar_wait(q_full, 0, p.err);
        for (int i = it > kStages ? it - kStages : 0; i < it; ++i)
          mbar_wait(&full[i % kStages], (uint32_t)(i / kStages) & 1u, p.err);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer ------------------
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_e4m3(kBlockM, kN);
        const uint32_t q_addr = smem_u32(sQ);
        const uint32_t k_addr = smem_u32(sK);
        bool ok = mbar_wait(q_full, 0, p.err);
        int it = 0;
        for (int s = 0; s < nseg && ok && !*abort_flag; ++s) {
          for (int kt = sSegLo[s]; kt < sSegHi[s]; ++kt, ++it) {
            const int st = it % kStages;
            const uint32_t ph = (uint32_t)(it / kStages) & 1u;
            const int b = it & 1;
            const uint32_t aph = (uint32_t)(it >> 1) & 1u;
            if (!mbar_wait(&full[st], ph, p.err) || !mbar_wait(&acc_empty[b], aph ^ 1u, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
              const uint64_t a = smem_desc(k_addr + st * C::kTileBytes + ks * 32, 16, C::kSBO, C::kSwizzle);
              const uint64_t bq = smem_desc(q_addr + ks * 32, 16, C::kSBO, C::kSwizzle);
              mma_e4m3_ss(tmem + (uint32_t)(b * kN), a, bq, idesc, ks > 0 ? 1u : 0u);
            }
            mma_commit(&empty[st]);
            mma_commit(&acc_full[b]);
          }
        }
        if (!ok) *abort_flag = 1;
        // all issued MMAs must finish before TMEM is released
        mma_commit(mma_done);
        mbar_wait(mma_done, 0, p.err);
      }
    } else {
      // ------------------------------------------------------------ epilogue --------------------
      constexpr int kTok = kSlice / HI;  // tokens in a warp's column slice
      const int quad = warp & 3;
      const int slice = (warp - 2) >> 2;
      const int row = quad * 32 + lane;  // key of the tile (TMEM lane)
      const int g0 = slice * kTok;       // first token of the slice (group-local)
      static_assert(kSlice % HI == 0 && kSlice % 32 == 0, "slice holds whole tokens");
      const float* wsl = sW + slice * kSlice;
      float* const srow = p.scores + (int64_t)(t0 + g0) * p.ld + row;  // used only where lim > 0
      int it = 0;
      bool ok = true;
      for (int s = 0; s < nseg && ok; ++s) {
        const int lo = sSegLo[s], hi = sSegHi[s];
        const int jn = sSegN[s];                                    // keys of the segment's longest token
        const int32_t* blk_s = sBlk + s * 2 * kMaxTpc - 2 * lo;     // page of (tile kt, half) at 2 kt + half
        const int32_t* lim_s = sLim + s * kMaxG + g0;
        for (int kt = lo; kt < hi; ++kt, ++it) {
          const int b = it & 1;
          const uint32_t aph = (uint32_t)(it >> 1) & 1u;
          const bool go = !*abort_flag && warp_wait(&acc_full[b], aph, p.err, lane);
          if (!__all_sync(0xffffffffu, go)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * kN + slice * kSlice);
          uint32_t acc[kSlice / 32][32];
#pragma unroll
          for (int q = 0; q < kSlice / 32; ++q) tmem_ld32(taddr + 32 * q, acc[q]);
          // key scale of this thread's key (< 0: the key lies outside the request), read before the
          // accumulator is released (the scale slot's lifetime depends on it)
          const int j = kt * kBlockM + row;
          float ks = -1.f;
          if (j < jn) {
            const int32_t blk = blk_s[2 * kt + (row >> 6)];
            if (blk >= 0)
              ks = p.scale_tma ? sScale[(it % kScaleRing) * kBlockM + row]
                               : __ldg(p.k_scale + (int64_t)blk * 64 + (j & 63));
          }
          tmem_wait_ld();
          // the slice is in registers: the accumulator may take the next MMA
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[b]);
#pragma unroll
          for (int k = 0; k < kTok; ++k) {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int h = 0; h < HI; h += 4) {
              const int c = k * HI + h;
              const float4 wv = lds_f4(wsl + c);
              const float x0 = __uint_as_float(acc[c / 32][c % 32]);
              const float x1 = __uint_as_float(acc[c / 32][c % 32 + 1]);
              const float x2 = __uint_as_float(acc[c / 32][c % 32 + 2]);
              const float x3 = __uint_as_float(acc[c / 32][c % 32 + 3]);
              ffma2(a0, a1, fmaxf(x0, 0.f), fmaxf(x1, 0.f), wv.x, wv.y);
              ffma2(a2, a3, x2 + fabsf(x2), x3 + fabsf(x3), wv.z, wv.w);
            }
            if (ks >= 0.f && j < lim_s[k])
              srow[(int64_t)k * p.ld + (int64_t)kt * kBlockM] = ks * ((a0 + a1) + (a2 + a3));
          }
        }
      }
    }
  }
  // ---------------- teardown: wait for outstanding MMAs, release TMEM -------------------------------
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DI, int HI>
static cudaError_t launch_t(const CUtensorMap& mq, const CUtensorMap& mk, const Params& p, int groups, int splits,
                            cudaStream_t stream) {
  using C = Cfg<DI, HI>;
  auto kern = indexer_kernel<DI, HI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(groups, splits), kThreads, C::kSmem, stream>>>(mq, mk, p);
  return cudaGetLastError();
}

}  // namespace indexer

// Called by the C ABI after argument checks. Encodes the tensor maps and launches.
cudaError_t launch_indexer(const hs_indexer_args* a, int num_sms, cudaStream_t stream, const char** why) {
  using namespace indexer;
  CUtensorMap mq, mk;
  const int DI = a->Di, HI = a->Hi;
  const CUtensorMapSwizzle sw = DI == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if (!encode_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->q, DI, (uint64_t)a->T * HI, DI, DI, kN, sw)) {
    *why = "cuTensorMapEncodeTiled failed for q";
    return cudaErrorInvalidValue;
  }
  if (!encode_2d(&mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->k_cache, DI, (uint64_t)a->nblk * 64, DI, DI, 64, sw)) {
    *why = "cuTensorMapEncodeTiled failed for k_cache";
    return cudaErrorInvalidValue;
  }
  Params p;
  p.T = a->T;
  p.B = a->B;
  p.Hi = HI;
  p.Di = DI;
  p.q_scale = a->q_scale;
  p.weights = a->weights;
  p.k_scale = a->k_scale;
  p.nblk = a->nblk;
  p.block_table = a->block_table;
  p.bt_stride = a->bt_stride;
  p.token_req = a->token_req;
  p.token_kvlen = a->token_kvlen;
  p.scores = a->scores;
  p.ld = a->ld;
  p.err = a->err_flag;
  const int G = kN / HI;
  const int groups = (a->T + G - 1) / G;
  const int64_t keys_max = a->ld < (int64_t)a->bt_stride * 64 ? a->ld : (int64_t)a->bt_stride * 64;
  const int tiles_max = (int)((keys_max + kBlockM - 1) / kBlockM);
  // about three CTAs' worth of tiles per SM over the whole grid, 8..64 tiles each
  int64_t tpc = ((int64_t)groups * tiles_max + 3LL * num_sms - 1) / (3LL * num_sms);
  if (tpc < 8) tpc = 8;
  if (tpc > 64) tpc = 64;
  p.tiles_per_cta = (int)tpc;
  p.scale_tma = ((uintptr_t)a->k_scale & 15) == 0 ? 1 : 0;
  int splits = (int)((tiles_max + tpc - 1) / tpc);
  if (splits < 1) splits = 1;
  if (groups == 0) return cudaSuccess;
#define HS_IDX_CASE(D, H) \
  if (DI == D && HI == H) return launch_t<D, H>(mq, mk, p, groups, splits, stream);
  HS_IDX_CASE(128, 64)
  HS_IDX_CASE(128, 32)
  HS_IDX_CASE(128, 16)
  HS_IDX_CASE(128, 8)
  HS_IDX_CASE(64, 64)
  HS_IDX_CASE(64, 32)
  HS_IDX_CASE(64, 16)
  HS_IDX_CASE(64, 8)
#undef HS_IDX_CASE
  *why = "unsupported (Hi, Di)";
  return cudaErrorInvalidValue;
}

}  // namespace hs
