// indexer.cu — lightning-indexer scores as an FP8 tcgen05 GEMM with a fused epilogue.
//
// [P1] "vLLM v0.32.0 GLM-5.3 サービング ...", section 「DP8とTP8が不十分な理由」: the indexer
// scores every prior token to pick the tokens sparse MLA attends; section 「数字がうまくいく理由」:
// keys are 128 FP8 values with a 4-byte scale. Score (DSA lightning-indexer form):
//   s[t, j] = sum_h w[t,h] * max(0, q_scale[t,h] * k_scale[j] * <q[t,h,:], k[j,:]>),  j < n_t.
// Since both scales are positive, s = k_scale[j] * sum_h (w*q_scale)[t,h] * max(0, <q, k>):
// the GEMM runs on raw e4m3 codes and the scales are applied in the epilogue.
//
// Work split: query tokens are taken in groups of 256/Hi consecutive tokens (so the MMA's N is
// tokens x heads = 256); a group's work is the 128-key tiles of each request in it. The kernel is
// persistent: one CTA per SM takes an equal share of all (group, tile) units (every CTA derives
// the per-group tile counts from the token lengths itself), so requests of very different
// lengths still keep every SM busy to the end. Keys sit on the MMA's M (TMEM lanes), so each
// epilogue thread owns one key and does the ReLU, the weighted head sum and the causal mask in
// registers, then writes one coalesced score.
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
constexpr int kEpiWarps = 16;   // four per TMEM lane quarter: two per accumulator, each 128 columns
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxG = 32;      // tokens per group when Hi = 8
// Key scales of tile i sit in slot i % kScaleRing. The TMA warp refills a slot for tile i + 8 only
// after MMA of tile i + 2 released stage (i + 8) % kStages, and that MMA waited for every epilogue
// warp to have read tile i (scales included) from the accumulator it reuses: 8 slots never race.
constexpr int kScaleRing = kStages + 2;

struct Params {
  int32_t T, B, Hi, Di;
  int32_t t_base;          // first query token of this launch (calls with many groups are split)
  int32_t ngroups;         // token groups of this launch (<= kMaxGroups)
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
  int32_t scale_tma;  // k_scale is 16-byte aligned: the TMA warp copies each page's 64 scales to smem
  int32_t keep_scores;  // keys and their scales are read evict-first and the scores stored evict-last in L2
};

// Work map: every CTA stages the launch's token lengths in chunks, derives each group's number
// of key tiles (sum over its requests of ceil(longest visible length / 128)) and their exclusive
// prefix sum. CTA c then takes the units [c U / C, (c + 1) U / C) of the flattened
// (group, request, tile) list, which it walks in pieces of at most kMaxPieceTiles tiles.
constexpr int kMaxGroups = 2048;
constexpr int kMaxPieceTiles = 512;
constexpr int kMapChunk = 512;     // tokens staged per step of the work map (a multiple of every G)

// Shared-memory load issued where it is written: the folded head weights are the same for every
// tile, and letting the compiler hoist them out of the tile loop makes it spill them to local
// memory and reload them from there on every tile.
// The address is a shared-window address plus a compile-time byte offset, which the instruction
// takes as its immediate (no per-load address arithmetic).
template <int kOffset>
__device__ __forceinline__ float4 lds_f4(uint32_t saddr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4 + %5];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(saddr), "n"(kOffset));
  return v;
}

// Calls f(std::integral_constant<int, i>) for i = 0 .. N-1 (compile-time indices).
template <int I>
struct IntC {
  static constexpr int value = I;
};
template <int N, int I = 0, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  if constexpr (I < N) {
    f(IntC<I>{});
    static_for<N, I + 1>(f);
  }
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
  static constexpr int kOffK = kQBytes;                       // (the work map's staging aliases it)
  static constexpr int kOffW = kOffK + kStages * kTileBytes;
  static constexpr int kOffTok = kOffW + kN * 4;              // int32 x 2 x kMaxG
  static constexpr int kOffSeg = kOffTok + 2 * kMaxG * 4;     // int32 x 6 x kMaxG
  static constexpr int kOffBlk = kOffSeg + 6 * kMaxG * 4;     // int32 [2 * kMaxPieceTiles]
  static constexpr int kOffLim = kOffBlk + 2 * kMaxPieceTiles * 4;  // int32 [kMaxG][kMaxG]
  static constexpr int kOffScale = kOffLim + kMaxG * kMaxG * 4;     // float [kScaleRing][kBlockM]
  static constexpr int kOffGroup = kOffScale + kScaleRing * kBlockM * 4;  // int32 [kMaxGroups + 1]
  static constexpr int kOffBar = kOffGroup + (kMaxGroups + 4) * 4;
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffMisc + 256 + 1024;         // + alignment slack
  static_assert(2 * kMapChunk * 4 <= kStages * kTileBytes, "work-map staging fits the K stages");
};

// Block-wide exclusive prefix sum of one value per thread; also returns the total.
__device__ __forceinline__ int32_t block_scan_excl(int32_t v, int32_t* part, int32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) part[warp] = incl;
  __syncthreads();
  int32_t before = 0, all = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    const int32_t x = part[w];
    before += w < warp ? x : 0;
    all += x;
  }
  __syncthreads();
  total = all;
  return before + incl - v;
}

// The indexer's pipeline waits sleep in the barrier (a suspend-time hint) instead of spinning: the
// epilogue warps wait for their accumulator half of the time, and spinning warps take issue slots
// from the warps that compute on the same sub-partition. The hint bounds each sleep; the phase's
// completion ends it. Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000u)  // hint in ns
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, int32_t* err) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if ((it & 7) == 7 && globaltimer() - t0 > kWaitLimitNs) {
      flag_error(err, HS_FLAG_TIMEOUT);
      return false;
    }
  }
}

template <int DI, int HI>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const Params p) {
  using C = Cfg<DI, HI>;
  constexpr int G = C::G;
  extern __shared__ uint8_t smem_raw[];
  // aligned to 1024 bytes by pointer arithmetic on the shared array itself, so that the compiler
  // still knows every pointer derived from it is a shared-memory one (shared loads and stores
  // with 32-bit addresses, not generic ones)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sK = smem + C::kOffK;
  float* sW = (float*)(smem + C::kOffW);                 // (w * q_scale) [G][HI] of the current group
  int32_t* sTokN = (int32_t*)(smem + C::kOffTok);        // visible keys per token (0 = skip)
  int32_t* sTokSeg = sTokN + kMaxG;                      // segment of each token (-1 = none)
  int32_t* sSegReq = (int32_t*)(smem + C::kOffSeg);      // request of each segment
  int32_t* sSegN = sSegReq + kMaxG;                      // max visible keys in the segment
  int32_t* sSegBase = sSegN + kMaxG;                     // first unit of the segment within its group
  int32_t* sSegLo = sSegBase + kMaxG;                    // first tile of the current piece
  int32_t* sSegHi = sSegLo + kMaxG;                      // one past the last tile
  int32_t* sSegPg = sSegHi + kMaxG;                      // offset of the segment's pages in sBlk
  int32_t* sBlk = (int32_t*)(smem + C::kOffBlk);         // physical page of each of the piece's pages
  int32_t* sLim = (int32_t*)(smem + C::kOffLim);         // [segment][token]: visible keys, 0 = other request
  float* sScale = (float*)(smem + C::kOffScale);         // key scales of the tiles in flight
  int32_t* sGroupOff = (int32_t*)(smem + C::kOffGroup);  // exclusive prefix of the groups' tiles (+ total)
  uint64_t* bars = (uint64_t*)(smem + C::kOffBar);
  uint64_t* full = bars;                                 // [kStages]
  uint64_t* empty = bars + kStages;                      // [kStages]
  uint64_t* acc_full = bars + 2 * kStages;               // [2]
  uint64_t* acc_empty = acc_full + 2;                    // [2]
  uint64_t* q_full = acc_empty + 2;
  uint64_t* mma_done = q_full + 1;
  int32_t* misc = (int32_t*)(smem + C::kOffMisc);
  // misc: [0] nseg, [1] abort, [2] tmem base, [3] piece group, [4] piece first unit (group-local),
  //       [5] piece end unit, [6] group changed, [7..] scan partials
  volatile int32_t* abort_flag = misc + 1;
  int32_t* scan_part = misc + 8;                         // [kThreads / 32]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t nmax = p.ld < (int64_t)p.bt_stride * 64 ? p.ld : (int64_t)p.bt_stride * 64;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps / 2);  // the warps of that accumulator's parity
    }
    mbar_init(q_full, 1);
    mbar_init(mma_done, 1);
    mbar_fence_init();
    misc[1] = 0;
  }
  if (warp == 1) tmem_alloc((uint32_t*)&misc[2], 512);

  // ---------------- work map: tiles per group and their prefix sums ----------------------------
  {
    int32_t* cReq = (int32_t*)sK;         // staged tokens of one chunk
    int32_t* cLen = cReq + kMapChunk;
    const int Tl = p.T - p.t_base < p.ngroups * G ? p.T - p.t_base : p.ngroups * G;  // tokens of this launch
    for (int c0 = 0; c0 < p.ngroups * G; c0 += kMapChunk) {
      __syncthreads();
      for (int i = tid; i < kMapChunk; i += kThreads) {
        const int t = c0 + i;
        int32_t r = -1, n = 0;
        if (t < Tl) {
          r = p.token_req[p.t_base + t];
          n = p.token_kvlen[p.t_base + t];
          if (r < 0 || r >= p.B || n < 0 || (int64_t)n > nmax) n = 0;  // flagged by the piece setup
        }
        cReq[i] = r;
        cLen[i] = n;
      }
      __syncthreads();
      // one warp per group, one lane per token (G <= 32): a token adds the tiles of its request's
      // longest token if no earlier token of the group belongs to the same request
      static_assert(G <= 32, "a group fits in a warp");
      for (int gl = warp; gl < kMapChunk / G; gl += kThreads / 32) {
        const int g = c0 / G + gl;
        if (g >= p.ngroups) break;  // warp-uniform
        const int32_t r = lane < G ? cReq[gl * G + lane] : -1;
        const int32_t n = lane < G ? cLen[gl * G + lane] : 0;
        bool first = n > 0;
        int32_t m = n;
        for (int jj = 0; jj < G; ++jj) {
          const int32_t rj = __shfl_sync(0xffffffffu, r, jj), nj = __shfl_sync(0xffffffffu, n, jj);
          if (jj != lane && nj > 0 && rj == r) {
            if (jj < lane) first = false;
            m = nj > m ? nj : m;
          }
        }
        const int32_t tiles = __reduce_add_sync(0xffffffffu, (first ? (m + kBlockM - 1) / kBlockM : 0));
        if (lane == 0) sGroupOff[g] = tiles;
      }
    }
    __syncthreads();
    // exclusive prefix sum over the groups (each thread sums a run of consecutive groups)
    constexpr int kPer = (kMaxGroups + kThreads - 1) / kThreads;
    int32_t loc[kPer], sum = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int g = tid * kPer + u;
      loc[u] = g < p.ngroups ? sGroupOff[g] : 0;
      sum += loc[u];
    }
    int32_t total;
    int32_t run = block_scan_excl(sum, scan_part, total);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int g = tid * kPer + u;
      if (g < p.ngroups) sGroupOff[g] = run;
      run += loc[u];
    }
    if (tid == 0) sGroupOff[p.ngroups] = total;
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = (uint32_t)misc[2];
  const int64_t U = sGroupOff[p.ngroups];
  const int32_t u_lo = (int32_t)(U * blockIdx.x / gridDim.x), u_hi = (int32_t)(U * (blockIdx.x + 1) / gridDim.x);
  // first group of this CTA: the last group whose prefix is <= u_lo among groups with tiles
  int32_t cur_g = 0;
  {
    int lo = 0, hi = p.ngroups;  // find the largest g with sGroupOff[g] <= u_lo (g < ngroups)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sGroupOff[mid] <= u_lo) lo = mid;
      else hi = mid;
    }
    cur_g = lo;
  }
  int32_t cur_u = u_lo;
  int prev_g = -1;
  // per-role iteration counters, continued across pieces
  int it_prod = 0, it_mma = 0, it_epi = 0, q_loads = 0;

  while (cur_u < u_hi) {
    // skip groups without tiles
    while (cur_g < p.ngroups - 1 && sGroupOff[cur_g + 1] <= cur_u) ++cur_g;
    const int32_t g_off = sGroupOff[cur_g], g_tiles = sGroupOff[cur_g + 1] - g_off;
    const int32_t a = cur_u - g_off;
    int32_t b = (u_hi < g_off + g_tiles ? u_hi : g_off + g_tiles) - g_off;
    if (b - a > kMaxPieceTiles) b = a + kMaxPieceTiles;
    const bool new_group = cur_g != prev_g;
    const int t0 = cur_g * G;  // group's first token (launch-local)

    // ---------------- piece setup ---------------------------------------------------------------
    __syncthreads();  // the previous piece is fully consumed (epilogue waited for its last MMA)
    if (new_group) {
      if (tid < G) {
        const int t = t0 + tid;
        int32_t n = 0, r = -1;
        if (t < p.ngroups * G && p.t_base + t < p.T) {
          r = p.token_req[p.t_base + t];
          n = p.token_kvlen[p.t_base + t];
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
        // folded weight w * q_scale; every head takes its ReLU as x + |x| = 2 max(x, 0) (packed
        // fp32x2 adds, two heads per instruction), so the weight carries the factor 1/2 (exact)
        const int g = tid / HI, h = tid % HI, t = p.t_base + t0 + g;
        const float half = 0.5f;
        sW[tid] = (t < p.T) ? half * (p.weights[(int64_t)t * HI + h] * p.q_scale[(int64_t)t * HI + h]) : 0.f;
      }
      __syncthreads();
      if (tid == 0) {
        int nseg = 0;
        for (int g = 0; g < G; ++g) {
          const int r = sTokSeg[g];
          if (r < 0) continue;
          int s2 = 0;
          while (s2 < nseg && sSegReq[s2] != r) ++s2;
          if (s2 == nseg) {
            sSegReq[s2] = r;
            sSegN[s2] = 0;
            ++nseg;
          }
          sTokSeg[g] = s2;
          if (sTokN[g] > sSegN[s2]) sSegN[s2] = sTokN[g];
        }
        int base = 0;
        for (int s2 = 0; s2 < nseg; ++s2) {
          sSegBase[s2] = base;
          base += (sSegN[s2] + kBlockM - 1) / kBlockM;
        }
        misc[0] = nseg;
      }
      __syncthreads();
      // keys token g may see while the CTA scores segment s (0 when g belongs to another request)
      for (int i = tid; i < misc[0] * G; i += kThreads) {
        const int sg = i / G, g = i % G;
        sLim[sg * kMaxG + g] = sTokSeg[g] == sg ? sTokN[g] : 0;
      }
    }
    if (tid == 0) {
      // the piece's tile range within each segment, and where the segment's pages go in sBlk
      int pg = 0;
      for (int s2 = 0; s2 < misc[0]; ++s2) {
        const int tiles = (sSegN[s2] + kBlockM - 1) / kBlockM;
        int lo = a - sSegBase[s2], hi = b - sSegBase[s2];
        lo = lo < 0 ? 0 : (lo > tiles ? tiles : lo);
        hi = hi < 0 ? 0 : (hi > tiles ? tiles : hi);
        sSegLo[s2] = lo;
        sSegHi[s2] = hi;
        sSegPg[s2] = pg;
        pg += 2 * (hi - lo);
      }
    }
    __syncthreads();
    // stage the piece's block-table entries (2 pages per tile) so no warp waits on them later
    const int nseg = misc[0];
    for (int s2 = 0; s2 < nseg; ++s2) {
      const int r = sSegReq[s2];
      const int npg = 2 * (sSegHi[s2] - sSegLo[s2]);
      for (int i = tid; i < npg; i += kThreads) {
        const int page = 2 * sSegLo[s2] + i;
        int32_t blk = -1;
        if (page * 64 < sSegN[s2]) {
          blk = p.block_table[(int64_t)r * p.bt_stride + page];
          if (blk < 0 || (int64_t)blk >= p.nblk) {
            flag_error(p.err, HS_FLAG_BAD_BLOCK);
            blk = -1;
          }
        }
        sBlk[sSegPg[s2] + i] = blk;
      }
    }
    __syncthreads();

    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer ----------------
      if (lane == 0) {
        const uint64_t pol_first = l2_policy_evict_first();
        if (new_group) {
          if (prev_g < 0) {
            prefetch_tensormap(&map_q);
            prefetch_tensormap(&map_k);
          }
          mbar_arrive_expect_tx(q_full, C::kQBytes);
          tma_load_2d(sQ, &map_q, q_full, 0, (p.t_base + t0) * HI);
        }
        for (int s2 = 0; s2 < nseg && !*abort_flag; ++s2) {
          for (int kt = sSegLo[s2]; kt < sSegHi[s2]; ++kt, ++it_prod) {
            const int st = it_prod % kStages;
            const uint32_t ph = (uint32_t)(it_prod / kStages) & 1u;
            if (!mbar_wait_sleep(&empty[st], ph ^ 1u, p.err)) {
              *abort_flag = 1;
              break;
            }
            int32_t blk[2];
            uint32_t bytes = 0;
            for (int pg = 0; pg < 2; ++pg) {
              blk[pg] = sBlk[sSegPg[s2] + 2 * (kt - sSegLo[s2]) + pg];
              if (blk[pg] >= 0) bytes += 64 * DI + (p.scale_tma ? 64 * 4 : 0);
            }
            mbar_arrive_expect_tx(&full[st], bytes);
            for (int pg = 0; pg < 2; ++pg)
              if (blk[pg] >= 0) {
                void* kdst = sK + st * C::kTileBytes + pg * 64 * DI;
                float* sdst = sScale + (it_prod % kScaleRing) * kBlockM + pg * 64;
                const float* ssrc = p.k_scale + (int64_t)blk[pg] * 64;
                if (p.keep_scores) {
                  tma_load_2d_hint(kdst, &map_k, &full[st], 0, blk[pg] * 64, pol_first);
                  if (p.scale_tma) bulk_g2s_hint(sdst, ssrc, 64 * 4, &full[st], pol_first);
                } else {
                  tma_load_2d(kdst, &map_k, &full[st], 0, blk[pg] * 64);
                  if (p.scale_tma) bulk_g2s(sdst, ssrc, 64 * 4, &full[st]);
                }
              }
          }
        }
        // every issued copy must land before the CTA's shared memory is reused or released
        if (new_group) mbar_wait(q_full, (uint32_t)q_loads & 1u, p.err);
        for (int i = it_prod > kStages ? it_prod - kStages : 0; i < it_prod; ++i)
          mbar_wait(&full[i % kStages], (uint32_t)(i / kStages) & 1u, p.err);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer ------------------
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_e4m3(kBlockM, kN);
        const uint32_t q_addr = smem_u32(sQ);
        const uint32_t k_addr = smem_u32(sK);
        bool ok = !new_group || mbar_wait(q_full, (uint32_t)q_loads & 1u, p.err);
        for (int s2 = 0; s2 < nseg && ok && !*abort_flag; ++s2) {
          for (int kt = sSegLo[s2]; kt < sSegHi[s2]; ++kt, ++it_mma) {
            const int st = it_mma % kStages;
            const uint32_t ph = (uint32_t)(it_mma / kStages) & 1u;
            const int bb = it_mma & 1;
            const uint32_t aph = (uint32_t)(it_mma >> 1) & 1u;
            if (!mbar_wait_sleep(&full[st], ph, p.err) || !mbar_wait_sleep(&acc_empty[bb], aph ^ 1u, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
              const uint64_t da = smem_desc(k_addr + st * C::kTileBytes + ks * 32, 16, C::kSBO, C::kSwizzle);
              const uint64_t dq = smem_desc(q_addr + ks * 32, 16, C::kSBO, C::kSwizzle);
              mma_e4m3_ss(tmem + (uint32_t)(bb * kN), da, dq, idesc, ks > 0 ? 1u : 0u);
            }
            mma_commit(&empty[st]);
            mma_commit(&acc_full[bb]);
          }
        }
        if (!ok) *abort_flag = 1;
      }
    } else {
      // ------------------------------------------------------------ epilogue --------------------
      // Warps take alternate tiles, so that while one half waits for its TMEM loads the other half
      // computes: slot = (warp - 2) / 4 in 0..3; the warps of parity slot / 2 drain accumulator
      // (tile % 2) == parity, each its lane quarter and the columns [col0, col0 + 128) in two
      // chunks of 64 (chunk 1 is loaded after chunk 0 is reduced; then the accumulator is released).
      constexpr int kChunk = 64;
      constexpr int kTok = kChunk / HI;  // tokens in a chunk
      static_assert(kChunk % HI == 0, "a chunk holds whole tokens");
      const int quad = warp & 3;
      const int slot = (warp - 2) >> 2;
      const int parity = slot >> 1;
      const int col0 = (slot & 1) * (kN / 2);
      const int row = quad * 32 + lane;  // key of the tile (TMEM lane)
      const int g0 = col0 / HI;          // first token of this warp's columns (group-local)
      const uint32_t wsl = smem_u32(sW + col0);  // this warp's folded weights
      float* const srow = p.scores + (int64_t)(p.t_base + t0 + g0) * p.ld + row;  // used only where lim > 0
      bool ok = true;
      const bool keep = p.keep_scores != 0;
      const uint64_t pol_last = l2_policy_evict_last();
      for (int s2 = 0; s2 < nseg && ok; ++s2) {
        const int lo = sSegLo[s2], hi = sSegHi[s2];
        const int jn = sSegN[s2];                                     // keys of the segment's longest token
        const int32_t* blk_s = sBlk + sSegPg[s2] - 2 * lo;           // page of (tile kt, half) at 2 kt + half
        const int32_t* lim_s = sLim + s2 * kMaxG + g0;
        // only the tiles of this warp's parity: tile kt has the running tile number ie
        const int ie0 = it_epi - lo;
        it_epi += hi - lo;
        for (int kt = lo + ((parity - (ie0 + lo)) & 1); kt < hi; kt += 2) {
          const uint32_t ie = (uint32_t)(ie0 + kt);
          const int bb = parity;
          const uint32_t aph = (ie >> 1) & 1u;
          int gi = 1;
          if (lane == 0) gi = !*abort_flag && mbar_wait_sleep(&acc_full[bb], aph, p.err) ? 1 : 0;
          const bool go = __shfl_sync(0xffffffffu, gi, 0) != 0;
          if (!__all_sync(0xffffffffu, go)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(bb * kN + col0);
          uint32_t acc[kChunk / 32][32];
#pragma unroll
          for (int q = 0; q < kChunk / 32; ++q) tmem_ld32(taddr + 32 * q, acc[q]);
          // key scale of this thread's key (< 0: the key lies outside the request), read before the
          // accumulator is released (the scale slot's lifetime depends on it)
          const int j = kt * kBlockM + row;
          float ks = -1.f;
          if (j < jn) {
            const int32_t blk = blk_s[2 * kt + (row >> 6)];
            if (blk >= 0)
              ks = p.scale_tma ? sScale[(ie % kScaleRing) * kBlockM + row]
                               : __ldg(p.k_scale + (int64_t)blk * 64 + (j & 63));
          }
          auto token_score = [&](auto cc, auto kc) -> float {  // weighted ReLU sum of token kc of chunk cc
            constexpr int k = decltype(kc)::value;
            constexpr int wbase = decltype(cc)::value * kChunk;
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            static_for<HI / 4>([&](auto hc) {
              constexpr int c = k * HI + 4 * decltype(hc)::value;
              const float4 wv = lds_f4<4 * (wbase + c)>(wsl);
              const float x0 = __uint_as_float(acc[c / 32][c % 32]);
              const float x1 = __uint_as_float(acc[c / 32][c % 32 + 1]);
              const float x2 = __uint_as_float(acc[c / 32][c % 32 + 2]);
              const float x3 = __uint_as_float(acc[c / 32][c % 32 + 3]);
              const float2 r01 = __fadd2_rn(make_float2(x0, x1), make_float2(fabsf(x0), fabsf(x1)));
              const float2 r23 = __fadd2_rn(make_float2(x2, x3), make_float2(fabsf(x2), fabsf(x3)));
              ffma2(a0, a1, r01.x, r01.y, wv.x, wv.y);
              ffma2(a2, a3, r23.x, r23.y, wv.z, wv.w);
            });
            return (a0 + a1) + (a2 + a3);
          };
          float sc[2][kTok];
          tmem_wait_ld();
          static_for<kTok>([&](auto kc) { sc[0][decltype(kc)::value] = token_score(IntC<0>{}, kc); });
#pragma unroll
          for (int q = 0; q < kChunk / 32; ++q) tmem_ld32(taddr + kChunk + 32 * q, acc[q]);
          tmem_wait_ld();
          // both chunks are in registers: the accumulator may take the next MMA
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[bb]);
          static_for<kTok>([&](auto kc) { sc[1][decltype(kc)::value] = token_score(IntC<1>{}, kc); });
          if (ks >= 0.f) {
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
              for (int k = 0; k < kTok; ++k) {
                const int g = c2 * kTok + k;
                if (j < lim_s[g]) {
                  float* dst = srow + (int64_t)g * p.ld + (int64_t)kt * kBlockM;
                  if (keep) st_global_hint(dst, ks * sc[c2][k], pol_last);
                  else *dst = ks * sc[c2][k];
                }
              }
          }
        }
      }
      if (!ok) *abort_flag = 1;
    }
    if (new_group) ++q_loads;
    prev_g = cur_g;
    cur_u = g_off + b;
    __syncthreads();
    if (*abort_flag) break;
  }
  // ---------------- teardown: every issued MMA has finished, release TMEM ---------------------------
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      mma_commit(mma_done);
      mbar_wait(mma_done, 0, p.err);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DI, int HI>
static cudaError_t launch_t(const CUtensorMap& mq, const CUtensorMap& mk, Params p, int ctas, cudaStream_t stream) {
  using C = Cfg<DI, HI>;
  auto kern = indexer_kernel<DI, HI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const int G = C::G;
  const int groups = (p.T + G - 1) / G;
  for (int g0 = 0; g0 < groups; g0 += kMaxGroups) {  // each launch balances at most kMaxGroups groups
    p.t_base = g0 * G;
    p.ngroups = groups - g0 < kMaxGroups ? groups - g0 : kMaxGroups;
    kern<<<ctas, kThreads, C::kSmem, stream>>>(mq, mk, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace indexer

// Called by the C ABI after argument checks. Encodes the tensor maps and launches.
cudaError_t launch_indexer(const hs_indexer_args* a, int num_sms, bool keep_scores, cudaStream_t stream,
                           const char** why) {
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
  p.t_base = 0;
  p.ngroups = 0;
  p.scale_tma = ((uintptr_t)a->k_scale & 15) == 0 ? 1 : 0;
  p.keep_scores = keep_scores ? 1 : 0;
  if (a->T == 0) return cudaSuccess;
  const int ctas = num_sms;  // persistent: one CTA per SM, each an equal share of the tiles
#define HS_IDX_CASE(D, H) \
  if (DI == D && HI == H) return launch_t<D, H>(mq, mk, p, ctas, stream);
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
