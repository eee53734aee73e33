// mla.cu — sparse MLA forward in MQA form on tcgen05.
//
// [P1] "vLLM v0.32.0 GLM-5.3 サービング ...", sections 「再現方法と必要なフラグ」 and
// 「数字がうまくいく理由」: each query gathers its selected 656-byte FP8 latent rows once and every
// row serves all 64 heads; QK runs over 576 dims (512 latent + 64 RoPE), PV over the 512 latent
// dims. Per query token t, head h, over the valid entries i of idx[t, :]:
//   logit_i = scale * <q[t,h,:], [latent_i, rope_i]>,  out = softmax(logit) . latent,  lse = ln sum exp.
//
// One CTA per query token (448 threads), rows in 32-row tiles through a ring of four stages:
//   warps 0-7   gather the rows of each tile (warp w owns rows 4w..4w+3; lane l works on row
//               4w + l / 8 and loads 16-byte pieces l % 8 of its 128-byte spans), dequantise
//               latent = e4m3 * group scale to fp16 (exact e4m3 -> fp16 conversion, then
//               code * scale rounded once, with the scale split into two fp16 parts; see
//               dequant8_f16) and write it, with the bf16 RoPE part as stored, into a
//               128-byte-swizzled [dim block][row] tile, once PV of the tile that used the stage
//               four tiles before has completed. The whole tile is published with one proxy fence
//               and one barrier arrival per warp (per-block-pair publication cost more in fences
//               and waits than its overlap gained). The rows of tile i + 1 are loaded into the
//               registers tile i leaves, part by part as tile i is written; rows are prefetched into
//               L2 three tiles ahead;
//   warp 8      allocates TMEM, loads Q by TMA and issues S = Q . K^T (M = 64 heads, N = 32 rows,
//               K = 512 fp16 latent + 64 bf16 RoPE; A = Q, B = tile) as soon as a tile is written
//               and an S buffer is free, so QK of later tiles runs while the softmax works on
//               earlier ones;
//   warp 9      issues O^T += V^T . P^T (M = 128 dims x4, N = 64 heads, K = 32 rows) for each tile
//               once its P is written; its completion releases the stage. All PV
//               MMAs come from this one thread, so they accumulate in order without waiting on one
//               another; the same tile is the K-major B of QK and, read MN-major, the A of PV, so it
//               is dequantised once;
//   warps 10-13 first convert Q's latent dims to fp16 in shared memory (a head's row whose largest
//               value fp16 cannot hold at full precision is scaled by a power of two), then run the
//               online softmax: two threads share each head's row of S (one shuffle for the max); P
//               goes as fp16 into the stage's RoPE block, which QK no longer needs (K-major, 64-byte
//               swizzle). O^T lives in TMEM and is rescaled only when a head's running max grows by
//               more than 2^8 (lazy rescaling), after the previous tile's PV has completed; the final
//               pass divides by the row sum and writes bf16 straight from TMEM (neighbouring lanes
//               swap values so that each stores two adjacent dims of one head).
// TMEM: columns 0-127 hold four S buffers (64-row layout, 32 columns each), 128-383 hold O^T.
//
// Work split (launch_mla): one CTA per query when the queries fill their waves; otherwise, given a
// workspace, one persistent CTA per SM takes an equal share of all (query, 32-row tile) units, a
// query split between CTAs leaves a normalised partial and its LSE per CTA, and mla_merge_kernel
// combines them (split-KV decode: DCP's log-sum-exp merge on one GPU).
#include "common.cuh"

namespace hs {
namespace mla {

constexpr int kRows = 32;                  // rows per tile
constexpr int kStages = 4;
constexpr int kProdWarps = 8;
constexpr int kMmaWarp = kProdWarps;       // QK issuer; also allocates TMEM
constexpr int kPvWarp = kProdWarps + 1;    // PV issuer
constexpr int kSmThreads = 128;
constexpr int kThreads = 32 * (kProdWarps + 2 + 4);  // + QK warp, PV warp, 4 softmax warps
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;
constexpr int kQBlk = 8192;                // one [64 heads][128 B] swizzled block of Q
constexpr int kBlk = kRows * 128;          // one [32 rows][128 B] swizzled block of a stage
constexpr int kQBytes = 9 * kQBlk;         // 64 heads x 576 bf16
constexpr int kStageBytes = 9 * kBlk;      // 32 rows x (512 latent + 64 rope) fp16/bf16
constexpr int kBlocks = 9;                 // 8 latent dim blocks + the RoPE block (later P)
constexpr int kOffQ = 0;
constexpr int kOffStage = kQBytes;
constexpr int kOffValid = kOffStage + kStages * kStageBytes;  // uint8 [kStages][32]
constexpr int kOffAlpha = kOffValid + kStages * kRows;        // float [64]
constexpr int kOffInvL = kOffAlpha + 256;                     // float [64]
constexpr int kOffQe = kOffInvL + 256;                        // int [64]: per-head exponent of the current query
constexpr int kNumBars = 6 * kStages + 5;
constexpr int kOffBar = kOffQe + 256;
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort
constexpr int kSmem = kOffMisc + 16 + 1024;
constexpr float kRescaleThreshold = 8.0f;         // log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kScaleMax = 65504.f / 448.f;      // |code * scale| stays finite in fp16
constexpr float kScaleMin = 6.103515625e-05f;     // 2^-14: scales stay fp16 normals
static_assert(kSmem <= 232448, "shared memory");

struct Params {
  int32_t T, H, k;
  const __nv_bfloat16* q;  // [T][H][576], also loaded by TMA; read directly to rescale a head's row
  const uint8_t* kv;
  int64_t R;
  const int32_t* idx;
  const int32_t* idx_row;  // shared index sets: query t reads idx row idx_row[t] (NULL: row t)
  int32_t idx_rows;
  const int32_t* kvlen;    // entries j >= kvlen[t] are skipped (NULL: none)
  const int32_t* bt;
  int32_t bt_stride;
  const int32_t* token_req;
  float scale_log2;  // softmax_scale * log2(e)
  __nv_bfloat16* out;
  float* lse;
  int32_t* err;
  // Work split. Units are (query, 32-row tile) pairs, U = T * tiles per query in total. A CTA
  // takes the units [c U / C, (c + 1) U / C) (persistent launch, C CTAs) or exactly the units of
  // query c (one CTA per query). A query whose units span several CTAs leaves, from each, its
  // softmax-normalised partial output (bf16) and log-sum-exp in a workspace slot (2c for the
  // CTA's first query, 2c + 1 for its last); mla_merge_kernel combines them.
  int32_t persistent;
  int64_t U;
  __nv_bfloat16* part_out;  // [2C][H][512]
  float* part_lse;          // [2C][H]
};

// First unit of CTA c of a persistent launch over U units with C CTAs.
__host__ __device__ __forceinline__ int64_t unit_begin(int64_t c, int64_t U, int64_t C) { return c * U / C; }
// CTA of a persistent launch holding unit u: the largest c with unit_begin(c) <= u.
__device__ __forceinline__ int64_t unit_cta(int64_t u, int64_t U, int64_t C) { return ((u + 1) * C - 1) / U; }

// 8 e4m3 codes (two 32-bit words) -> 8 fp16 values code * scale, rounded once. The fp32 group
// scale is split into fp16 parts hi + lo (hi = fp16(scale), lo = fp16(scale - hi)); the
// e4m3 -> fp16 conversion is exact, t = code * lo is a correction of relative size 2^-11 whose own
// rounding is ~2^-22 of the result, and fma(code, hi, t) rounds the sum once. Rounding the scale
// to fp16 alone would give every value of a (row, group) the same relative error (up to 2^-11), a
// bias that large logits turn into a coherent shift of that row's softmax weight.
__device__ __forceinline__ uint4 dequant8_f16(uint32_t w0, uint32_t w1, uint32_t hi2, uint32_t lo2) {
  uint4 r;
  asm("{ .reg .b16 a, b, c, d; .reg .b32 x, y, z, u, tx, ty, tz, tu;\n"
      " mov.b32 {a, b}, %4; mov.b32 {c, d}, %5;\n"
      " cvt.rn.f16x2.e4m3x2 x, a; cvt.rn.f16x2.e4m3x2 y, b; cvt.rn.f16x2.e4m3x2 z, c; cvt.rn.f16x2.e4m3x2 u, d;\n"
      " mul.rn.f16x2 tx, x, %7; mul.rn.f16x2 ty, y, %7; mul.rn.f16x2 tz, z, %7; mul.rn.f16x2 tu, u, %7;\n"
      " fma.rn.f16x2 %0, x, %6, tx; fma.rn.f16x2 %1, y, %6, ty; fma.rn.f16x2 %2, z, %6, tz; fma.rn.f16x2 %3, u, %6, tu; }"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "r"(w0), "r"(w1), "r"(hi2), "r"(lo2));
  return r;
}

// The rows of one tile a producer lane holds: four 16-byte latent pieces (bytes 128 j + 16 (l % 8)
// of its row, j = 0..3), its 16-byte RoPE piece and the row's four group scales.
struct TileRegs {
  uint4 lat[4];
  uint4 rope;
  uint4 scl;
};

// Segment walk shared by every role: the CTA's units [u0, u1) as queries q with tiles [ta, tb).
struct Seg {
  int64_t q;
  int ta, tb;
};
__device__ __forceinline__ Seg next_seg(int64_t& u, int64_t u1, int ntq) {
  Seg g;
  g.q = u / ntq;
  g.ta = (int)(u - g.q * ntq);
  g.tb = (int)((u1 - g.q * ntq) < ntq ? (u1 - g.q * ntq) : ntq);
  u = g.q * ntq + g.tb;
  return g;
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap map_q, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sStage = smem + kOffStage;
  uint8_t* sValid = smem + kOffValid;
  float* sAlpha = (float*)(smem + kOffAlpha);
  float* sInvL = (float*)(smem + kOffInvL);
  int32_t* sQe = (int32_t*)(smem + kOffQe);
  uint64_t* bars = (uint64_t*)(smem + kOffBar);
  uint64_t* full = bars + 0;                       // [4] producers wrote the stage's tile -> QK, softmax
  uint64_t* empty = full + kStages;                // [4] PV of the stage's tile complete -> producers, softmax
  uint64_t* s_full = empty + kStages;              // [4] QK done -> softmax
  uint64_t* s_free = s_full + kStages;             // [4] softmax read S -> QK
  uint64_t* p_ready = s_free + kStages;            // [4] softmax wrote P (and rescaled O^T) -> PV
  uint64_t* q_full = p_ready + kStages;
  uint64_t* mma_done = q_full + 1;                 // QK issuer's MMAs drained
  uint64_t* pv_drain = q_full + 2;                 // PV issuer's MMAs drained
  uint64_t* q_ready = q_full + 3;                  // Q converted to fp16 (latent dims) -> QK issuer
  uint64_t* q_free = q_full + 4;                   // QK MMAs of a query finished reading Q -> QK issuer
  uint32_t* misc = (uint32_t*)(smem + kOffMisc);
  volatile uint32_t* abort_flag = misc + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = p.k;
  const int ntq = (k + kRows - 1) / kRows;  // tiles per query
  // this CTA's units; every role walks them as segments (query, tiles [ta, tb)) in the same order,
  // and counts tiles globally (gi) for the stage and barrier phases
  int64_t u0, u1;
  if (p.persistent) {
    u0 = unit_begin(blockIdx.x, p.U, gridDim.x);
    u1 = unit_begin(blockIdx.x + 1, p.U, gridDim.x);
  } else {
    u0 = (int64_t)blockIdx.x * ntq;
    u1 = u0 + ntq;
  }
  const int ntot = (int)(u1 - u0);  // tiles of this CTA

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], kProdWarps);
      mbar_init(&empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
      mbar_init(&p_ready[i], 4);
    }
    mbar_init(q_full, 1);
    mbar_init(mma_done, 1);
    mbar_init(pv_drain, 1);
    mbar_init(q_ready, 4);
    mbar_init(q_free, 1);
    mbar_fence_init();
    misc[1] = 0;
  }
  if (warp == kMmaWarp) tmem_alloc(&misc[0], 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp < kProdWarps) {
    // ================================================================ gather + dequantise ======
    // Warp w owns rows 4w .. 4w+3 of every tile; lane l works on row 4w + rl, rl = l / 8, and
    // loads bytes 128 j + 16 c8 (c8 = l % 8, j = 0..3) of its latent codes: 16 codes of dim block
    // 2j + c8 / 4, i.e. 16-byte chunks 2 (c8 % 4) and 2 (c8 % 4) + 1 of that block's fp16 row
    // (group scale j). Its RoPE piece is bytes 16 c8 of the row's RoPE part (chunk c8 of the RoPE
    // block); each lane also loads its row's four scales (the eight lanes of a row read the same
    // 16 bytes, one transaction). Lanes 0-3 carry the index pipeline of rows 4w .. 4w+3:
    //   tile i+5: index entries (and visible lengths)   tile i+4: block-table entries
    //   tile i+1 .. i+3: rows prefetched into L2 by the TMA engine (one 656-byte bulk prefetch
    //             per row, three tiles ahead)
    //   tile i+1: row data loaded into registers, each part as soon as tile i's part in those
    //             registers has been written
    //   tile i  : dequantised into stage i % 4 once PV of tile i-4 has completed.
    // Every loaded value is first used one step after its load, so no step waits on a load
    // issued in the same step.
    // Loads are volatile so they are issued here and not next to their first use.
    const int rl = lane >> 3, c8 = lane & 7;
    const int row = warp * 4 + rl;   // this lane's row within a tile
    int64_t la_q = u0 / ntq;
    int la_t = (int)(u0 - la_q * ntq), la_n = 0;
    // lanes 0-3: index entry of row 4 * warp + lane of the CTA's next lookahead tile (tiles are
    // visited in order) and, with a block table, the request of its query
    auto ld_idx = [&](int32_t& req, int32_t& lim) -> int32_t {
      req = 0;
      lim = 0x7FFFFFFF;
      const bool live = la_n < ntot;
      const int64_t q = la_q;
      const int e = la_t * kRows + warp * 4 + lane;
      if (++la_t == ntq) {
        la_t = 0;
        ++la_q;
      }
      ++la_n;
      if (lane >= 4 || !live || e >= k) return -1;
      int64_t r = q;
      if (p.idx_row) {
        r = ldg_nc_s32(p.idx_row + q);
        if (r < 0 || r >= p.idx_rows) {
          flag_error(p.err, HS_FLAG_BAD_INDEX);
          return -1;
        }
      }
      if (p.bt) req = ldg_nc_s32(p.token_req + q);
      const int32_t j = ldg_nc_s32(p.idx + r * k + e);
      if (p.kvlen) lim = ldg_nc_s32(p.kvlen + q);  // applied one step later, in ld_blk
      return j;
    };
    auto ld_blk = [&](int32_t& j, int32_t req, int32_t lim) -> int32_t {  // lanes 0-3: block-table entry of entry j (j if none)
      if (j >= lim) j = -1;  // beyond the query's visible length
      if (lane >= 4 || j < 0 || !p.bt) return j;
      const int32_t page = j >> 6;
      return page < p.bt_stride ? ldg_nc_s32(p.bt + (int64_t)req * p.bt_stride + page) : -1;
    };
    auto phys_row = [&](int32_t j, int32_t b) -> int64_t {  // lanes 0-3: physical row, -1 if none
      if (lane >= 4 || j < 0) return -1;
      const int64_t r = p.bt ? (b >= 0 ? (int64_t)b * 64 + (j & 63) : -1) : (int64_t)j;
      if (r < 0 || r >= p.R) {
        flag_error(p.err, HS_FLAG_BAD_INDEX);
        return -1;
      }
      return r;
    };
    auto prefetch_rows = [&](int64_t r) {
      if (r >= 0) bulk_prefetch_l2(p.kv + r * HS_KV_ROW_BYTES, HS_KV_ROW_BYTES);
    };
    // this lane's row of a tile from the lanes 0-3 row values
    auto row_of = [&](int64_t rows_lane) -> int64_t { return __shfl_sync(0xffffffffu, rows_lane, rl); };
    auto ld_lat = [&](int64_t r, int j) -> uint4 {
      return r >= 0 ? ldg_nc_v4(p.kv + r * HS_KV_ROW_BYTES + 128 * j + 16 * c8) : make_uint4(0, 0, 0, 0);
    };
    auto ld_rope = [&](int64_t r) -> uint4 {
      return r >= 0 ? ldg_nc_v4(p.kv + r * HS_KV_ROW_BYTES + HS_D_LATENT + 16 + 16 * c8) : make_uint4(0, 0, 0, 0);
    };
    auto ld_scl = [&](int64_t r) -> uint4 {
      return r >= 0 ? ldg_nc_v4(p.kv + r * HS_KV_ROW_BYTES + HS_D_LATENT) : make_uint4(0, 0, 0, 0);
    };
    auto ld_tile = [&](TileRegs& t, int64_t rows_lane) {
      const int64_t r = row_of(rows_lane);
#pragma unroll
      for (int j = 0; j < 4; ++j) t.lat[j] = ld_lat(r, j);
      t.rope = ld_rope(r);
      t.scl = ld_scl(r);
    };
    auto wait_empty = [&](int s, int i) -> bool {
      int go = 1;
      if (lane == 0) go = !*abort_flag && mbar_wait(&empty[s], ((uint32_t)(i >> 2) & 1u) ^ 1u, p.err);
      go = __shfl_sync(0xffffffffu, go, 0);
      if (!go && lane == 0) *abort_flag = 1;
      return go != 0;
    };
    // Writes tile i (in t, rows cur_rows on lanes 0-3) into stage i % 4 and loads tile i + 1
    // (rows next_rows) into t part by part as each part is written; false on abort.
    auto publish = [&](int i, TileRegs& t, int64_t cur_rows, int64_t next_rows) -> bool {
      const int s = i & 3;
      const int64_t nr = row_of(next_rows);
      if (!wait_empty(s, i)) return false;  // PV of tile i - 4 complete
      uint8_t* st = sStage + s * kStageBytes;
      if (lane < 4) sValid[s * kRows + warp * 4 + lane] = cur_rows >= 0 ? 1 : 0;
      bool range_ok = true;
      const float scales[4] = {__uint_as_float(t.scl.x), __uint_as_float(t.scl.y), __uint_as_float(t.scl.z),
                               __uint_as_float(t.scl.w)};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float scale = scales[j];
        range_ok &= scale == 0.f || (fabsf(scale) >= kScaleMin && fabsf(scale) <= kScaleMax);
        const __half shi = __float2half_rn(scale);
        const __half2 h2 = __half2half2(shi);
        const __half2 l2 = __float2half2_rn(scale - __half2float(shi));  // scale - hi is exact in fp32
        const uint32_t h2u = *reinterpret_cast<const uint32_t*>(&h2);
        const uint32_t l2u = *reinterpret_cast<const uint32_t*>(&l2);
        const uint4 v = t.lat[j];
        const uint4 lo = dequant8_f16(v.x, v.y, h2u, l2u);
        const uint4 hi = dequant8_f16(v.z, v.w, h2u, l2u);
        uint8_t* blk = st + (2 * j + (c8 >> 2)) * kBlk;
        *reinterpret_cast<uint4*>(blk + sw128_offset(row, 32 * (c8 & 3))) = lo;
        *reinterpret_cast<uint4*>(blk + sw128_offset(row, 32 * (c8 & 3) + 16)) = hi;
        t.lat[j] = ld_lat(nr, j);
      }
      // RoPE block (bf16 as stored); it held P of tile i - 4
      *reinterpret_cast<uint4*>(st + 8 * kBlk + sw128_offset(row, 16 * c8)) = t.rope;
      if (!range_ok) flag_error(p.err, HS_FLAG_RANGE);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[s]);
      t.rope = ld_rope(nr);
      t.scl = ld_scl(nr);
      return true;
    };
    // prologue: index entries of tiles 0-5, block-table entries of tiles 0-4; tile 0 into the
    // registers, tiles 1-3 prefetched into L2
    int32_t jt[6], rq[6], lm[6];
#pragma unroll
    for (int x = 0; x < 6; ++x) jt[x] = ld_idx(rq[x], lm[x]);
    int32_t bt[5];
#pragma unroll
    for (int x = 0; x < 5; ++x) bt[x] = ld_blk(jt[x], rq[x], lm[x]);
    int64_t rowc = phys_row(jt[0], bt[0]);  // lanes 0-3: rows of the tile in the registers
    TileRegs A;
    ld_tile(A, rowc);
    int64_t r1 = phys_row(jt[1], bt[1]);
    int64_t r2 = phys_row(jt[2], bt[2]);
    int64_t r3 = phys_row(jt[3], bt[3]);
    prefetch_rows(r1);
    prefetch_rows(r2);
    prefetch_rows(r3);
    int32_t j4 = jt[4], b4 = bt[4];
    int32_t j5 = jt[5], q5 = rq[5], l5 = lm[5];
    for (int i = 0; i < ntot; ++i) {
      const int64_t n1 = r1;
      if (!publish(i, A, rowc, n1)) break;
      rowc = n1;
      const int64_t r4 = phys_row(j4, b4);
      prefetch_rows(r4);
      r1 = r2;
      r2 = r3;
      r3 = r4;
      b4 = ld_blk(j5, q5, l5);
      j4 = j5;
      j5 = ld_idx(q5, l5);
    }
  } else if (warp == kMmaWarp) {
    // ================================================================ QK issuer =================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(64, kRows, 0, 0);       // latent dims: fp16
      constexpr uint32_t idesc_qk_rope = idesc_bf16(64, kRows, 0, 0); // RoPE dims: bf16
      prefetch_tensormap(&map_q);
      const uint32_t q_addr = smem_u32(sQ), st_addr = smem_u32(sStage);
      bool ok = true;
      int seg = 0, i = 0;  // segment and global tile counters
#pragma unroll 1
      for (int64_t u = u0; u < u1 && ok; ++seg) {
        const Seg g = next_seg(u, u1, ntq);
        if (seg > 0) {  // the previous query's QK MMAs must have read Q before it is replaced
          mma_commit(q_free);
          if (!mbar_wait(q_free, (uint32_t)(seg - 1) & 1u, p.err)) {
            ok = false;
            break;
          }
        }
        mbar_arrive_expect_tx(q_full, kQBytes);
#pragma unroll 1
        for (int db = 0; db < 9; ++db)
          tma_load_2d(sQ + db * kQBlk, &map_q, q_full, db * 64, (int32_t)(g.q * p.H));
        if (!mbar_wait(q_ready, (uint32_t)seg & 1u, p.err)) {
          ok = false;
          break;
        }
#pragma unroll 1
        for (int jt = g.ta; jt < g.tb; ++jt, ++i) {
          const int s = i & 3;
          const uint32_t ph = (uint32_t)(i >> 2) & 1u;
          if (*abort_flag || !mbar_wait(&s_free[s], ph ^ 1u, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sa = st_addr + (uint32_t)(s * kStageBytes);
          const uint32_t d = tmem + kColS + kRows * s;
          if (!mbar_wait(&full[s], ph, p.err)) {  // the whole tile written by all producer warps
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int db = 0; db < kBlocks; ++db) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = smem_desc(q_addr + db * kQBlk + kk * 32, 16, 1024, 2);
              const uint64_t b = smem_desc(sa + db * kBlk + kk * 32, 16, 1024, 2);
              mma_bf16_ss(d, a, b, db < 8 ? idesc_qk : idesc_qk_rope, (db | kk) != 0 ? 1u : 0u);
            }
          }
          if (!ok) break;
          mma_commit(&s_full[s]);
        }
      }
      if (!ok) *abort_flag = 1;
      mma_commit(mma_done);
      mbar_wait(mma_done, 0, p.err);
      if (seg > 0) mbar_wait(q_full, (uint32_t)(seg - 1) & 1u, p.err);  // the last Q copy has landed
    }
  } else if (warp == kPvWarp) {
    // ================================================================ PV issuer =================
    // O^T += V^T . P^T for each tile once the softmax warps have written its P: the stage read
    // MN-major as A (M = 128 dims x4 M-tiles, K = 32 rows in two steps), P^T from the stage's
    // RoPE block as B (K-major, 64-byte swizzle, N = 64 heads). The first tile of a query starts
    // O^T afresh. One commit per tile marks its PV complete, which releases the whole stage
    // (the producers refill it, and a softmax warp about to rescale O^T waits for it).
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_f16(128, 64, 1, 0);
      const uint32_t st_addr = smem_u32(sStage);
      bool ok = true;
      int i = 0;
#pragma unroll 1
      for (int64_t u = u0; u < u1 && ok;) {
        const Seg g = next_seg(u, u1, ntq);
#pragma unroll 1
        for (int jt = g.ta; jt < g.tb; ++jt, ++i) {
          const int s = i & 3;
          if (*abort_flag || !mbar_wait(&p_ready[s], (uint32_t)(i >> 2) & 1u, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = st_addr + (uint32_t)(s * kStageBytes);
          const uint32_t p_addr = sa + 8 * kBlk;  // P of this tile in the stage's RoPE block
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int kk = 0; kk < kRows / 16; ++kk) {
              const uint64_t a = smem_desc(sa + (uint32_t)(2 * mt * kBlk + kk * 2048), kBlk, 1024, 2);
              const uint64_t b = smem_desc(p_addr + kk * 32, 16, 512, 4);
              mma_bf16_ss(tmem + kColO + 64 * mt, a, b, idesc_pv, (jt > g.ta || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit(&empty[s]);  // the tile's PV is complete: the stage (and P in it) may be refilled
        }
      }
      if (!ok) *abort_flag = 1;
      mma_commit(pv_drain);
      mbar_wait(pv_drain, 0, p.err);
    }
  } else {
    // ================================================================ softmax / epilogue ========
    // Head h = 16 * quad + (lane % 16); lanes l and l + 16 share it, each owning 16 of the tile's
    // 32 columns (TMEM 16x32bx2 load), so the running max is agreed by one shuffle.
    const int quad = warp & 3;
    const int hl = lane & 15, half = lane >> 4;
    const int h = quad * 16 + hl;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int sm_tid = tid - (kThreads - kSmThreads);
    bool ok = true;
    int seg = 0, i = 0;  // segment and global tile counters
    // true once PV of global tile j has completed (its commit releases the stage)
    auto wait_pv = [&](int j) -> bool {
      return warp_wait(&empty[j & 3], (uint32_t)(j >> 2) & 1u, p.err, lane);
    };
#pragma unroll 1
    for (int64_t u = u0; u < u1 && ok; ++seg) {
      const Seg g = next_seg(u, u1, ntq);
      const int64_t q = g.q;
      const int ta = g.ta, tb = g.tb;
      // Q's latent dims (blocks 0-7) bf16 -> fp16 in place. Chunk c = sm_tid + 128 j (16 bytes) is
      // dim block j / 4 of head row (sm_tid / 8) + 16 (j % 4), so the 8 lanes sm_tid & ~7 .. + 7
      // hold all of a row's chunks and agree on its largest |q| with three shuffles. A row whose
      // largest value lies outside [2^-6, 2^15) (rare: fp16 would overflow, or lose precision to its
      // subnormal range) is then rewritten from global memory scaled by an exact power of two 2^e
      // that puts its largest value in [2^14, 2^15), RoPE block included (bf16, exact); the softmax
      // multiplies that head's logits by 2^-e. Other rows keep e = 0.
      float sc_log2;  // softmax scale * log2(e) * 2^-e of this thread's head
      {
        const bool qok = warp_wait(q_full, (uint32_t)seg & 1u, p.err, lane);
        bool finite = true;
        if (qok) {
          uint32_t rmax[4] = {0u, 0u, 0u, 0u};  // packed maxima of |bf16| bit patterns (NaN above inf)
          uint4* q4 = reinterpret_cast<uint4*>(sQ);
#pragma unroll 4
          for (int j = 0; j < 32; ++j) {
            const int c = sm_tid + kSmThreads * j;
            uint4 v = q4[c];
            uint32_t* w = &v.x;
#pragma unroll
            for (int uu = 0; uu < 4; ++uu) {
              rmax[j & 3] = __vmaxu2(rmax[j & 3], w[uu] & 0x7FFF7FFFu);
              const float lo = __uint_as_float(w[uu] << 16), hi = __uint_as_float(w[uu] & 0xFFFF0000u);
              const __half2 h2 = __floats2half2_rn(lo, hi);
              w[uu] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            q4[c] = v;
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) {
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) rmax[r] = __vmaxu2(rmax[r], __shfl_xor_sync(0xffffffffu, rmax[r], o));
            const uint32_t amax = max(rmax[r] & 0xFFFFu, rmax[r] >> 16);
            const int row = (sm_tid >> 3) + 16 * r;
            finite &= amax < 0x7F80u || row >= p.H;
            int e = 0;
            if (amax >= 0x4700u && amax < 0x7F80u) e = 14 - ((int)(amax >> 7) - 127);       // >= 2^15
            else if (amax >= 0x0080u && amax < 0x3C80u) e = 14 - ((int)(amax >> 7) - 127);  // normal, < 2^-6
            else if (amax > 0u && amax < 0x0080u) e = 126;  // bf16 subnormals only
            if (row >= p.H) e = 0;  // rows of the next query (or beyond the tensor): not computed here
            e = e < -126 ? -126 : (e > 126 ? 126 : e);
            if ((sm_tid & 7) == 0) sQe[row] = e;
            if (e != 0) {
              // rare: rewrite the row from global memory, 9 chunks per lane (lane & 7 = chunk column)
              const float f = __uint_as_float((uint32_t)(e + 127) << 23);  // 2^e
              const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) + (q * p.H + row) * HS_D_QK * 2;
#pragma unroll 1
              for (int b = 0; b < 9; ++b) {
                const int chunk = sm_tid & 7;
                uint4 v = ldg_nc_v4(src + b * 128 + 16 * chunk);
                uint32_t* w = &v.x;
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                  const float lo = __uint_as_float(w[uu] << 16) * f, hi = __uint_as_float(w[uu] & 0xFFFF0000u) * f;
                  if (b < 8) {
                    const __half2 h2 = __floats2half2_rn(lo, hi);
                    w[uu] = *reinterpret_cast<const uint32_t*>(&h2);
                  } else {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                    w[uu] = *reinterpret_cast<const uint32_t*>(&b2);
                  }
                }
                *reinterpret_cast<uint4*>(sQ + b * kQBlk + sw128_offset(row, 16 * chunk)) = v;
              }
            }
          }
        }
        if (!finite) flag_error(p.err, HS_FLAG_RANGE);
        if (!qok) *abort_flag = 1;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_ready);
        named_bar(1, kSmThreads);  // every row's exponent written (QK has already been released)
        sc_log2 = p.scale_log2 * __uint_as_float((uint32_t)(127 - sQe[h]) << 23);
      }
      float m_ref = -INFINITY, l_part = 0.f;
#pragma unroll 1
      for (int jt = ta; jt < tb; ++jt, ++i) {
        const int s = i & 3;
        const uint32_t ph = (uint32_t)(i >> 2) & 1u;
        // every exit decision is taken by all four softmax warps together (no partial barriers)
        // (the RoPE block barrier also orders the producers' row-validity bytes before the reads below)
        bool w = !*abort_flag && warp_wait(&s_full[s], ph, p.err, lane) &&
                 warp_wait(&full[s], ph, p.err, lane);
        if (named_bar_or(1, kSmThreads, !w)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        uint32_t xr[16];
        tmem_ld16x2_16(tmem + lane_base + kColS + kRows * s, xr);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[s]);
        // logits in log2 units, in place (as float bits); masked rows become -inf
        float mt = -INFINITY;
        {
          const uint4 vv = *reinterpret_cast<const uint4*>(sValid + s * kRows + 16 * half);
          const uint32_t w4[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const bool valid = (w4[c >> 2] >> (8 * (c & 3))) & 0xFFu;
            const float v = valid ? __uint_as_float(xr[c]) * sc_log2 : -INFINITY;
            xr[c] = __float_as_uint(v);
            mt = fmaxf(mt, v);
          }
        }
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        const bool need = mt > m_ref + kRescaleThreshold;
        const float m_new = need ? mt : m_ref;
        // (the first tile of a query starts O^T afresh: PV does not accumulate into it)
        const bool any = named_bar_or(1, kSmThreads, need && jt > ta);
        const float alpha = need ? fast_exp2(m_ref - m_new) : 1.f;
        l_part *= alpha;
        m_ref = m_new;
        {
          // P goes into this stage's RoPE block as [head][32 rows] fp16 (64-byte rows, 64-byte
          // swizzle): QK of the tile has finished reading the block (s_full), and the producers do
          // not refill it before PV of the tile releases it. This thread writes rows 16 half ..
          // 16 half + 15 of head h: two 16-byte chunks.
          uint8_t* sPt = sStage + s * kStageBytes + 8 * kBlk;
          float psum = 0.f;
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t pk[4];
#pragma unroll
            for (int uu = 0; uu < 4; ++uu) {
              const int c = ch * 8 + 2 * uu;
              const float x0 = __uint_as_float(xr[c]), x1 = __uint_as_float(xr[c + 1]);
              const float p0 = x0 == -INFINITY ? 0.f : fast_exp2(x0 - m_ref);
              const float p1 = x1 == -INFINITY ? 0.f : fast_exp2(x1 - m_ref);
              psum += p0 + p1;
              const __half2 h2 = __floats2half2_rn(p0, p1);
              pk[uu] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(sPt + sw64_offset(h, (2 * half + ch) * 16)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
          l_part += psum;
        }
        // rescale O^T columns of the heads whose reference max moved, once PV of the previous tile
        // (and so every earlier one: they complete in order) has finished accumulating into it
        if (any) {
          if (!wait_pv(i - 1)) *abort_flag = 1;
          if (half == 0) sAlpha[h] = alpha;
          named_bar(1, kSmThreads);
          tc_fence_after();
#pragma unroll 1
          for (int part = 0; part < 8; ++part) {  // 4 M-tiles x 2 halves of 32 head columns
            uint32_t o[32];
            const uint32_t oa = tmem + lane_base + kColO + 32 * part;
            const float* al = sAlpha + 32 * (part & 1);
            tmem_ld32(oa, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * al[c]);
            tmem_st32(oa, o);
          }
          tmem_wait_st();
        }
        // P (and the corrected O^T) of this warp are ready; the PV warp waits for all four
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_ready[s]);
      }
      // ---- the query's normalisation and output (final, or a partial for the merge) ----
      if (ok) {
        const bool w = wait_pv(i - 1);
        if (named_bar_or(1, kSmThreads, !w)) {
          ok = false;
          *abort_flag = 1;
        }
      }
      tc_fence_after();
      const bool whole = ta == 0 && tb == ntq;
      const int64_t slot = seg == 0 ? 2 * (int64_t)blockIdx.x : 2 * (int64_t)blockIdx.x + 1;
      __nv_bfloat16* obase = whole ? p.out + q * p.H * HS_D_LATENT : p.part_out + slot * p.H * HS_D_LATENT;
      float* lbase = whole ? (p.lse ? p.lse + q * p.H : nullptr) : p.part_lse + slot * p.H;
      const float l_sum = l_part + __shfl_xor_sync(0xffffffffu, l_part, 16);
      if (half == 0) {
        sInvL[h] = l_sum > 0.f ? 1.f / l_sum : 0.f;
        if (lbase && h < p.H) lbase[h] = l_sum > 0.f ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
      }
      named_bar(1, kSmThreads);
      if (ok) {
        // O^T holds dims on TMEM lanes and heads on columns; the output rows are heads. This thread
        // owns dim 128 mt + 32 quad + lane of every M-tile mt. Neighbouring lanes swap values so
        // that each holds two adjacent dims of one head (even lanes: even heads, odd lanes: odd
        // heads) and writes them with one 4-byte store; a warp's store covers 64 contiguous bytes
        // of each of two head rows.
        const int odd = lane & 1;
#pragma unroll 1
        for (int mt4 = 0; mt4 < 4; ++mt4) {
#pragma unroll 1
          for (int hh = 0; hh < 2 && 32 * hh < p.H; ++hh) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + kColO + 64 * mt4 + 32 * hh, o);
            tmem_wait_ld();
            const int d0 = mt4 * 128 + quad * 32 + (lane & ~1);  // the pair's first dim
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float e = __uint_as_float(o[2 * j]), f = __uint_as_float(o[2 * j + 1]);
              const float mine = odd ? f : e;  // head 2j + odd at this dim
              const float give = odd ? e : f;  // the other head at this dim
              const float got = __shfl_xor_sync(0xffffffffu, give, 1);  // this head at the partner's dim
              const int hd = 32 * hh + 2 * j + odd;
              if (hd < p.H) {
                const float il = sInvL[hd];
                const float lo = odd ? got : mine, hi = odd ? mine : got;
                *reinterpret_cast<__nv_bfloat162*>(obase + (int64_t)hd * HS_D_LATENT + d0) =
                    __floats2bfloat162_rn(lo * il, hi * il);
              }
            }
          }
        }
        // O^T is read out before this warp's first P arrival of the next query lets PV overwrite it
        tc_fence_before();
      }
    }
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Combines the partial outputs of every query whose units were split between CTAs of a
// persistent launch: with partial (O_s, lse_s) per CTA s, lse = ln sum_s exp(lse_s) and
// out = sum_s exp(lse_s - lse) O_s (each O_s is already normalised by its own softmax sum).
// One CTA per (query, 8 heads); queries held by a single CTA were written by mla_kernel and are
// skipped. Every part's vectors are loaded before any is combined, so a thread has up to
// 2 x kMaxParts 16-byte loads in flight.
constexpr int kMergeThreads = 256;
constexpr int kMergeHeads = 8;
constexpr int kMaxParts = 8;
__global__ void __launch_bounds__(kMergeThreads)
    mla_merge_kernel(const Params p, int32_t C) {
  const int64_t q = blockIdx.x;
  const int h0 = blockIdx.y * kMergeHeads;
  const int ntq = (p.k + kRows - 1) / kRows;
  const int64_t ca = unit_cta(q * ntq, p.U, C), cb = unit_cta(q * ntq + ntq - 1, p.U, C);
  if (ca == cb || h0 >= p.H) return;
  __shared__ float w[kMaxParts][kMergeHeads];  // merge weight of each part and head
  __shared__ int64_t base[kMaxParts];          // slot of each part in part_out / part_lse
  const int nparts = (int)(cb - ca + 1);
  if (nparts > kMaxParts) {  // cannot happen for launch sizes the host chooses; never silently wrong
    if (threadIdx.x == 0) flag_error(p.err, HS_FLAG_BAD_STATE);
    return;
  }
  if (threadIdx.x < nparts) {
    // slot of CTA c for this query: its first query -> 2c, else its last -> 2c + 1
    const int64_t c = ca + threadIdx.x;
    base[threadIdx.x] = unit_begin(c, p.U, C) / ntq == q ? 2 * c : 2 * c + 1;
  }
  __syncthreads();
  const int nh = p.H - h0 < kMergeHeads ? p.H - h0 : kMergeHeads;
  if (threadIdx.x < nh) {
    const int h = h0 + threadIdx.x;
    float m = -INFINITY;
    for (int s = 0; s < nparts; ++s) m = fmaxf(m, p.part_lse[base[s] * p.H + h]);
    float z = 0.f;
    float e[kMaxParts];
#pragma unroll
    for (int s = 0; s < kMaxParts; ++s) {
      e[s] = 0.f;
      if (s < nparts) {
        const float l = p.part_lse[base[s] * p.H + h];
        e[s] = (m == -INFINITY || l == -INFINITY) ? 0.f : __expf(l - m);
        z += e[s];
      }
    }
#pragma unroll
    for (int s = 0; s < kMaxParts; ++s)
      if (s < nparts) w[s][threadIdx.x] = z > 0.f ? e[s] / z : 0.f;
    if (p.lse) p.lse[q * p.H + h] = z > 0.f ? m + __logf(z) : -INFINITY;
  }
  __syncthreads();
  // 8 output values (16 bytes) per vector, 64 vectors per head
  constexpr int kVec = HS_D_LATENT / 8;
  constexpr int kPer = kMergeHeads * kVec / kMergeThreads;  // vectors per thread
  const int nvec = nh * kVec;
  uint4 x[kMaxParts][kPer];
#pragma unroll
  for (int s = 0; s < kMaxParts; ++s) {
    if (s < nparts) {
      const __nv_bfloat16* src = p.part_out + (base[s] * p.H + h0) * HS_D_LATENT;
#pragma unroll
      for (int b = 0; b < kPer; ++b) {
        const int v = threadIdx.x + b * kMergeThreads;
        x[s][b] = v < nvec ? ldg_nc_v4(src + 8 * (int64_t)v) : make_uint4(0, 0, 0, 0);
      }
    }
  }
#pragma unroll
  for (int b = 0; b < kPer; ++b) {
    const int v = threadIdx.x + b * kMergeThreads;
    if (v >= nvec) continue;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxParts; ++s) {
      if (s < nparts) {
        const float ws = w[s][v / kVec];
        const uint32_t xs[4] = {x[s][b].x, x[s][b].y, x[s][b].z, x[s][b].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[2 * e] += ws * __uint_as_float(xs[e] << 16);
          acc[2 * e + 1] += ws * __uint_as_float(xs[e] & 0xFFFF0000u);
        }
      }
    }
    uint4 o;
    uint32_t* os = &o.x;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
      os[e] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(p.out + (q * p.H + h0) * HS_D_LATENT + 8 * (int64_t)v) = o;
  }
}

}  // namespace mla

// Workspace of the persistent launch on a device with `sms` SMs: two partial slots per CTA.
uint64_t mla_workspace_bytes(int32_t H, int sms) {
  return (uint64_t)2 * sms * H * (HS_D_LATENT * 2 + 4);
}

cudaError_t launch_mla(const hs_mla_args* a, int sms, cudaStream_t stream, const char** why) {
  using namespace mla;
  CUtensorMap mq;
  if (!encode_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->q, HS_D_QK, (uint64_t)a->T * a->H, HS_D_QK * 2, 64, 64,
                 CU_TENSOR_MAP_SWIZZLE_128B)) {
    *why = "cuTensorMapEncodeTiled failed for q";
    return cudaErrorInvalidValue;
  }
  Params p;
  p.T = a->T;
  p.H = a->H;
  p.k = a->k;
  p.q = reinterpret_cast<const __nv_bfloat16*>(a->q);
  p.kv = a->kv_pool;
  p.R = a->R;
  p.idx = a->idx;
  p.idx_row = a->idx_row;
  p.idx_rows = a->idx_rows;
  p.kvlen = a->token_kvlen;
  p.bt = a->block_table;
  p.bt_stride = a->bt_stride;
  p.token_req = a->token_req;
  p.scale_log2 = a->softmax_scale * kLog2e;
  p.out = reinterpret_cast<__nv_bfloat16*>(a->out);
  p.lse = a->lse;
  p.err = a->err_flag;
  p.persistent = 0;
  p.U = 0;
  p.part_out = nullptr;
  p.part_lse = nullptr;
  if (a->T == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int ntq = (a->k + kRows - 1) / kRows;
  const int64_t U = (int64_t)a->T * ntq;
  // One CTA per query keeps every SM busy when the queries fill whole waves; otherwise (fewer
  // queries than SMs, or a last wave mostly empty) the persistent split pays for its per-query
  // set-up at the split points and for the merge. The split is used when one CTA per query would
  // leave more than a quarter of the SM-time of its waves idle.
  const int64_t waves = (a->T + sms - 1) / sms;
  const bool split = a->workspace && 4 * (int64_t)a->T < 3 * waves * sms;
  if (!split) {  // one CTA per query
    mla_kernel<<<a->T, kThreads, kSmem, stream>>>(mq, p);
    return cudaGetLastError();
  }
  // persistent: one CTA per SM, each an equal share of the units; at most 4 CTAs per query, so
  // a query is split into at most 5 parts (tiny batches use fewer CTAs)
  int64_t C64 = sms;
  if (C64 > U) C64 = U;
  if (C64 > 4LL * a->T) C64 = 4LL * a->T;
  const int C = (int)C64;
  p.persistent = 1;
  p.U = U;
  p.part_out = reinterpret_cast<__nv_bfloat16*>(a->workspace);
  p.part_lse = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(a->workspace) +
                                        (uint64_t)2 * sms * a->H * HS_D_LATENT * 2);
  mla_kernel<<<C, kThreads, kSmem, stream>>>(mq, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mla_merge_kernel<<<dim3((unsigned)a->T, (unsigned)((a->H + kMergeHeads - 1) / kMergeHeads)), kMergeThreads, 0, stream>>>(
      p, C);
  return cudaGetLastError();
}

}  // namespace hs
