// mla.cu — sparse MLA forward in MQA form on tcgen05, the gathered rows on the MMA's M side.
//
// [P1] "vLLM v0.32.0 GLM-5.3 サービング ...", sections 「再現方法と必要なフラグ」 and
// 「数字がうまくいく理由」: each query gathers its selected 656-byte FP8 latent rows once and every
// row serves all 64 heads; QK runs over 576 dims (512 latent + 64 RoPE), PV over the 512 latent
// dims. Per query token t, head h, over the valid entries i of idx[t, :]:
//   logit_i = scale * <q[t,h,:], [latent_i, rope_i]>,  out = softmax(logit) . latent,  lse = ln sum exp.
//
// The gathered rows are the M side of QK, and the dims the M side of PV:
//   S^T = K . Q^T   M = 64 gathered rows, N = 64 heads, K = 512 fp16 latent + 64 bf16 RoPE dims;
//   O^T += V^T . P  M = 128 dims (x4), N = 64 heads, K = 64 rows;
// 52 MMAs per 64-row tile (36 + 16). With M = 64 rows each QK MMA covers twice the rows that one
// with the 64 heads on M and 32 rows on N did, at the same cost (~45 cycles: shared-memory operand
// bandwidth and a fixed cost per instruction dominate shapes this small).
//
// One CTA per query token (512 threads), or, given a workspace and too few queries to fill the
// SMs' waves, one persistent CTA per SM taking an equal share of all (query, 64-row tile) units.
// Two tile slots live in shared memory beside the query's 64 x 576 Q (72 KB), each as nine
// 128-byte-swizzled [64 rows][64 dims] blocks (fp16 latent blocks 0-7, bf16 RoPE block 8): the
// producers fill one while the other goes through QK, softmax and PV. A slot is released to its
// next tile chunk by chunk, a chunk being a 128-dim latent group (two blocks), as PV drains it.
// Roles by warp; warp w runs on SM sub-partition w % 4 and reads TMEM lanes 32 (w % 4) .. + 31:
//   warps 1-3, 5-7, 13, 14 (producers 0-7, on sub-partitions 1-3): producer p owns rows
//               8p .. 8p+7 of every tile; in each of two passes a lane works on row 8p + 4 pass +
//               l / 8 and loads the 16-byte pieces l % 8 of its 128-byte spans (coalesced 16-byte
//               loads of random 656-byte rows), each lane from the index and block-table entries
//               of its own rows. They dequantise latent = e4m3 * group scale to fp16 (exact
//               e4m3 -> fp16 conversion, then code * scale rounded once, with the scale split into
//               two fp16 parts; see dequant8_f16) and write chunk c of tile i once PV of tile i-2
//               has finished with it. Rows are loaded into registers one tile ahead and prefetched
//               into L2 by the TMA engine two tiles ahead. Chunk 3 carries the RoPE block (bf16 as
//               stored) and each row's validity;
//   warp 0      allocates TMEM, loads Q by TMA and issues S^T chunk by chunk as the producers
//               publish them;
//   warp 4      issues O^T += V^T . P once P is written (the slot's latent blocks read MN-major as
//               A, P as an MN-major B) and commits after each chunk, which releases that chunk;
//   warps 8-11  first convert Q's latent dims to fp16 in shared memory (a head's row whose largest
//               value fp16 cannot hold at full precision is scaled by a power of two), then run
//               the online softmax: thread (warp w, lane l) owns tile row 16 (w % 4) + l % 16 and
//               heads 32 (l / 16) .. + 31. A head's reference max is shared by all rows and only
//               moves when some logit exceeds it by more than 2^8 (lazy rescaling): the check is
//               one OR-barrier per tile; when it fires the tile's exact per-head maxima are taken
//               (a transposing butterfly within each half-warp, then across the four warps) and
//               O^T's columns are rescaled once the previous tile's PV has completed. P goes as
//               fp16 [row][64 heads] into the slot's RoPE block, which QK has finished with. Each
//               thread keeps its row's running sums; the last pass adds them per head, divides and
//               writes bf16 straight from TMEM.
// The two MMA-issuing warps share sub-partition 0 with the quarter-0 softmax warp only: warps that
// run long ALU sequences on a sub-partition (the dequantisation) take the issue slots a lone
// issuing thread needs, and measured on this GPU that feeds the tensor core up to ten times slower.
// TMEM: columns 0-127 hold two S^T buffers (64-row layout: tile row 16 q + r in lane 32 q + r),
// 128-383 hold O^T (4 x [128 dims][64 heads]).
//
// A query split between CTAs leaves, from each, a normalised partial and its LSE in the workspace;
// mla_merge_kernel combines them (split-KV decode: DCP's log-sum-exp merge on one GPU).
#include "common.cuh"

namespace hs {
namespace mla {

constexpr int kRows = 64;                  // rows per tile (the M of S^T = K . Q^T)
constexpr int kSlots = 2;                  // tiles in shared memory: one is filled while the other is used
// Warp roles by sub-partition (see the header).
constexpr int kQkWarp = 0;                 // QK issuer; also allocates TMEM and loads Q
constexpr int kPvWarp = 4;                 // PV issuer
constexpr int kSmWarp0 = 8;                // softmax warps 8-11 (lane quarters 0-3)
constexpr int kSmWarps = 4;
constexpr int kSmThreads = 32 * kSmWarps;
constexpr int kProdWarps = 8;              // on sub-partitions 1-3: warps 1-3, 5-7, 13, 14
constexpr int kThreads = 512;              // warps 12 and 15 have no role
// producer index of warp w (0-7), or -1
__host__ __device__ constexpr int producer_index(int w) {
  return (w % 4 == 0 || (w >= 8 && w < 12) || w == 15) ? -1 : (w < 8 ? w - 1 - w / 4 : w - 7);
}
constexpr uint32_t kColS = 0;              // two S^T buffers of 64 columns
constexpr uint32_t kColO = 128;
constexpr int kQBlk = 8192;                // one [64 heads][128 B] swizzled block of Q
constexpr int kBlk = kRows * 128;          // one [64 rows][128 B] swizzled block of a tile
constexpr int kQBytes = 9 * kQBlk;         // 64 heads x 576 bf16
constexpr int kTileBytes = 9 * kBlk;       // 64 rows x (512 latent fp16 + 64 rope bf16)
constexpr int kOffQ = 0;
constexpr int kOffTile = kQBytes;                        // kSlots tiles
constexpr int kOffValid = kOffTile + kSlots * kTileBytes;  // uint8 [kSlots][64]
constexpr int kOffM = kOffValid + kSlots * kRows;        // float [3][2][64]: running max, max + threshold, exponent offset
constexpr int kOffC = kOffM + 3 * 2 * 64 * 4;            // float [64]: softmax scale * log2(e) * 2^-e per head
constexpr int kOffAlpha = kOffC + 256;                   // float [64]
constexpr int kOffInvL = kOffAlpha + 256;                // float [64]
constexpr int kOffQe = kOffInvL + 256;                   // int [64]: per-head exponent of the current query
constexpr int kOffRed = kOffQe + 256;                    // float [4][64]: per-warp partial maxima / sums
constexpr int kNumBars = 2 * 4 * kSlots + 3 * kSlots + 5;
constexpr int kOffBar = kOffRed + 4 * 64 * 4;
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort
constexpr int kSmem = kOffMisc + 16 + 1024;
constexpr float kRescaleThreshold = 8.0f;         // log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kScaleMax = 65504.f / 448.f;      // |code * scale| stays finite in fp16
constexpr float kScaleMin = 6.103515625e-05f;     // 2^-14: scales stay fp16 normals
static_assert(kSmem <= 232448, "shared memory");
static_assert(kOffTile % 1024 == 0 && kTileBytes % 1024 == 0, "swizzled blocks need 1024-byte alignment");

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
  // Work split. Units are (query, 64-row tile) pairs, U = T * tiles per query in total. A CTA
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

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Per-head reduction over the 16 lanes of a half-warp that hold 16 rows of S^T with the same 32
// heads hb .. hb + 31 (lane bits 0-3 = row, lane bit 4 = head half), so that lane l ends with heads
// hb + (l % 16) and hb + 16 + (l % 16) reduced over those 16 rows. pair_step takes the values of
// heads hb + 16 g .. + 15: a lane whose bit 0 is b keeps head hb + 16 g + 2m + b, sends the other of
// the pair to its partner lane and stores the combination in r[8 g + m], which then stands for head
// hb + 2 (8 g + m) + b. finish runs the remaining steps over lane bits 1-3 on r[0..7] and r[8..15]
// separately (each step a lane keeps half of its values and sends the other half to its partner).
template <bool kMax>
__device__ __forceinline__ void half_transpose_pair_step(const float (&x)[16], float (&r)[16], int g, int lane) {
  const bool up = (lane & 1) != 0;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float a = x[2 * m], b = x[2 * m + 1];
    const float got = __shfl_xor_sync(0xffffffffu, up ? a : b, 1);
    r[8 * g + m] = kMax ? fmaxf(up ? b : a, got) : (up ? b : a) + got;
  }
}
template <bool kMax>
__device__ __forceinline__ void half_transpose_finish(float (&r)[16], int lane) {
#pragma unroll
  for (int base = 0; base < 16; base += 8) {
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) {
      const bool up = (lane & (2 * o)) != 0;
#pragma unroll
      for (int i = 0; i < o; ++i) {
        const float send = up ? r[base + i] : r[base + i + o];
        const float keep = up ? r[base + i + o] : r[base + i];
        const float got = __shfl_xor_sync(0xffffffffu, send, 2 * o);
        r[base + i] = kMax ? fmaxf(keep, got) : keep + got;
      }
    }
  }
}

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

// The 16-byte pieces of one latent group that a producer lane holds for its two rows of a tile,
// and those rows' scales of that group.
struct Chunk {
  uint4 v[2];
  float s[2];
  uint32_t ok;  // bit ps: the row of pass ps exists (else its values count as zeros)
};
struct Rope {
  uint4 v[2];
  uint32_t ok;
};

__global__ void __launch_bounds__(kThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap map_q, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sTile = smem + kOffTile;     // slot s at sTile + s * kTileBytes
  uint8_t* sValid = smem + kOffValid;   // [slot][row]
  float* sM = (float*)(smem + kOffM);   // [2][64] running max per head (log2 units), two versions
  float* sThr = sM + 128;               // [2][64] running max + threshold
  float* sMe = sThr + 128;              // [2][64] running max, 0 where it is -inf (exponent offset)
  float* sC = (float*)(smem + kOffC);
  float* sAlpha = (float*)(smem + kOffAlpha);
  float* sInvL = (float*)(smem + kOffInvL);
  int32_t* sQe = (int32_t*)(smem + kOffQe);
  float* sRed = (float*)(smem + kOffRed);
  uint64_t* bars = (uint64_t*)(smem + kOffBar);
  uint64_t* chunk_full = bars + 0;            // [slot][4] producers wrote chunk c -> QK (chunk 3: softmax too)
  uint64_t* chunk_free = bars + 4 * kSlots;   // [slot][4] PV finished with chunk c -> producers (chunk 3: softmax)
  uint64_t* s_full = bars + 8 * kSlots;       // [slot] S^T of the slot's tile complete -> softmax
  uint64_t* s_free = s_full + kSlots;         // [slot] softmax read S^T -> QK
  uint64_t* p_ready = s_free + kSlots;        // [slot] softmax wrote P (and rescaled O^T) -> PV
  uint64_t* q_full = p_ready + kSlots;        // Q landed (TMA)
  uint64_t* q_ready = q_full + 1;             // Q converted to fp16 (latent dims) -> QK issuer
  uint64_t* q_free = q_full + 2;              // QK MMAs of a query finished reading Q -> QK issuer
  uint64_t* mma_done = q_full + 3;            // QK issuer's MMAs drained
  uint64_t* pv_drain = q_full + 4;            // PV issuer's MMAs drained
  uint32_t* misc = (uint32_t*)(smem + kOffMisc);
  volatile uint32_t* abort_flag = misc + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = p.k;
  const int ntq = (k + kRows - 1) / kRows;  // tiles per query
  // this CTA's units; every role walks them as segments (query, tiles [ta, tb)) in the same order,
  // and counts tiles globally (i): tile i uses slot i % 2, and each slot's barriers complete one
  // phase per use, so the phase parity of tile i is (i / 2) % 2
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
    for (int s = 0; s < kSlots; ++s) {
      for (int c = 0; c < 4; ++c) {
        mbar_init(&chunk_full[4 * s + c], kProdWarps);
        mbar_init(&chunk_free[4 * s + c], 1);
      }
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], kSmWarps);
      mbar_init(&p_ready[s], kSmWarps);
    }
    mbar_init(q_full, 1);
    mbar_init(q_ready, kSmWarps);
    mbar_init(q_free, 1);
    mbar_init(mma_done, 1);
    mbar_init(pv_drain, 1);
    mbar_fence_init();
    misc[1] = 0;
  }
  if (warp == kQkWarp) tmem_alloc(&misc[0], 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  const int pw = producer_index(warp);
  if (pw >= 0) {
    // ================================================================ gather + dequantise ======
    // Lane l of producer pw works on rows 8 pw + 4 pass + rl (rl = l / 8, pass 0-1) and on bytes 16 c8 (c8 = l % 8)
    // of each 128-byte span of them: the 16 codes of latent group c there become fp16 dims
    // 16 c8 .. + 15 of that group, i.e. 16-byte chunks 2 (c8 % 4) and 2 (c8 % 4) + 1 of block
    // 2c + c8 / 4. Lanes with c8 >= 4 store their second chunk first, so that in each store the
    // eight lanes of a row hit eight different bank groups. Each lane reads the index and
    // block-table entries of its own rows (the eight lanes of a row read the same words): no value
    // crosses lanes, since shuffles queue behind the tensor core's shared-memory traffic.
    const int rl = lane >> 3, c8 = lane & 7;
    const bool swp = c8 >= 4;
    int64_t la_q = u0 / ntq;
    int la_t = (int)(u0 - la_q * ntq), la_n = 0;
    // Index entries of this lane's rows of the CTA's next lookahead tile (tiles are visited in
    // order), with, given a block table, the request of its query and its visible length. Every
    // load reads a valid address (entry 0 of query 0 where there is no entry) and `val` says which
    // entries exist: a load under a condition with a constant on the other path makes that write
    // wait for the load.
    struct Ent {
      int32_t j[2];
      int32_t req, lim;
      uint32_t val;
    };
    auto ld_idx = [&](Ent& E) {
      const bool live = la_n < ntot;
      const int64_t q = live ? la_q : 0;
      const int e0 = la_t * kRows + pw * 8 + rl;
      if (++la_t == ntq) {
        la_t = 0;
        ++la_q;
      }
      ++la_n;
      int64_t r = q;
      bool row_ok = true;
      if (p.idx_row) {  // shared index sets: the query's idx row (its value forms the address)
        r = ldg_nc_s32(p.idx_row + q);
        if (r < 0 || r >= p.idx_rows) {
          if (live && lane == 0) flag_error(p.err, HS_FLAG_BAD_INDEX);
          row_ok = false;
          r = 0;
        }
      }
      E.req = 0;
      E.lim = 0x7FFFFFFF;
      if (p.bt) E.req = ldg_nc_s32(p.token_req + q);
      if (p.kvlen) E.lim = ldg_nc_s32(p.kvlen + q);  // applied one step later, in ld_blk
      E.val = 0u;
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        const int e = e0 + 4 * ps;
        const bool ok = live && row_ok && e < k;
        E.val |= ok ? 1u << ps : 0u;
        E.j[ps] = ldg_nc_s32(p.idx + r * k + (ok ? e : 0));
      }
    };
    // one tile later: entries that do not exist or lie beyond the query's visible length become -1,
    // and the block-table entries are read (page clamped into the table; checked in phys_row)
    auto ld_blk = [&](Ent& E, int32_t (&b)[2]) {
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        if (!((E.val >> ps) & 1u) || E.j[ps] >= E.lim) E.j[ps] = -1;
        b[ps] = 0;
        if (p.bt) {
          const int32_t page = E.j[ps] >= 0 ? E.j[ps] >> 6 : 0;
          b[ps] = ldg_nc_s32(p.bt + (int64_t)E.req * p.bt_stride + (page < p.bt_stride ? page : 0));
        }
      }
    };
    // physical row of entry j (block entry b), -1 if none; an entry that names no row is flagged
    auto phys_row = [&](int32_t j, int32_t b) -> int32_t {
      if (j < 0) return -1;
      const int64_t r = p.bt ? (((j >> 6) < p.bt_stride && b >= 0) ? (int64_t)b * 64 + (j & 63) : -1) : (int64_t)j;
      if (r < 0 || r >= p.R) {
        if (c8 == 0) flag_error(p.err, HS_FLAG_BAD_INDEX);
        return -1;
      }
      return (int32_t)r;
    };
    // the rows are prefetched into L2 by the TMA engine, one bulk prefetch per row (lane c8 = 0)
    auto prefetch_rows = [&](const int32_t (&rows)[2]) {
      if (c8 == 0) {
#pragma unroll
        for (int ps = 0; ps < 2; ++ps)
          if (rows[ps] >= 0) bulk_prefetch_l2(p.kv + (int64_t)rows[ps] * HS_KV_ROW_BYTES, HS_KV_ROW_BYTES);
      }
    };
    // Loads are unconditional (a padding row reads row 0 instead, whose values are then replaced by
    // zeros where they are used), for the reason given above.
    auto ld_chunk = [&](Chunk& ch, const int32_t (&rows)[2], int c) {
      ch.ok = 0u;
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        const int32_t r = rows[ps];
        ch.ok |= r >= 0 ? 1u << ps : 0u;
        const uint8_t* src = p.kv + (int64_t)(r >= 0 ? r : 0) * HS_KV_ROW_BYTES;
        ch.v[ps] = ldg_nc_v4(src + 128 * c + 16 * c8);
        ch.s[ps] = ldg_nc_f32(src + HS_D_LATENT + 4 * c);
      }
    };
    auto ld_rope = [&](Rope& rp, const int32_t (&rows)[2]) {
      rp.ok = 0u;
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        const int32_t r = rows[ps];
        rp.ok |= r >= 0 ? 1u << ps : 0u;
        rp.v[ps] = ldg_nc_v4(p.kv + (int64_t)(r >= 0 ? r : 0) * HS_KV_ROW_BYTES + HS_D_LATENT + 16 + 16 * c8);
      }
    };
    // chunk c of tile i may be written once PV of tile i - 2 (the slot's previous tile) has
    // finished with it (every lane waits, so no result has to be broadcast)
    auto wait_free = [&](int c, int i) -> bool {
      const bool go = !*abort_flag && mbar_wait(&chunk_free[4 * (i & 1) + c], ((uint32_t)(i >> 1) & 1u) ^ 1u, p.err);
      if (!go && lane == 0) *abort_flag = 1;
      return __all_sync(0xffffffffu, go);
    };
    bool range_ok = true;
    auto st_chunk = [&](uint8_t* tile, const Chunk& ch, int c) {
      uint8_t* blk = tile + (2 * c + (c8 >> 2)) * kBlk;
      const uint32_t b0 = 32 * (c8 & 3) + (swp ? 16 : 0);
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        const int row = 8 * pw + 4 * ps + rl;
        const bool live = (ch.ok >> ps) & 1u;
        const float scale = live ? ch.s[ps] : 0.f;
        range_ok &= scale == 0.f || (fabsf(scale) >= kScaleMin && fabsf(scale) <= kScaleMax);
        const __half shi = __float2half_rn(scale);
        const __half2 h2 = __half2half2(shi);
        const __half2 l2 = __float2half2_rn(scale - __half2float(shi));  // scale - hi is exact in fp32
        const uint32_t h2u = *reinterpret_cast<const uint32_t*>(&h2);
        const uint32_t l2u = *reinterpret_cast<const uint32_t*>(&l2);
        const uint4 v = live ? ch.v[ps] : make_uint4(0, 0, 0, 0);
        const uint4 d0 = dequant8_f16(swp ? v.z : v.x, swp ? v.w : v.y, h2u, l2u);
        const uint4 d1 = dequant8_f16(swp ? v.x : v.z, swp ? v.y : v.w, h2u, l2u);
        *reinterpret_cast<uint4*>(blk + sw128_offset(row, b0)) = d0;
        *reinterpret_cast<uint4*>(blk + sw128_offset(row, b0 ^ 16u)) = d1;
      }
    };
    auto publish = [&](int c, int i) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&chunk_full[4 * (i & 1) + c]);
    };
    // Pipeline, entering tile i: physical rows of tiles i (rc) and i + 1 (rn), index and
    // block-table entries of tile i + 2 (E2, b2), index entries of tile i + 3 (E3).
    Ent E0, E1, E2, E3;
    ld_idx(E0);
    ld_idx(E1);
    ld_idx(E2);
    ld_idx(E3);
    int32_t b0[2], b1[2], b2[2];
    ld_blk(E0, b0);
    ld_blk(E1, b1);
    ld_blk(E2, b2);
    int32_t rc[2], rn[2];
#pragma unroll
    for (int ps = 0; ps < 2; ++ps) {
      rc[ps] = phys_row(E0.j[ps], b0[ps]);
      rn[ps] = phys_row(E1.j[ps], b1[ps]);
    }
    prefetch_rows(rc);
    prefetch_rows(rn);
    // the rows of a tile are loaded into registers one tile ahead: chunk c of tile i + 1 as soon as
    // chunk c of tile i has been written
    Chunk C[4];
    Rope rp;
#pragma unroll
    for (int c = 0; c < 4; ++c) ld_chunk(C[c], rc, c);
    ld_rope(rp, rc);
#pragma unroll 1
    for (int i = 0; i < ntot; ++i) {
      uint8_t* tile = sTile + (i & 1) * kTileBytes;
      int32_t r2[2];
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) r2[ps] = phys_row(E2.j[ps], b2[ps]);
      prefetch_rows(r2);
      int32_t b3[2];
      ld_blk(E3, b3);
      Ent E4;
      ld_idx(E4);
      bool go = true;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (!wait_free(c, i)) {
          go = false;
          break;
        }
        st_chunk(tile, C[c], c);
        if (c == 3) {
          // the RoPE block (it held P of tile i - 2) and the rows' validity
#pragma unroll
          for (int ps = 0; ps < 2; ++ps)
            *reinterpret_cast<uint4*>(tile + 8 * kBlk + sw128_offset(8 * pw + 4 * ps + rl, 16 * c8)) =
                ((rp.ok >> ps) & 1u) ? rp.v[ps] : make_uint4(0, 0, 0, 0);
          if (c8 == 0) {
#pragma unroll
            for (int ps = 0; ps < 2; ++ps) sValid[(i & 1) * kRows + 8 * pw + 4 * ps + rl] = rc[ps] >= 0 ? 1 : 0;
          }
        }
        publish(c, i);
        ld_chunk(C[c], rn, c);
        if (c == 3) ld_rope(rp, rn);
      }
      if (!go) break;
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        rc[ps] = rn[ps];
        rn[ps] = r2[ps];
        b2[ps] = b3[ps];
      }
      E2 = E3;
      E3 = E4;
    }
    if (!range_ok) flag_error(p.err, HS_FLAG_RANGE);
  } else if (warp == kQkWarp) {
    // ================================================================ QK issuer =================
    // S^T = K . Q^T into the slot's S buffer: A = the tile (K-major, M = 64 rows), B = Q (K-major,
    // N = 64 heads); chunk c's two blocks as soon as the producers publish them, chunk 3 with the
    // RoPE block.
    if (lane == 0) {
      constexpr uint32_t idesc_lat = idesc_f16(kRows, 64, 0, 0);   // latent dims: fp16
      constexpr uint32_t idesc_rope = idesc_bf16(kRows, 64, 0, 0); // RoPE dims: bf16
      prefetch_tensormap(&map_q);
      const uint32_t q_addr = smem_u32(sQ);
      const uint64_t qd = smem_desc(q_addr, 16, 1024, 2);
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
          const int s = i & 1;
          const uint32_t ph = (uint32_t)(i >> 1) & 1u;
          if (*abort_flag || !mbar_wait(&s_free[s], ph ^ 1u, p.err)) {
            ok = false;
            break;
          }
          const uint64_t td = smem_desc(smem_u32(sTile + s * kTileBytes), 16, 1024, 2);
          const uint32_t d = tmem + kColS + 64 * s;
#pragma unroll 1
          for (int c = 0; c < 4 && ok; ++c) {
            if (!mbar_wait(&chunk_full[4 * s + c], ph, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // descriptors advance by adding (byte offset / 16) to their start-address field
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
              const int db = 2 * c + bb;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(d, td + (uint64_t)((db * kBlk + kk * 32) >> 4), qd + (uint64_t)((db * kQBlk + kk * 32) >> 4),
                            idesc_lat, (db | kk) != 0 ? 1u : 0u);
            }
            if (c == 3) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(d, td + (uint64_t)((8 * kBlk + kk * 32) >> 4), qd + (uint64_t)((8 * kQBlk + kk * 32) >> 4),
                            idesc_rope, 1u);
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
    // O^T += V^T . P for each tile once the softmax warps have written its P: A = latent blocks
    // 2 mt, 2 mt + 1 of the slot read MN-major (M = 128 dims, K = 16 rows per MMA), B = P from the
    // slot's RoPE block (MN-major [row][64 heads], N = 64). The first tile of a query starts O^T
    // afresh. The commit after chunk mt releases it to the producers; the last one also releases
    // P's block and tells a softmax warp about to rescale O^T that the tile's PV is complete.
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_f16(128, 64, 1, 1);
      bool ok = true;
      int i = 0;
#pragma unroll 1
      for (int64_t u = u0; u < u1 && ok;) {
        const Seg g = next_seg(u, u1, ntq);
#pragma unroll 1
        for (int jt = g.ta; jt < g.tb; ++jt, ++i) {
          const int s = i & 1;
          if (*abort_flag || !mbar_wait(&p_ready[s], (uint32_t)(i >> 1) & 1u, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t t_addr = smem_u32(sTile + s * kTileBytes);
          const uint64_t ad = smem_desc(t_addr, kBlk, 1024, 2);
          const uint64_t pd = smem_desc(t_addr + 8 * kBlk, kBlk, 1024, 2);
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int kk = 0; kk < kRows / 16; ++kk)
              mma_bf16_ss(tmem + kColO + 64 * mt, ad + (uint64_t)((2 * mt * kBlk + kk * 2048) >> 4),
                          pd + (uint64_t)((kk * 2048) >> 4), idesc_pv, (jt > g.ta || kk > 0) ? 1u : 0u);
            mma_commit(&chunk_free[4 * s + mt]);
          }
        }
      }
      if (!ok) *abort_flag = 1;
      mma_commit(pv_drain);
      mbar_wait(pv_drain, 0, p.err);
    }
  } else if (warp >= kSmWarp0 && warp < kSmWarp0 + kSmWarps) {
    // ================================================================ softmax / epilogue ========
    // S^T of a 64-row tile sits in the 64-row TMEM layout: tile row 16 q + r (q = the warp's lane
    // quarter, r < 16) in lane 32 q + r. Thread (warp w, lane l) owns row 16 (w % 4) + (l % 16) and
    // heads hb .. hb + 31, hb = 32 (l / 16), read with one TMEM 16x32bx2 load per tile (the second
    // half-warp 32 columns further on) and kept in registers for the check, the maxima and P.
    const int quad = warp & 3;            // TMEM lane quarter this warp may access
    const int row = quad * 16 + (lane & 15);
    const int hb = 32 * (lane >> 4);
    const bool lead = quad == 0;          // this warp finalises per-head values (heads l, l + 32)
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int sm_tid = tid - kSmWarp0 * 32;
    bool ok = true;
    int seg = 0, i = 0;  // segment and global tile counters
    // true once PV of global tile j has completed (its last commit releases chunk 3 of its slot)
    auto wait_pv = [&](int j) -> bool {
      return warp_wait_all(&chunk_free[4 * (j & 1) + 3], (uint32_t)(j >> 1) & 1u, p.err);
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
      // multiplies that head's logits by 2^-e. Other rows keep e = 0. The same lanes reset the
      // head's softmax state for the query.
      bool qscaled;  // some head of this query has e != 0: per-head scales from sC
      {
        const bool qok = warp_wait_all(q_full, (uint32_t)seg & 1u, p.err);
        bool finite = true, scaled = false;
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
              w[uu] = pack_half2(lo, hi);
            }
            q4[c] = v;
          }
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) rmax[rr] = __vmaxu2(rmax[rr], __shfl_xor_sync(0xffffffffu, rmax[rr], o));
            const uint32_t amax = max(rmax[rr] & 0xFFFFu, rmax[rr] >> 16);
            const int qrow = (sm_tid >> 3) + 16 * rr;
            finite &= amax < 0x7F80u || qrow >= p.H;
            int e = 0;
            if (amax >= 0x4700u && amax < 0x7F80u) e = 14 - ((int)(amax >> 7) - 127);       // >= 2^15
            else if (amax >= 0x0080u && amax < 0x3C80u) e = 14 - ((int)(amax >> 7) - 127);  // normal, < 2^-6
            else if (amax > 0u && amax < 0x0080u) e = 126;  // bf16 subnormals only
            if (qrow >= p.H) e = 0;  // rows of the next query (or beyond the tensor): not computed here
            e = e < -126 ? -126 : (e > 126 ? 126 : e);
            if ((sm_tid & 7) == 0) {
              sQe[qrow] = e;
              sC[qrow] = p.scale_log2 * __uint_as_float((uint32_t)(127 - e) << 23);
              sM[qrow] = -INFINITY;
              sThr[qrow] = -INFINITY;
              sMe[qrow] = 0.f;
            }
            scaled |= e != 0;
            if (e != 0) {
              // rare: rewrite the row from global memory, 9 chunks per lane (lane & 7 = chunk column)
              const float f = __uint_as_float((uint32_t)(e + 127) << 23);  // 2^e
              const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) + (q * p.H + qrow) * HS_D_QK * 2;
#pragma unroll 1
              for (int b = 0; b < 9; ++b) {
                const int chunk = sm_tid & 7;
                uint4 v = ldg_nc_v4(src + b * 128 + 16 * chunk);
                uint32_t* w = &v.x;
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                  const float lo = __uint_as_float(w[uu] << 16) * f, hi = __uint_as_float(w[uu] & 0xFFFF0000u) * f;
                  if (b < 8) {
                    w[uu] = pack_half2(lo, hi);
                  } else {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                    w[uu] = *reinterpret_cast<const uint32_t*>(&b2);
                  }
                }
                *reinterpret_cast<uint4*>(sQ + b * kQBlk + sw128_offset(qrow, 16 * chunk)) = v;
              }
            }
          }
        }
        if (!finite) flag_error(p.err, HS_FLAG_RANGE);
        if (!qok) *abort_flag = 1;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_ready);
        // every head's exponent, scale and reset state written (QK has already been released)
        qscaled = named_bar_or(1, kSmThreads, scaled);
      }
      const float csc = p.scale_log2;
      auto cof = [&](int h) -> float { return qscaled ? sC[h] : csc; };
      float l[32];  // this row's sums of P for heads hb .. hb + 31
#pragma unroll
      for (int c = 0; c < 32; ++c) l[c] = 0.f;
      int v = 0;  // version of the per-head state in sM / sThr / sMe
#pragma unroll 1
      for (int jt = ta; jt < tb; ++jt, ++i) {
        const int s = i & 1;
        const uint32_t ph = (uint32_t)(i >> 1) & 1u;
        // the load's address is the warp's; the second half-warp reads 32 columns further on
        const uint32_t s_col = tmem + lane_base + kColS + 64 * s;
        // every exit decision is taken by all four softmax warps together (no partial barriers);
        // chunk 3's barrier also orders the producers' row-validity bytes before the read below
        bool w = !*abort_flag && warp_wait_all(&s_full[s], ph, p.err) && warp_wait_all(&chunk_full[4 * s + 3], ph, p.err);
        if (named_bar_or(1, kSmThreads, !w)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const bool valid = sValid[s * kRows + row] != 0;
        // this row's 32 logits, in one TMEM load (the second half-warp's columns are 32 further on)
        uint32_t x[32];
        tmem_ld16x2_32(s_col, x);
        tmem_wait_ld();
        // S^T has been read: QK of the tile after next may overwrite this buffer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[s]);
        // does a logit of this row exceed its head's reference max by more than the threshold?
        bool need = false;
        if (valid) {
          const float* thr = sThr + 64 * v + hb;
#pragma unroll
          for (int c = 0; c < 32; ++c) need |= __uint_as_float(x[c]) * cof(hb + c) > thr[c];
        }
        const bool moved = named_bar_or(1, kSmThreads, need);
        if (moved) {
          // the tile's exact per-head maxima: over this warp's 16 rows by a transposing butterfly
          // within each half-warp (lane l ends with heads hb + l % 16 and hb + 16 + l % 16), then
          // over the four warps
          float mx[16];
          {
            // first butterfly step straight from the logits (see half_transpose_pair_step)
            const bool up = (lane & 1) != 0;
#pragma unroll
            for (int k2 = 0; k2 < 16; ++k2) {
              const float a = valid ? __uint_as_float(x[2 * k2]) * cof(hb + 2 * k2) : -INFINITY;
              const float b = valid ? __uint_as_float(x[2 * k2 + 1]) * cof(hb + 2 * k2 + 1) : -INFINITY;
              const float got = __shfl_xor_sync(0xffffffffu, up ? a : b, 1);
              mx[k2] = fmaxf(up ? b : a, got);
            }
          }
          half_transpose_finish<true>(mx, lane);
          sRed[quad * 64 + hb + (lane & 15)] = mx[0];
          sRed[quad * 64 + hb + 16 + (lane & 15)] = mx[8];
          named_bar(1, kSmThreads);
          if (lead) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int h = 32 * hh + lane;
              const float tm = fmaxf(fmaxf(sRed[h], sRed[64 + h]), fmaxf(sRed[128 + h], sRed[192 + h]));
              const float mo = sM[64 * v + h];
              const bool up = tm > mo + kRescaleThreshold;
              const float mn = up ? tm : mo;
              sM[64 * (v ^ 1) + h] = mn;
              sThr[64 * (v ^ 1) + h] = mn + kRescaleThreshold;
              sMe[64 * (v ^ 1) + h] = mn == -INFINITY ? 0.f : mn;
              sAlpha[h] = up ? fast_exp2(mo - mn) : 1.f;  // 0 when the head had no row before
            }
          }
          named_bar(1, kSmThreads);
          v ^= 1;
#pragma unroll
          for (int c = 0; c < 32; ++c) l[c] *= sAlpha[hb + c];
        }
        // P = 2^(logit - max) as fp16 into the slot's RoPE block as [row][64 heads] (128-byte rows,
        // 128-byte swizzle): QK of the tile has finished reading the block (s_full), and the
        // producers do not refill it before PV of the tile releases it. This thread's 32 heads are
        // four 16-byte chunks.
        {
          const float* me = sMe + 64 * v + hb;
          uint8_t* sP = sTile + s * kTileBytes + 8 * kBlk;
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            float p0 = 0.f, p1 = 0.f;
            if (valid) {
              p0 = fast_exp2(fmaf(__uint_as_float(x[2 * c]), cof(hb + 2 * c), -me[2 * c]));
              p1 = fast_exp2(fmaf(__uint_as_float(x[2 * c + 1]), cof(hb + 2 * c + 1), -me[2 * c + 1]));
            }
            l[2 * c] += p0;
            l[2 * c + 1] += p1;
            pk[c] = pack_half2(p0, p1);
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            *reinterpret_cast<uint4*>(sP + sw128_offset(row, 2 * hb + 16 * jj)) =
                make_uint4(pk[4 * jj], pk[4 * jj + 1], pk[4 * jj + 2], pk[4 * jj + 3]);
        }
        // rescale O^T's columns (this warp's 32 dims of each M-tile) when the maxima moved, once PV
        // of the previous tile (and so every earlier one: they complete in order) has finished
        if (moved && jt > ta) {
          if (!wait_pv(i - 1)) *abort_flag = 1;
          tc_fence_after();
#pragma unroll 1
          for (int gq = 0; gq < 4; ++gq) {
            float al[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) al[c] = sAlpha[16 * gq + c];
#pragma unroll 1
            for (int mt = 0; mt < 4; ++mt) {
              uint32_t o[16];
              const uint32_t oa = tmem + lane_base + kColO + 64 * mt + 16 * gq;
              tmem_ld16(oa, o);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * al[c]);
              tmem_st16(oa, o);
            }
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
      // per-head sums: this warp's 16 rows by the transposing butterfly, then the four warps
      {
        float ls[16];
#pragma unroll
        for (int gq = 0; gq < 2; ++gq) {
          float lh[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) lh[c] = l[16 * gq + c];
          half_transpose_pair_step<false>(lh, ls, gq, lane);
        }
        half_transpose_finish<false>(ls, lane);
        sRed[quad * 64 + hb + (lane & 15)] = ls[0];
        sRed[quad * 64 + hb + 16 + (lane & 15)] = ls[8];
      }
      named_bar(1, kSmThreads);
      if (lead) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int h = 32 * hh + lane;
          const float lsum = (sRed[h] + sRed[64 + h]) + (sRed[128 + h] + sRed[192 + h]);
          sInvL[h] = lsum > 0.f ? 1.f / lsum : 0.f;
          if (lbase && h < p.H) lbase[h] = lsum > 0.f ? (sMe[64 * v + h] + log2f(lsum)) * kLn2 : -INFINITY;
        }
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
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll 1
          for (int hh = 0; hh < 2 && 32 * hh < p.H; ++hh) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + kColO + 64 * mt + 32 * hh, o);
            tmem_wait_ld();
            const int d0 = mt * 128 + quad * 32 + (lane & ~1);  // the pair's first dim
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
  if (warp == kQkWarp) {
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
