// mla.cu — sparse MLA forward in MQA form on tcgen05.
//
// [P1] "vLLM v0.32.0 GLM-5.3 サービング ...", sections 「再現方法と必要なフラグ」 and
// 「数字がうまくいく理由」: each query gathers its selected 656-byte FP8 latent rows once and every
// row serves all 64 heads; QK runs over 576 dims (512 latent + 64 RoPE), PV over the 512 latent
// dims. Per query token t, head h, over the valid entries i of idx[t, :]:
//   logit_i = scale * <q[t,h,:], [latent_i, rope_i]>,  out = softmax(logit) . latent,  lse = ln sum exp.
//
// One CTA per query token (416 threads):
//   warps 0-7   gather 64 rows per tile (thread = one row x one 128-element scale group), with
//               16-byte loads, dequantise latent = e4m3 * group scale to bf16 and write it, with
//               the bf16 RoPE part, into a 128-byte-swizzled [dim block][row] tile (2 stages);
//   warp 8      allocates TMEM and issues the MMAs:
//                 S   = Q . K^T        M = 64 heads, N = 64 rows, K = 576  (A = Q, B = tile)
//                 O^T += V^T . P^T     M = 128 dims (x4), N = 64 heads, K = 64 rows
//               The same tile serves as the K-major B of the first and, read MN-major, as the A of
//               the second, so it is dequantised once;
//   warps 9-12  online softmax: each of the 64 head threads owns one row of S (thread-local max
//               and sum); P goes to shared memory as bf16. O^T lives in TMEM and is rescaled only
//               when a head's running max grows by more than 2^8 (lazy rescaling); the final pass
//               divides by the row sum and writes bf16.
// TMEM: columns 0-127 hold two S buffers (64-row layout), 128-383 hold O^T.
#include "common.cuh"

namespace hs {
namespace mla {

constexpr int kRows = 64;
constexpr int kProdWarps = 8;
constexpr int kMmaWarp = kProdWarps;
constexpr int kSmThreads = 128;
constexpr int kThreads = 32 * (kProdWarps + 1 + 4);
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;
constexpr int kBlk = 8192;                 // one [64 rows][128 B] swizzled block
constexpr int kQBytes = 9 * kBlk;          // 64 heads x 576 bf16
constexpr int kStageBytes = 9 * kBlk;      // 64 rows x (512 latent + 64 rope) bf16
constexpr int kPBytes = kBlk;              // 64 heads x 64 rows bf16
constexpr int kOffQ = 0;
constexpr int kOffStage = kQBytes;
constexpr int kOffP = kOffStage + 2 * kStageBytes;
constexpr int kOffValid = kOffP + kPBytes;          // uint8 [2][64]
constexpr int kOffAlpha = kOffValid + 128;          // float [64]
constexpr int kOffInvL = kOffAlpha + 256;           // float [64]
constexpr int kOffBar = kOffInvL + 256;             // 12 barriers
constexpr int kOffMisc = kOffBar + 12 * 8;          // tmem base, abort
constexpr int kSmem = kOffMisc + 16 + 1024;
constexpr float kRescaleThreshold = 8.0f;           // log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Params {
  int32_t T, H, k;
  const uint8_t* kv;
  int64_t R;
  const int32_t* idx;
  const int32_t* bt;
  int32_t bt_stride;
  const int32_t* token_req;
  float scale_log2;  // softmax_scale * log2(e)
  __nv_bfloat16* out;
  float* lse;
  int32_t* err;
};

__device__ __forceinline__ uint32_t dequant2(uint16_t codes, float scale) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)codes, __NV_E4M3);
  float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
  return *reinterpret_cast<uint32_t*>(&b);
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap map_q, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sStage = smem + kOffStage;
  uint8_t* sP = smem + kOffP;
  uint8_t* sValid = smem + kOffValid;
  float* sAlpha = (float*)(smem + kOffAlpha);
  float* sInvL = (float*)(smem + kOffInvL);
  uint64_t* bars = (uint64_t*)(smem + kOffBar);
  uint64_t* full = bars + 0;      // [2] producers -> MMA, softmax
  uint64_t* empty = bars + 2;     // [2] PV done with the stage -> producers
  uint64_t* s_full = bars + 4;    // [2] QK done -> softmax
  uint64_t* s_free = bars + 6;    // [2] softmax read S -> MMA
  uint64_t* p_ready = bars + 8;   // softmax wrote P (and corrected O) -> MMA
  uint64_t* pv_done = bars + 9;   // PV done -> softmax
  uint64_t* q_full = bars + 10;
  uint64_t* mma_done = bars + 11;
  uint32_t* misc = (uint32_t*)(smem + kOffMisc);
  volatile uint32_t* abort_flag = misc + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x;
  const int k = p.k;
  const int ntiles = (k + kRows - 1) / kRows;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full[i], kProdWarps);
      mbar_init(&empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
    }
    mbar_init(p_ready, 4);
    mbar_init(pv_done, 1);
    mbar_init(q_full, 1);
    mbar_init(mma_done, 1);
    mbar_fence_init();
    misc[1] = 0;
  }
  if (warp == kMmaWarp) tmem_alloc(&misc[0], 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp < kProdWarps) {
    // ================================================================ gather + dequantise ======
    const int row = tid >> 2;   // 0..63
    const int grp = tid & 3;    // 128-element scale group
    const int req = p.bt ? p.token_req[t] : 0;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i & 1;
      int go = 1;
      if (lane == 0) go = !*abort_flag && mbar_wait(&empty[s], ((uint32_t)(i >> 1) & 1u) ^ 1u, p.err);
      if (!__shfl_sync(0xffffffffu, go, 0)) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      const int e = i * kRows + row;
      bool valid = false;
      int64_t prow = 0;
      if (e < k) {
        const int32_t j = p.idx[(int64_t)t * k + e];
        if (j >= 0) {
          if (p.bt) {
            const int32_t page = j >> 6;
            int32_t blk = -1;
            if (page < p.bt_stride) blk = p.bt[(int64_t)req * p.bt_stride + page];
            prow = (int64_t)blk * 64 + (j & 63);
            valid = blk >= 0 && prow < p.R;
          } else {
            prow = j;
            valid = prow < p.R;
          }
          if (!valid && grp == 0) flag_error(p.err, HS_FLAG_BAD_INDEX);
        }
      }
      uint4 lat[8], rope[2];
      float scale = 0.f;
      if (valid) {
        const uint8_t* src = p.kv + prow * HS_KV_ROW_BYTES;
        const uint4* l4 = reinterpret_cast<const uint4*>(src + grp * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) lat[c] = __ldg(l4 + c);
        scale = __ldg(reinterpret_cast<const float*>(src + HS_D_LATENT) + grp);
        const uint4* r4 = reinterpret_cast<const uint4*>(src + HS_D_LATENT + 16);
        rope[0] = __ldg(r4 + 2 * grp);
        rope[1] = __ldg(r4 + 2 * grp + 1);
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) lat[c] = make_uint4(0, 0, 0, 0);
        rope[0] = rope[1] = make_uint4(0, 0, 0, 0);
      }
      uint8_t* st = sStage + s * kStageBytes;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        // 16 latent dims grp*128 + c*16 .. +15 -> dim block 2*grp + c/4, 16-byte chunks 2*(c%4), +1
        uint8_t* blk = st + (2 * grp + (c >> 2)) * kBlk;
        const int ch = (c & 3) * 2;
        uint4 lo, hi;
        lo.x = dequant2((uint16_t)(lat[c].x & 0xFFFF), scale);
        lo.y = dequant2((uint16_t)(lat[c].x >> 16), scale);
        lo.z = dequant2((uint16_t)(lat[c].y & 0xFFFF), scale);
        lo.w = dequant2((uint16_t)(lat[c].y >> 16), scale);
        hi.x = dequant2((uint16_t)(lat[c].z & 0xFFFF), scale);
        hi.y = dequant2((uint16_t)(lat[c].z >> 16), scale);
        hi.z = dequant2((uint16_t)(lat[c].w & 0xFFFF), scale);
        hi.w = dequant2((uint16_t)(lat[c].w >> 16), scale);
        *reinterpret_cast<uint4*>(blk + sw128_offset(row, ch * 16)) = lo;
        *reinterpret_cast<uint4*>(blk + sw128_offset(row, ch * 16 + 16)) = hi;
      }
      uint8_t* rb = st + 8 * kBlk;
      *reinterpret_cast<uint4*>(rb + sw128_offset(row, (2 * grp) * 16)) = rope[0];
      *reinterpret_cast<uint4*>(rb + sw128_offset(row, (2 * grp + 1) * 16)) = rope[1];
      if (grp == 0) sValid[s * kRows + row] = valid ? 1 : 0;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[s]);
    }
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer ================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(64, kRows, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(128, 64, 1, 0);
      prefetch_tensormap(&map_q);
      mbar_arrive_expect_tx(q_full, kQBytes);
#pragma unroll 1
      for (int db = 0; db < 9; ++db) tma_load_2d(sQ + db * kBlk, &map_q, q_full, db * 64, t * p.H);
      const uint32_t q_addr = smem_u32(sQ), st_addr = smem_u32(sStage), p_addr = smem_u32(sP);
      bool ok = mbar_wait(q_full, 0, p.err);
      auto issue_pv = [&](int j) -> bool {
        if (!mbar_wait(p_ready, (uint32_t)j & 1u, p.err)) return false;
        tc_fence_after();
        const uint32_t sa = st_addr + (uint32_t)((j & 1) * kStageBytes);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = smem_desc(sa + (uint32_t)(2 * mt * kBlk + kk * 2048), kBlk, 1024, 2);
            const uint64_t b = smem_desc(p_addr + kk * 32, 16, 1024, 2);
            mma_bf16_ss(tmem + kColO + 64 * mt, a, b, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(pv_done);
        mma_commit(&empty[j & 1]);
        return true;
      };
#pragma unroll 1
      for (int i = 0; i < ntiles && ok; ++i) {
        const int s = i & 1;
        const uint32_t ph = (uint32_t)(i >> 1) & 1u;
        if (!mbar_wait(&full[s], ph, p.err) || !mbar_wait(&s_free[s], ph ^ 1u, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = st_addr + (uint32_t)(s * kStageBytes);
        const uint32_t d = tmem + kColS + 64 * s;
#pragma unroll
        for (int db = 0; db < 9; ++db) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = smem_desc(q_addr + db * kBlk + kk * 32, 16, 1024, 2);
            const uint64_t b = smem_desc(sa + db * kBlk + kk * 32, 16, 1024, 2);
            mma_bf16_ss(d, a, b, idesc_qk, (db | kk) != 0 ? 1u : 0u);
          }
        }
        mma_commit(&s_full[s]);
        if (i >= 1 && !issue_pv(i - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && ntiles > 0) ok = issue_pv(ntiles - 1);
      if (!ok) *abort_flag = 1;
      mma_commit(mma_done);
      mbar_wait(mma_done, 0, p.err);
      mbar_wait(q_full, 0, p.err);
    }
  } else {
    // ================================================================ softmax / epilogue ========
    const int quad = warp & 3;
    const int h = quad * 16 + lane;           // head row owned by lanes 0..15
    const bool head_thread = lane < 16;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = true;
#pragma unroll 1
    for (int i = 0; i < ntiles; ++i) {
      const int s = i & 1;
      const uint32_t ph = (uint32_t)(i >> 1) & 1u;
      // every exit decision is taken by all four softmax warps together (no partial barriers)
      bool w = !*abort_flag && warp_wait(&s_full[s], ph, p.err, lane) && warp_wait(&full[s], ph, p.err, lane);
      if (named_bar_or(1, kSmThreads, !w)) {
        ok = false;
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      uint32_t xr[64];
      tmem_ld32(tmem + lane_base + kColS + 64 * s, *reinterpret_cast<uint32_t(*)[32]>(&xr[0]));
      tmem_ld32(tmem + lane_base + kColS + 64 * s + 32, *reinterpret_cast<uint32_t(*)[32]>(&xr[32]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[s]);
      // logits in log2 units, in place (as float bits); masked rows become -inf
      float mt = -INFINITY;
      {
        const uint4* vld4 = reinterpret_cast<const uint4*>(sValid + s * kRows);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint4 vv = vld4[q4];
          const uint32_t w4[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int col = q4 * 16 + c;
            const bool valid = (w4[c >> 2] >> (8 * (c & 3))) & 0xFFu;
            const float v = valid ? __uint_as_float(xr[col]) * p.scale_log2 : -INFINITY;
            xr[col] = __float_as_uint(v);
            mt = fmaxf(mt, v);
          }
        }
      }
      if (!head_thread) mt = -INFINITY;
      const bool need = mt > m_ref + kRescaleThreshold;
      const float m_new = need ? mt : m_ref;
      w = i == 0 || warp_wait(pv_done, (uint32_t)(i - 1) & 1u, p.err, lane);
      if (named_bar_or(1, kSmThreads, !w)) {
        ok = false;
        *abort_flag = 1;
        break;
      }
      const bool any = named_bar_or(1, kSmThreads, need && i > 0);
      const float alpha = need ? exp2f(m_ref - m_new) : 1.f;
      l_sum *= alpha;
      m_ref = m_new;
      if (head_thread) {
        float psum = 0.f;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t pk[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = ch * 8 + 2 * u;
            const float x0 = __uint_as_float(xr[c]), x1 = __uint_as_float(xr[c + 1]);
            const float p0 = x0 == -INFINITY ? 0.f : exp2f(x0 - m_ref);
            const float p1 = x1 == -INFINITY ? 0.f : exp2f(x1 - m_ref);
            psum += p0 + p1;
            __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
            pk[u] = *reinterpret_cast<uint32_t*>(&b2);
          }
          *reinterpret_cast<uint4*>(sP + sw128_offset(h, ch * 16)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        l_sum += psum;
      }
      // rescale O^T columns of the heads whose reference max moved (after P: fewer live registers)
      if (any) {
        if (head_thread) sAlpha[h] = alpha;
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
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready);
    }
    // ---- final normalisation and output ----
    if (ok && ntiles > 0) {
      const bool w = warp_wait(pv_done, (uint32_t)(ntiles - 1) & 1u, p.err, lane);
      if (named_bar_or(1, kSmThreads, !w)) {
        ok = false;
        *abort_flag = 1;
      }
    }
    tc_fence_after();
    if (head_thread) {
      sInvL[h] = l_sum > 0.f ? 1.f / l_sum : 0.f;
      if (p.lse && h < p.H)
        p.lse[(int64_t)t * p.H + h] = l_sum > 0.f ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
    }
    named_bar(1, kSmThreads);
    if (ok && ntiles > 0) {
#pragma unroll 1
      for (int part = 0; part < 8; ++part) {  // 4 M-tiles (128 dims each) x 2 halves of 32 heads
        uint32_t o[32];
        const int mt4 = part >> 1, h0 = 32 * (part & 1);
        tmem_ld32(tmem + lane_base + kColO + 64 * mt4 + h0, o);
        tmem_wait_ld();
        const int d = mt4 * 128 + quad * 32 + lane;
        __nv_bfloat16* dst = p.out + ((int64_t)t * p.H + h0) * HS_D_LATENT + d;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (h0 + c < p.H)
            dst[(int64_t)c * HS_D_LATENT] = __float2bfloat16_rn(__uint_as_float(o[c]) * sInvL[h0 + c]);
      }
    } else if (ntiles == 0) {
      for (int hh = 0; hh < p.H; ++hh)
        for (int d = quad * 32 + lane; d < HS_D_LATENT; d += 128)
          p.out[((int64_t)t * p.H + hh) * HS_D_LATENT + d] = __float2bfloat16_rn(0.f);
    }
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace mla

cudaError_t launch_mla(const hs_mla_args* a, cudaStream_t stream, const char** why) {
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
  p.kv = a->kv_pool;
  p.R = a->R;
  p.idx = a->idx;
  p.bt = a->block_table;
  p.bt_stride = a->bt_stride;
  p.token_req = a->token_req;
  p.scale_log2 = a->softmax_scale * kLog2e;
  p.out = reinterpret_cast<__nv_bfloat16*>(a->out);
  p.lse = a->lse;
  p.err = a->err_flag;
  if (a->T == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  mla_kernel<<<a->T, kThreads, kSmem, stream>>>(mq, p);
  return cudaGetLastError();
}

}  // namespace hs
