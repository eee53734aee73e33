// append.cu — FP8 KV append: new tokens into the paged 656-byte MLA rows and the indexer keys.
//
// [P1] "vLLM v0.32.0 GLM-5.3 サービング ...", section 「数字がうまくいく理由」: a token's MLA KV is a
// 656-byte FP8 row and its indexer key is 128 FP8 values with a 4-byte scale. Row layout
// [512 x e4m3][4 x fp32 group scales][64 x bf16 RoPE]; key layout e4m3 [Di] + fp32 scale. For each
// 128-dim latent group and for each key, in IEEE binary32:
//   scale = max(amax / 448, 2^-14),   code = e4m3(x / scale)  (round to nearest even, saturating)
// with x the bf16 input. The divisions are IEEE-rounded (not approximate) and the conversion is
// the native cvt.rn.satfinite, so the codes are exactly those of the binary32 definition.
//
// One warp per token: lane l quantises latent values 16 l .. 16 l + 15 (a 128-dim group is 8 lanes,
// its amax three shuffles) and writes them as one 16-byte store; lanes 0-7 copy the RoPE part; the
// key is spread over the whole warp. Warps stride over the tokens with the next token's inputs
// loaded while the current one is quantised. Memory-bound: 2,208 bytes of traffic per token.
#include "common.cuh"

namespace hs {
namespace append {

constexpr int kWarps = 8;
constexpr int kCtasPerSm = 4;  // registers for the prefetched token: 64 a thread
constexpr float kScaleFloor = 6.103515625e-05f;  // 2^-14

struct Params {
  int32_t T, B, Di, bt_stride;
  const uint16_t* latent;     // bf16 [T, 512] or null
  const uint16_t* rope;       // bf16 [T, 64]
  const uint16_t* key;        // bf16 [T, Di] or null
  const int32_t* token_req;
  const int32_t* token_pos;
  const int32_t* bt;
  uint8_t* kv;
  int64_t R;
  uint8_t* k_cache;
  float* k_scale;
  int64_t nblk;
  int32_t* err;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// two binary32 values -> two e4m3 codes, `first` in the lower byte
__device__ __forceinline__ uint32_t e4m3x2(float first, float second) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(second), "f"(first));
  return d;
}

__device__ __forceinline__ float quant_scale(float amax) {
  return fmaxf(__fdiv_rn(amax, 448.0f), kScaleFloor);
}

// One token's inputs as a lane holds them: latent values 16 l .. 16 l + 15, RoPE piece l (lanes
// 0-7), key values (Di / 32 per lane), and the token's request and position.
struct TokenIn {
  uint4 la, lb, rp;
  uint2 k;
  int32_t r, pos;
};

__device__ __forceinline__ TokenIn load_token(const Params& p, int64_t t, int lane) {
  TokenIn in;
  in.r = p.token_req[t];
  in.pos = p.token_pos[t];
  if (p.latent) {
    const uint4* src = reinterpret_cast<const uint4*>(p.latent + t * HS_D_LATENT) + 2 * lane;
    in.la = src[0];
    in.lb = src[1];
    if (lane < 8) in.rp = reinterpret_cast<const uint4*>(p.rope + t * HS_D_ROPE)[lane];
  }
  if (p.key) {
    if (p.Di == 128) {
      in.k = reinterpret_cast<const uint2*>(p.key + t * 128)[lane];
    } else {
      in.k.x = reinterpret_cast<const uint32_t*>(p.key + t * 64)[lane];
      in.k.y = 0u;
    }
  }
  return in;
}

__global__ void __launch_bounds__(32 * kWarps, kCtasPerSm) append_kernel(const Params p) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kWarps;
  int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= p.T) return;
  TokenIn cur = load_token(p, t, lane);
  for (; t < p.T; t += stride) {
    // the next token's loads are in flight while this one is quantised and stored
    TokenIn nxt;
    if (t + stride < p.T) nxt = load_token(p, t + stride, lane);
    const int32_t r = cur.r, pos = cur.pos;
    bool ok = !(r < 0 || r >= p.B || pos < 0 || pos / 64 >= p.bt_stride);
    if (!ok) {
      if (lane == 0) flag_error(p.err, HS_FLAG_BAD_INDEX);
    } else {
      const int32_t blk = p.bt[(int64_t)r * p.bt_stride + pos / 64];
      const int64_t row = (int64_t)blk * 64 + (pos & 63);
      if (blk < 0 || (p.latent && row >= p.R) || (p.key && blk >= p.nblk)) {
        if (lane == 0) flag_error(p.err, HS_FLAG_BAD_BLOCK);
      } else {
        if (p.latent) {
          const uint32_t w[8] = {cur.la.x, cur.la.y, cur.la.z, cur.la.w, cur.lb.x, cur.lb.y, cur.lb.z, cur.lb.w};
          float x[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            x[2 * i] = bf16_lo(w[i]);
            x[2 * i + 1] = bf16_hi(w[i]);
          }
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          const float s = quant_scale(amax);
          uint32_t c[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            c[i] = e4m3x2(__fdiv_rn(x[4 * i], s), __fdiv_rn(x[4 * i + 1], s)) |
                   (e4m3x2(__fdiv_rn(x[4 * i + 2], s), __fdiv_rn(x[4 * i + 3], s)) << 16);
          uint8_t* dst = p.kv + row * HS_KV_ROW_BYTES;
          *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(c[0], c[1], c[2], c[3]);
          if ((lane & 7) == 0) *reinterpret_cast<float*>(dst + HS_D_LATENT + 4 * (lane >> 3)) = s;
          if (lane < 8) reinterpret_cast<uint4*>(dst + HS_D_LATENT + 16)[lane] = cur.rp;
        }
        if (p.key) {
          const float x0 = bf16_lo(cur.k.x), x1 = bf16_hi(cur.k.x);
          const float x2 = p.Di == 128 ? bf16_lo(cur.k.y) : 0.f, x3 = p.Di == 128 ? bf16_hi(cur.k.y) : 0.f;
          float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          const float s = quant_scale(amax);
          const uint32_t lo = e4m3x2(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
          if (p.Di == 128) {
            const uint32_t hi = e4m3x2(__fdiv_rn(x2, s), __fdiv_rn(x3, s));
            reinterpret_cast<uint32_t*>(p.k_cache + row * 128)[lane] = lo | (hi << 16);
          } else {
            reinterpret_cast<uint16_t*>(p.k_cache + row * 64)[lane] = (uint16_t)lo;
          }
          if (lane == 0) p.k_scale[row] = s;
        }
      }
    }
    cur = nxt;
  }
}

}  // namespace append

cudaError_t launch_append(const hs_kv_append_args* a, int sms, cudaStream_t stream) {
  using namespace append;
  Params p;
  p.T = a->T;
  p.B = a->B;
  p.Di = a->Di;
  p.bt_stride = a->bt_stride;
  p.latent = reinterpret_cast<const uint16_t*>(a->latent);
  p.rope = reinterpret_cast<const uint16_t*>(a->rope);
  p.key = reinterpret_cast<const uint16_t*>(a->index_key);
  p.token_req = a->token_req;
  p.token_pos = a->token_pos;
  p.bt = a->block_table;
  p.kv = a->kv_pool;
  p.R = a->R;
  p.k_cache = a->k_cache;
  p.k_scale = a->k_scale;
  p.nblk = a->nblk;
  p.err = a->err_flag;
  if (a->T == 0) return cudaSuccess;
  int64_t blocks = ((int64_t)a->T + kWarps - 1) / kWarps;
  // two waves of resident CTAs (measured faster than one); warps stride over the rest
  if (blocks > 2LL * kCtasPerSm * sms) blocks = 2LL * kCtasPerSm * sms;
  append_kernel<<<(unsigned)blocks, 32 * kWarps, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace hs
