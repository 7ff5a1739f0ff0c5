// The per-block quantising store of kv_quant_append, shared by the append
// kernel and the fused decode step (a decode kernel that stores each
// sequence's new token itself). Every fp32 step is an explicitly rounded
// intrinsic, so the codes, scales and zero points are the same bit for bit
// whatever the translation unit's contraction flags.
//
// The quantiser is the asymmetric per-channel formula of the heterogeneous
// engine article (section 2.6), applied per (physical block, kv head,
// channel) as in its section 2.4; fp8 pools take E4M3 codes with one
// symmetric scale max|x| / 448 per (physical block, kv head, channel),
// rounded to nearest-even and saturated (the pages name FP8 among the formats
// to add, TFFInfer section 9.3, without fixing a scheme).
#pragma once

#include "pa_common.cuh"

namespace pa {

__device__ __forceinline__ int32_t sat_rint_i32(float x) {
  // rintf then convert; cvt.rni.s32.f32 saturates and maps NaN to 0.
  return __float2int_rn(x);
}

template <int KV>
__device__ __forceinline__ int read_code(const uint8_t* page_codes, int D, int slot, int c) {
  if (KV == PA_KV_UINT8) return page_codes[slot * D + c];
  const uint8_t byte = page_codes[slot * (D / 2) + c / 2];
  return (c & 1) ? (byte >> 4) : (byte & 15);
}

// Lanes per channel: the tokens of a block are spread over tok_lanes<BS>()
// lanes (token s goes to lane s % lanes), 8 tokens a thread, so a thread
// quantises 8 tokens instead of all BS and the per-channel min / max is a
// shuffle reduction over the lanes. Eight keeps a decode step's append (one
// block per sequence, K and V of every kv head) within one wave of threads:
// batch 64 x 8 kv heads x 2 x 256 threads for 16-token blocks.
template <int BS>
constexpr int tok_lanes() {
  return BS / 8;
}

// min / max over the lanes of one channel, with the sequential rule of the
// quantiser: the running value starts at token 0 and a token replaces it only
// when it compares below (above); so a NaN counts only as token 0, and the
// other values give the same result in any order (+-0 ties change neither
// the scale nor the zero point).
template <int TL>
__device__ __forceinline__ void channel_min_max(float& mn, float& mx, float v0) {
#pragma unroll
  for (int o = 1; o < TL; o <<= 1) {
    const float a = __shfl_xor_sync(0xffffffffu, mn, o), b = __shfl_xor_sync(0xffffffffu, mx, o);
    if (a < mn) mn = a;
    if (b > mx) mx = b;
  }
  if (v0 != v0) mn = mx = v0;  // token 0 is NaN
}

// Store one channel's share of the block `page` (one kv head's K or V block)
// after `old_cnt` stored tokens and up to `valid` tokens: the calling thread
// is token lane ts (tokens s = ts + lanes * j) of channel c. The lanes of a
// channel must be adjacent lanes of one warp and every lane of the warp must
// call (the min / max and the uint4 byte pairing are shuffles). New token s
// comes from src[((row0 + s) * Hkv + h) * D + c] (bf16).
template <int KV, int BS>
__device__ __forceinline__ void append_block(const PoolDev& pool, long long page, int is_v, int c, int ts,
                                             int lane, int old_cnt, int valid, const __nv_bfloat16* src,
                                             long long row0, int Hkv, int h) {
  constexpr int kTokLanes = tok_lanes<BS>();
  constexpr int NJ = BS / kTokLanes;  // tokens per thread: s = ts + kTokLanes * j
  static_assert(BS % kTokLanes == 0 && kTokLanes >= 1 && kTokLanes <= 32, "token lanes");
  const int D = pool.head_dim;
  uint8_t* codes = is_v ? pool.v : pool.k;
  float* scales = is_v ? pool.v_scale : pool.k_scale;
  int32_t* zps = is_v ? pool.v_zp : pool.k_zp;
  if (KV == PA_KV_BF16) {
    uint16_t* dst = reinterpret_cast<uint16_t*>(page_of(codes, page, pool.stride));
    const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int s = ts + kTokLanes * j;
      if (s >= old_cnt && s < valid) dst[s * D + c] = s16[((row0 + s) * Hkv + h) * D + c];
    }
    return;
  }

  if (KV == PA_KV_FP8) {
    // stored tokens enter as float(value(code)) * scale, new ones as bf16
    uint8_t* pc = page_of(codes, page, pool.stride);
    float* psc = page_of(scales, page, pool.stride);
    const float old_scale = psc[c];
    float vals[NJ];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int s = ts + kTokLanes * j;
      float x = 0.0f;
      if (s < old_cnt) {
        x = __fmul_rn(e4m3_to_float(pc[s * D + c]), old_scale);
      } else if (s < valid) {
        x = __bfloat162float(src[((row0 + s) * Hkv + h) * D + c]);
      }
      vals[j] = x;
      if (s < valid && fabsf(x) > amax) amax = fabsf(x);
    }
#pragma unroll
    for (int o = 1; o < kTokLanes; o <<= 1) {
      const float a = __shfl_xor_sync(0xffffffffu, amax, o);
      if (a > amax) amax = a;
    }
    float scale = __fdiv_rn(amax, 448.0f);
    if (!(scale > 0.0f)) scale = 1.0f;
    // (a channel's lanes, and so every reader of its old codes and scale,
    // are in one warp: the shuffles above ordered those reads first)
    __syncwarp();
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int s = ts + kTokLanes * j;
      if (s < valid) pc[s * D + c] = float_to_e4m3(__fdiv_rn(vals[j], scale));
    }
    if (ts == 0) psc[c] = scale;
    return;
  }

  constexpr int L = (KV == PA_KV_UINT4) ? 15 : 255;
  uint8_t* pc = page_of(codes, page, pool.stride);
  float* psc = page_of(scales, page, pool.stride);
  int32_t* pzp = page_of(zps, page, pool.stride);
  float vals[NJ];
  const float old_scale = psc[c];
  const int32_t old_zp = pzp[c];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int s = ts + kTokLanes * j;
    float x = 0.0f;
    if (s < old_cnt) {
      const int32_t diff = read_code<KV>(pc, D, s, c) - old_zp;
      x = __fmul_rn(__int2float_rn(diff), old_scale);
    } else if (s < valid) {
      x = __bfloat162float(src[((row0 + s) * Hkv + h) * D + c]);
    }
    vals[j] = x;
    if (s < valid) {
      if (x < mn) mn = x;
      if (x > mx) mx = x;
    }
  }
  // token 0 (always valid) is j = 0 of the channel's lane ts = 0
  channel_min_max<kTokLanes>(mn, mx, __shfl_sync(0xffffffffu, vals[0], lane & ~(kTokLanes - 1)));
  const float r = __fsub_rn(mx, mn);
  float scale = __fdiv_rn(r, (float)L);
  if (!(scale > 0.0f)) {
    scale = __fdiv_rn(fabsf(mn), (float)L);
    if (!(scale > 0.0f)) scale = 1.0f;
  }
  const int32_t zp = sat_rint_i32(rintf(__fdiv_rn(-mn, scale)));
  int code[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    long long t = (long long)sat_rint_i32(rintf(__fdiv_rn(vals[j], scale))) + (long long)zp;
    t = t < 0 ? 0 : (t > L ? L : t);
    code[j] = (int)t;
  }
  // the lanes of a channel, and of the channel sharing its uint4 bytes, are
  // in one warp and have read their old codes, scale and zero point (the
  // shuffles above ordered those reads before these stores)
  __syncwarp();
  if (KV == PA_KV_UINT8) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int s = ts + kTokLanes * j;
      if (s < valid) pc[s * D + c] = (uint8_t)code[j];
    }
  } else {
    // channels 2i (low nibble) and 2i+1 (high nibble) of one byte: the odd
    // channel's lane is kTokLanes lanes up
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int s = ts + kTokLanes * j;
      const int other = __shfl_xor_sync(0xffffffffu, code[j], kTokLanes);
      if (s < valid && (c & 1) == 0) pc[s * (D / 2) + c / 2] = (uint8_t)(code[j] | (other << 4));
    }
  }
  if (ts == 0) {
    psc[c] = scale;
    pzp[c] = zp;
  }
}

}  // namespace pa
