// kv_quant_append: store new tokens' K/V into their physical blocks.
//
// Addressing follows the paged KV cache of the TFFInfer article (section
// 3.6.4: logical token t -> slot t % block_size of block page_table[t /
// block_size]); the quantiser is the asymmetric per-channel formula of the
// heterogeneous engine article (section 2.6), applied per (physical block,
// kv head, channel) as in its section 2.4. fp8 pools take E4M3 codes (OCP
// 8-bit floating point) with one symmetric scale max|x| / 448 per (physical
// block, kv head, channel), rounded to nearest-even and saturated to +-448
// (the pages name FP8 among the formats to add, TFFInfer section 9.3,
// without fixing a scheme).
//
// This translation unit is compiled with --fmad=false and uses explicitly
// rounded intrinsics so every fp32 step is one IEEE operation in the stated
// order: codes, scales and zero points are bit-exact across implementations.
#include "pa_common.cuh"
#include "pa_kernels.h"

namespace pa {

namespace {

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

// One thread block per (sequence, touched-block slot x, tensor/head z); a
// warp holds 32 / kTokLanes channels x kTokLanes token lanes.
// grid = (X, batch, 2 * Hkv), block = head_dim * kTokLanes threads.
template <int KV, int BS>
__global__ void __launch_bounds__(128 * tok_lanes<BS>()) kv_append_kernel(PoolDev pool, const __nv_bfloat16* k_new,
                                                                    const __nv_bfloat16* v_new,
                                                                    const int32_t* cu_new,
                                                                    const int32_t* ctx_lens,
                                                                    const int32_t* block_table,
                                                                    int32_t max_blocks) {
  constexpr int kTokLanes = tok_lanes<BS>();
  constexpr int NJ = BS / kTokLanes;  // tokens per thread: s = ts + kTokLanes * j
  static_assert(BS % kTokLanes == 0 && kTokLanes >= 1 && kTokLanes <= 32, "token lanes");
  // programmatic stream serialization: start early, touch memory only after
  // the preceding kernel has completed
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.y;
  const int is_v = blockIdx.z & 1;
  const int h = blockIdx.z >> 1;
  const int lane = threadIdx.x & 31;
  const int ts = lane & (kTokLanes - 1);
  const int c = (threadIdx.x >> 5) * (32 / kTokLanes) + (lane / kTokLanes);  // channel
  const int D = pool.head_dim;
  const int Hkv = pool.num_kv_heads;
  const bool lead = threadIdx.x == 0;

  const int32_t c0 = cu_new[b], c1 = cu_new[b + 1];
  const int n_new = c1 - c0;
  if (n_new < 0) {
    if (blockIdx.x == 0 && lead && blockIdx.z == 0) set_error(pool.err, PA_DEVERR_APPEND);
    return;
  }
  if (n_new == 0) return;
  const int ctx = ctx_lens[b];
  const long long total = (long long)ctx + n_new;
  if (ctx < 0 || total > (long long)max_blocks * BS) {
    if (blockIdx.x == 0 && lead && blockIdx.z == 0) set_error(pool.err, PA_DEVERR_SEQ_LEN);
    return;
  }
  const int first_blk = ctx / BS;
  const int last_blk = (int)((total - 1) / BS);
  const __nv_bfloat16* src = is_v ? v_new : k_new;
  uint8_t* codes = is_v ? pool.v : pool.k;
  float* scales = is_v ? pool.v_scale : pool.k_scale;
  int32_t* zps = is_v ? pool.v_zp : pool.k_zp;

  for (int blk = first_blk + blockIdx.x; blk <= last_blk; blk += gridDim.x) {
    const int phys = block_table[(long long)b * max_blocks + blk];
    if (phys < 0 || phys >= pool.num_blocks) {
      if (lead && !is_v && h == 0) set_error(pool.err, PA_DEVERR_BLOCK_TABLE);
      continue;
    }
    const int first = blk * BS;
    const int old_cnt = ctx > first ? min(ctx - first, BS) : 0;
    const int valid = (int)min((long long)BS, total - first);
    const long long page = (long long)phys * Hkv + h;
    // row of the new-token array holding logical position first + s
    const long long row0 = (long long)c0 + first - ctx;

    if (KV == PA_KV_BF16) {
      uint16_t* dst = reinterpret_cast<uint16_t*>(page_of(codes, page, pool.stride));
      const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src);
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int s = ts + kTokLanes * j;
        if (s >= old_cnt && s < valid) dst[s * D + c] = s16[((row0 + s) * Hkv + h) * D + c];
      }
      continue;
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
      continue;
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
}

template <int KV, int BS>
cudaError_t launch_append_t(const PoolDev& pool, const void* k_new, const void* v_new,
                            const int32_t* cu_new, const int32_t* ctx_lens,
                            const int32_t* block_table, int batch, int max_blocks,
                            int blocks_per_seq, cudaStream_t stream) {
  static std::atomic<unsigned long long> ready{0};  // per instantiation, per device
  const cudaError_t e = prepare_kernel(kv_append_kernel<KV, BS>, 0, ready);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks_per_seq, batch, 2 * pool.num_kv_heads);
  cfg.blockDim = dim3(pool.head_dim * tok_lanes<BS>());
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kv_append_kernel<KV, BS>, pool,
                            static_cast<const __nv_bfloat16*>(k_new),
                            static_cast<const __nv_bfloat16*>(v_new), cu_new, ctx_lens, block_table,
                            max_blocks);
}

}  // namespace

cudaError_t launch_append(int kv_dtype, const PoolDev& pool, const void* k_new, const void* v_new,
                          const int32_t* cu_new, const int32_t* ctx_lens,
                          const int32_t* block_table, int batch, int max_blocks,
                          int blocks_per_seq, cudaStream_t stream) {
#define PA_APPEND_CASE(KVT, BSV)                                                              \
  if (kv_dtype == KVT && pool.block_size == BSV)                                              \
    return launch_append_t<KVT, BSV>(pool, k_new, v_new, cu_new, ctx_lens, block_table, batch, \
                                     max_blocks, blocks_per_seq, stream);
  PA_APPEND_CASE(PA_KV_BF16, 16)
  PA_APPEND_CASE(PA_KV_BF16, 32)
  PA_APPEND_CASE(PA_KV_UINT8, 16)
  PA_APPEND_CASE(PA_KV_UINT8, 32)
  PA_APPEND_CASE(PA_KV_UINT4, 16)
  PA_APPEND_CASE(PA_KV_UINT4, 32)
  PA_APPEND_CASE(PA_KV_FP8, 16)
  PA_APPEND_CASE(PA_KV_FP8, 32)
#undef PA_APPEND_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
