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
// The per-block quantising store is append_block (pa_quant.cuh): explicitly
// rounded intrinsics, so every fp32 step is one IEEE operation in the stated
// order and codes, scales and zero points are bit-exact across
// implementations (this translation unit is also compiled with --fmad=false).
#include "pa_common.cuh"
#include "pa_kernels.h"
#include "pa_quant.cuh"

namespace pa {

namespace {

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

    append_block<KV, BS>(pool, page, is_v, c, ts, lane, old_cnt, valid, src, row0, Hkv, h);
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
