// Decode kernels for bf16 pools: one translation unit per KV format, so the
// formats compile in parallel (the kernels live in pa_decode_kernels.cuh).
#include "pa_decode_kernels.cuh"

namespace pa {

cudaError_t launch_decode_bf16(const PoolDev& pool, const PoolMaps& maps, const void* q,
                               const int32_t* block_table, const int32_t* seq_lens, float* out,
                               void* workspace, DecodeLaunch& L, cudaStream_t stream) {
  return launch_decode_kv<PA_KV_BF16>(pool, maps, q, block_table, seq_lens, out, workspace, L, stream);
}

}  // namespace pa
