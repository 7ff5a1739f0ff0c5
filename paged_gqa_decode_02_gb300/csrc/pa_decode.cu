// Host-side decode entry points: TMA descriptors of a pool, workspace size,
// occupancy, and the launch by KV format (the kernels are instantiated per
// format in pa_decode_<format>.cu).
#include "pa_decode_kernels.cuh"

namespace pa {

bool make_pool_maps(int kv_dtype, const PoolDev& pool, PoolMaps& maps) {
  maps.valid = 0;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  auto encode = reinterpret_cast<CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill)>(fn);
  const bool u8 = kv_dtype != PA_KV_BF16;  // quantised records: rows of 128 bytes
  if (u8 && pool.head_dim != 128) return false;
  const unsigned long long pages = (unsigned long long)pool.num_blocks * pool.num_kv_heads;
  const int rpp = u8 ? (int)(pool.stride / 128) : 2 * pool.block_size;  // rows per record
  const unsigned long long rows = pages * (unsigned long long)rpp;
  if (rows >= (1ull << 31) || rpp > 256) return false;  // row coordinates are int32; box <= 256 rows
  const cuuint64_t gdim[2] = {(cuuint64_t)(u8 ? 128 : pool.head_dim), (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)(u8 ? 128 : pool.head_dim * 2)};
  const cuuint32_t box[2] = {u8 ? 128u : 64u, (cuuint32_t)rpp};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(&maps.rec, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                      (void*)pool.k, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  maps.rows_per_page = rpp;
  maps.valid = 1;
  return true;
}

size_t decode_workspace_bytes(int num_ctas, int batch, int num_kv_heads, int group, int head_dim) {
  const size_t slots = (size_t)num_ctas + (size_t)batch * num_kv_heads;
  return align256(sizeof(unsigned long long) * (size_t)batch * num_kv_heads) +
         align256(sizeof(int32_t) * ((size_t)batch + 1)) + align256(sizeof(float) * slots * group) +
         align256(sizeof(float) * slots * group * head_dim);
}

int decode_ctas_per_sm(int kv_dtype, int block_size, int head_dim, int group, bool tensor_cores) {
  size_t smem = kv_dtype == PA_KV_BF16
                    ? (tensor_cores ? smem_bytes_kv<PA_KV_BF16, true>(head_dim, block_size, group)
                                    : smem_bytes_kv<PA_KV_BF16, false>(head_dim, block_size, group))
                : kv_dtype == PA_KV_UINT8
                    ? (tensor_cores && head_dim == 128 ? smem_bytes_kv<PA_KV_UINT8, true>(head_dim, block_size, group)
                                                       : smem_bytes_kv<PA_KV_UINT8, false>(head_dim, block_size, group))
                : kv_dtype == PA_KV_UINT4
                    ? (tensor_cores && head_dim == 128 ? smem_bytes_kv<PA_KV_UINT4, true>(head_dim, block_size, group)
                                                       : smem_bytes_kv<PA_KV_UINT4, false>(head_dim, block_size, group))
                    : (tensor_cores && head_dim == 128 ? smem_bytes_kv<PA_KV_FP8, true>(head_dim, block_size, group)
                                                       : smem_bytes_kv<PA_KV_FP8, false>(head_dim, block_size, group));
  const size_t per_sm = 227 * 1024;
  int n = (int)(per_sm / (smem + 1024));
  return n < 1 ? 1 : (n > 4 ? 4 : n);
}

cudaError_t launch_decode(int kv_dtype, const PoolDev& pool, const PoolMaps& maps, const void* q,
                          const int32_t* block_table, const int32_t* seq_lens, float* out,
                          void* workspace, DecodeLaunch& L, cudaStream_t stream) {
  if (kv_dtype == PA_KV_BF16) return launch_decode_bf16(pool, maps, q, block_table, seq_lens, out, workspace, L, stream);
  if (kv_dtype == PA_KV_UINT8) return launch_decode_uint8(pool, maps, q, block_table, seq_lens, out, workspace, L, stream);
  if (kv_dtype == PA_KV_UINT4) return launch_decode_uint4(pool, maps, q, block_table, seq_lens, out, workspace, L, stream);
  if (kv_dtype == PA_KV_FP8) return launch_decode_fp8(pool, maps, q, block_table, seq_lens, out, workspace, L, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
