// Internal launch interface between the C ABI (pa_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

struct PoolDev;
struct PoolMaps;

// Geometry of the decode launch: how the (sequence, kv head, block) work
// list is cut into partitions and where partial results go.
struct DecodeLaunch {
  int num_ctas;         // partitions = thread blocks of the decode kernel
  int group;            // Hq / Hkv
  int num_q_heads;
  int batch;
  int max_blocks;
  float scale_log2;     // softmax_scale * log2(e)
  bool tensor_cores;    // bf16 pools: mma consumer fed by swizzled 2-D TMA
  bool fused_combine;   // merge split units inside the decode kernel
  bool early_plan;      // plan before waiting on the preceding kernel
  unsigned long long epoch;  // per-call tag of the merge tickets (40 bits, never 0)
  int unit_cost;        // phantom pages per (sequence, kv head) unit in the partition
  // several query tokens per sequence (n_q > 1): batch counts virtual
  // sequences (sequence x column group, n_cg per sequence), group is
  // tpg * g_heads columns (tpg query tokens x g_heads heads)
  int n_q;
  int n_cg;
  int tpg;
  int g_heads;
  // fused decode step (n_q == 1): store each sequence's last token from
  // k_new / v_new (bf16 [batch][Hkv][D]) before attending; null otherwise
  const void* k_new;
  const void* v_new;
  // workspace carve-up
  int32_t* pre_cost;    // [batch + 1] per-head cost-line prefix of the sequences
  float* part_o;        // [num_ctas + batch*Hkv][group][D]
  float* part_lse;      // [num_ctas + batch*Hkv][group]
};

cudaError_t launch_append(int kv_dtype, const PoolDev& pool, const void* k_new, const void* v_new,
                          const int32_t* cu_new, const int32_t* ctx_lens,
                          const int32_t* block_table, int batch, int max_blocks,
                          int blocks_per_seq, cudaStream_t stream);

// Bytes of workspace for a given partition count.
size_t decode_workspace_bytes(int num_ctas, int batch, int num_kv_heads, int group, int head_dim);

// Thread blocks of the decode kernel that fit on one SM for this shape.
int decode_ctas_per_sm(int kv_dtype, int block_size, int head_dim, int group, bool tensor_cores);

// Encode the TMA descriptors of a bf16 pool, or of a uint8 pool with head_dim
// 128 (false if the driver call fails, the shape is not served or the pool is
// too large for 32-bit row coordinates).
bool make_pool_maps(int kv_dtype, const PoolDev& pool, PoolMaps& maps);

// Per-format launches (one translation unit each).
cudaError_t launch_decode_bf16(const PoolDev& pool, const PoolMaps& maps, const void* q,
                               const int32_t* block_table, const int32_t* seq_lens, float* out,
                               void* workspace, DecodeLaunch& L, cudaStream_t stream);
cudaError_t launch_decode_uint8(const PoolDev& pool, const PoolMaps& maps, const void* q,
                                const int32_t* block_table, const int32_t* seq_lens, float* out,
                                void* workspace, DecodeLaunch& L, cudaStream_t stream);
cudaError_t launch_decode_uint4(const PoolDev& pool, const PoolMaps& maps, const void* q,
                                const int32_t* block_table, const int32_t* seq_lens, float* out,
                                void* workspace, DecodeLaunch& L, cudaStream_t stream);
cudaError_t launch_decode_fp8(const PoolDev& pool, const PoolMaps& maps, const void* q,
                              const int32_t* block_table, const int32_t* seq_lens, float* out,
                              void* workspace, DecodeLaunch& L, cudaStream_t stream);

// Carve the workspace and launch decode + combine.
cudaError_t launch_decode(int kv_dtype, const PoolDev& pool, const PoolMaps& maps, const void* q,
                          const int32_t* block_table, const int32_t* seq_lens, float* out,
                          void* workspace, DecodeLaunch& L, cudaStream_t stream);

}  // namespace pa
