// C ABI of libpagedattn: pool lifetime, argument validation, dispatch.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <new>

#include "pa_common.cuh"
#include "pa_kernels.h"
#include "pagedattn.h"

struct pa_pool {
  pa::PoolMaps maps;  // first: 64-byte aligned member
  pa_pool_desc desc;
  int32_t decode_path;
  bool fused_combine;
  bool early_plan;
  int32_t unit_cost;  // partition: phantom pages per unit; < 0 = the kernel's default
  void* slab;
  size_t slab_bytes;
  pa::PoolDev dev;
  size_t kv_bytes;
  size_t meta_bytes;
  int sm_count;
};

namespace {

thread_local char g_last_error[512] = "";

// Tags of decode calls: the split-KV merge tickets in the workspace carry the
// tag of the call that wrote them, so stale tickets never need clearing.
std::atomic<unsigned long long> g_epoch{0};

unsigned long long next_epoch() {
  unsigned long long e = (g_epoch.fetch_add(1) + 1) & ((1ull << 40) - 1);
  return e ? e : next_epoch();
}

pa_status fail(pa_status s, const char* fmt, const char* detail = "") {
  snprintf(g_last_error, sizeof g_last_error, fmt, detail);
  return s;
}

pa_status cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_last_error, sizeof g_last_error, "%s: %s", where, cudaGetErrorString(e));
  return PA_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// value v into `per` consecutive floats of each of `pages` records `stride` floats apart
__global__ void fill_scales(float* p, size_t pages, int per, size_t stride, float v) {
  const size_t n = pages * per;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[(i / per) * stride + i % per] = v;
}

// Diagnostic: one thread waits, with the kernels' bounded wait, on a fresh
// mbarrier that nothing ever arrives at, and records the expiry as every
// kernel wait does.
__global__ void selftest_bounded_wait(uint32_t* err, long long limit_cycles) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  pa::mbar_init(&bar, 1);
  pa::fence_mbar_init();
  if (!pa::mbar_wait_bounded(&bar, 0, limit_cycles)) pa::set_error(err, PA_DEVERR_TIMEOUT);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sets the pool's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  cudaError_t err = cudaSuccess;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) err = cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// Default phantom pages per unit of the cost-balanced partition: the fixed
// work of a unit (query load, state deposit and merge, row or partial write)
// in page times of the pool's decode kernel, as measured on GB300 over the
// Qwen-shaped bf16, uint8 and fp8 workloads and the prefix-sharing mix
// (quantised pages are short to stream and costly to decode, so a unit weighs
// more: 10 for uint8, 14 for fp8, whose pages stream faster still).
int32_t default_unit_cost(const pa_pool* p) {
  return p->desc.kv_dtype == PA_KV_UINT8 ? 10 : (p->desc.kv_dtype == PA_KV_FP8 ? 14 : 6);
}

bool uses_tensor_cores(const pa_pool* p) {
  return p->maps.valid && p->decode_path != PA_DECODE_CUDA_CORE;
}

int auto_splits(const pa_pool* p, int group) {
  return p->sm_count * pa::decode_ctas_per_sm(p->desc.kv_dtype, p->desc.block_size,
                                              p->desc.head_dim, group, uses_tensor_cores(p));
}

}  // namespace

extern "C" {

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_OOM: return "out of device memory or workspace too small";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_DEVICE_BOUNDS: return "device-side bounds violation";
    case PA_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char* pa_last_error(void) { return g_last_error; }

pa_status pa_create_pool(const pa_pool_desc* d, pa_pool** out) {
  g_last_error[0] = 0;
  if (!d || !out) return fail(PA_ERR_INVALID_ARG, "null descriptor or output pointer%s");
  *out = nullptr;
  if (d->num_blocks < 1 || d->num_kv_heads < 1 || d->device < 0)
    return fail(PA_ERR_INVALID_ARG, "num_blocks, num_kv_heads must be >= 1 and device >= 0%s");
  if (d->block_size != 16 && d->block_size != 32)
    return fail(PA_ERR_UNSUPPORTED, "block_size must be 16 or 32%s");
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128%s");
  if (d->kv_dtype != PA_KV_BF16 && d->kv_dtype != PA_KV_UINT8 && d->kv_dtype != PA_KV_UINT4 &&
      d->kv_dtype != PA_KV_FP8)
    return fail(PA_ERR_UNSUPPORTED, "unknown kv_dtype%s");
  DeviceGuard dg(d->device);
  if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
  const size_t pages = (size_t)d->num_blocks * d->num_kv_heads;
  const size_t elem_bits = d->kv_dtype == PA_KV_BF16 ? 16 : (d->kv_dtype == PA_KV_UINT4 ? 4 : 8);
  const size_t codes_bytes = (size_t)d->block_size * d->head_dim * elem_bits / 8;  // one of K or V
  const size_t meta_bytes = d->kv_dtype == PA_KV_BF16 ? 0 : (size_t)d->head_dim * 4;  // one metadata array
  // K scale, K zp, V scale, V zp; fp8 pools hold no zero points
  const int meta_arrays = d->kv_dtype == PA_KV_FP8 ? 2 : 4;
  const size_t stride = 2 * codes_bytes + meta_arrays * meta_bytes;  // one page record
  const size_t slab = 256 + pages * stride;
  pa_pool* p = new (std::nothrow) pa_pool();
  if (!p) return fail(PA_ERR_OOM, "host allocation failed%s");
  p->desc = *d;
  p->kv_bytes = pages * codes_bytes;
  p->meta_bytes = pages * meta_bytes;
  cudaError_t e = cudaMalloc(&p->slab, slab);
  if (e != cudaSuccess) {
    delete p;
    cudaGetLastError();
    return fail(PA_ERR_OOM, "cudaMalloc of the pool failed%s");
  }
  p->slab_bytes = slab;
  uint8_t* base = static_cast<uint8_t*>(p->slab);
  p->dev.err = reinterpret_cast<uint32_t*>(base);
  uint8_t* rec = base + 256;
  p->dev.stride = (long long)stride;
  p->dev.k = rec;
  p->dev.v = rec + codes_bytes;
  p->dev.k_scale = nullptr;
  p->dev.k_zp = nullptr;
  p->dev.v_scale = nullptr;
  p->dev.v_zp = nullptr;
  if (meta_bytes && meta_arrays == 2) {
    p->dev.k_scale = reinterpret_cast<float*>(rec + 2 * codes_bytes);
    p->dev.v_scale = reinterpret_cast<float*>(rec + 2 * codes_bytes + meta_bytes);
  } else if (meta_bytes) {
    p->dev.k_scale = reinterpret_cast<float*>(rec + 2 * codes_bytes);
    p->dev.k_zp = reinterpret_cast<int32_t*>(rec + 2 * codes_bytes + meta_bytes);
    p->dev.v_scale = reinterpret_cast<float*>(rec + 2 * codes_bytes + 2 * meta_bytes);
    p->dev.v_zp = reinterpret_cast<int32_t*>(rec + 2 * codes_bytes + 3 * meta_bytes);
  }
  p->dev.num_blocks = d->num_blocks;
  p->dev.num_kv_heads = d->num_kv_heads;
  p->dev.block_size = d->block_size;
  p->dev.head_dim = d->head_dim;
  e = cudaMemset(p->slab, 0, slab);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, d->device);
  if (e == cudaSuccess && meta_bytes) {
    // scales start at 1.0 so an untouched page dequantises to its (zero) codes
    const size_t n = pages * d->head_dim;
    const unsigned grid = (unsigned)((n + 255) / 256 < 65535 ? (n + 255) / 256 : 65535);
    fill_scales<<<grid, 256>>>(p->dev.k_scale, pages, d->head_dim, stride / 4, 1.0f);
    fill_scales<<<grid, 256>>>(p->dev.v_scale, pages, d->head_dim, stride / 4, 1.0f);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
  }
  if (e != cudaSuccess) {
    cudaFree(p->slab);
    delete p;
    return cuda_fail(e, "pool initialisation");
  }
  p->decode_path = PA_DECODE_AUTO;
  p->fused_combine = false;
  p->early_plan = false;
  p->unit_cost = -1;
  p->maps.valid = 0;
  pa::make_pool_maps(d->kv_dtype, p->dev, p->maps);
  *out = p;
  return PA_OK;
}

pa_status pa_destroy(pa_pool* p) {
  g_last_error[0] = 0;
  if (!p) return PA_OK;
  DeviceGuard dg(p->desc.device);
  cudaError_t e = cudaDeviceSynchronize();
  cudaError_t e2 = cudaFree(p->slab);
  delete p;
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFree");
  return PA_OK;
}

pa_status pa_pool_view(const pa_pool* p, pa_pool_buffers* out) {
  if (!p || !out) return fail(PA_ERR_INVALID_ARG, "null pool or output%s");
  out->k = p->dev.k;
  out->v = p->dev.v;
  out->k_scale = p->dev.k_scale;
  out->k_zp = p->dev.k_zp;
  out->v_scale = p->dev.v_scale;
  out->v_zp = p->dev.v_zp;
  out->page_stride = (size_t)p->dev.stride;
  out->num_pages = (size_t)p->desc.num_blocks * p->desc.num_kv_heads;
  return PA_OK;
}

pa_status pa_copy_blocks(pa_pool* p, const int32_t* src, const int32_t* dst, int32_t n, void* stream) {
  g_last_error[0] = 0;
  if (!p || n < 0 || (n > 0 && (!src || !dst))) return fail(PA_ERR_INVALID_ARG, "null pool or block lists, or n < 0%s");
  for (int32_t i = 0; i < n; ++i)
    if (src[i] < 0 || src[i] >= p->desc.num_blocks || dst[i] < 0 || dst[i] >= p->desc.num_blocks || src[i] == dst[i])
      return fail(PA_ERR_INVALID_ARG, "block id out of range, or a block copied onto itself%s");
  if (n == 0) return PA_OK;
  DeviceGuard dg(p->desc.device);
  if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
  // a block's records (one per kv head) are contiguous: one copy per block
  const size_t bytes = (size_t)p->desc.num_kv_heads * (size_t)p->dev.stride;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int32_t i = 0; i < n; ++i) {
    const cudaError_t e = cudaMemcpyAsync(p->dev.k + (size_t)dst[i] * bytes, p->dev.k + (size_t)src[i] * bytes, bytes,
                                          cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "block copy");
  }
  return PA_OK;
}

size_t pa_pool_block_bytes(const pa_pool* p) {
  return p ? (size_t)p->desc.num_kv_heads * (size_t)p->dev.stride : 0;
}

pa_status pa_swap_blocks(pa_pool* p, void* host_buffer, int32_t num_host_blocks, const int32_t* blocks,
                         const int32_t* slots, int32_t n, int32_t direction, void* stream) {
  g_last_error[0] = 0;
  if (!p || !host_buffer || num_host_blocks < 0 || n < 0 || (n > 0 && (!blocks || !slots)))
    return fail(PA_ERR_INVALID_ARG, "null pool, buffer or id lists, or a negative count%s");
  if (direction != PA_SWAP_OUT && direction != PA_SWAP_IN)
    return fail(PA_ERR_INVALID_ARG, "direction must be PA_SWAP_OUT or PA_SWAP_IN%s");
  for (int32_t i = 0; i < n; ++i)
    if (blocks[i] < 0 || blocks[i] >= p->desc.num_blocks || slots[i] < 0 || slots[i] >= num_host_blocks)
      return fail(PA_ERR_INVALID_ARG, "block id or host slot out of range%s");
  if (n == 0) return PA_OK;
  DeviceGuard dg(p->desc.device);
  if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
  // a block's records (one per kv head) are contiguous: one copy per block
  const size_t bytes = pa_pool_block_bytes(p);
  uint8_t* host = static_cast<uint8_t*>(host_buffer);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int32_t i = 0; i < n; ++i) {
    uint8_t* dev = p->dev.k + (size_t)blocks[i] * bytes;
    uint8_t* hst = host + (size_t)slots[i] * bytes;
    const cudaError_t e = direction == PA_SWAP_OUT
                              ? cudaMemcpyAsync(hst, dev, bytes, cudaMemcpyDeviceToHost, s)
                              : cudaMemcpyAsync(dev, hst, bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "block swap copy");
  }
  return PA_OK;
}

pa_status pa_selftest_wait_timeout(int32_t device, int64_t limit_cycles, uint32_t* flags) {
  g_last_error[0] = 0;
  if (!flags || device < 0 || limit_cycles < 1 || limit_cycles > 4000000000LL)
    return fail(PA_ERR_INVALID_ARG, "null flags, negative device or limit outside [1, 4e9] cycles%s");
  *flags = 0;
  DeviceGuard dg(device);
  if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
  uint32_t* word = nullptr;
  cudaError_t e = cudaMalloc(&word, sizeof(uint32_t));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc");
  e = cudaMemset(word, 0, sizeof(uint32_t));
  if (e == cudaSuccess) {
    selftest_bounded_wait<<<1, 32>>>(word, (long long)limit_cycles);
    e = cudaGetLastError();
  }
  uint32_t host = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&host, word, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  cudaFree(word);
  if (e != cudaSuccess) return cuda_fail(e, "bounded-wait self-test");
  *flags = host;
  return PA_OK;
}

// The bandwidth calibration read: grid-stride 16-byte streaming loads, XOR
// folded per thread; the fold is stored only if it equals a constant.
__global__ void __launch_bounds__(512) stream_read_kernel(const int4* __restrict__ src, size_t n16,
                                                          uint32_t* sink) {
  uint32_t acc = 0;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x) {
    const int4 v = __ldcs(src + i);
    acc ^= (uint32_t)(v.x ^ v.y ^ v.z ^ v.w);
  }
  if (acc == 0x9E3779B9u) atomicOr(sink, acc);
}

pa_status pa_stream_read(const void* src, size_t bytes, uint32_t* sink, void* stream) {
  g_last_error[0] = 0;
  if (!src || !sink || !aligned16(src) || (bytes & 15u))
    return fail(PA_ERR_INVALID_ARG, "null pointer, src not 16-byte aligned or bytes not a multiple of 16%s");
  if (bytes == 0) return PA_OK;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  stream_read_kernel<<<4 * sms, 512, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const int4*>(src),
                                                                              bytes / 16, sink);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "stream_read launch");
  return PA_OK;
}

pa_status pa_get_device_error(pa_pool* p, void* stream, uint32_t* flags) {
  g_last_error[0] = 0;
  if (!p || !flags) return fail(PA_ERR_INVALID_ARG, "null pool or flags%s");
  DeviceGuard dg(p->desc.device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, p->dev.err, sizeof host, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(p->dev.err, 0, sizeof host, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  *flags = host;
  if (host & PA_DEVERR_TIMEOUT) return fail(PA_ERR_TIMEOUT, "a kernel wait timed out%s");
  if (host) return fail(PA_ERR_DEVICE_BOUNDS, "a kernel met a bad table entry or length%s");
  return PA_OK;
}

pa_status pa_append_kv(pa_pool* p, const void* k_new, const void* v_new, const int32_t* cu_new,
                       const int32_t* ctx_lens, const int32_t* block_table, int32_t batch,
                       int32_t max_blocks, int32_t max_new_per_seq, void* stream) {
  g_last_error[0] = 0;
  if (!p) return fail(PA_ERR_INVALID_ARG, "null pool%s");
  if (batch < 0 || max_blocks < 0 || max_new_per_seq < 0)
    return fail(PA_ERR_INVALID_ARG, "negative batch, max_blocks or max_new_per_seq%s");
  if (batch == 0) return PA_OK;
  if (!k_new || !v_new || !cu_new || !ctx_lens || !block_table || max_blocks == 0)
    return fail(PA_ERR_INVALID_ARG, "null device pointer or max_blocks == 0%s");
  DeviceGuard dg(p->desc.device);
  if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
  const int bs = p->desc.block_size;
  long long max_new = max_new_per_seq > 0 ? max_new_per_seq : (long long)max_blocks * bs;
  long long touched = (max_new + bs - 1) / bs + 1;
  if (touched > max_blocks) touched = max_blocks;
  if (touched < 1) touched = 1;
  if (touched > 65535) touched = 65535;
  cudaError_t e = pa::launch_append(p->desc.kv_dtype, p->dev, k_new, v_new, cu_new, ctx_lens,
                                    block_table, batch, max_blocks, (int)touched,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_quant_append launch");
  return PA_OK;
}

pa_status pa_pool_set_decode_path(pa_pool* p, int32_t path) {
  g_last_error[0] = 0;
  if (!p) return fail(PA_ERR_INVALID_ARG, "null pool%s");
  const int kernel = path & 3;
  if (path < 0 || (path & ~(3 | PA_DECODE_FUSED_COMBINE | PA_DECODE_EARLY_PLAN)) ||
      kernel > PA_DECODE_TENSOR_CORE)
    return fail(PA_ERR_INVALID_ARG, "unknown decode path%s");
  if (kernel == PA_DECODE_TENSOR_CORE && !p->maps.valid)
    return fail(PA_ERR_UNSUPPORTED, "the tensor-core decode path serves bf16 pools and quantised pools of head_dim 128%s");
  p->decode_path = kernel;
  p->fused_combine = (path & PA_DECODE_FUSED_COMBINE) != 0;
  p->early_plan = (path & PA_DECODE_EARLY_PLAN) != 0;
  return PA_OK;
}

pa_status pa_pool_set_unit_cost(pa_pool* p, int32_t unit_cost_pages) {
  g_last_error[0] = 0;
  if (!p) return fail(PA_ERR_INVALID_ARG, "null pool%s");
  if (unit_cost_pages > 4096) return fail(PA_ERR_INVALID_ARG, "unit cost above 4096 pages%s");
  p->unit_cost = unit_cost_pages < 0 ? -1 : unit_cost_pages;
  return PA_OK;
}

int32_t pa_decode_num_splits(const pa_pool* p, int32_t num_splits) {
  if (!p || num_splits < 0) return 0;
  return num_splits > 0 ? num_splits : auto_splits(p, 8);
}

size_t pa_decode_workspace_bytes(const pa_pool* p, int32_t batch, int32_t num_q_heads,
                                 int32_t num_splits) {
  if (!p || batch < 0 || num_q_heads < 1 || num_splits < 0) return 0;
  const int Hkv = p->desc.num_kv_heads;
  if (num_q_heads % Hkv) return 0;
  const int group = num_q_heads / Hkv;
  const int ctas = num_splits > 0 ? num_splits : auto_splits(p, group);
  return pa::decode_workspace_bytes(ctas, batch, Hkv, group, p->desc.head_dim);
}

// pa_decode, and with k_new / v_new the fused decode step (pa_decode_step).
static pa_status decode_impl(pa_pool* p, const void* q, const int32_t* block_table, const int32_t* seq_lens,
                             int32_t batch, int32_t num_q_heads, int32_t max_blocks, float softmax_scale,
                             float* out, void* workspace, size_t workspace_bytes, int32_t num_splits,
                             const void* k_new, const void* v_new, void* stream) {
  if (!p) return fail(PA_ERR_INVALID_ARG, "null pool%s");
  if (batch < 0 || max_blocks < 0 || num_splits < 0)
    return fail(PA_ERR_INVALID_ARG, "negative batch, max_blocks or num_splits%s");
  if (num_q_heads < 1 || num_q_heads % p->desc.num_kv_heads)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads%s");
  const int group = num_q_heads / p->desc.num_kv_heads;
  if (group > 8) return fail(PA_ERR_UNSUPPORTED, "GQA group size above 8%s");
  if (!isfinite(softmax_scale)) return fail(PA_ERR_INVALID_ARG, "softmax_scale is not finite%s");
  if (batch == 0) return PA_OK;
  if (!q || !block_table || !seq_lens || !out || !workspace || max_blocks == 0)
    return fail(PA_ERR_INVALID_ARG, "null device pointer or max_blocks == 0%s");
  if (!aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(PA_ERR_INVALID_ARG, "q and out must be 16-byte aligned and workspace 256-byte aligned%s");
  const int ctas = num_splits > 0 ? num_splits : auto_splits(p, group);
  const size_t need = pa::decode_workspace_bytes(ctas, batch, p->desc.num_kv_heads, group,
                                                 p->desc.head_dim);
  if (workspace_bytes < need) return fail(PA_ERR_OOM, "workspace smaller than pa_decode_workspace_bytes()%s");
  DeviceGuard dg(p->desc.device);
  if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
  pa::DecodeLaunch L = {};
  L.num_ctas = ctas;
  L.group = group;
  L.num_q_heads = num_q_heads;
  L.batch = batch;
  L.max_blocks = max_blocks;
  L.scale_log2 = softmax_scale * 1.4426950408889634f;
  L.tensor_cores = uses_tensor_cores(p);
  L.fused_combine = p->fused_combine;
  L.early_plan = p->early_plan;
  L.epoch = next_epoch();
  L.unit_cost = p->unit_cost >= 0 ? p->unit_cost : default_unit_cost(p);
  L.k_new = k_new;
  L.v_new = v_new;
  cudaError_t e = pa::launch_decode(p->desc.kv_dtype, p->dev, p->maps, q, block_table, seq_lens, out,
                                    workspace, L, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "paged_gqa_decode launch");
  return PA_OK;
}

pa_status pa_decode(pa_pool* p, const void* q, const int32_t* block_table,
                    const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                    int32_t max_blocks, float softmax_scale, float* out, void* workspace,
                    size_t workspace_bytes, int32_t num_splits, void* stream) {
  g_last_error[0] = 0;
  return decode_impl(p, q, block_table, seq_lens, batch, num_q_heads, max_blocks, softmax_scale, out, workspace,
                     workspace_bytes, num_splits, nullptr, nullptr, stream);
}

pa_status pa_decode_step(pa_pool* p, const void* k_new, const void* v_new, const void* q,
                         const int32_t* block_table, const int32_t* seq_lens, int32_t batch,
                         int32_t num_q_heads, int32_t max_blocks, float softmax_scale, float* out,
                         void* workspace, size_t workspace_bytes, int32_t num_splits, void* stream) {
  g_last_error[0] = 0;
  if (batch > 0 && (!k_new || !v_new)) return fail(PA_ERR_INVALID_ARG, "null k_new or v_new%s");
  return decode_impl(p, q, block_table, seq_lens, batch, num_q_heads, max_blocks, softmax_scale, out, workspace,
                     workspace_bytes, num_splits, k_new, v_new, stream);
}

// Column groups of several query tokens: tokens per group (as many whole
// tokens' heads as fit in 8 columns) and groups per sequence.
static void multi_groups(int n_q, int group, int* tpg, int* n_cg) {
  int t = 8 / group;
  if (t < 1) t = 1;
  if (t > n_q) t = n_q;
  *tpg = t;
  *n_cg = (n_q + t - 1) / t;
}

size_t pa_decode_multi_workspace_bytes(const pa_pool* p, int32_t batch, int32_t n_q, int32_t num_q_heads,
                                       int32_t num_splits) {
  if (!p || batch < 0 || n_q < 1 || num_q_heads < 1 || num_splits < 0) return 0;
  const int Hkv = p->desc.num_kv_heads;
  if (num_q_heads % Hkv || num_q_heads / Hkv > 8) return 0;
  int tpg, n_cg;
  multi_groups(n_q, num_q_heads / Hkv, &tpg, &n_cg);
  const int cols = tpg * (num_q_heads / Hkv);
  // the kernel for several query tokens is built for 8 columns
  const int ctas = num_splits > 0 ? num_splits : auto_splits(p, 8);
  return pa::decode_workspace_bytes(ctas, batch * n_cg, Hkv, cols, p->desc.head_dim);
}

pa_status pa_decode_multi(pa_pool* p, const void* q, const int32_t* block_table, const int32_t* seq_lens,
                          int32_t batch, int32_t n_q, int32_t num_q_heads, int32_t max_blocks,
                          float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                          int32_t num_splits, void* stream) {
  g_last_error[0] = 0;
  if (!p) return fail(PA_ERR_INVALID_ARG, "null pool%s");
  if (batch < 0 || max_blocks < 0 || num_splits < 0 || n_q < 1)
    return fail(PA_ERR_INVALID_ARG, "negative batch, max_blocks or num_splits, or n_q < 1%s");
  if ((long long)batch * n_q > (1 << 30)) return fail(PA_ERR_INVALID_ARG, "batch * n_q too large%s");
  if (num_q_heads < 1 || num_q_heads % p->desc.num_kv_heads)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads%s");
  const int group = num_q_heads / p->desc.num_kv_heads;
  if (group > 8) return fail(PA_ERR_UNSUPPORTED, "GQA group size above 8%s");
  if (!isfinite(softmax_scale)) return fail(PA_ERR_INVALID_ARG, "softmax_scale is not finite%s");
  if (batch == 0) return PA_OK;
  if (!q || !block_table || !seq_lens || !out || !workspace || max_blocks == 0)
    return fail(PA_ERR_INVALID_ARG, "null device pointer or max_blocks == 0%s");
  if (!aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(PA_ERR_INVALID_ARG, "q and out must be 16-byte aligned and workspace 256-byte aligned%s");
  if (n_q == 1)
    return pa_decode(p, q, block_table, seq_lens, batch, num_q_heads, max_blocks, softmax_scale, out, workspace,
                     workspace_bytes, num_splits, stream);
  int tpg, n_cg;
  multi_groups(n_q, group, &tpg, &n_cg);
  const int cols = tpg * group;
  // the kernel for several query tokens is built for 8 columns
  const int ctas = num_splits > 0 ? num_splits : auto_splits(p, 8);
  const size_t need = pa::decode_workspace_bytes(ctas, batch * n_cg, p->desc.num_kv_heads, cols, p->desc.head_dim);
  if (workspace_bytes < need) return fail(PA_ERR_OOM, "workspace smaller than pa_decode_multi_workspace_bytes()%s");
  DeviceGuard dg(p->desc.device);
  if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
  pa::DecodeLaunch L = {};
  L.num_ctas = ctas;
  L.group = cols;
  L.num_q_heads = num_q_heads;
  L.batch = batch * n_cg;
  L.max_blocks = max_blocks;
  L.scale_log2 = softmax_scale * 1.4426950408889634f;
  L.tensor_cores = uses_tensor_cores(p);
  L.fused_combine = false;
  L.early_plan = p->early_plan;
  L.epoch = next_epoch();
  L.unit_cost = p->unit_cost >= 0 ? p->unit_cost : default_unit_cost(p);
  L.n_q = n_q;
  L.n_cg = n_cg;
  L.tpg = tpg;
  L.g_heads = group;
  cudaError_t e = pa::launch_decode(p->desc.kv_dtype, p->dev, p->maps, q, block_table, seq_lens, out,
                                    workspace, L, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "paged_gqa_decode (several query tokens) launch");
  return PA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ decode without allocation
//
// Some callers cannot call cudaMalloc at all: code running under an allocator
// that forbids device allocations on the hot path, processes whose memory is
// reserved up front, or callers that have no allocator handle to give us.
// pa_decode_noalloc serves them: its split-KV scratch is a fixed array in
// this library's device image (allocated once, when the library's module is
// loaded on a device, and held until the process exits), so a call needs no
// workspace from the caller and allocates nothing.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

}  // namespace

extern "C" pa_status pa_decode_noalloc(pa_pool* p, const void* q, const int32_t* block_table,
                                       const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                       int32_t max_blocks, float softmax_scale, float* out,
                                       int32_t num_splits, void* stream) {
  g_last_error[0] = 0;
  if (!p) return fail(PA_ERR_INVALID_ARG, "null pool%s");
  // Argument errors and the empty batch get pa_decode's own answer, before the
  // scratch's address is looked up (which selects the device and loads the
  // module): such a call has no side effect.
  if (batch <= 0 || num_q_heads < 1 || num_splits < 0 || max_blocks <= 0 || !isfinite(softmax_scale) || !q ||
      !block_table || !seq_lens || !out)
    return pa_decode(p, q, block_table, seq_lens, batch, num_q_heads, max_blocks, softmax_scale, out, nullptr, 0,
                     num_splits, stream);
  const int dev = p->desc.device;
  if (dev >= kNoAllocMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device ordinal above 63%s");
  const size_t need = pa_decode_workspace_bytes(p, batch, num_q_heads, num_splits);
  if (batch > 0 && need == 0) return fail(PA_ERR_INVALID_ARG, "invalid batch, head count or split count%s");
  if (need > kNoAllocScratchBytes) {
    snprintf(g_last_error, sizeof g_last_error,
             "pa_decode_noalloc: this batch needs %zu bytes of split-KV scratch but the static "
             "scratch holds %zu; use pa_decode with a caller workspace or fewer splits",
             need, kNoAllocScratchBytes);
    return PA_ERR_OOM;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    scratch = g_noalloc_ptr[dev];
    if (!scratch) {
      // first call on this device: look up the array's device address with the
      // pool's device current (the host-side name is not a device address)
      DeviceGuard dg(dev);
      if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
      cudaError_t e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
      if (e != cudaSuccess || !scratch) return cuda_fail(e, "cudaGetSymbolAddress of the static scratch");
      g_noalloc_ptr[dev] = scratch;
    }
  }
  return pa_decode(p, q, block_table, seq_lens, batch, num_q_heads, max_blocks, softmax_scale, out,
                   scratch, kNoAllocScratchBytes, num_splits, stream);
}
