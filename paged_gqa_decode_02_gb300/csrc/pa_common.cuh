// Shared device helpers for the paged-attention kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <atomic>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

// Pool geometry and device addresses, passed by value to every kernel. A
// page (one block of one kv head) is one contiguous record
// [K][V][K scale][K zp][V scale][V zp]; each pointer addresses its component
// in page 0, and page n's component sits n * stride bytes further on.
struct PoolDev {
  uint8_t* k;       // codes or bf16 elements [bs][D] (uint4: [bs][D/2])
  uint8_t* v;
  float* k_scale;   // [D] (quantised pools)
  int32_t* k_zp;
  float* v_scale;
  int32_t* v_zp;
  uint32_t* err;    // device error word
  long long stride; // bytes from one page record to the next
  int32_t num_blocks;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t head_dim;
};

template <typename T>
__host__ __device__ __forceinline__ T* page_of(T* base, long long page, long long stride) {
  return reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(base) + page * stride);
}

// TMA descriptor of a pool's page records viewed as a 2-D tensor of rows,
// 128-byte swizzle. bf16: rows of head_dim elements (2*bs rows per record, K
// then V), boxes of 64 channels x 2*bs rows (two per record for head_dim 128).
// uint8 (head_dim 128): rows of 128 bytes (stride/128 rows per record, codes
// then metadata), one box per record.
struct PoolMaps {  // aligned as its CUtensorMap member
  CUtensorMap rec;
  int32_t rows_per_page;
  int32_t valid;
};

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bits) { atomicOr(err, bits); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------- mbarrier / bulk copy (PTX)
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy writes to global memory before
// later async-proxy (TMA) accesses that are ordered after it (through an
// mbarrier arrive / wait, for another thread of the block).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// roughly `limit_cycles` SM clocks. Returns false on timeout. The default,
// 2e8 clocks (about 0.1 s at 2 GHz), is far above the longest wait of a
// healthy launch: every wait starts after the wait on the preceding kernel,
// and the longest, the merger's wait for a slice's first unit, covers at most
// one slice's pages (a slice of 100 k pages streams in about 20 ms).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit_cycles = 200000000LL) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit_cycles) return false;
  }
}

// Create an L2 eviction policy for data read once.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D TMA bulk copy global -> shared, completing on an mbarrier. Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Bring `bytes` of global memory into L2 without waiting for it (address
// 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* src_gmem, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

// Prefetch a TMA descriptor (kernel parameter) into the descriptor cache.
__device__ __forceinline__ void prefetch_tensormap(const void* desc) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(desc) : "memory");
}

// One-time per-device launch set-up of a kernel (host side): its dynamic
// shared memory limit, and the shared-memory carveout pinned to the maximum.
// Every kernel of the library uses the same carveout because an SM runs
// thread blocks of two kernels side by side (as a programmatic dependent
// launch does with a kernel and the one after it) only while their carveouts
// agree; otherwise the later kernel's blocks wait for the SM to drain.
template <typename Kernel>
inline cudaError_t prepare_kernel(Kernel kern, int dyn_smem_bytes, std::atomic<unsigned long long>& ready) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (ready.load(std::memory_order_acquire) & bit) return cudaSuccess;
  if (dyn_smem_bytes > 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem_bytes);
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  ready.fetch_or(bit, std::memory_order_release);
  return cudaSuccess;
}

// Programmatic dependent launch controls (no-ops without the launch attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}


}  // namespace pa

namespace pa {

// ---------------------------------------------------------------- tensor-core helpers (PTX)
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose an 8x8 b16 matrix held in the mma fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 2-D TMA tensor load (tile mode) into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void* dst_smem, const void* tmap, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst_smem)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

}  // namespace pa

namespace pa {

// D = A(16x16, row) * B(16x8, col) + D, f16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte permute: bytes of {b, a} numbered 0..3 (a) and 4..7 (b); nibble i of
// sel picks byte i of the result.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Two bytes of w (chosen by sel, see prmt) as two exact f16 integers 0..255.
// The IEEE-754 binary16 identity behind it: exponent field 25 (bias 15, so a
// scale of 2^10) with ten mantissa bits m is the value 1024 + m, so the bit
// pattern 0x6400 | XX is exactly 1024 + XX, and one f16 subtraction of 1024
// (exact: both operands are integers below 2048) leaves XX. This is the
// usual bit-level integer-to-half conversion of low-precision dequantisation
// kernels, here written from the format's definition.
__device__ __forceinline__ uint32_t bytes_to_f16x2(uint32_t w, uint32_t sel) {
  const uint32_t x = prmt(w, 0x64646464u, sel);
  __half2 h = *reinterpret_cast<const __half2*>(&x);
  h = __hsub2(h, __halves2half2(__ushort_as_half((unsigned short)0x6400), __ushort_as_half((unsigned short)0x6400)));
  return *reinterpret_cast<uint32_t*>(&h);
}

// 2^x by the special-function unit (PTX ex2.approx.ftz.f32: relative error
// about 2^-22, a subnormal result flushes to zero, 2^-inf = 0), for the
// per-page softmax weights whose f16 high + remainder split keeps 22 bits.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// lo, hi rounded to nearest-even f16 and packed (lo in the lower half): one cvt
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// the two halves of an f16 pair widened exactly to fp32
__device__ __forceinline__ float2 unpack_f16(uint32_t w) {
  float2 r;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.f32.f16 %0, lo;\n cvt.f32.f16 %1, hi;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(w));
  return r;
}

// E4M3 (OCP 8-bit floating point: bias 7, 3 mantissa bits, no infinities,
// largest finite 448) through the hardware conversions. Every E4M3 value is
// an f16 value, so widening is exact.
// Two codes (bits 0-7 and 8-15 of w) -> f16x2 (low half from bits 0-7).
// Two E4M3 codes widened exactly to an f16 pair (every E4M3 value is an f16
// value): the codes in the low (_lo) or high (_hi) 16 bits of w, the lower
// byte to the lower half. The half is taken as a register view, no shift.
__device__ __forceinline__ uint32_t e4m3x2_lo_to_f16x2(uint32_t w) {
  uint32_t d;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n}" : "=r"(d) : "r"(w));
  return d;
}
__device__ __forceinline__ uint32_t e4m3x2_hi_to_f16x2(uint32_t w) {
  uint32_t d;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.f16x2.e4m3x2 %0, hi;\n}" : "=r"(d) : "r"(w));
  return d;
}

__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(__half(h));
}

// fp32 -> E4M3, round to nearest-even, saturated to +-448 (finite inputs).
__device__ __forceinline__ uint8_t float_to_e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

}  // namespace pa
