// Device helpers shared by the CSA2 kernels: the device status word, FP4/FP8
// scalar conversions written from the format definitions, and small PTX wrappers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_fp4.h>

#include "csa2.h"

namespace csa2 {

// First device-side error of the process (0 = none); read and cleared by
// csa2_sync_status().
__device__ int g_dev_error = 0;

__device__ __forceinline__ void set_dev_error(int code) { atomicCAS(&g_dev_error, 0, code); }

// ---------------------------------------------------------------- loads
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// Eight consecutive source values (f32 or bf16) as float; p is 16-byte aligned.
template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&x)[8]);

template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&x)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t* p, float (&x)[8]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&x)[4]);

template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&x)[4]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
}

template <>
__device__ __forceinline__ void load4<uint16_t>(const uint16_t* p, float (&x)[4]) {
  const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
  x[0] = __uint_as_float(a.x << 16);
  x[1] = __uint_as_float(a.x & 0xFFFF0000u);
  x[2] = __uint_as_float(a.y << 16);
  x[3] = __uint_as_float(a.y & 0xFFFF0000u);
}

__device__ __forceinline__ float load_elem(const void* p, int dtype, size_t i) {
  return dtype == CSA2_F32 ? __ldg(static_cast<const float*>(p) + i)
                           : bf16_bits_to_float(__ldg(static_cast<const uint16_t*>(p) + i));
}

// ---------------------------------------------------------------- E4M3 / E8M0
// float8_e4m3fn code -> float (finite codes; exponent bias 7, subnormals m/8*2^-6).
__device__ __forceinline__ float e4m3_decode(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  const float mag = e == 0 ? (float)m * 0.001953125f /* 2^-9 */
                           : __uint_as_float(((e - 7u + 127u) << 23) | (m << 20));
  return (c & 0x80u) ? -mag : mag;
}

// Nearest E4M3 value (ties to even), saturating to the largest finite value.
__device__ __forceinline__ uint32_t e4m3_encode_satfinite(float v) {
  return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// 2^(e-127) for an E8M0 byte (e < 255), including the subnormal 2^-127.
__device__ __forceinline__ float e8m0_decode(uint32_t e) {
  return e == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// ---------------------------------------------------------------- ordered keys
// Monotone map of a float to uint32 (larger float -> larger key); -0 equals +0.
__device__ __forceinline__ uint32_t float_order_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Selection key of slot i with score s: (order(s) << 32) | (2^32-1 - i). Keys are
// distinct, and a larger key is a higher score, then a lower slot.
__device__ __forceinline__ unsigned long long topk_key(float s, uint32_t slot) {
  return ((unsigned long long)float_order_key(s) << 32) | (unsigned long long)(0xFFFFFFFFu - slot);
}

// ---------------------------------------------------------------- launch ordering
// Programmatic dependent launch: a kernel waits for the kernel before it in the
// stream (its completion and memory) before touching global memory, then lets the
// kernel after it launch. A kernel launched behind a kernel that never triggers
// starts after that kernel ends, as without these calls; without a programmatic
// dependency the wait returns at once.
__device__ __forceinline__ void pdl_wait_and_release() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// The two halves, for a kernel that lets the next one launch only near its end (the
// streaming scan: a cluster kernel placed next to its last blocks could find no room
// for its last clusters until its own first ones ended).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// ---------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint32_t smem_u32addr(const void* p) { return smem_u32(p); }

// 16 bytes from global to shared memory (shared address dst), asynchronously: no
// register holds the data, so many copies can be in flight per thread.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// ---------------------------------------------------------------- L2 policy, mbarriers, bulk copies
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of the given parity; false after about budget_ns (error
// recorded) or when another thread of the block has given up (*abort set).
__device__ __forceinline__ bool mbar_wait_bounded_ns(uint32_t bar, uint32_t parity, volatile int* abort,
                                                     uint64_t budget_ns) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u) {
      if (*abort) return false;
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > budget_ns) {
        set_dev_error(CSA2_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

// The kernels' waits: about one second.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort) {
  return mbar_wait_bounded_ns(bar, parity, abort, 1000000000ull);
}

__device__ __forceinline__ void tma_load_rows(uint32_t dst, const void* tmap, int32_t x, int32_t y, uint32_t bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;\n" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace csa2
