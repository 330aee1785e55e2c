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
