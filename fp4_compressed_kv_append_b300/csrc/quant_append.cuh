// kv_quant_append: ratio-2 merge (optional), E2M1/E4M3-16 packing of the 512-channel
// latent and MXFP4 (E2M1/E8M0-32) packing of the 128-channel indexer key.
//
// Pages: "Le cache KV en FP4 -- les 890 octets", sections "Cache principal"
// (eq. 288) and "Cles d'indexeur" (eq. 68); "compresse le KV-Cache de 4 fois",
// item 2 (two consecutive positions merged with learned per-channel weights).
//
// One warp per output entry. Lane l owns latent channels [16l, 16l+16) -- exactly
// one E4M3 scale block -- and indexer channels [4l, 4l+4); eight lanes form one
// 32-channel MXFP4 block. All loads are 16-byte vectors; every lane stores 8 bytes
// of latent codes (one 256-byte coalesced row per warp), one scale byte and
// 2 bytes of key codes.
#pragma once

#include "common.cuh"

namespace csa2 {

constexpr int kAppendWarps = 8;

// Lane l's share of one packed entry.
struct PackedLane {
  uint32_t lo, hi;     // 16 latent codes
  uint32_t s_code;     // their E4M3 scale
  uint32_t kc;         // 4 indexer-key codes
  uint32_t x_code;     // the E8M0 scale of the lane's 32-channel key block
};

// One entry: ratio-2 merge (optional), then both packings. Lane l of the warp.
// Needs only the source token, not the cache position, so the loads do not wait
// for the sequence length.
template <typename Tin>
__device__ __forceinline__ PackedLane quant_entry(const Tin* __restrict__ lat, const Tin* __restrict__ ikey, int T,
                                                  int ratio, const float* __restrict__ w0l,
                                                  const float* __restrict__ w1l, const float* __restrict__ w0i,
                                                  const float* __restrict__ w1i, int b, int e, int lane) {
  PackedLane P;
  const size_t tok = (size_t)b * T + (size_t)e * ratio;

  // ---- latent: one 16-channel block per lane
  float x[16];
  {
    const Tin* p = lat + tok * 512 + 16 * lane;
    float a[8], c[8];
    load8(p, a);
    load8(p + 8, c);
#pragma unroll
    for (int i = 0; i < 8; ++i) { x[i] = a[i]; x[8 + i] = c[i]; }
    if (ratio == 2) {
      float y[16], u0[8], u1[8];
      load8(p + 512, u0);
      load8(p + 520, u1);
#pragma unroll
      for (int i = 0; i < 8; ++i) { y[i] = u0[i]; y[8 + i] = u1[i]; }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float w0 = __ldg(w0l + 16 * lane + i), w1 = __ldg(w1l + 16 * lane + i);
        x[i] = __fadd_rn(__fmul_rn(w0, x[i]), __fmul_rn(w1, y[i]));
      }
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint32_t s_code = e4m3_encode_satfinite(__fdiv_rn(amax, 6.0f));
  const float s = e4m3_decode(s_code);
  uint32_t lo = 0, hi = 0;
  if (s != 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) lo |= e2m1_encode(__fdiv_rn(x[i], s)) << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i) hi |= e2m1_encode(__fdiv_rn(x[8 + i], s)) << (4 * i);
  }
  P.lo = lo;
  P.hi = hi;
  P.s_code = s_code;

  // ---- indexer key: four channels per lane, eight lanes per 32-channel block
  float z[4];
  {
    const Tin* p = ikey + tok * 128 + 4 * lane;
    load4(p, z);
    if (ratio == 2) {
      float y[4];
      load4(p + 128, y);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float w0 = __ldg(w0i + 4 * lane + i), w1 = __ldg(w1i + 4 * lane + i);
        z[i] = __fadd_rn(__fmul_rn(w0, z[i]), __fmul_rn(w1, y[i]));
      }
    }
  }
  float am = fmaxf(fmaxf(fabsf(z[0]), fabsf(z[1])), fmaxf(fabsf(z[2]), fabsf(z[3])));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
  // X = floor(log2 amax) - 2 from the exponent field, clamped to [-127, 127]
  // (a zero or subnormal amax gives -127; a finite amax never exceeds 125).
  const int ef = (int)((__float_as_uint(am) >> 23) & 0xFFu);
  const int X = ef == 0 ? -127 : max(ef - 127 - 2, -127);
  const float inv = __uint_as_float((uint32_t)(127 - X) << 23);  // 2^-X, exact
  uint32_t kc = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) kc |= e2m1_encode(z[i] * inv) << (4 * i);
  P.kc = kc;
  P.x_code = (uint32_t)(X + 127);
  return P;
}

// Lane l's stores of an entry at cache slot `slot` (row index b * cap + position).
__device__ __forceinline__ void store_entry(const PackedLane& P, uint8_t* __restrict__ lat_codes,
                                            uint8_t* __restrict__ lat_scales, uint8_t* __restrict__ idx_codes,
                                            uint8_t* __restrict__ idx_scales, int64_t slot, int lane) {
  *reinterpret_cast<uint2*>(lat_codes + slot * 256 + 8 * lane) = make_uint2(P.lo, P.hi);
  lat_scales[slot * 32 + lane] = (uint8_t)P.s_code;
  *reinterpret_cast<uint16_t*>(idx_codes + slot * 64 + 2 * lane) = (uint16_t)P.kc;
  if ((lane & 7) == 0) idx_scales[slot * 4 + (lane >> 3)] = (uint8_t)P.x_code;
}

template <typename Tin>
__global__ void __launch_bounds__(kAppendWarps * 32)
k_quant_append(const Tin* __restrict__ lat, const Tin* __restrict__ ikey, int T, int ratio,
               const float* __restrict__ w0l, const float* __restrict__ w1l,
               const float* __restrict__ w0i, const float* __restrict__ w1i,
               uint8_t* __restrict__ lat_codes, uint8_t* __restrict__ lat_scales,
               uint8_t* __restrict__ idx_codes, uint8_t* __restrict__ idx_scales,
               int32_t* __restrict__ len, int64_t cap, int n_new) {
  pdl_wait_and_release();
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  const int b = blockIdx.y;
  const int64_t base = len[b];  // in flight while the entry is packed
  PackedLane P{};
  if (e < n_new) P = quant_entry(lat, ikey, T, ratio, w0l, w1l, w0i, w1i, b, e, lane);
  const bool refused = base < 0 || base + n_new > cap;  // the whole append of this sequence is refused
  if (refused && blockIdx.x == 0 && threadIdx.x == 0) set_dev_error(CSA2_ERR_BOUNDS);
  if (e < n_new && !refused)
    store_entry(P, lat_codes, lat_scales, idx_codes, idx_scales, (int64_t)b * cap + base + e, lane);
  // a single block per sequence advances len itself (every thread has read it)
  if (gridDim.x == 1) {
    __syncthreads();
    if (threadIdx.x == 0 && !refused) len[b] = (int32_t)(base + n_new);
  }
}

// Advance len[b] by n_new after an append (refused appends leave len unchanged).
__global__ void k_bump_len(int32_t* len, int batch, int64_t cap, int n_new) {
  pdl_wait_and_release();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) {
    const int64_t l = len[b];
    if (l >= 0 && l + n_new <= cap) len[b] = (int32_t)(l + n_new);
  }
}

}  // namespace csa2
