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
// 2 bytes of key codes. A warp packs up to kAppendPerWarp entries in turn, with the
// ratio-2 merge weights of its channels loaded once into registers. E2M1 codes come
// from the hardware pair conversion (round to nearest even, saturating at 6, the
// sign kept on zero), two values per instruction.
#pragma once

#include "common.cuh"

namespace csa2 {

constexpr int kAppendWarps = 8;
constexpr int kAppendPerWarp = 4;
constexpr int kAppendBlockEntries = kAppendWarps * kAppendPerWarp;

// Lane l's share of one packed entry.
struct PackedLane {
  uint32_t lo, hi;     // 16 latent codes
  uint32_t s_code;     // their E4M3 scale
  uint32_t kc;         // 4 indexer-key codes
  uint32_t x_code;     // the E8M0 scale of the lane's 32-channel key block
};

// Merge weights of lane l's channels (ratio 2).
struct LaneWeights {
  float l0[16], l1[16], i0[4], i1[4];
};

// Eight E2M1 codes of v[0..7], v[2j] in the low nibble of byte j.
__device__ __forceinline__ uint32_t e2m1x8(const float* v) {
  uint32_t r = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    r |= (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(v[2 * j], v[2 * j + 1]), __NV_E2M1, cudaRoundNearest)
         << (8 * j);
  return r;
}

// One entry: ratio-2 merge (optional), then both packings. Lane l of the warp.
// Needs only the source token, not the cache position.
template <typename Tin>
__device__ __forceinline__ PackedLane quant_entry(const Tin* __restrict__ lat, const Tin* __restrict__ ikey, int T,
                                                  int ratio, const LaneWeights& W, int b, int e, int lane) {
  PackedLane P;
  const size_t tok = (size_t)b * T + (size_t)e * ratio;

  // ---- loads: latent (one 16-channel block per lane) and key (4 channels), both tokens
  float x[16], y[16], z[4], zy[4];
  {
    const Tin* p = lat + tok * 512 + 16 * lane;
    float a[8], c[8];
    load8(p, a);
    load8(p + 8, c);
#pragma unroll
    for (int i = 0; i < 8; ++i) { x[i] = a[i]; x[8 + i] = c[i]; }
    if (ratio == 2) {
      load8(p + 512, a);
      load8(p + 520, c);
#pragma unroll
      for (int i = 0; i < 8; ++i) { y[i] = a[i]; y[8 + i] = c[i]; }
    }
    const Tin* pk = ikey + tok * 128 + 4 * lane;
    load4(pk, z);
    if (ratio == 2) load4(pk + 128, zy);
  }
  if (ratio == 2) {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __fadd_rn(__fmul_rn(W.l0[i], x[i]), __fmul_rn(W.l1[i], y[i]));
#pragma unroll
    for (int i = 0; i < 4; ++i) z[i] = __fadd_rn(__fmul_rn(W.i0[i], z[i]), __fmul_rn(W.i1[i], zy[i]));
  }

  // ---- latent: s = E4M3(amax / 6), codes E2M1(x / s)
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint32_t s_code = e4m3_encode_satfinite(__fdiv_rn(amax, 6.0f));
  const float s = e4m3_decode(s_code);
  uint32_t lo = 0, hi = 0;
  if (s != 0.f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __fdiv_rn(x[i], s);
    lo = e2m1x8(x);
    hi = e2m1x8(x + 8);
  }
  P.lo = lo;
  P.hi = hi;
  P.s_code = s_code;

  // ---- indexer key: four channels per lane, eight lanes per 32-channel block
  float am = fmaxf(fmaxf(fabsf(z[0]), fabsf(z[1])), fmaxf(fabsf(z[2]), fabsf(z[3])));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
  // X = floor(log2 amax) - 2 from the exponent field, clamped to [-127, 127]
  // (a zero or subnormal amax gives -127; a finite amax never exceeds 125).
  const int ef = (int)((__float_as_uint(am) >> 23) & 0xFFu);
  const int X = ef == 0 ? -127 : max(ef - 127 - 2, -127);
  const float inv = __uint_as_float((uint32_t)(127 - X) << 23);  // 2^-X, exact
  float zs[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) zs[i] = z[i] * inv;
  P.kc = (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(zs[0], zs[1]), __NV_E2M1, cudaRoundNearest) |
         ((uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(zs[2], zs[3]), __NV_E2M1, cudaRoundNearest) << 8);
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

// Block x of sequence b packs entries [kAppendBlockEntries x, +kAppendBlockEntries);
// warp w takes entries w, w + kAppendWarps, ... of that range.
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
  const int b = blockIdx.y;
  const int64_t base = len[b];  // in flight while the first entry is packed
  LaneWeights W;
  if (ratio == 2) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(w0l + 16 * lane) + i);
      const float4 c = __ldg(reinterpret_cast<const float4*>(w1l + 16 * lane) + i);
      W.l0[4 * i] = a.x; W.l0[4 * i + 1] = a.y; W.l0[4 * i + 2] = a.z; W.l0[4 * i + 3] = a.w;
      W.l1[4 * i] = c.x; W.l1[4 * i + 1] = c.y; W.l1[4 * i + 2] = c.z; W.l1[4 * i + 3] = c.w;
    }
    const float4 a = __ldg(reinterpret_cast<const float4*>(w0i + 4 * lane));
    const float4 c = __ldg(reinterpret_cast<const float4*>(w1i + 4 * lane));
    W.i0[0] = a.x; W.i0[1] = a.y; W.i0[2] = a.z; W.i0[3] = a.w;
    W.i1[0] = c.x; W.i1[1] = c.y; W.i1[2] = c.z; W.i1[3] = c.w;
  }
  const bool refused = base < 0 || base + n_new > cap;  // the whole append of this sequence is refused
  if (refused && blockIdx.x == 0 && threadIdx.x == 0) set_dev_error(CSA2_ERR_BOUNDS);
  const int e0 = blockIdx.x * kAppendBlockEntries + (threadIdx.x >> 5);
#pragma unroll 1
  for (int j = 0; j < kAppendPerWarp; ++j) {
    const int e = e0 + j * kAppendWarps;
    if (e >= n_new) break;
    const PackedLane P = quant_entry(lat, ikey, T, ratio, W, b, e, lane);
    if (!refused)
      store_entry(P, lat_codes, lat_scales, idx_codes, idx_scales, (int64_t)b * cap + base + e, lane);
  }
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
