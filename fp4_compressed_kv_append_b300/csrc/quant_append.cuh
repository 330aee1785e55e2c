// kv_quant_append: ratio-2 merge (optional), E2M1/E4M3-16 packing of the 512-channel
// latent and MXFP4 (E2M1/E8M0-32) packing of the 128-channel indexer key.
//
// Pages: "Le cache KV en FP4 -- les 890 octets", sections "Cache principal"
// (eq. 288) and "Cles d'indexeur" (eq. 68); "compresse le KV-Cache de 4 fois",
// item 2 (two consecutive positions merged with learned per-channel weights).
//
// The block's source tokens (a contiguous run of rows per sequence) are first
// bulk-copied into shared memory by one thread, so the whole block's input is in
// flight at once; the warps then pack from shared memory.
//
// One warp per output entry. Lane l owns latent channels [16l, 16l+16) -- exactly
// one E4M3 scale block -- and indexer channels [4l, 4l+4); eight lanes form one
// 32-channel MXFP4 block. All loads are 16-byte vectors; every lane stores 8 bytes
// of latent codes (one 256-byte coalesced row per warp), one scale byte and
// 2 bytes of key codes. A warp packs up to kAppendPerWarp entries in turn; the block
// loads the ratio-2 merge weights once into shared memory. E2M1 codes come
// from the hardware pair conversion (round to nearest even, saturating at 6, the
// sign kept on zero), two values per instruction; the latent's division by its
// scale is bracketed (e2m1_div16) so that the correctly rounded division runs only
// next to tie points.
#pragma once

#include "common.cuh"

namespace csa2 {

constexpr int kAppendWarps = 8;
constexpr int kAppendPerWarp = 2;  // 16 entries a block: a 40 KB stage (bf16, ratio 2), four blocks per SM
constexpr int kAppendBlockEntries = kAppendWarps * kAppendPerWarp;

// Lane l's share of one packed entry.
struct PackedLane {
  uint32_t lo, hi;     // 16 latent codes
  uint32_t s_code;     // their E4M3 scale
  uint32_t kc;         // 4 indexer-key codes
  uint32_t x_code;     // the E8M0 scale of the lane's 32-channel key block
};

// Merge weights of a block's layer (ratio 2), in shared memory, transposed so that
// the lanes of a warp read consecutive words: [i][lane] holds latent channel 16 lane + i
// and key channel 4 lane + i.
struct MergeWeights {
  float l0[16][32], l1[16][32], i0[4][32], i1[4][32];
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

// E2M1 codes of fl32(x[i] / s) for a 16-channel block (s > 0), with few divisions:
// q = x * fl32(1/s) is within about two ulps of the quotient, so q * (1 - 2^-20) and
// q * (1 + 2^-20) lie on either side of fl32(x / s). E2M1 rounding is monotone, so
// where the codes of the two agree they are the code of the quotient; a block with a
// value so close to a tie point that they differ takes the correctly rounded division.
__device__ __forceinline__ void e2m1_div16(const float (&x)[16], float s, uint32_t& lo, uint32_t& hi) {
  constexpr float kDown = 1.0f - 0x1p-20f, kUp = 1.0f + 0x1p-20f;
  const float r = __frcp_rn(s);
  float a[16], c[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float q = x[i] * r;
    a[i] = q * kDown;
    c[i] = q * kUp;
  }
  const uint32_t a0 = e2m1x8(a), a1 = e2m1x8(a + 8), c0 = e2m1x8(c), c1 = e2m1x8(c + 8);
  if (a0 == c0 && a1 == c1) {
    lo = a0;
    hi = a1;
    return;
  }
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(x[i], s);
  lo = e2m1x8(q);
  hi = e2m1x8(q + 8);
}

// Eight / four consecutive source values from shared memory (16- / 8-byte aligned).
template <typename T>
__device__ __forceinline__ void load8_shared(const T* p, float (&x)[8]);
template <>
__device__ __forceinline__ void load8_shared<float>(const float* p, float (&x)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <>
__device__ __forceinline__ void load8_shared<uint16_t>(const uint16_t* p, float (&x)[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <typename T>
__device__ __forceinline__ void load4_shared(const T* p, float (&x)[4]);
template <>
__device__ __forceinline__ void load4_shared<float>(const float* p, float (&x)[4]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
}
template <>
__device__ __forceinline__ void load4_shared<uint16_t>(const uint16_t* p, float (&x)[4]) {
  const uint2 a = *reinterpret_cast<const uint2*>(p);
  x[0] = __uint_as_float(a.x << 16);
  x[1] = __uint_as_float(a.x & 0xFFFF0000u);
  x[2] = __uint_as_float(a.y << 16);
  x[3] = __uint_as_float(a.y & 0xFFFF0000u);
}

// One entry: ratio-2 merge (optional), then both packings. Lane l of the warp.
// Needs only the source token, not the cache position. lat / ikey are the block's
// staged rows in shared memory; tok is the entry's first token among them.
template <typename Tin>
__device__ __forceinline__ PackedLane quant_entry(const Tin* lat, const Tin* ikey, int tok, int ratio,
                                                  const MergeWeights& W, int lane) {
  PackedLane P;

  // ---- loads: latent (one 16-channel block per lane) and key (4 channels), both tokens
  float x[16], y[16], z[4], zy[4];
  {
    const Tin* p = lat + (size_t)tok * 512 + 16 * lane;
    float a[8], c[8];
    load8_shared(p, a);
    load8_shared(p + 8, c);
#pragma unroll
    for (int i = 0; i < 8; ++i) { x[i] = a[i]; x[8 + i] = c[i]; }
    if (ratio == 2) {
      load8_shared(p + 512, a);
      load8_shared(p + 520, c);
#pragma unroll
      for (int i = 0; i < 8; ++i) { y[i] = a[i]; y[8 + i] = c[i]; }
    }
    const Tin* pk = ikey + (size_t)tok * 128 + 4 * lane;
    load4_shared(pk, z);
    if (ratio == 2) load4_shared(pk + 128, zy);
  }
  if (ratio == 2) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      x[i] = __fadd_rn(__fmul_rn(W.l0[i][lane], x[i]), __fmul_rn(W.l1[i][lane], y[i]));
#pragma unroll
    for (int i = 0; i < 4; ++i)
      z[i] = __fadd_rn(__fmul_rn(W.i0[i][lane], z[i]), __fmul_rn(W.i1[i][lane], zy[i]));
  }

  // ---- latent: s = E4M3(amax / 6), codes E2M1(x / s)
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint32_t s_code = e4m3_encode_satfinite(__fdiv_rn(amax, 6.0f));
  const float s = e4m3_decode(s_code);
  uint32_t lo = 0, hi = 0;
  if (s != 0.f) e2m1_div16(x, s, lo, hi);
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

// Block bx of sequence b packs entries [kAppendBlockEntries bx, +kAppendBlockEntries);
// warp w takes entries w, w + kAppendWarps, ... of that range. With own_len (the
// append has a single block per sequence) the block advances len itself.
template <typename Tin>
__device__ __forceinline__ void append_block(const Tin* __restrict__ lat, const Tin* __restrict__ ikey, int T,
                                             int ratio, const float* __restrict__ w0l, const float* __restrict__ w1l,
                                             const float* __restrict__ w0i, const float* __restrict__ w1i,
                                             uint8_t* __restrict__ lat_codes, uint8_t* __restrict__ lat_scales,
                                             uint8_t* __restrict__ idx_codes, uint8_t* __restrict__ idx_scales,
                                             int32_t* __restrict__ len, int64_t cap, int n_new, int bx, int b,
                                             bool own_len) {
  const int lane = threadIdx.x & 31;
  const int64_t base = len[b];  // in flight while the tokens are copied
  __shared__ MergeWeights W;
  __shared__ unsigned long long stage_bar;
  __shared__ int stage_abort;
  extern __shared__ __align__(16) unsigned char append_stage[];
  Tin* st_lat = reinterpret_cast<Tin*>(append_stage);            // [ratio * kAppendBlockEntries][512]
  Tin* st_key = st_lat + (size_t)ratio * kAppendBlockEntries * 512;  // [ratio * kAppendBlockEntries][128]
  const int e_begin = bx * kAppendBlockEntries;
  const int ntok = max(0, min(kAppendBlockEntries, n_new - e_begin)) * ratio;
  const uint32_t sbar = smem_u32(&stage_bar);
  if (threadIdx.x == 0 && ntok > 0) {
    mbar_init(sbar, 1);
    stage_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    const size_t tok0 = (size_t)b * T + (size_t)e_begin * ratio;
    const uint32_t nlat = (uint32_t)ntok * 512u * (uint32_t)sizeof(Tin), nkey = (uint32_t)ntok * 128u * (uint32_t)sizeof(Tin);
    const uint64_t pol = l2_evict_first_policy();
    mbar_arrive_expect_tx(sbar, nlat + nkey);
    bulk_load(smem_u32(st_lat), lat + tok0 * 512, nlat, sbar, pol);
    bulk_load(smem_u32(st_key), ikey + tok0 * 128, nkey, sbar, pol);
  }
  if (ratio == 2) {  // the block loads the weights once (16-byte vectors), transposing them
    for (int i = threadIdx.x; i < 2 * 512 / 4; i += blockDim.x) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(i < 128 ? w0l : w1l) + (i & 127));
      float* dst = i < 128 ? &W.l0[0][0] : &W.l1[0][0];
      const int c0 = 4 * (i & 127);
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) dst[((c0 + u) & 15) * 32 + ((c0 + u) >> 4)] = vv[u];
    }
    for (int i = threadIdx.x; i < 2 * 128 / 4; i += blockDim.x) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(i < 32 ? w0i : w1i) + (i & 31));
      float* dst = i < 32 ? &W.i0[0][0] : &W.i1[0][0];
      const int c0 = 4 * (i & 31);
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) dst[((c0 + u) & 3) * 32 + ((c0 + u) >> 2)] = vv[u];
    }
  }
  __syncthreads();  // the weights and the barrier's initialisation
  if (ntok > 0 && !mbar_wait_bounded(sbar, 0u, &stage_abort)) {
    volatile int again = 0;  // a wait ran out (recorded): let the copy land before going on
    mbar_wait_bounded(sbar, 0u, &again);
  }
  const bool refused = base < 0 || base + n_new > cap;  // the whole append of this sequence is refused
  if (refused && bx == 0 && threadIdx.x == 0) set_dev_error(CSA2_ERR_BOUNDS);
  const int e0 = bx * kAppendBlockEntries + (threadIdx.x >> 5);
#pragma unroll 1
  for (int j = 0; j < kAppendPerWarp; ++j) {
    const int e = e0 + j * kAppendWarps;
    if (e >= n_new) break;
    const PackedLane P = quant_entry(st_lat, st_key, (e - e_begin) * ratio, ratio, W, lane);
    if (!refused)
      store_entry(P, lat_codes, lat_scales, idx_codes, idx_scales, (int64_t)b * cap + base + e, lane);
  }
  if (own_len) {  // every thread has read len
    __syncthreads();
    if (threadIdx.x == 0 && !refused) len[b] = (int32_t)(base + n_new);
  }
}

// Dynamic shared memory of an append block: its source tokens (latent and key rows).
template <typename Tin>
constexpr size_t append_stage_bytes(int ratio) {
  return (size_t)ratio * kAppendBlockEntries * (512 + 128) * sizeof(Tin);
}

template <typename Tin>
__global__ void __launch_bounds__(kAppendWarps * 32, 4)
k_quant_append(const Tin* __restrict__ lat, const Tin* __restrict__ ikey, int T, int ratio,
               const float* __restrict__ w0l, const float* __restrict__ w1l,
               const float* __restrict__ w0i, const float* __restrict__ w1i,
               uint8_t* __restrict__ lat_codes, uint8_t* __restrict__ lat_scales,
               uint8_t* __restrict__ idx_codes, uint8_t* __restrict__ idx_scales,
               int32_t* __restrict__ len, int64_t cap, int n_new) {
  pdl_wait_and_release();
  append_block(lat, ikey, T, ratio, w0l, w1l, w0i, w1i, lat_codes, lat_scales, idx_codes, idx_scales, len, cap,
               n_new, (int)blockIdx.x, (int)blockIdx.y, gridDim.x == 1);
}

// ---------------------------------------------------------------- multi-layer store
// csa2_store_append: T source tokens of each of up to kStoreMaxLayers layers, each
// into its own cache with its own ratio and merge weights ("Le compte par couche":
// layers 2, 8 and 14 at ratio 2 and layer 20 at ratio 1), in one launch: the blocks
// of layer l are [block0, block0 + ceil(n_new / kAppendBlockEntries)) along x;
// k_store_bump then advances every layer's lengths.
constexpr int kStoreMaxLayers = 8;

struct StoreLayer {
  const void* lat;
  const void* ikey;
  const float *w0l, *w1l, *w0i, *w1i;
  uint8_t *lat_codes, *lat_scales, *idx_codes, *idx_scales;
  int32_t* len;
  int64_t cap;
  int ratio, n_new, block0;
};

struct StoreArgs {
  StoreLayer L[kStoreMaxLayers];
  int n_layers, T;
};

template <typename Tin>
__global__ void __launch_bounds__(kAppendWarps * 32, 4) k_store_append(const __grid_constant__ StoreArgs a) {
  pdl_wait_and_release();
  int l = 0;
  for (int i = 1; i < a.n_layers; ++i)
    if ((int)blockIdx.x >= a.L[i].block0) l = i;
  const StoreLayer& L = a.L[l];
  append_block(static_cast<const Tin*>(L.lat), static_cast<const Tin*>(L.ikey), a.T, L.ratio, L.w0l, L.w1l, L.w0i,
               L.w1i, L.lat_codes, L.lat_scales, L.idx_codes, L.idx_scales, L.len, L.cap, L.n_new,
               (int)blockIdx.x - L.block0, (int)blockIdx.y, false);
}

// Block l advances layer l's lengths (refused appends leave len unchanged).
__global__ void k_store_bump(const __grid_constant__ StoreArgs a, int batch) {
  pdl_wait_and_release();
  const StoreLayer& L = a.L[blockIdx.x];
  for (int b = threadIdx.x; b < batch; b += blockDim.x) {
    const int64_t l = L.len[b];
    if (l >= 0 && l + L.n_new <= L.cap) L.len[b] = (int32_t)(l + L.n_new);
  }
}

// ---------------------------------------------------------------- FP8 window rows
// csa2_swa_quant: one warp per row of 512 values, lane l the 16-value block l: X =
// floor(log2 amax) - 8 (clamped to [-127, 127]) from the exponent field, E8M0 byte
// X + 127, value codes E4M3(x * 2^-X), nearest-even, saturating at 448 ("Le cache KV
// en FP4", "La contrepartie : la fenetre glissante": FP8 with 512/16 scale bytes).
constexpr int kSwaWarps = 8;

template <typename Tin>
__global__ void __launch_bounds__(kSwaWarps * 32)
k_swa_quant(const Tin* __restrict__ rows, int64_t n_rows, uint8_t* __restrict__ codes,
            uint8_t* __restrict__ scales) {
  pdl_wait_and_release();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kSwaWarps + (threadIdx.x >> 5);
  if (r >= n_rows) return;
  float x[16];
  {
    float a[8], c[8];
    load8(rows + r * 512 + 16 * lane, a);
    load8(rows + r * 512 + 16 * lane + 8, c);
#pragma unroll
    for (int i = 0; i < 8; ++i) { x[i] = a[i]; x[8 + i] = c[i]; }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  const int X = ef == 0 ? -127 : min(max(ef - 127 - 8, -127), 127);
  // 2^-X as two exact factors (2^-X alone leaves the float range when X = -127)
  const float f1 = __uint_as_float((uint32_t)(127 - X / 2) << 23);
  const float f2 = __uint_as_float((uint32_t)(127 - (X - X / 2)) << 23);
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t v = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) v |= e4m3_encode_satfinite((x[4 * q + u] * f1) * f2) << (8 * u);
    w[q] = v;
  }
  *reinterpret_cast<uint4*>(codes + r * 512 + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
  scales[r * 32 + lane] = (uint8_t)(X + 127);
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
