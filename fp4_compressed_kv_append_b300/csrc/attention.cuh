// sparse_latent_attn: gather the selected cache entries, dequantise them, and run
// multi-head attention in which every key is also its value (one 512-d latent).
//
// Pages: "compresse le KV-Cache de 4 fois", section "Mecanismes", item 1 (one
// 512-dimensional latent shared by keys and values); "890 octets de cache KV par
// token", "Troisiemement" (E2M1 values with an E4M3 scale per 16 channels; a
// 128-token sliding window kept outside the global cache).
//
// A cluster of two 256-thread blocks per (sequence, group of 16 heads) walks the
// selected keys, then the window rows, in chunks of 64 with an online softmax,
// block r taking half r of the chunks; block 1 then hands its (max, sum, O) to
// block 0 through distributed shared memory and block 0 writes the merged
// result -- nothing partial goes through global memory. Per chunk:
//  * the raw codes and scales of the chunk's entries were gathered into shared
//    memory by cp.async during the previous chunk; they are dequantised to fp16
//    (exact: an E2M1 value times an E4M3 scale has at most 6 significant bits and
//    lies in [2^-10, 2688]); window rows (bf16) are converted directly;
//  * S = Q V^T on the tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate):
//    warp (kg, dg) covers keys 32kg..32kg+31 over dims 128dg..128dg+127 with its
//    query fragments held in registers; the four dim-group partials meet in
//    shared memory;
//  * softmax in base 2 with a running max per head; P is rounded to fp16;
//  * O += P V, warp w owning output dims 64w..64w+63.
// Queries are scaled per head by a power of two 2^s so that fp16 keeps their
// bits (fp32 queries are split into fp16 hi + lo parts); the factor is undone in
// the logit coefficient.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace csa2 {

constexpr int kAttnThreads = 256;  // 8 warps
constexpr int kAttnChunk = 64;     // keys per chunk
constexpr int kAttnHeads = 16;     // heads per block
constexpr float kLog2e = 1.4426950408889634f;

// shared-memory layout (bytes)
constexpr int kAttnV = 0;                                     // [64 keys][512] fp16, swizzled; Q first
constexpr int kAttnRawPitch = 272;                           // bytes per raw code row (padded)
constexpr int kAttnRawC = kAttnV + kAttnChunk * 1024;         // [64][272] codes
constexpr int kAttnRawS = kAttnRawC + kAttnChunk * kAttnRawPitch;  // [64][32] E4M3 scales
constexpr int kAttnSPitch = 68;                               // floats per S-partial row
constexpr int kAttnSPart = kAttnRawS + kAttnChunk * 32;       // [4 dg][16 heads][68] f32
constexpr int kAttnP = kAttnSPart + 4 * kAttnHeads * kAttnSPitch * 4;  // [16][64] fp16, swizzled
constexpr int kAttnRedM = kAttnP + kAttnHeads * 128;          // [8 warps][16] f32
constexpr int kAttnRedL = kAttnRedM + 8 * kAttnHeads * 4;     // [8 warps][16] f32
constexpr int kAttnCoef = kAttnRedL + 8 * kAttnHeads * 4;     // [16] f32
constexpr int kAttnKeyOk = kAttnCoef + kAttnHeads * 4;        // [64] i32
constexpr int kAttnXO = kAttnV;                              // partner partials: [32][256] f32 (end)
constexpr int kAttnXML = kAttnSPart;                          // partner m, l per head: [2][16] f32
constexpr int kAttnSmem = kAttnKeyOk + kAttnChunk * 4;

__device__ __forceinline__ uint32_t swz(int row, int chunk, int chunks_per_row) {
  return (uint32_t)(row * chunks_per_row * 16 + ((chunk ^ (row & 7)) << 4));
}

// 16-byte chunk c of a 1024-byte row (keys, or query heads): the chunk index is
// XORed with the row (8 consecutive rows of one chunk column hit 8 bank groups,
// as ldmatrix reads them) and with its own bits 4-5 (the four threads that
// dequantise chunks c, c+16, c+32, c+48 of one row hit 4 bank groups).
__device__ __forceinline__ uint32_t swzv(int row, int chunk) {
  return (uint32_t)(row * 1024 + ((chunk ^ (row & 7) ^ ((chunk >> 4) & 3)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}


// Issue the gathers of the raw codes and scales of index chunk c.
__device__ __forceinline__ void attn_prefetch_chunk(unsigned char* smem, const uint8_t* lat_codes,
                                                    const uint8_t* lat_scales, const int32_t* idxrow, int k,
                                                    int c, int n_b, size_t seq_row0) {
  const int tid = threadIdx.x;
  {
    const int kk = tid >> 2, part = tid & 3;  // 4 x 64 bytes of codes per key
    const int j = c * kAttnChunk + kk;
    const int pos = j < k ? __ldg(idxrow + j) : -1;
    if (pos >= 0 && pos < n_b) {
      const uint8_t* src = lat_codes + (seq_row0 + pos) * 256 + 64 * part;
      const uint32_t dst = smem_u32(smem + kAttnRawC + kk * kAttnRawPitch + 64 * part);
#pragma unroll
      for (int i = 0; i < 4; ++i) cp_async16(dst + 16 * i, src + 16 * i);
    }
  }
  if (tid < 2 * kAttnChunk) {
    const int kk = tid >> 1, half = tid & 1;
    const int j = c * kAttnChunk + kk;
    const int pos = j < k ? __ldg(idxrow + j) : -1;
    if (pos >= 0 && pos < n_b)
      cp_async16(smem_u32(smem + kAttnRawS + kk * 32 + 16 * half), lat_scales + (seq_row0 + pos) * 32 + 16 * half);
  }
  cp_async_commit();
}

template <int NPART>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttnThreads, NPART == 1 ? 2 : 1)
k_sparse_attn(const void* __restrict__ q, int q_dtype, float scale, const uint8_t* __restrict__ lat_codes,
              const uint8_t* __restrict__ lat_scales, const int32_t* __restrict__ len, int64_t cap,
              const int32_t* __restrict__ idx, int k, const uint16_t* __restrict__ swa,
              const uint8_t* __restrict__ swa_codes, const uint8_t* __restrict__ swa_scales, int W, int H,
              float* __restrict__ out) {
  pdl_wait_and_release();
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* vs = smem + kAttnV;
  float* spart = reinterpret_cast<float*>(smem + kAttnSPart);
  unsigned char* ps = smem + kAttnP;
  float* red_m = reinterpret_cast<float*>(smem + kAttnRedM);
  float* red_l = reinterpret_cast<float*>(smem + kAttnRedL);
  float* coef = reinterpret_cast<float*>(smem + kAttnCoef);
  int* key_ok = reinterpret_cast<int*>(smem + kAttnKeyOk);

  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int half = (int)cluster.block_rank();  // 0 or 1: which half of the chunks
  const int hg = blockIdx.x >> 1, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int kg = w & 1, dg = w >> 1;
  const int n_b = (int)min((int64_t)__ldg(len + b), cap);
  const size_t seq_row0 = (size_t)b * cap;
  const int32_t* idxrow = idx ? idx + (size_t)b * k : nullptr;
  const int n_idx_chunks = (k + kAttnChunk - 1) / kAttnChunk;
  const int n_chunks = n_idx_chunks + (W + kAttnChunk - 1) / kAttnChunk;
  const int c_begin = half == 0 ? 0 : (n_chunks + 1) / 2;
  const int c_end = half == 0 ? (n_chunks + 1) / 2 : n_chunks;

  if (c_begin < n_idx_chunks && c_begin < c_end)
    attn_prefetch_chunk(smem, lat_codes, lat_scales, idxrow, k, c_begin, n_b, seq_row0);

  // ---- queries: per-head 2^s, fp16 parts into the V area, then register fragments
  {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = 2 * w + hh;
      const size_t base = ((size_t)b * H + hg * kAttnHeads + h) * 512 + 16 * lane;
      float x[16];
      if (q_dtype == CSA2_F32) {
        const float4* p4 = reinterpret_cast<const float4*>(static_cast<const float*>(q) + base);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 v = __ldg(p4 + i);
          x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
        }
      } else {
        const uint4* p4 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(q) + base);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint4 v = __ldg(p4 + i);
          const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            x[8 * i + 2 * j] = __uint_as_float(ww[j] << 16);
            x[8 * i + 2 * j + 1] = __uint_as_float(ww[j] & 0xFFFF0000u);
          }
        }
      }
      float mx = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(x[i]));
      mx = warp_max(mx);
      int sq = 0;
      if (mx > 0.f) {
        const int e = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;  // floor(log2) for normal mx
        sq = min(max(14 - e, -100), 100);
      }
      const float f = __uint_as_float((uint32_t)(sq + 127) << 23);  // 2^sq, exact
      if (lane == 0) coef[h] = scale * kLog2e * __uint_as_float((uint32_t)(127 - sq) << 23);
#pragma unroll
      for (int part = 0; part < NPART; ++part) {
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float v[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float y = x[2 * i + j] * f;
            const float hi = __half2float(__float2half_rn(y));
            v[j] = part == 0 ? hi : y - hi;
          }
          o[i] = pack_half2(v[0], v[1]);
        }
        unsigned char* qs = vs + part * (kAttnHeads * 1024);
        *reinterpret_cast<uint4*>(qs + swzv(h, 2 * lane)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(qs + swzv(h, 2 * lane + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  }
  __syncthreads();
  uint32_t qf[NPART][8][4];
#pragma unroll
  for (int part = 0; part < NPART; ++part) {
    const uint32_t qb = smem_u32(vs + part * (kAttnHeads * 1024));
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      ldsm_x4(qb + swzv(lane & 15, 16 * dg + 2 * ks + (lane >> 4)), qf[part][ks][0], qf[part][ks][1],
              qf[part][ks][2], qf[part][ks][3]);
  }
  const float cf0 = coef[g], cf1 = coef[g + 8];
  __syncthreads();  // the V area is free again

  float oacc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads g, g+8

  for (int c = c_begin; c < c_end; ++c) {
    // ---- chunk keys -> fp16 V rows
    {
      const int kk = tid >> 2, qq = tid & 3;  // key kk, dims 128qq .. 128qq+127
      bool ok = false;
      if (c < n_idx_chunks) {
        cp_async_wait_all();
        __syncthreads();
        const int j = c * kAttnChunk + kk;
        const int pos = j < k ? __ldg(idxrow + j) : -1;
        if (pos >= n_b) set_dev_error(CSA2_ERR_BOUNDS);
        ok = pos >= 0 && pos < n_b;
        if (ok) {
          const unsigned char* rc = smem + kAttnRawC + kk * kAttnRawPitch + 64 * qq;
          const unsigned char* rs = smem + kAttnRawS + kk * 32 + 8 * qq;
          const uint2 sc8 = *reinterpret_cast<const uint2*>(rs);
#pragma unroll
          for (int i0 = 0; i0 < 4; ++i0) {  // 16 code bytes = 32 dims = 2 scale blocks
            const int i = (i0 + qq) & 3;     // rotated: the four threads of a row read distinct banks
            const uint4 cv = *reinterpret_cast<const uint4*>(rc + 16 * i);
            const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              const int sidx = 2 * i + hb;
              const uint32_t sbyte = ((sidx < 4 ? sc8.x : sc8.y) >> (8 * (sidx & 3))) & 0xFFu;
              const __half2 s2 = __float2half2_rn(e4m3_decode(sbyte));
              uint32_t o[8];
#pragma unroll
              for (int wv = 0; wv < 2; ++wv) {
                const uint32_t word = cw[2 * hb + wv];
#pragma unroll
                for (int by = 0; by < 4; ++by) {
                  const __half2_raw r =
                      __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((word >> (8 * by)) & 0xFFu), __NV_E2M1);
                  const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&r), s2);
                  o[4 * wv + by] = *reinterpret_cast<const uint32_t*>(&v);
                }
              }
              const int chunk = 16 * qq + 4 * i + 2 * hb;
              *reinterpret_cast<uint4*>(vs + swzv(kk, chunk)) = make_uint4(o[0], o[1], o[2], o[3]);
              *reinterpret_cast<uint4*>(vs + swzv(kk, chunk + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
            }
          }
        }
      } else {
        __syncthreads();
        const int wr = (c - n_idx_chunks) * kAttnChunk + kk;
        ok = wr < W;
        if (ok && swa_codes) {  // FP8 window row: E4M3 values times the block's 2^(e - 127)
          const size_t wrow = (size_t)b * W + wr;
          const uint2 sv = __ldg(reinterpret_cast<const uint2*>(swa_scales + wrow * 32 + 8 * qq));
#pragma unroll 2
          for (int i = 0; i < 8; ++i) {  // blocks 8 qq + i: dims 128 qq + 16 i ..
            const float f = e8m0_decode(((i < 4 ? sv.x : sv.y) >> (8 * (i & 3))) & 0xFFu);
            const uint4 cv = __ldg(reinterpret_cast<const uint4*>(swa_codes + wrow * 512 + 128 * qq) + i);
            const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
            uint32_t o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint32_t byte2 = (cw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
              o[e] = pack_half2(e4m3_decode(byte2 & 0xFFu) * f, e4m3_decode(byte2 >> 8) * f);
            }
            *reinterpret_cast<uint4*>(vs + swzv(kk, 16 * qq + 2 * i)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(vs + swzv(kk, 16 * qq + 2 * i + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        } else if (ok) {
          const uint4* src = reinterpret_cast<const uint4*>(swa + ((size_t)b * W + wr) * 512 + 128 * qq);
#pragma unroll 4
          for (int i = 0; i < 16; ++i) {
            const uint4 v = __ldg(src + i);
            const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              o[e] = pack_half2(bf16_bits_to_float(vw[e] & 0xFFFFu), bf16_bits_to_float(vw[e] >> 16));
            *reinterpret_cast<uint4*>(vs + swzv(kk, 16 * qq + i)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
      if (!ok) {
#pragma unroll 4
        for (int i = 0; i < 16; ++i)
          *reinterpret_cast<uint4*>(vs + swzv(kk, 16 * qq + i)) = make_uint4(0, 0, 0, 0);
      }
      if (qq == 0) key_ok[kk] = ok ? 1 : 0;
    }
    __syncthreads();
    if (c + 1 < n_idx_chunks && c + 1 < c_end)
      attn_prefetch_chunk(smem, lat_codes, lat_scales, idxrow, k, c + 1, n_b, seq_row0);

    // ---- S partial = Q V^T over this warp's keys (32kg..) and dims (128dg..)
    {
      float sacc[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
      const uint32_t vb = smem_u32(vs);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int key = 32 * kg + 16 * jj + (lane & 7) + ((lane >> 4) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(vb + swzv(key, 16 * dg + 2 * ks + ((lane >> 3) & 1)), b0, b1, b2, b3);
#pragma unroll
          for (int part = 0; part < NPART; ++part) {
            mma_f16(sacc[2 * jj], qf[part][ks][0], qf[part][ks][1], qf[part][ks][2], qf[part][ks][3], b0, b1);
            mma_f16(sacc[2 * jj + 1], qf[part][ks][0], qf[part][ks][1], qf[part][ks][2], qf[part][ks][3], b2, b3);
          }
        }
      }
      float* sp = spart + dg * kAttnHeads * kAttnSPitch;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = 32 * kg + 8 * j + 2 * t4;
        *reinterpret_cast<float2*>(sp + g * kAttnSPitch + key) = make_float2(sacc[j][0], sacc[j][1]);
        *reinterpret_cast<float2*>(sp + (g + 8) * kAttnSPitch + key) = make_float2(sacc[j][2], sacc[j][3]);
      }
    }
    __syncthreads();

    // ---- softmax: warp w finishes keys 8w..8w+7 (heads g, g+8)
    float alpha0, alpha1;
    {
      const int key = 8 * w + 2 * t4;
      float s[4] = {0.f, 0.f, 0.f, 0.f};  // (g, key), (g, key+1), (g+8, key), (g+8, key+1)
#pragma unroll
      for (int d = 0; d < 4; ++d) {
        const float* sp = spart + d * kAttnHeads * kAttnSPitch;
        const float2 a = *reinterpret_cast<const float2*>(sp + g * kAttnSPitch + key);
        const float2 bq = *reinterpret_cast<const float2*>(sp + (g + 8) * kAttnSPitch + key);
        s[0] += a.x; s[1] += a.y; s[2] += bq.x; s[3] += bq.y;
      }
      const bool ok0 = key_ok[key] != 0, ok1 = key_ok[key + 1] != 0;
      s[0] = ok0 ? s[0] * cf0 : -INFINITY;
      s[1] = ok1 ? s[1] * cf0 : -INFINITY;
      s[2] = ok0 ? s[2] * cf1 : -INFINITY;
      s[3] = ok1 ? s[3] * cf1 : -INFINITY;
      float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      if (t4 == 0) {
        red_m[w * kAttnHeads + g] = mx0;
        red_m[w * kAttnHeads + g + 8] = mx1;
      }
      __syncthreads();
      float M0 = m0, M1 = m1;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        M0 = fmaxf(M0, red_m[i * kAttnHeads + g]);
        M1 = fmaxf(M1, red_m[i * kAttnHeads + g + 8]);
      }
      const float Z0 = M0 == -INFINITY ? 0.f : M0, Z1 = M1 == -INFINITY ? 0.f : M1;
      alpha0 = exp2f(m0 - Z0);  // m = -inf -> 0 (O and l are still 0)
      alpha1 = exp2f(m1 - Z1);
      m0 = M0;
      m1 = M1;
      const __half2 p01 = __floats2half2_rn(exp2f(s[0] - Z0), exp2f(s[1] - Z0));
      const __half2 p23 = __floats2half2_rn(exp2f(s[2] - Z1), exp2f(s[3] - Z1));
      const float2 f01 = __half22float2(p01), f23 = __half22float2(p23);
      float ls0 = f01.x + f01.y, ls1 = f23.x + f23.y;
      *reinterpret_cast<__half2*>(ps + swz(g, key >> 3, 8) + (key & 7) * 2) = p01;
      *reinterpret_cast<__half2*>(ps + swz(g + 8, key >> 3, 8) + (key & 7) * 2) = p23;
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, 1);
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, 2);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, 1);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, 2);
      if (t4 == 0) {
        red_l[w * kAttnHeads + g] = ls0;
        red_l[w * kAttnHeads + g + 8] = ls1;
      }
      __syncthreads();
      float L0 = 0.f, L1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        L0 += red_l[i * kAttnHeads + g];
        L1 += red_l[i * kAttnHeads + g + 8];
      }
      l0 = l0 * alpha0 + L0;
      l1 = l1 * alpha1 + L1;
    }

    // ---- O = alpha O + P V (warp w: dims 64w .. 64w+63)
    {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        oacc[j][0] *= alpha0; oacc[j][1] *= alpha0;
        oacc[j][2] *= alpha1; oacc[j][3] *= alpha1;
      }
      const uint32_t pb = smem_u32(ps), vb = smem_u32(vs);
#pragma unroll
      for (int ks = 0; ks < kAttnChunk / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(pb + swz(lane & 15, 2 * ks + (lane >> 4), 8), a0, a1, a2, a3);
        const int key = 16 * ks + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + swzv(key, (64 * w + 16 * jj) / 8 + (lane >> 4)), b0, b1, b2, b3);
          mma_f16(oacc[2 * jj], a0, a1, a2, a3, b0, b1);
          mma_f16(oacc[2 * jj + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
  }

  // ---- merge the two halves (block 1 hands (m, l, O) to block 0), normalise, store
  cluster.sync();  // both halves are done with their shared memory
  float* xo = cluster.map_shared_rank(reinterpret_cast<float*>(smem + kAttnXO), 0);
  float* xml = cluster.map_shared_rank(reinterpret_cast<float*>(smem + kAttnXML), 0);
  if (half == 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) xo[(4 * j + e) * kAttnThreads + tid] = oacc[j][e];
    if (w == 0 && t4 == 0) {
      xml[g] = m0;
      xml[g + 8] = m1;
      xml[16 + g] = l0;
      xml[16 + g + 8] = l1;
    }
  }
  cluster.sync();  // no block touches the other's shared memory after this point
  if (half == 1) return;
  {
    const float pm0 = xml[g], pm1 = xml[g + 8], pl0 = xml[16 + g], pl1 = xml[16 + g + 8];
    const float M0 = fmaxf(m0, pm0), M1 = fmaxf(m1, pm1);
    const float Z0 = M0 == -INFINITY ? 0.f : M0, Z1 = M1 == -INFINITY ? 0.f : M1;
    const float a0 = exp2f(m0 - Z0), b0 = exp2f(pm0 - Z0), a1 = exp2f(m1 - Z1), b1 = exp2f(pm1 - Z1);
    const float L0 = l0 * a0 + pl0 * b0, L1 = l1 * a1 + pl1 * b1;
    const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
    float* o0 = out + ((size_t)b * H + hg * kAttnHeads + g) * 512;
    float* o1 = o0 + 8 * 512;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int d = 64 * w + 8 * j + 2 * t4;
      const float x0 = (oacc[j][0] * a0 + xo[(4 * j + 0) * kAttnThreads + tid] * b0) * inv0;
      const float x1 = (oacc[j][1] * a0 + xo[(4 * j + 1) * kAttnThreads + tid] * b0) * inv0;
      const float x2 = (oacc[j][2] * a1 + xo[(4 * j + 2) * kAttnThreads + tid] * b1) * inv1;
      const float x3 = (oacc[j][3] * a1 + xo[(4 * j + 3) * kAttnThreads + tid] * b1) * inv1;
      *reinterpret_cast<float2*>(o0 + d) = make_float2(x0, x1);
      *reinterpret_cast<float2*>(o1 + d) = make_float2(x2, x3);
    }
  }
}

}  // namespace csa2
