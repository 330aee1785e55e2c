// sparse_latent_attn: gather the selected cache entries, dequantise them, and run
// multi-head attention in which every key is also its value (one 512-d latent).
//
// Pages: "compresse le KV-Cache de 4 fois", section "Mecanismes", item 1 (one
// 512-dimensional latent shared by keys and values); "890 octets de cache KV par
// token", "Troisiemement" (E2M1 values with an E4M3 scale per 16 channels; a
// 128-token sliding window kept outside the global cache).
//
// Split-key ("flash-decoding") form: one 256-thread block per (sequence, 128 keys).
// The block dequantises its 128 keys to fp16 in shared memory -- exact, since an
// E2M1 value times an E4M3 scale has at most 6 significant bits and lies in
// [2^-10, 2688] -- and runs S = Q V^T and O = P V on the tensor cores
// (mma.sync m16n8k16, fp16 inputs, fp32 accumulation). Queries are scaled per head
// by a power of two so that fp16 keeps their bits; that factor is undone on the
// logits. fp32 queries are split into two fp16 parts (hi + lo). Each block writes an
// unnormalised partial (o, running max m, sum l); k_attn_combine merges the splits.
#pragma once

#include "common.cuh"

namespace csa2 {

constexpr int kAttnThreads = 256;  // 8 warps
constexpr int kAttnKeys = 128;     // keys per block
constexpr float kLog2e = 1.4426950408889634f;

template <int HT>
struct AttnShape {
  static constexpr int H = 16 * HT;
  static constexpr int NKG = 8 / HT;        // key groups (GEMM1) / dim groups (GEMM2)
  static constexpr int KW = kAttnKeys / NKG;
  static constexpr int NT1 = KW / 8;        // n8 tiles of S per warp
  static constexpr int DW = 512 / NKG;
  static constexpr int NT2 = DW / 8;        // n8 tiles of O per warp
  static constexpr size_t q_bytes = (size_t)H * 1024;
  static constexpr size_t v_bytes = (size_t)kAttnKeys * 1024;
  static constexpr size_t p_bytes = (size_t)H * 256;
  static constexpr size_t red_bytes = (size_t)2 * NKG * H * 4;
  static constexpr size_t smem = q_bytes + v_bytes + p_bytes + red_bytes + H * 4 + kAttnKeys * 4;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk, int chunks_per_row) {
  return (uint32_t)(row * chunks_per_row * 16 + ((chunk ^ (row & 7)) << 4));
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

// Write Q (one part) of sequence b into shared memory, scaled by 2^sq[h].
// part 0: fp16(q*2^sq) (the only part for bf16 q); part 1: fp16 of the remainder.
template <int H>
__device__ void attn_load_q(const void* q, int q_dtype, int b, const float* sq_pow,
                            unsigned char* qs, int part) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int h = wid; h < H; h += 8) {
    const float f = sq_pow[h];
    const size_t base = ((size_t)b * H + h) * 512 + 16 * lane;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float v[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float x = load_elem(q, q_dtype, base + 2 * i + j) * f;
        const float hi = __half2float(__float2half_rn(x));
        v[j] = part == 0 ? hi : x - hi;
      }
      w[i] = pack_half2(v[0], v[1]);
    }
    // lane covers dims [16 lane, 16 lane + 16) = chunks 2 lane, 2 lane + 1
    *reinterpret_cast<uint4*>(qs + swz(h, 2 * lane, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(qs + swz(h, 2 * lane + 1, 64)) = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

template <int HT>
__global__ void __launch_bounds__(kAttnThreads, 1)
k_sparse_attn_mma(const void* __restrict__ q, int q_dtype, float scale,
                  const uint8_t* __restrict__ lat_codes, const uint8_t* __restrict__ lat_scales,
                  const int32_t* __restrict__ len, int64_t cap, const int32_t* __restrict__ idx,
                  int k, const uint16_t* __restrict__ swa, int W, int n_idx_splits,
                  float* __restrict__ part_o, float* __restrict__ part_ml) {
  using S = AttnShape<HT>;
  constexpr int H = S::H;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* qs = smem;
  unsigned char* vs = qs + S::q_bytes;
  unsigned char* ps = vs + S::v_bytes;
  float* red_m = reinterpret_cast<float*>(ps + S::p_bytes);
  float* red_l = red_m + S::NKG * H;
  float* sq_pow = red_l + S::NKG * H;                 // per-head 2^sq
  int* key_ok = reinterpret_cast<int*>(sq_pow + H);   // per key: 1 valid, 0 empty

  const int b = blockIdx.y, split = blockIdx.x, n_splits = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;

  // ---- per-head power-of-two scale of the queries
  for (int h = wid; h < H; h += 8) {
    float mx = 0.f;
    const size_t base = ((size_t)b * H + h) * 512;
    for (int d = lane; d < 512; d += 32) mx = fmaxf(mx, fabsf(load_elem(q, q_dtype, base + d)));
    mx = warp_max(mx);
    if (lane == 0) {
      int sq = 0;
      if (mx > 0.f) {
        const int e = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;  // floor(log2) for normals
        sq = min(max(14 - e, -100), 100);
      }
      sq_pow[h] = __uint_as_float((uint32_t)(sq + 127) << 23);  // exact 2^sq
    }
  }

  // ---- the 128 keys of this split, dequantised to fp16 (rows swizzled)
  const bool window_split = split >= n_idx_splits;
  const int n_b = (int)min((int64_t)__ldg(len + b), cap);  // never past the capacity
  {
    const int kk = tid >> 1, hf = tid & 1;
    bool ok = false;
    if (!window_split) {
      const int j = split * kAttnKeys + kk;
      const int pos = j < k ? __ldg(idx + (size_t)b * k + j) : -1;
      if (pos >= n_b) set_dev_error(CSA2_ERR_BOUNDS);
      ok = pos >= 0 && pos < n_b;
      if (ok) {
        const size_t row = (size_t)b * cap + pos;
        const uint4* cp = reinterpret_cast<const uint4*>(lat_codes + row * 256 + 128 * hf);
        const uint4* sp = reinterpret_cast<const uint4*>(lat_scales + row * 32 + 16 * hf);
        const uint4 sv = __ldg(sp);
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {  // 16 code bytes = 32 dims = 2 scale blocks
          const uint4 cv = __ldg(cp + c8);
          const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {   // one 16-dim scale block = 2 chunks of 8 dims
            const int sidx = 2 * c8 + hb;
            const float sf = e4m3_decode((sw[sidx >> 2] >> (8 * (sidx & 3))) & 0xFFu);
            const __half2 s2 = __float2half2_rn(sf);
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
            const int chunk = 32 * hf + 4 * c8 + 2 * hb;
            *reinterpret_cast<uint4*>(vs + swz(kk, chunk, 64)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(vs + swz(kk, chunk + 1, 64)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
      }
    } else {
      const int wr = (split - n_idx_splits) * kAttnKeys + kk;
      ok = wr < W;
      if (ok) {
        const uint4* src = reinterpret_cast<const uint4*>(swa + ((size_t)b * W + wr) * 512 + 256 * hf);
#pragma unroll 4
        for (int c = 0; c < 32; ++c) {
          const uint4 v = __ldg(src + c);
          const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            o[i] = pack_half2(bf16_bits_to_float(vw[i] & 0xFFFFu), bf16_bits_to_float(vw[i] >> 16));
          *reinterpret_cast<uint4*>(vs + swz(kk, 32 * hf + c, 64)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
    if (!ok) {
      for (int c = 0; c < 32; ++c)
        *reinterpret_cast<uint4*>(vs + swz(kk, 32 * hf + c, 64)) = make_uint4(0, 0, 0, 0);
    }
    if (hf == 0) key_ok[kk] = ok ? 1 : 0;
  }
  __syncthreads();

  // ---- S = Q V^T  (warp: head tile ht, keys [kg*KW, kg*KW + KW))
  const int ht = wid % HT, kg = wid / HT;
  float sacc[S::NT1][4];
#pragma unroll
  for (int j = 0; j < S::NT1; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
  const int n_parts = q_dtype == CSA2_F32 ? 2 : 1;
  for (int part = 0; part < n_parts; ++part) {
    __syncthreads();
    attn_load_q<H>(q, q_dtype, b, sq_pow, qs, part);
    __syncthreads();
    const uint32_t qb = smem_u32(qs), vb = smem_u32(vs);
#pragma unroll 2
    for (int ks = 0; ks < 32; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(qb + swz(ht * 16 + (lane & 15), 2 * ks + (lane >> 4), 64), a0, a1, a2, a3);
#pragma unroll
      for (int jj = 0; jj < S::NT1 / 2; ++jj) {
        const int key = kg * S::KW + 16 * jj + (lane & 7) + ((lane >> 4) << 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(vb + swz(key, 2 * ks + ((lane >> 3) & 1), 64), b0, b1, b2, b3);
        mma_f16(sacc[2 * jj], a0, a1, a2, a3, b0, b1);
        mma_f16(sacc[2 * jj + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }

  // ---- softmax over this split's keys (base-2 logits)
  const int h0 = ht * 16 + g, h1 = h0 + 8;
  const float c0 = scale * kLog2e / sq_pow[h0], c1 = scale * kLog2e / sq_pow[h1];
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int j = 0; j < S::NT1; ++j) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = kg * S::KW + 8 * j + 2 * t4 + e;
      const bool okk = key_ok[key] != 0;
      sacc[j][e] = okk ? sacc[j][e] * c0 : -INFINITY;
      sacc[j][2 + e] = okk ? sacc[j][2 + e] * c1 : -INFINITY;
      mx0 = fmaxf(mx0, sacc[j][e]);
      mx1 = fmaxf(mx1, sacc[j][2 + e]);
    }
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  if (t4 == 0) { red_m[kg * H + h0] = mx0; red_m[kg * H + h1] = mx1; }
  __syncthreads();
  float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
  for (int i = 0; i < S::NKG; ++i) { M0 = fmaxf(M0, red_m[i * H + h0]); M1 = fmaxf(M1, red_m[i * H + h1]); }
  const float Z0 = M0 == -INFINITY ? 0.f : M0, Z1 = M1 == -INFINITY ? 0.f : M1;
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int j = 0; j < S::NT1; ++j) {
    const __half2 p01 = __floats2half2_rn(exp2f(sacc[j][0] - Z0), exp2f(sacc[j][1] - Z0));
    const __half2 p23 = __floats2half2_rn(exp2f(sacc[j][2] - Z1), exp2f(sacc[j][3] - Z1));
    const float2 f01 = __half22float2(p01), f23 = __half22float2(p23);
    l0 += f01.x + f01.y;
    l1 += f23.x + f23.y;
    const int key = kg * S::KW + 8 * j + 2 * t4;  // chunk key/8, element key%8
    *reinterpret_cast<__half2*>(ps + swz(h0, key >> 3, 16) + (key & 7) * 2) = p01;
    *reinterpret_cast<__half2*>(ps + swz(h1, key >> 3, 16) + (key & 7) * 2) = p23;
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (t4 == 0) { red_l[kg * H + h0] = l0; red_l[kg * H + h1] = l1; }
  __syncthreads();

  // ---- O = P V  (warp: head tile ht, dims [dg*DW, dg*DW + DW))
  const int dg = wid / HT;
  float oacc[S::NT2][4];
#pragma unroll
  for (int j = 0; j < S::NT2; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
  {
    const uint32_t pb = smem_u32(ps), vb = smem_u32(vs);
#pragma unroll
    for (int ks = 0; ks < kAttnKeys / 16; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(pb + swz(ht * 16 + (lane & 15), 2 * ks + (lane >> 4), 16), a0, a1, a2, a3);
      const int key = 16 * ks + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int jj = 0; jj < S::NT2 / 2; ++jj) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz(key, (dg * S::DW + 16 * jj) / 8 + (lane >> 4), 64), b0, b1, b2, b3);
        mma_f16(oacc[2 * jj], a0, a1, a2, a3, b0, b1);
        mma_f16(oacc[2 * jj + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }

  // ---- partial results
  const size_t pbase = ((size_t)b * n_splits + split) * H;
  float* o0 = part_o + (pbase + h0) * 512;
  float* o1 = part_o + (pbase + h1) * 512;
#pragma unroll
  for (int j = 0; j < S::NT2; ++j) {
    const int d = dg * S::DW + 8 * j + 2 * t4;
    *reinterpret_cast<float2*>(o0 + d) = make_float2(oacc[j][0], oacc[j][1]);
    *reinterpret_cast<float2*>(o1 + d) = make_float2(oacc[j][2], oacc[j][3]);
  }
  if (dg == 0 && t4 == 0) {
    float L0 = 0.f, L1 = 0.f;
#pragma unroll
    for (int i = 0; i < S::NKG; ++i) { L0 += red_l[i * H + h0]; L1 += red_l[i * H + h1]; }
    part_ml[(pbase + h0) * 2] = M0;
    part_ml[(pbase + h0) * 2 + 1] = L0;
    part_ml[(pbase + h1) * 2] = M1;
    part_ml[(pbase + h1) * 2 + 1] = L1;
  }
}

// Merge the split partials: o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
__global__ void __launch_bounds__(128)
k_attn_combine(const float* __restrict__ part_o, const float* __restrict__ part_ml, int n_splits,
               int H, float* __restrict__ out) {
  const int b = blockIdx.y, h = blockIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, part_ml[(((size_t)b * n_splits + s) * H + h) * 2]);
  float L = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (M != -INFINITY) {
    for (int s = 0; s < n_splits; ++s) {
      const size_t ph = ((size_t)b * n_splits + s) * H + h;
      const float m = part_ml[ph * 2];
      if (m == -INFINITY) continue;
      const float wgt = exp2f(m - M);
      L += wgt * part_ml[ph * 2 + 1];
      const float4 v = *reinterpret_cast<const float4*>(part_o + ph * 512 + 4 * threadIdx.x);
      acc[0] += wgt * v.x; acc[1] += wgt * v.y; acc[2] += wgt * v.z; acc[3] += wgt * v.w;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  *reinterpret_cast<float4*>(out + ((size_t)b * H + h) * 512 + 4 * threadIdx.x) =
      make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
}

}  // namespace csa2
