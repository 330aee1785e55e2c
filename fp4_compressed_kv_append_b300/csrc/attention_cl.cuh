// sparse_latent_attn, key-split form: one cluster of C blocks per (sequence, group
// of 64 heads); block r takes keys 128r .. 128r+127 of the row's list (the k
// selected entries, then the W window rows) for all 64 heads, so every selected
// entry is gathered and dequantised once per sequence.
//
// Pages: "compresse le KV-Cache de 4 fois", section "Mecanismes", item 1 (one
// 512-dimensional latent shared by keys and values); "890 octets de cache KV par
// token", "Troisiemement" (E2M1 values with an E4M3 scale per 16 channels; a
// 128-token sliding window kept outside the global cache).
//
// Per block (512 threads, 16 warps; shared memory: Q 64 KB + V 128 KB):
//  * thread t loads a quarter of key t/4 (64 code bytes, 8 E4M3 bytes) into
//    registers at once, then the queries (per-head 2^s scaling as in the chunked
//    form; fp32 queries as fp16 hi + lo, the lo part kept in registers) go to
//    shared memory, then the keys are dequantised to fp16 (exact) into V;
//  * S = Q V^T (mma.sync m16n8k16): warp (mt, kg) covers heads 16mt.. and keys
//    32kg.. over all 512 dims;
//  * softmax over the block's keys (base 2, max per head over the four key
//    groups through shared memory), P rounded to fp16 and kept in the Q area;
//  * O = P V: warp (mt, dq) owns heads 16mt.. and dims 128dq..;
//  * the unnormalised O, max and sum of every block are staged in its shared
//    memory; after a cluster barrier block r merges heads [64r/C, 64(r+1)/C) of
//    all C blocks (distributed shared memory: the weights in one round of remote
//    loads, then every partial row of a thread's items in flight at once).
#pragma once

#include <cooperative_groups.h>

#include "attention.cuh"

namespace csa2 {

constexpr int kAclThreads = 512;
constexpr int kAclKeys = 128;   // keys per block
constexpr int kAclHeads = 64;   // heads per block
constexpr int kAclMaxBlocks = 8;
constexpr int kAclQ = 0;                                  // [64 heads][512] fp16 (swzv); later P [64][128]
constexpr int kAclV = kAclQ + kAclHeads * 1024;           // [128 keys][512] fp16 (swzv)
constexpr int kAclRedM = kAclV + kAclKeys * 1024;         // [4 key groups][64] f32
constexpr int kAclRedL = kAclRedM + 4 * kAclHeads * 4;    // [4][64] f32
constexpr int kAclCoef = kAclRedL + 4 * kAclHeads * 4;    // [64] f32
constexpr int kAclM = kAclCoef + kAclHeads * 4;           // [64] f32: this block's max per head
constexpr int kAclL = kAclM + kAclHeads * 4;              // [64] f32: this block's sum per head
constexpr int kAclKeyOk = kAclL + kAclHeads * 4;          // [128] i32
constexpr int kAclSmem = kAclKeyOk + kAclKeys * 4;
constexpr int kAclOPitch = 520;                           // floats per staged O row (bank spread)
constexpr int kAclO = 0;                                  // [64][520] f32 over Q and V, after O = P V
static_assert(kAclO + kAclHeads * kAclOPitch * 4 <= kAclRedM, "staged O fits over Q and V");
static_assert((kAclMaxBlocks + 1) * kAclHeads * 4 <= kAclM - kAclRedM, "merge weights fit over RedM, RedL and Coef");

// P [64 heads][128 keys] fp16: 16-byte chunk c of row h.
__device__ __forceinline__ uint32_t acl_pidx(int h, int c) { return (uint32_t)(h * 256 + ((c ^ (h & 7)) << 4)); }

template <int NPART>
__global__ void __launch_bounds__(kAclThreads, 1)
k_sparse_attn_cl(const void* __restrict__ q, int q_dtype, float scale, const uint8_t* __restrict__ lat_codes,
                 const uint8_t* __restrict__ lat_scales, const int32_t* __restrict__ len, int64_t cap,
                 const int32_t* __restrict__ idx, int k, const uint16_t* __restrict__ swa, int W, int H,
                 float* __restrict__ out) {
  extern __shared__ __align__(128) unsigned char smem[];
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int r = (int)cluster.block_rank();
  const int hg = blockIdx.x / C, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  unsigned char* qs = smem + kAclQ;
  unsigned char* vs = smem + kAclV;
  float* red_m = reinterpret_cast<float*>(smem + kAclRedM);
  float* red_l = reinterpret_cast<float*>(smem + kAclRedL);
  float* coef = reinterpret_cast<float*>(smem + kAclCoef);
  float* m_blk = reinterpret_cast<float*>(smem + kAclM);
  float* l_blk = reinterpret_cast<float*>(smem + kAclL);
  int* key_ok = reinterpret_cast<int*>(smem + kAclKeyOk);

  const int n_b = (int)min((int64_t)__ldg(len + b), cap);
  const size_t seq_row0 = (size_t)b * cap;

  // ---- this thread's quarter of key kk (dims 128qq .. 128qq+127): codes and scales,
  // loaded after the query loads are in flight
  const int kk = tid >> 2, qq = tid & 3;
  const int j = r * kAclKeys + kk;  // position in the row's key list
  int kind = 0;                     // 0 none, 1 cache entry, 2 window row
  uint4 cv[4];
  uint2 sc8 = make_uint2(0u, 0u);

  // ---- queries: heads 4w .. 4w+3 (lane: dims 16 lane .. 16 lane + 15); every load first
  uint32_t qlo[4][8];  // fp32 queries: the fp16 remainder, stored after the first S pass
  {
    float x[4][16];
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      const size_t base = ((size_t)b * H + hg * kAclHeads + 4 * w + hh) * 512 + 16 * lane;
      if (q_dtype == CSA2_F32) {
        const float4* p4 = reinterpret_cast<const float4*>(static_cast<const float*>(q) + base);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 v = __ldg(p4 + i);
          x[hh][4 * i] = v.x; x[hh][4 * i + 1] = v.y; x[hh][4 * i + 2] = v.z; x[hh][4 * i + 3] = v.w;
        }
      } else {
        const uint4* p4 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(q) + base);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint4 v = __ldg(p4 + i);
          const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x[hh][8 * i + 2 * e] = __uint_as_float(ww[e] << 16);
            x[hh][8 * i + 2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
          }
        }
      }
    }
    if (j < k) {
      const int pos = idx ? __ldg(idx + (size_t)b * k + j) : -1;
      if (pos >= n_b) set_dev_error(CSA2_ERR_BOUNDS);
      if (pos >= 0 && pos < n_b) {
        kind = 1;
        const uint4* src = reinterpret_cast<const uint4*>(lat_codes + (seq_row0 + pos) * 256 + 64 * qq);
#pragma unroll
        for (int i = 0; i < 4; ++i) cv[i] = __ldg(src + i);
        sc8 = __ldg(reinterpret_cast<const uint2*>(lat_scales + (seq_row0 + pos) * 32 + 8 * qq));
      }
    } else if (j < k + W) {
      kind = 2;
    }
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      const int h = 4 * w + hh;
      float mx = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(x[hh][i]));
      mx = warp_max(mx);
      int sq = 0;
      if (mx > 0.f) {
        const int e = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;  // floor(log2) for normal mx
        sq = min(max(14 - e, -100), 100);
      }
      const float f = __uint_as_float((uint32_t)(sq + 127) << 23);  // 2^sq, exact
      if (lane == 0) coef[h] = scale * kLog2e * __uint_as_float((uint32_t)(127 - sq) << 23);
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float y0 = x[hh][2 * i] * f, y1 = x[hh][2 * i + 1] * f;
        const float h0 = __half2float(__float2half_rn(y0)), h1 = __half2float(__float2half_rn(y1));
        o[i] = pack_half2(h0, h1);
        qlo[hh][i] = NPART == 2 ? pack_half2(y0 - h0, y1 - h1) : 0u;
      }
      *reinterpret_cast<uint4*>(qs + swzv(h, 2 * lane)) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(qs + swzv(h, 2 * lane + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }

  // ---- keys -> fp16 V rows (invalid keys: zero rows)
  if (kind == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // 16 code bytes = 32 dims = 2 scale blocks
      const uint32_t cw[4] = {cv[i].x, cv[i].y, cv[i].z, cv[i].w};
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
            const __half2_raw rr =
                __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((word >> (8 * by)) & 0xFFu), __NV_E2M1);
            const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&rr), s2);
            o[4 * wv + by] = *reinterpret_cast<const uint32_t*>(&v);
          }
        }
        const int chunk = 16 * qq + 4 * i + 2 * hb;
        *reinterpret_cast<uint4*>(vs + swzv(kk, chunk)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(vs + swzv(kk, chunk + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  } else if (kind == 2) {
    const uint4* src = reinterpret_cast<const uint4*>(swa + ((size_t)b * W + (j - k)) * 512 + 128 * qq);
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
  } else {
#pragma unroll 4
    for (int i = 0; i < 16; ++i) *reinterpret_cast<uint4*>(vs + swzv(kk, 16 * qq + i)) = make_uint4(0, 0, 0, 0);
  }
  if (qq == 0) key_ok[kk] = kind != 0 ? 1 : 0;
  __syncthreads();

  // ---- S = Q V^T: warp (mt, kg): heads 16mt .. 16mt+15, keys 32kg .. 32kg+31
  const int mt = w & 3, kg = w >> 2;
  float sacc[4][4];
#pragma unroll
  for (int jn = 0; jn < 4; ++jn) sacc[jn][0] = sacc[jn][1] = sacc[jn][2] = sacc[jn][3] = 0.f;
#pragma unroll
  for (int part = 0; part < NPART; ++part) {
    if (part == 1) {  // the fp16 remainder of fp32 queries replaces the first part
      __syncthreads();
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const int h = 4 * w + hh;
        *reinterpret_cast<uint4*>(qs + swzv(h, 2 * lane)) =
            make_uint4(qlo[hh][0], qlo[hh][1], qlo[hh][2], qlo[hh][3]);
        *reinterpret_cast<uint4*>(qs + swzv(h, 2 * lane + 1)) =
            make_uint4(qlo[hh][4], qlo[hh][5], qlo[hh][6], qlo[hh][7]);
      }
      __syncthreads();
    }
    const uint32_t qb = smem_u32(qs), vb = smem_u32(vs);
#pragma unroll 4
    for (int ks = 0; ks < 32; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(qb + swzv(16 * mt + (lane & 15), 2 * ks + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int key = 32 * kg + 16 * jj + (lane & 7) + ((lane >> 4) << 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(vb + swzv(key, 2 * ks + ((lane >> 3) & 1)), b0, b1, b2, b3);
        mma_f16(sacc[2 * jj], a0, a1, a2, a3, b0, b1);
        mma_f16(sacc[2 * jj + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }

  // ---- softmax over this block's keys (heads h0 = 16mt + g, h1 = h0 + 8)
  const int h0 = 16 * mt + g, h1 = h0 + 8;
  {
    const float cf0 = coef[h0], cf1 = coef[h1];
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int jn = 0; jn < 4; ++jn) {
      const int key = 32 * kg + 8 * jn + 2 * t4;
      const bool ok0 = key_ok[key] != 0, ok1 = key_ok[key + 1] != 0;
      sacc[jn][0] = ok0 ? sacc[jn][0] * cf0 : -INFINITY;
      sacc[jn][1] = ok1 ? sacc[jn][1] * cf0 : -INFINITY;
      sacc[jn][2] = ok0 ? sacc[jn][2] * cf1 : -INFINITY;
      sacc[jn][3] = ok1 ? sacc[jn][3] * cf1 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(sacc[jn][0], sacc[jn][1]));
      mx1 = fmaxf(mx1, fmaxf(sacc[jn][2], sacc[jn][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    if (t4 == 0) {
      red_m[kg * kAclHeads + h0] = mx0;
      red_m[kg * kAclHeads + h1] = mx1;
    }
    __syncthreads();  // (also: every warp is done reading Q, so P may overwrite it)
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      M0 = fmaxf(M0, red_m[i * kAclHeads + h0]);
      M1 = fmaxf(M1, red_m[i * kAclHeads + h1]);
    }
    const float Z0 = M0 == -INFINITY ? 0.f : M0, Z1 = M1 == -INFINITY ? 0.f : M1;
    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
    for (int jn = 0; jn < 4; ++jn) {
      const int key = 32 * kg + 8 * jn + 2 * t4;
      const __half2 p01 = __floats2half2_rn(exp2f(sacc[jn][0] - Z0), exp2f(sacc[jn][1] - Z0));
      const __half2 p23 = __floats2half2_rn(exp2f(sacc[jn][2] - Z1), exp2f(sacc[jn][3] - Z1));
      const float2 f01 = __half22float2(p01), f23 = __half22float2(p23);
      ls0 += f01.x + f01.y;
      ls1 += f23.x + f23.y;
      *reinterpret_cast<__half2*>(qs + acl_pidx(h0, key >> 3) + (key & 7) * 2) = p01;
      *reinterpret_cast<__half2*>(qs + acl_pidx(h1, key >> 3) + (key & 7) * 2) = p23;
    }
    ls0 += __shfl_xor_sync(0xffffffffu, ls0, 1);
    ls0 += __shfl_xor_sync(0xffffffffu, ls0, 2);
    ls1 += __shfl_xor_sync(0xffffffffu, ls1, 1);
    ls1 += __shfl_xor_sync(0xffffffffu, ls1, 2);
    if (t4 == 0) {
      red_l[kg * kAclHeads + h0] = ls0;
      red_l[kg * kAclHeads + h1] = ls1;
      if (kg == 0) {
        m_blk[h0] = M0;
        m_blk[h1] = M1;
      }
    }
  }
  __syncthreads();
  if (tid < kAclHeads) l_blk[tid] = red_l[tid] + red_l[kAclHeads + tid] + red_l[2 * kAclHeads + tid] +
                                    red_l[3 * kAclHeads + tid];

  // ---- O = P V: warp (mt, dq): heads 16mt .., dims 128dq .. 128dq+127
  const int dq = w >> 2;
  float oacc[16][4];
#pragma unroll
  for (int jn = 0; jn < 16; ++jn) oacc[jn][0] = oacc[jn][1] = oacc[jn][2] = oacc[jn][3] = 0.f;
  {
    const uint32_t pb = smem_u32(qs), vb = smem_u32(vs);
#pragma unroll 2
    for (int ks = 0; ks < kAclKeys / 16; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(pb + acl_pidx(16 * mt + (lane & 15), 2 * ks + (lane >> 4)), a0, a1, a2, a3);
      const int key = 16 * ks + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swzv(key, 16 * dq + 2 * jj + (lane >> 4)), b0, b1, b2, b3);
        mma_f16(oacc[2 * jj], a0, a1, a2, a3, b0, b1);
        mma_f16(oacc[2 * jj + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
  // ---- merge: block r finishes heads [64r/C, 64(r+1)/C) of all C blocks. Every
  // block stages its unnormalised O over its own Q and V; after a cluster barrier
  // block r reads the max and sum of its heads from every block (one round of
  // remote loads into shared memory), then each thread loads the C partial rows
  // of its items with all loads in flight at once.
  __syncthreads();  // every warp is done with P and V: stage O over them
  {
    float* os = reinterpret_cast<float*>(smem + kAclO);
#pragma unroll
    for (int jn = 0; jn < 16; ++jn) {
      const int d = 128 * dq + 8 * jn + 2 * t4;
      *reinterpret_cast<float2*>(os + h0 * kAclOPitch + d) = make_float2(oacc[jn][0], oacc[jn][1]);
      *reinterpret_cast<float2*>(os + h1 * kAclOPitch + d) = make_float2(oacc[jn][2], oacc[jn][3]);
    }
  }
  cluster.sync();  // every block's O, max and sum are staged
  const int hb0 = r * kAclHeads / C, nh = (r + 1) * kAclHeads / C - hb0;
  float* wa = reinterpret_cast<float*>(smem + kAclRedM);  // [C][nh]: weight of block c for head hb0 + i (over RedM, RedL, Coef)
  float* winv = wa + kAclMaxBlocks * kAclHeads;            // [nh]: 1 / merged sum
  if (tid < nh) {
    const int h = hb0 + tid;
    float mc[kAclMaxBlocks], lc[kAclMaxBlocks];
#pragma unroll
    for (int c = 0; c < kAclMaxBlocks; ++c) {
      mc[c] = c < C ? cluster.map_shared_rank(m_blk, (unsigned)c)[h] : -INFINITY;
      lc[c] = c < C ? cluster.map_shared_rank(l_blk, (unsigned)c)[h] : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < kAclMaxBlocks; ++c) M = fmaxf(M, mc[c]);
    const float Z = M == -INFINITY ? 0.f : M;
    float L = 0.f;
#pragma unroll
    for (int c = 0; c < kAclMaxBlocks; ++c) {
      const float a = exp2f(mc[c] - Z);  // a block with no valid key (or none at all): 0
      L += a * lc[c];
      if (c < C) wa[c * kAclHeads + tid] = a;
    }
    winv[tid] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  {
    constexpr int kPer = 2;  // items (head, 4 dims) per thread per round
    const int items = nh * 128;
    for (int it0 = tid; it0 < items; it0 += kPer * kAclThreads) {
      float4 v[kPer][kAclMaxBlocks];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int it = it0 + u * kAclThreads;
        const int hl = it >> 7, d4 = it & 127;
#pragma unroll
        for (int c = 0; c < kAclMaxBlocks; ++c)
          if (c < C && it < items)
            v[u][c] = *reinterpret_cast<const float4*>(
                cluster.map_shared_rank(reinterpret_cast<float*>(smem + kAclO), (unsigned)c) +
                (hb0 + hl) * kAclOPitch + 4 * d4);
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int it = it0 + u * kAclThreads;
        if (it < items) {
          const int hl = it >> 7, d4 = it & 127;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int c = 0; c < kAclMaxBlocks; ++c) {
            if (c < C) {
              const float a = wa[c * kAclHeads + hl];
              acc.x += a * v[u][c].x;
              acc.y += a * v[u][c].y;
              acc.z += a * v[u][c].z;
              acc.w += a * v[u][c].w;
            }
          }
          const float inv = winv[hl];
          *reinterpret_cast<float4*>(out + ((size_t)b * H + hg * kAclHeads + hb0 + hl) * 512 + 4 * d4) =
              make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
      }
    }
  }
  cluster.sync();  // no block leaves while another reads its shared memory
}

}  // namespace csa2
