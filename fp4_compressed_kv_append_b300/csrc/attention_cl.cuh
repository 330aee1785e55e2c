// sparse_latent_attn, key-split form: C blocks per (sequence, group of 64 heads,
// layer), C from 1 to 8 (a cluster when C > 1). The row's key list (the k selected
// entries, then the W window rows) is dealt out key by key: block r takes list
// positions r, r + C, r + 2C, ..., in chunks of 128, so every selected entry is
// gathered and dequantised once per sequence and the window rows spread evenly over
// the blocks.
//
// Pages: "compresse le KV-Cache de 4 fois", section "Mecanismes", item 1 (one
// 512-dimensional latent shared by keys and values); "890 octets de cache KV par
// token", "Troisiemement" (E2M1 values with an E4M3 scale per 16 channels; a
// 128-token sliding window kept outside the global cache).
//
// Per block (512 threads, 16 warps; shared memory: Q 64 KB, V 128 KB, S 32 KB; all
// 512 columns of tensor memory):
//  * the queries (per-head 2^s scaling as in the chunked form; fp32 queries as fp16
//    hi + lo, the lo part kept in registers) are staged once in shared memory and
//    serve every chunk;
//  * per chunk: thread t holds a quarter of key t/4 (64 code bytes, 8 E4M3 bytes,
//    loaded while the previous chunk's S^T was on the tensor cores) and dequantises it to fp16
//    (exact) into V; S^T = V Q^T on the 5th-generation tensor cores (one thread
//    issues 32 tcgen05.mma, M = 128 keys, N = 64 heads, K = 16 each, into tensor
//    memory; fp32 queries: a second pass with the fp16 remainder); the logits are
//    read back with tcgen05.ld and staged as S; softmax per head (base 2; eight
//    lanes per head) against a running reference exponent, P rounded to fp16 and
//    written over S; O^T += V^T P^T on the tensor cores (V read in place as an
//    MN-major operand, P K-major, four M = 128 blocks of dims, accumulated in tensor
//    memory over the chunks);
//  * the reference exponent of a head moves only when a chunk's maximum passes it by
//    more than kAclLazy (so P <= 2^kAclLazy in fp16); when it moves, the head's
//    accumulated O and sum are scaled by 2^(old - new) in tensor memory first;
//  * C = 1: O / sum is written straight from the registers. C > 1: the unnormalised
//    O, reference and sum of every block are staged in its shared memory; after a
//    cluster barrier block r merges heads [64r/C, 64(r+1)/C) of all C blocks
//    (distributed shared memory: the weights in one round of remote loads, then
//    every partial row of a thread's items in flight at once).
#pragma once

#include <cooperative_groups.h>

#include "attention.cuh"
#include "indexer_scan_tc.cuh"

namespace csa2 {

constexpr int kAclThreads = 512;
constexpr int kAclKeys = 128;   // keys per chunk
constexpr int kAclHeads = 64;   // heads per block
constexpr int kAclMaxBlocks = 8;
constexpr float kAclLazy = 8.f;
constexpr int kAclQ = 0;                                  // Q [64 heads][512] fp16, K-major 128-byte swizzle
constexpr int kAclV = kAclQ + kAclHeads * 1024;           // V [128 keys][512] fp16, K-major 128-byte swizzle
constexpr int kAclSSt = kAclV + kAclKeys * 1024;          // S [64 heads][128 keys] f32
constexpr int kAclP = kAclSSt;                            // P [64 heads][128 keys] fp16 over S (after every read of S)
constexpr int kAclCoef = kAclSSt + kAclHeads * kAclKeys * 4;  // [64] f32: log2(e) x scale / 2^s of the head's queries
constexpr int kAclM = kAclCoef + kAclHeads * 4;           // [64] f32: reference exponent per head (running)
constexpr int kAclL = kAclM + kAclHeads * 4;              // [64] f32: sum per head (running)
constexpr int kAclFac = kAclL + kAclHeads * 4;            // [64] f32: this chunk's rescale factor per head
constexpr int kAclKeyOk = kAclFac + kAclHeads * 4;        // [128] i32
constexpr int kAclBar = kAclKeyOk + kAclKeys * 4;         // mbarrier (8 B), tensor-memory base (4 B), abort (4 B),
                                                          // MMA commits issued (4 B)
constexpr int kAclSmem = kAclBar + 32 + 1024;             // + slack to align the base to 1024 bytes
static_assert(kAclSmem <= 232448, "one block per SM, within the per-block limit");
// tensor memory: O^T in columns 0..255 (four blocks of 128 dims: lanes = dims, columns
// 64 mb .. 64 mb + 63 = heads), S^T in columns 256..319 (lanes = keys, columns = heads)
constexpr int kAclTmemCols = 512;
constexpr uint32_t kAclSCol = 256;
// instruction descriptors, kind::f16: D f32, A = B = f16, M = 128, N = 64. S: both
// operands K-major. O: A (V^T) MN-major, B (P^T) K-major.
constexpr uint32_t kAclIDesc = (1u << 4) | ((uint32_t)(kAclHeads >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
constexpr uint32_t kAclIDescPV = kAclIDesc | (1u << 15);
static_assert(kAclHeads * kAclKeys * 2 <= kAclHeads * kAclKeys * 4, "P fits over S");
constexpr int kAclOPitch = 520;                           // floats per staged O row (bank spread)
constexpr int kAclO = 0;                                  // [64][520] f32 over Q and V, after the last chunk
static_assert(kAclO + kAclHeads * kAclOPitch * 4 <= kAclSSt, "staged O fits over Q and V");
static_assert((kAclMaxBlocks + 1) * kAclHeads * 4 <= kAclHeads * kAclKeys * 4, "merge weights fit over S");

// The tensor core's K-major, 128-byte-swizzled operand layout: 16-byte chunk c (dims
// 8c .. 8c+7) of row r sits in the 64-dim block c/8, in row r of that block (128 B
// per row, blocks of `rows` rows), at chunk (c mod 8) XOR (r mod 8).
__device__ __forceinline__ uint32_t acl_kidx(int r, int c, int rows) {
  return (uint32_t)((c >> 3) * (rows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}
__device__ __forceinline__ uint32_t acl_vidx(int key, int c) { return acl_kidx(key, c, kAclKeys); }
__device__ __forceinline__ uint32_t acl_qidx(int h, int c) { return acl_kidx(h, c, kAclHeads); }

// Shared-memory matrix descriptor, 128-byte swizzle, with an explicit leading-
// dimension byte offset (the stride between 64-element swizzle atoms along M or N of
// an MN-major operand) and the 1,024-byte stride between 8-row groups.
__device__ __forceinline__ uint64_t smem_desc_sw128_lbo(uint32_t saddr, uint32_t lbo_bytes) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// D[tmem] (+)= A[smem descriptor] x B[smem descriptor], kind::f16.
__device__ __forceinline__ void tc_mma_f16_ss(uint32_t d_taddr, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_taddr),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// Per-layer operands of one launch: layer blockIdx.z of the grid. Layers launched
// together share the cache, k, W, H and the query type; each has its own queries,
// selection, window rows and output.
constexpr int kAclMaxLayers = 4;
struct AclLayers {
  const void* q[kAclMaxLayers];
  const int32_t* idx[kAclMaxLayers];
  const uint16_t* swa[kAclMaxLayers];
  const uint8_t* swa_codes[kAclMaxLayers];
  const uint8_t* swa_scales[kAclMaxLayers];
  float* out[kAclMaxLayers];
};

// Grid: (C x H/64, batch, layers); launched as clusters of C blocks along x when C > 1.
// NPART == 2 (fp32 queries) needs one chunk per block: its second pass overwrites Q.
template <int NPART>
__global__ void __launch_bounds__(kAclThreads, 1)
k_sparse_attn_cl(const __grid_constant__ AclLayers layers, int q_dtype, float scale,
                 const uint8_t* __restrict__ lat_codes, const uint8_t* __restrict__ lat_scales,
                 const int32_t* __restrict__ len, int64_t cap, int k, int W, int H, int q_early, int C) {
  const int li = blockIdx.z;
  const void* __restrict__ q = layers.q[li];
  const int32_t* __restrict__ idx = layers.idx[li];
  const uint16_t* __restrict__ swa = layers.swa[li];
  const uint8_t* __restrict__ swa_codes = layers.swa_codes[li];
  const uint8_t* __restrict__ swa_scales = layers.swa_scales[li];
  float* __restrict__ out = layers.out[li];
  extern __shared__ __align__(1024) unsigned char acl_smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(acl_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int r = blockIdx.x % C, hg = blockIdx.x / C, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int n_list = k + W;
  const int nch = (n_list + kAclKeys * C - 1) / (kAclKeys * C);  // chunks of this block (the same in all)
  if (NPART == 2 && nch > 1) {  // (uniform over the grid: no block reaches a cluster barrier)
    if (tid == 0) set_dev_error(CSA2_ERR_ARG);
    return;
  }
  unsigned char* qs = smem + kAclQ;
  unsigned char* vs = smem + kAclV;
  float* coef = reinterpret_cast<float*>(smem + kAclCoef);
  float* m_blk = reinterpret_cast<float*>(smem + kAclM);
  float* l_blk = reinterpret_cast<float*>(smem + kAclL);
  float* fac_s = reinterpret_cast<float*>(smem + kAclFac);
  int* key_ok = reinterpret_cast<int*>(smem + kAclKeyOk);
  const uint32_t bar = smem_u32addr(smem + kAclBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kAclBar + 8);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kAclBar + 12);
  volatile uint32_t* n_commits = reinterpret_cast<volatile uint32_t*>(smem + kAclBar + 16);
  if (tid == 0) {
    mbar_init(bar, 1);
    *abort = 0;
    *n_commits = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (tid < kAclHeads) {
    m_blk[tid] = -INFINITY;
    l_blk[tid] = 0.f;
  }
  // q_early (set by the decode step when the kernel before this one is its own Top-k,
  // which does not write the queries, and every kernel before that has completed by
  // the time this one starts): the queries are loaded and staged before waiting for
  // the Top-k. Otherwise everything waits for the previous kernel first.
  if (!q_early) pdl_wait_and_release();
  const size_t seq_row0 = (size_t)b * cap;

  // ---- this thread's quarter of key kk (dims 128qq .. 128qq+127) of a chunk: the
  // selection is read one chunk ahead of the codes and scales
  const int kk = tid >> 2, qq = tid & 3;
  int n_b = 0;
  int kind = 0;  // 0 none, 1 cache entry, 2 window row
  int j_cur = 0;  // list position of this thread's key in the current chunk
  uint2 cv[8];    // codes of the 16-dim groups 4m + qq, m = 0..7
  uint4 sc[2];    // the entry's 32 E4M3 bytes
  auto list_pos = [&](int t) { return (kAclKeys * t + kk) * C + r; };
  auto read_sel = [&](int t) {  // the selected position for chunk t (-1: none or not a cache entry)
    const int j = list_pos(t);
    return (t < nch && j < k && idx) ? __ldg(idx + (size_t)b * k + j) : -1;
  };
  auto load_keys = [&](int t, int pos) {
    const int j = list_pos(t);
    j_cur = j;
    kind = 0;
    if (j < k) {
      if (pos >= n_b) set_dev_error(CSA2_ERR_BOUNDS);
      if (pos >= 0 && pos < n_b) {
        kind = 1;
        const uint2* src = reinterpret_cast<const uint2*>(lat_codes + (seq_row0 + pos) * 256) + qq;
#pragma unroll
        for (int m = 0; m < 8; ++m) cv[m] = __ldg(src + 4 * m);
        const uint4* ss = reinterpret_cast<const uint4*>(lat_scales + (seq_row0 + pos) * 32);
        sc[0] = __ldg(ss);
        sc[1] = __ldg(ss + 1);
      }
    } else if (j < n_list) {
      kind = 2;
    }
  };
  int pos_next = -1;  // the selection of the next chunk, read a chunk ahead
  auto start_keys = [&]() {
    n_b = (int)min((int64_t)__ldg(len + b), cap);
    const int p0 = read_sel(0);
    pos_next = read_sel(1);
    load_keys(0, p0);
  };

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
    if (!q_early) start_keys();  // in flight while the queries are scaled
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
      {  // lanes 4..7 of each eight store their odd chunk first: distinct 16-byte positions
        const bool sw = ((lane >> 2) & 1) != 0;
        const uint4 lo4 = make_uint4(o[0], o[1], o[2], o[3]), hi4 = make_uint4(o[4], o[5], o[6], o[7]);
        *reinterpret_cast<uint4*>(qs + acl_qidx(h, 2 * lane + (sw ? 1 : 0))) = sw ? hi4 : lo4;
        *reinterpret_cast<uint4*>(qs + acl_qidx(h, 2 * lane + (sw ? 0 : 1))) = sw ? lo4 : hi4;
      }
    }
    if (q_early) {
      pdl_wait_and_release();  // the selected indices (and the cache) are ready from here on
      start_keys();
    }
  }
  if (w == 0) tc_alloc(smem_u32addr(tmem_slot), kAclTmemCols);

  uint32_t n_wait = 0;  // phases of the MMA barrier waited for so far
  for (int t = 0; t < nch; ++t) {
    if (t > 0) {  // O^T += V^T P^T of the previous chunk is done with V and P
      mbar_wait_bounded(bar, n_wait & 1u, abort);
      ++n_wait;
      tc_fence_after();
    }
    // ---- keys -> fp16 V rows (invalid keys: zero rows). Thread qq of a key takes the
    // 16-dim groups 4m + qq: the eight lanes of one store (two keys x four threads) then
    // write eight distinct 16-byte positions of the swizzled rows.
    if (kind == 1) {
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint32_t sw = m < 4 ? (m == 0 ? sc[0].x : m == 1 ? sc[0].y : m == 2 ? sc[0].z : sc[0].w)
                                  : (m == 4 ? sc[1].x : m == 5 ? sc[1].y : m == 6 ? sc[1].z : sc[1].w);
        const __half2 s2 = __float2half2_rn(e4m3_decode((sw >> (8 * qq)) & 0xFFu));  // scale of group 4m + qq
        const uint32_t cw[2] = {cv[m].x, cv[m].y};
        uint32_t o[8];
#pragma unroll
        for (int wv = 0; wv < 2; ++wv) {
#pragma unroll
          for (int by = 0; by < 4; ++by) {
            const __half2_raw rr =
                __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((cw[wv] >> (8 * by)) & 0xFFu), __NV_E2M1);
            const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&rr), s2);
            o[4 * wv + by] = *reinterpret_cast<const uint32_t*>(&v);
          }
        }
        const int chunk = 2 * (4 * m + qq);
        *reinterpret_cast<uint4*>(vs + acl_vidx(kk, chunk)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(vs + acl_vidx(kk, chunk + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    } else if (kind == 2 && swa_codes) {  // FP8 window row: E4M3 values times the block's 2^(e - 127)
      const size_t wrow = (size_t)b * W + (j_cur - k);
      const uint4* ss = reinterpret_cast<const uint4*>(swa_scales + wrow * 32);
      const uint4 s0 = __ldg(ss), s1 = __ldg(ss + 1);
      uint4 cw4[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) cw4[m] = __ldg(reinterpret_cast<const uint4*>(swa_codes + wrow * 512) + 4 * m + qq);
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int g = 4 * m + qq;  // the 16-value block
        const uint32_t sw = m < 4 ? (m == 0 ? s0.x : m == 1 ? s0.y : m == 2 ? s0.z : s0.w)
                                  : (m == 4 ? s1.x : m == 5 ? s1.y : m == 6 ? s1.z : s1.w);
        const float f = e8m0_decode((sw >> (8 * qq)) & 0xFFu);
        const uint32_t cw[4] = {cw4[m].x, cw4[m].y, cw4[m].z, cw4[m].w};
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t byte2 = (cw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
          o[e] = pack_half2(e4m3_decode(byte2 & 0xFFu) * f, e4m3_decode(byte2 >> 8) * f);
        }
        *reinterpret_cast<uint4*>(vs + acl_vidx(kk, 2 * g)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(vs + acl_vidx(kk, 2 * g + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    } else if (kind == 2) {  // bf16 window row: two rounds of eight loads
      const uint4* src = reinterpret_cast<const uint4*>(swa + ((size_t)b * W + (j_cur - k)) * 512);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint4 v8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ii = 8 * half + i;
          v8[i] = __ldg(src + 2 * (4 * (ii >> 1) + qq) + (ii & 1));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ii = 8 * half + i;
          const uint32_t vw[4] = {v8[i].x, v8[i].y, v8[i].z, v8[i].w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = pack_half2(bf16_bits_to_float(vw[e] & 0xFFFFu), bf16_bits_to_float(vw[e] >> 16));
          *reinterpret_cast<uint4*>(vs + acl_vidx(kk, 2 * (4 * (ii >> 1) + qq) + (ii & 1))) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    } else {
#pragma unroll 4
      for (int i = 0; i < 16; ++i)
        *reinterpret_cast<uint4*>(vs + acl_vidx(kk, 2 * (4 * (i >> 1) + qq) + (i & 1))) = make_uint4(0, 0, 0, 0);
    }
    if (qq == 0) key_ok[kk] = kind != 0 ? 1 : 0;

    // ---- S^T = V Q^T on the tensor cores (tcgen05, M = 128 keys, N = 64 heads, K = 512
    // in 32 steps): one thread issues, the accumulator lives in tensor memory
    fence_proxy_async_smem();  // this thread's Q and V stores, for the tensor core's reads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
#pragma unroll
    for (int part = 0; part < NPART; ++part) {
      if (part == 1) {  // the fp16 remainder of fp32 queries replaces the first part
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const int h = 4 * w + hh;
          const bool sw = ((lane >> 2) & 1) != 0;
          const uint4 lo4 = make_uint4(qlo[hh][0], qlo[hh][1], qlo[hh][2], qlo[hh][3]);
          const uint4 hi4 = make_uint4(qlo[hh][4], qlo[hh][5], qlo[hh][6], qlo[hh][7]);
          *reinterpret_cast<uint4*>(qs + acl_qidx(h, 2 * lane + (sw ? 1 : 0))) = sw ? hi4 : lo4;
          *reinterpret_cast<uint4*>(qs + acl_qidx(h, 2 * lane + (sw ? 0 : 1))) = sw ? lo4 : hi4;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
      }
      if (tid == 0 && !*abort) {  // (after a wait that ran out, nothing more is issued)
        const uint32_t vb = smem_u32addr(vs), qb = smem_u32addr(qs);
#pragma unroll 4
        for (int ks = 0; ks < 32; ++ks) {  // dims 16 ks .. 16 ks + 15: block ks/4, 32 bytes per step
          const uint64_t da = smem_desc_sw128(vb + (ks >> 2) * (kAclKeys * 128) + (ks & 3) * 32);
          const uint64_t db = smem_desc_sw128(qb + (ks >> 2) * (kAclHeads * 128) + (ks & 3) * 32);
          tc_mma_f16_ss(tmem + kAclSCol, da, db, kAclIDesc, (part > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(bar);
        *n_commits = *n_commits + 1;
      }
      if (part == NPART - 1 && t + 1 < nch) {  // while the MMAs run: the next chunk's codes and
        const int p = pos_next;                // scales, and the selection after it
        pos_next = read_sel(t + 2);
        load_keys(t + 1, p);
      }
      mbar_wait_bounded(bar, n_wait & 1u, abort);  // the MMAs are done reading Q and V (or abort is set)
      ++n_wait;
      tc_fence_after();
    }

    // ---- logits: warp w reads keys 32(w%4) .. and heads 16(w/4) .. of S^T, scales and
    // masks them, and stages them as S [head][key] (f32)
    {
      const int key = 32 * (w & 3) + lane, hc = 16 * (w >> 2);
      uint32_t v[16];
      tc_ld16(tmem + ((uint32_t)(32 * (w & 3)) << 16) + kAclSCol + (uint32_t)hc, v);
      tc_wait_ld();
      const bool ok = key_ok[key] != 0;
      float* sst = reinterpret_cast<float*>(smem + kAclSSt);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        sst[(hc + i) * kAclKeys + key] = ok ? __uint_as_float(v[i]) * coef[hc + i] : -INFINITY;
    }
    tc_fence_before();
    __syncthreads();

    // ---- softmax over this chunk's keys against the head's running reference:
    // thread (h, seg) takes keys 16 seg .. 16 seg + 15 of head h; the eight segments
    // of a head are eight consecutive lanes
    int rescale;
    {
      const int h = tid >> 3, seg = tid & 7;
      const float4* sr = reinterpret_cast<const float4*>(smem + kAclSSt) + (h * kAclKeys + 16 * seg) / 4;
      // read j takes keys 16 seg + 4 jj .., jj = (j + seg / 2) mod 4: the eight lanes
      // of a read hit eight distinct 16-byte positions
      float x[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 tt = sr[(j + (seg >> 1)) & 3];
        x[4 * j] = tt.x; x[4 * j + 1] = tt.y; x[4 * j + 2] = tt.z; x[4 * j + 3] = tt.w;
      }
      float M = x[0];
#pragma unroll
      for (int i = 1; i < 16; ++i) M = fmaxf(M, x[i]);
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float ref_old = m_blk[h];
      const bool move = M > ref_old + kAclLazy;  // (never for a chunk with no valid key)
      const float ref = move ? M : ref_old;
      const float fac = move ? exp2f(ref_old - ref) : 1.f;  // 0 while nothing was accumulated
      const float Z = ref == -INFINITY ? 0.f : ref;
      uint2 pw[4];
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 p01 = __floats2half2_rn(exp2f(x[4 * j] - Z), exp2f(x[4 * j + 1] - Z));
        const __half2 p23 = __floats2half2_rn(exp2f(x[4 * j + 2] - Z), exp2f(x[4 * j + 3] - Z));
        const float2 f01 = __half22float2(p01), f23 = __half22float2(p23);
        ls += (f01.x + f01.y) + (f23.x + f23.y);
        pw[j] = make_uint2(*reinterpret_cast<const uint32_t*>(&p01), *reinterpret_cast<const uint32_t*>(&p23));
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
      rescale = __syncthreads_or(move && t > 0);  // every read of S (and of m_blk) is done: P goes over S
      unsigned char* ps = smem + kAclP;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int jj = (j + (seg >> 1)) & 3;  // keys 16 seg + 4 jj .. + 3
        *reinterpret_cast<uint2*>(ps + acl_qidx(h, 2 * seg + (jj >> 1)) + (jj & 1) * 8) = pw[j];
      }
      if (seg == 0) {
        m_blk[h] = ref;
        l_blk[h] = l_blk[h] * fac + ls;
        fac_s[h] = fac;
      }
    }
    fence_proxy_async_smem();  // this thread's P stores, for the tensor core's reads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (rescale) {  // a reference moved: O^T (dims of this thread's lane, all heads) times 2^(old - new)
      const uint32_t ta = tmem + ((uint32_t)(32 * (w & 3)) << 16) + (uint32_t)(64 * (w >> 2));
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t v[16];
        tc_ld16(ta + 16 * q4, v);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * fac_s[16 * q4 + i]);
        tc_st16(ta + 16 * q4, v);
      }
      tc_wait_st();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
    // ---- O^T += V^T P^T on the tensor cores: M = 128 dims (four blocks), N = 64 heads,
    // K = 128 keys in 8 steps. A = V read in place as an MN-major operand (dims run
    // along its 128-byte rows; 64-dim atoms 16 KB apart, 8-key groups 1 KB apart); B = P,
    // K-major (rows = heads).
    if (tid == 0 && !*abort) {
      const uint32_t vb = smem_u32addr(vs), pb = smem_u32addr(smem + kAclP);
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
        for (int ks = 0; ks < kAclKeys / 16; ++ks) {  // keys 16 ks .. 16 ks + 15
          const uint64_t da = smem_desc_sw128_lbo(vb + 2 * mb * (kAclKeys * 128) + ks * 2048, kAclKeys * 128);
          const uint64_t db = smem_desc_sw128(pb + (ks >> 2) * (kAclHeads * 128) + (ks & 3) * 32);
          tc_mma_f16_ss(tmem + 64 * mb, da, db, kAclIDescPV, (t > 0 || ks > 0) ? 1u : 0u);
        }
      }
      tc_commit(bar);
      *n_commits = *n_commits + 1;
    }
  }
  mbar_wait_bounded(bar, n_wait & 1u, abort);  // the last MMAs are done (or abort is set)
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // warp w: dims 128 (w / 4) + 32 (w % 4) + lane, all 64 heads
  float ov[64];
  {
    const uint32_t ta = tmem + ((uint32_t)(32 * (w & 3)) << 16) + (uint32_t)(64 * (w >> 2));
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint32_t v[16];
      tc_ld16(ta + 16 * q4, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) ov[16 * q4 + i] = __uint_as_float(v[i]);
    }
    tc_wait_ld();
  }
  tc_fence_before();
  __syncthreads();  // every read of tensor memory is done; Q, V and S are free
  if (*abort) {
    // a wait ran out (CSA2_ERR_TIMEOUT is recorded): let the last committed MMAs finish
    // (again with a limit) before the tensor memory is freed; the outputs of this
    // block are then meaningless, but every barrier below is still reached
    if (tid == 0 && *n_commits > 0) {
      volatile int again = 0;
      mbar_wait_bounded(bar, (*n_commits - 1u) & 1u, &again);
    }
    __syncthreads();
  }
  if (w == 0) {
    tc_fence_after();
    tc_dealloc(tmem, kAclTmemCols);
  }
  const int d = 128 * (w >> 2) + 32 * (w & 3) + lane;
  if (C == 1) {  // the whole row in this block: O / sum, from the registers
    if (tid < kAclHeads) {
      const float L = l_blk[tid];
      fac_s[tid] = L > 0.f ? 1.f / L : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < kAclHeads; ++h) out[((size_t)b * H + hg * kAclHeads + h) * 512 + d] = ov[h] * fac_s[h];
    return;
  }
  // ---- merge: block r finishes heads [64r/C, 64(r+1)/C) of all C blocks. Every
  // block stages its unnormalised O over its own Q and V; after a cluster barrier
  // block r reads the reference and sum of its heads from every block (one round of
  // remote loads into shared memory), then each thread loads the C partial rows of
  // its items with all loads in flight at once.
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  {
    float* os = reinterpret_cast<float*>(smem + kAclO);
#pragma unroll
    for (int h = 0; h < kAclHeads; ++h) os[h * kAclOPitch + d] = ov[h];
  }
  cluster.sync();  // every block's O, reference and sum are staged
  const int hb0 = r * kAclHeads / C, nh = (r + 1) * kAclHeads / C - hb0;
  float* wa = reinterpret_cast<float*>(smem + kAclSSt);  // [C][nh]: weight of block c for head hb0 + i (over S)
  float* winv = wa + kAclMaxBlocks * kAclHeads;           // [nh]: 1 / merged sum
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
