// indexer_score, streaming form on the 5th-generation tensor cores (tcgen05).
//
// Pages: "Le cache KV en FP4", section "Les ingredients", item 2 (the 128-channel
// indexer key scores positions) and section "Cles d'indexeur" (eq. 68: E2M1 with an
// E8M0 scale per 32 channels).
//
// A ring of shared-memory stages like the mma.sync form's, here of 128 entries (a
// producer warp streams one TMA box of codes, 64-byte swizzle, and their E8M0 bytes
// per stage); the rest is per entry:
//  * two groups of four converter warps take the stages in turn; thread r of a
//    group owns entry r of its stage (TMEM lane r): it turns the entry's 64 code
//    bytes into 128 fp16 values (exact) and writes them to an A buffer in tensor
//    memory (tcgen05.st, 64 columns), and writes its 32 bytes of the query tile B
//    (shared memory, 128-byte swizzle, K-major): B[k][4 blk + h] = q_h[k] 2^s_h
//    when channel k lies in 32-channel block blk, else 0 (fp32 queries: a second
//    set of 16 rows with the fp16 remainder);
//  * one thread issues D = A B as eight tcgen05.mma (M = 128 entries, N = 16 or
//    32, K = 16, fp16 in, fp32 accumulate in tensor memory), then tcgen05.commit
//    to the "D ready" and "A free" barriers;
//  * the converting thread reads its D row back (tcgen05.ld: the four block dots
//    of each head), applies the E8M0 scales (exact powers of two), the ReLU and
//    the head weights, and writes the score.
// Buffers: 3 A (64 columns) + 4 D (16 columns; 2 x 32 for fp32 queries) of a
// 256-column tensor-memory allocation, 3 B tiles, 8 stages. Every mbarrier wait
// gives up after about a second (CSA2_ERR_TIMEOUT) and the block then drains its
// copies and MMAs before freeing tensor memory.
#pragma once

#include "indexer_scan.cuh"

namespace csa2 {

constexpr int kTcConvWarps = 8;                           // two groups of four
constexpr int kTcThreads = (kTcConvWarps + 2) * 32;       // + producer warp + MMA warp
constexpr int kTcStages = 8;
constexpr int kTcStageBytes = 9216;                       // 8192 codes + 512 E8M0 (+ pad)
constexpr int kTcNA = 3;
constexpr int kTcTmemCols = 256;

template <int NPART>
struct TcShape {
  static constexpr int N = 16 * NPART;                    // D columns
  static constexpr int ND = NPART == 1 ? 4 : 2;           // D buffers
  static constexpr int BBytes = N * 256;                  // N rows x 128 fp16
  static constexpr int BOff = kTcStages * kTcStageBytes;  // 73,728: 1024-aligned
  static constexpr int BarOff = BOff + kTcNA * BBytes;
  // full[8] empty[8] afull[3] aempty[3] dfull[ND] dempty[ND] done
  static constexpr int NBars = 2 * kTcStages + 2 * kTcNA + 2 * ND + 1;
  static constexpr int MiscOff = BarOff + 8 * NBars;      // tmem base (4 B), abort (4 B)
  static constexpr int Smem = MiscOff + 16 + 1024;        // + alignment slack
  static constexpr int DCol0 = kTcNA * 64;                // D buffers after the A buffers
  // instruction descriptor, kind::f16: D f32, A = B = f16, both K-major, M = 128
  static constexpr uint32_t IDesc = (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
};

// ------------------------------------------------------------------ tcgen05 helpers
__device__ __forceinline__ void tc_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
      "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]), "r"(v[32])
      : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

// D[tmem] (+)= A[tmem] x B[smem descriptor], kind::f16.
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_taddr),
      "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
               : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle (8-row groups of
// 1024 bytes), start address in 16-byte units.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) /* LBO (unused) */ |
         ((uint64_t)(1024 >> 4) << 32) /* SBO */ | ((uint64_t)1 << 46) /* descriptor version */ |
         ((uint64_t)2 << 61) /* 128-byte swizzle */;
}

// Byte offset of 16-byte chunk c (0..15: channels 8c..8c+7) of row n in a B tile of
// N rows: two 128-byte-swizzled atoms of 64 channels.
template <int N>
__device__ __forceinline__ uint32_t btile_off(int n, int c) {
  return (uint32_t)((c >> 3) * (N * 128) + n * 128 + (((c & 7) ^ (n & 7)) << 4));
}

// Every lane of a warp waits; the warp goes on only if all of them saw the phase
// (a lane that timed out makes the whole warp give up, so the .sync.aligned
// tensor-memory instructions after it are never reached by part of a warp).
__device__ __forceinline__ bool warp_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

struct TcQ {        // this converter thread's part of the query tile of one sequence
  uint32_t v[16];   // NPART 1: rows n, chunks 2cp, 2cp+1 (8 words); NPART 2: also row n + 16
  float winv[4];    // w_h * 2^-s_h
};

// Query tile values of sequence b for converter thread t (0..127): row n = t / 8,
// channels 16 cp .. 16 cp + 15 with cp = t % 8 (and row n + 16 for the fp32 remainder).
template <int NPART>
__device__ __forceinline__ void tc_setup_q(int b, const TmaScanArgs& a, int t, int lane, TcQ& Q) {
  const size_t qb = (size_t)b * CSA2_INDEXER_HEADS * CSA2_INDEXER_DIM;
  float f[CSA2_INDEXER_HEADS];
#pragma unroll
  for (int h = 0; h < CSA2_INDEXER_HEADS; ++h) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fabsf(load_elem(a.q_idx, a.q_dtype, qb + h * 128 + lane + 32 * i)));
    m = warp_max(m);
    int s = 0;
    if (m > 0.f) {
      const int e = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;
      s = min(max(14 - e, -100), 100);
    }
    f[h] = __uint_as_float((uint32_t)(127 + s) << 23);
    Q.winv[h] = __ldg(a.w + (size_t)b * CSA2_INDEXER_HEADS + h) * __uint_as_float((uint32_t)(127 - s) << 23);
  }
  const int n = t >> 3, cp = t & 7;
  const int blk = n >> 2, h = n & 3;
  float fh = f[0];
#pragma unroll
  for (int hh = 1; hh < CSA2_INDEXER_HEADS; ++hh) fh = h == hh ? f[hh] : fh;
  const bool live = (cp >> 1) == blk;  // channels 16cp.. lie in block cp/2
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // channel pair 16cp + 2i, +1
    float x0 = 0.f, x1 = 0.f;
    if (live) {
      x0 = load_elem(a.q_idx, a.q_dtype, qb + h * 128 + 16 * cp + 2 * i) * fh;
      x1 = load_elem(a.q_idx, a.q_dtype, qb + h * 128 + 16 * cp + 2 * i + 1) * fh;
    }
    const float h0 = __half2float(__float2half_rn(x0)), h1 = __half2float(__float2half_rn(x1));
    Q.v[i] = f16x2_bits(h0, h1);
    if constexpr (NPART == 2) Q.v[8 + i] = f16x2_bits(x0 - h0, x1 - h1);
  }
}

template <int NPART>
__global__ void __launch_bounds__(kTcThreads, 2)
k_indexer_scan_tc(const __grid_constant__ CUtensorMap tmap, const TmaScanArgs a) {
  pdl_wait_and_release();
  using S = TcShape<NPART>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32addr(smem);
  const uint32_t bar = sbase + S::BarOff;
  auto bar_full = [&](int s) { return bar + 8 * s; };
  auto bar_empty = [&](int s) { return bar + 8 * (kTcStages + s); };
  auto bar_afull = [&](int i) { return bar + 8 * (2 * kTcStages + i); };
  auto bar_aempty = [&](int i) { return bar + 8 * (2 * kTcStages + kTcNA + i); };
  auto bar_dfull = [&](int i) { return bar + 8 * (2 * kTcStages + 2 * kTcNA + i); };
  auto bar_dempty = [&](int i) { return bar + 8 * (2 * kTcStages + 2 * kTcNA + S::ND + i); };
  const uint32_t bar_done = bar + 8 * (2 * kTcStages + 2 * kTcNA + 2 * S::ND);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::MiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + S::MiscOff + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kProducer = kTcConvWarps, kMma = kTcConvWarps + 1;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 4);
    }
    for (int i = 0; i < kTcNA; ++i) {
      mbar_init(bar_afull(i), 4);
      mbar_init(bar_aempty(i), 1);
    }
    for (int i = 0; i < S::ND; ++i) {
      mbar_init(bar_dfull(i), 1);
      mbar_init(bar_dempty(i), 4);
    }
    mbar_init(bar_done, 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == kMma) tc_alloc(smem_u32addr(tmem_slot), kTcTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t t_begin = (int64_t)blockIdx.x * a.total_tiles / gridDim.x;
  const int64_t t_end = (int64_t)(blockIdx.x + 1) * a.total_tiles / gridDim.x;
  const int b0 = (int)(t_begin / a.tiles_per_seq);
  const int64_t e00 = (t_begin - (int64_t)b0 * a.tiles_per_seq) * kTmaRows;
  const int64_t seq_rows = a.tiles_per_seq * kTmaRows;

  if (warp == kProducer) {
    // ---------------- producer: one lane streams the stages
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      asm volatile("prefetch.tensormap [%0];\n" ::"l"(&tmap) : "memory");
      uint32_t it = 0;
      int b = b0;
      int64_t e0 = e00, n_b = min((int64_t)__ldg(a.len + b), a.cap);
      for (int64_t t = t_begin; t < t_end; ++t) {
        if (e0 < n_b) {
          const uint32_t s = it % kTcStages, ph = (it / kTcStages) & 1u;
          if (!mbar_wait_bounded(bar_empty(s), ph ^ 1u, abort)) break;
          const uint32_t st = sbase + s * kTcStageBytes;
          const int64_t row = (int64_t)b * a.cap + e0;
          mbar_arrive_expect_tx(bar_full(s), kTmaRows * 64 + kTmaRows * 4);
          tma_load_rows(st, &tmap, 0, (int32_t)row, bar_full(s), pol);
          bulk_load(st + kTmaRows * 64, a.scales + row * 4, kTmaRows * 4, bar_full(s), pol);
          ++it;
        }
        e0 += kTmaRows;
        if (e0 >= seq_rows && t + 1 < t_end) {
          e0 = 0;
          ++b;
          n_b = min((int64_t)__ldg(a.len + b), a.cap);
        }
      }
      for (uint32_t j = (it > kTcStages ? it - kTcStages : 0); j < it; ++j) {  // every copy lands
        volatile int no_abort = 0;
        mbar_wait_bounded(bar_full(j % kTcStages), (j / kTcStages) & 1u, &no_abort);
      }
    }
  } else if (warp == kMma) {
    // ---------------- MMA issuer: one lane
    if (lane == 0) {
      uint32_t it = 0;
      int b = b0;
      int64_t e0 = e00, n_b = min((int64_t)__ldg(a.len + b), a.cap);
      for (int64_t t = t_begin; t < t_end; ++t) {
        if (e0 < n_b) {
          const uint32_t ab = it % kTcNA, d = it % S::ND;
          if (!mbar_wait_bounded(bar_afull(ab), (it / kTcNA) & 1u, abort)) break;
          if (!mbar_wait_bounded(bar_dempty(d), ((it / S::ND) & 1u) ^ 1u, abort)) break;
          tc_fence_after();
          const uint32_t b_saddr = sbase + S::BOff + ab * S::BBytes;
          const uint32_t d_taddr = tmem + S::DCol0 + d * S::N, a_taddr = tmem + ab * 64;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {  // channels 16 ks .. 16 ks + 15: atom ks/4, 32 bytes per step
            const uint64_t bd = smem_desc_sw128(b_saddr + (ks >> 2) * (S::N * 128) + (ks & 3) * 32);
            tc_mma_f16_ts(d_taddr, a_taddr + 8 * ks, bd, S::IDesc, ks > 0 ? 1u : 0u);
          }
          tc_commit(bar_dfull(d));
          tc_commit(bar_aempty(ab));
          ++it;
        }
        e0 += kTmaRows;
        if (e0 >= seq_rows && t + 1 < t_end) {
          e0 = 0;
          ++b;
          n_b = min((int64_t)__ldg(a.len + b), a.cap);
        }
      }
      tc_commit(bar_done);  // arrives once every MMA issued above has completed
      volatile int no_abort = 0;
      mbar_wait_bounded(bar_done, 0u, &no_abort);
    }
  } else {
    // ---------------- converters: group g takes tiles it % 2 == g; thread r = entry r
    const int g = warp >> 2, r = 32 * (warp & 3) + lane;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t swz = (uint32_t)((r >> 1) & 3);
    TcQ Q;
    int setup_b = -1;
    // the tile whose epilogue is pending
    bool pend = false;
    uint32_t p_it = 0, p_sw = 0;
    int p_b = 0;
    int64_t p_e = 0, p_n = 0;
    auto epilogue = [&]() {
      const uint32_t d = p_it % S::ND;
      if (!warp_wait_bounded(bar_dfull(d), (p_it / S::ND) & 1u, abort)) return false;
      tc_fence_after();
      uint32_t v[16], v2[16];
      tc_ld16(tmem + lane_base + S::DCol0 + d * S::N, v);
      if constexpr (NPART == 2) tc_ld16(tmem + lane_base + S::DCol0 + d * S::N + 16, v2);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dempty(d));
      float sc[4];
      e8m0x4_decode(p_sw, sc);
      float score = 0.f;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float p = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float x = __uint_as_float(v[4 * j + h]);
          if constexpr (NPART == 2) x += __uint_as_float(v2[4 * j + h]);
          p = fmaf(x, sc[j], p);
        }
        score = fmaf(Q.winv[h], fmaxf(p, 0.f), score);
      }
      if (p_e < p_n) a.scores[(size_t)p_b * a.cap + p_e] = score;
      return true;
    };
    uint32_t it = 0;
    int b = b0;
    int64_t e0 = e00, n_b = min((int64_t)__ldg(a.len + b), a.cap);
    bool ok = true;
    for (int64_t t = t_begin; t < t_end && ok; ++t) {
      if (e0 < n_b) {
        if ((int)(it & 1u) == g) {
          if (b != setup_b) {
            if (pend) {  // the pending tile belongs to the previous sequence's weights
              ok = epilogue();
              pend = false;
              if (!ok) break;
            }
            tc_setup_q<NPART>(b, a, r, lane, Q);
            setup_b = b;
          }
          const uint32_t s = it % kTcStages;
          if (!warp_wait_bounded(bar_full(s), (it / kTcStages) & 1u, abort)) break;
          const unsigned char* st = smem + s * kTcStageBytes;
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 q4 = *reinterpret_cast<const uint4*>(st + 64 * r + 16 * ((uint32_t)j ^ swz));
            w[4 * j] = q4.x; w[4 * j + 1] = q4.y; w[4 * j + 2] = q4.z; w[4 * j + 3] = q4.w;
          }
          const uint32_t sw = *reinterpret_cast<const uint32_t*>(st + kTmaRows * 64 + 4 * r);
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_empty(s));
          const uint32_t ab = it % kTcNA;
          if (!warp_wait_bounded(bar_aempty(ab), ((it / kTcNA) & 1u) ^ 1u, abort)) break;
          tc_fence_after();
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {  // channels 64 hf .. 64 hf + 63: columns 32 hf ..
            uint32_t A[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint32_t o[4];
              e2m1x8_to_f16x2(w[8 * hf + j], o);
              A[4 * j] = o[0]; A[4 * j + 1] = o[1]; A[4 * j + 2] = o[2]; A[4 * j + 3] = o[3];
            }
            tc_st32(tmem + lane_base + ab * 64 + 32 * hf, A);
          }
          {  // this thread's 32 (64) bytes of the query tile
            unsigned char* bt = smem + S::BOff + ab * S::BBytes;
            const int n = r >> 3, cp = r & 7;
            *reinterpret_cast<uint4*>(bt + btile_off<S::N>(n, 2 * cp)) = make_uint4(Q.v[0], Q.v[1], Q.v[2], Q.v[3]);
            *reinterpret_cast<uint4*>(bt + btile_off<S::N>(n, 2 * cp + 1)) =
                make_uint4(Q.v[4], Q.v[5], Q.v[6], Q.v[7]);
            if constexpr (NPART == 2) {
              *reinterpret_cast<uint4*>(bt + btile_off<S::N>(n + 16, 2 * cp)) =
                  make_uint4(Q.v[8], Q.v[9], Q.v[10], Q.v[11]);
              *reinterpret_cast<uint4*>(bt + btile_off<S::N>(n + 16, 2 * cp + 1)) =
                  make_uint4(Q.v[12], Q.v[13], Q.v[14], Q.v[15]);
            }
          }
          tc_wait_st();
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_afull(ab));
          if (pend) {
            ok = epilogue();
            if (!ok) break;
          }
          pend = true;
          p_it = it;
          p_sw = sw;
          p_b = b;
          p_e = e0 + r;
          p_n = n_b;
        }
        ++it;
      }
      e0 += kTmaRows;
      if (e0 >= seq_rows && t + 1 < t_end) {
        e0 = 0;
        ++b;
        n_b = min((int64_t)__ldg(a.len + b), a.cap);
      }
    }
    if (ok && pend) epilogue();
  }

  // ---------------- teardown: every MMA has completed (the MMA lane waited for it)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMma) tc_dealloc(tmem, kTcTmemCols);
}

}  // namespace csa2
