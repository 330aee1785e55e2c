// indexer_score: score_t = sum_h w_h * max(0, q_h . k_t) over the 4 indexer heads,
// k_t the MXFP4 key (E2M1 codes times the E8M0 scale of each 32-channel block).
//
// Pages: "Le cache KV en FP4", section "Les ingredients", item 2 (the 128-channel
// indexer key scores positions) and section "Cles d'indexeur" (eq. 68: E2M1 with an
// E8M0 scale per 32 channels).
//
// The scan reads 68 bytes per entry and does 4 x 128 multiply-adds on them, more
// arithmetic per byte than the CUDA cores can sustain at HBM speed, so the
// contraction runs on the tensor cores (mma.sync m16n8k16, fp16 operands, fp32
// accumulation) and the CUDA cores only unpack codes and finish the epilogue.
//
//  * Operand A (16 entries x 16 channels): unscaled E2M1 values, converted from
//    the packed codes with cvt.rn.f16x2.e2m1x2 -- exact in fp16.
//  * Operand B (16 channels x 8 columns): the queries, scaled per head by a power
//    of two 2^s_h so that fp16 keeps every bit of a bf16 query (fp32 queries are
//    split into fp16 hi + lo parts, a second n-tile). Column n = 2*h + jj holds
//    head h restricted to block jj of a pair of 32-channel blocks (zero
//    elsewhere), so one MMA keeps two E8M0 blocks apart and every column is used.
//  * Epilogue: lane t4 of a quad holds head t4's four block dots of its two rows;
//    it multiplies each by the block's exact power-of-two scale (E8M0 -> bf16 by
//    cvt.rn.bf16x2.ue8m0x2), adds them, applies the ReLU and the head weight (with
//    2^-s_h folded in), and two quad shuffles sum the heads.
//
// Lane (g = lane/4, t4 = lane%4) of a warp loads, for entries g + 8r (r = 0..3),
// the 32-bit word t4 of each 16-byte block of codes -- so a k-step's channels
// (8 t4 + 2 kq + {0,1} of a block) sit in the right fragment slots without any
// shuffle. Each warp walks a contiguous range of 32-entry tiles (two m16 row
// tiles), prefetching the next tile's registers while it computes the current one.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace csa2 {

constexpr int kScanWarps = 8;
constexpr int kScanThreads = kScanWarps * 32;
constexpr int kScanTile = 32;  // entries per warp iteration

// ------------------------------------------------------------------ PTX helpers

// Policy for the scores: a decode step's scores are read back at once by its Top-k,
// so they are kept in L2 ahead of the streamed keys (evict-last); scores returned to a
// caller are stored with the normal priority.
__device__ __forceinline__ uint64_t l2_scores_policy(int scratch) {
  uint64_t p;
  if (scratch) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(p));
  else asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}

__device__ __forceinline__ void st_score(float* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;\n" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

// 32-bit read-only load, L2 evict-first (the keys are streamed once).
__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p, uint64_t pol) {
  uint32_t v;
  asm volatile("ld.global.nc.L2::cache_hint.b32 %0, [%1], %2;\n" : "=r"(v) : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}

// Four bytes = eight E2M1 codes -> four f16x2 (the low nibble of a byte in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n .reg .b8 c0, c1, c2, c3;\n"
      " mov.b32 {c0, c1, c2, c3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, c0;\n"
      " cvt.rn.f16x2.e2m1x2 %1, c1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, c2;\n"
      " cvt.rn.f16x2.e2m1x2 %3, c3;\n}\n"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ------------------------------------------------------------------ tile registers
struct ScanTile {
  uint32_t w[4][4];  // [row r = entry g + 8r][block j]: code word t4 of block j
  uint32_t s[4];     // the entry's four E8M0 bytes
  int b;             // sequence
  int64_t e0;        // first entry (or candidate slot) of the tile
  uint32_t flags;    // bit r: slot in range; bit 4+r: entry valid
};

struct ScanArgs {
  const void* q_idx;
  int q_dtype;
  const float* w;
  const uint8_t* codes;
  const uint8_t* scales;
  int64_t cap;
  const int32_t* len;
  const int32_t* cand;
  int P;
  float* scores;
  int scratch;  // the scores are a decode step's scratch (see l2_scores_policy)
  int64_t stride;
  int64_t tiles_per_seq;
  int64_t total_tiles;
};

__device__ __forceinline__ void scan_load_tile(ScanTile& T, int64_t t, const ScanArgs& a, int g, int t4,
                                               uint64_t pol) {
  T.b = (int)(t / a.tiles_per_seq);
  T.e0 = (t - (int64_t)T.b * a.tiles_per_seq) * kScanTile;
  const int64_t n_b = min((int64_t)__ldg(a.len + T.b), a.cap);
  const int64_t n = a.cand ? (int64_t)a.P : n_b;
  T.flags = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int64_t e = T.e0 + g + 8 * r;
    int64_t pos = e;
    bool in = e < n, ok = in;
    if (a.cand && in) {
      pos = __ldg(a.cand + (size_t)T.b * a.P + e);
      ok = pos >= 0 && pos < n_b;
      if (pos >= n_b && t4 == 0) set_dev_error(CSA2_ERR_BOUNDS);
    }
    T.flags |= (in ? 1u : 0u) << r;
    T.flags |= (ok ? 1u : 0u) << (4 + r);
    if (ok) {
      const size_t row = (size_t)T.b * a.cap + pos;
      const uint8_t* cp = a.codes + row * 64 + 4 * t4;
#pragma unroll
      for (int j = 0; j < 4; ++j) T.w[r][j] = ldg_stream_u32(cp + 16 * j, pol);
      T.s[r] = ldg_stream_u32(a.scales + row * 4, pol);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) T.w[r][j] = 0;
      T.s[r] = 0;
    }
  }
}

// Query fragments of sequence b. NPART = 1 (bf16 queries) or 2 (fp32: hi, lo).
template <int NPART>
__device__ __forceinline__ void scan_setup(int b, const ScanArgs& a, int lane, int g, int t4,
                                           uint32_t (&bf)[2][4][NPART][2], float& wsel) {
  const size_t qb = (size_t)b * CSA2_INDEXER_HEADS * CSA2_INDEXER_DIM;
  float f[CSA2_INDEXER_HEADS], winv[CSA2_INDEXER_HEADS];
#pragma unroll
  for (int h = 0; h < CSA2_INDEXER_HEADS; ++h) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fabsf(load_elem(a.q_idx, a.q_dtype, qb + h * 128 + lane + 32 * i)));
    m = warp_max(m);
    int s = 0;
    if (m > 0.f) {
      const int e = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;  // floor(log2 m) for normal m
      s = min(max(14 - e, -100), 100);
    }
    f[h] = __uint_as_float((uint32_t)(127 + s) << 23);     // 2^s, exact
    winv[h] = __ldg(a.w + (size_t)b * CSA2_INDEXER_HEADS + h) * __uint_as_float((uint32_t)(127 - s) << 23);
  }
  wsel = winv[0];
#pragma unroll
  for (int h = 1; h < CSA2_INDEXER_HEADS; ++h) wsel = t4 == h ? winv[h] : wsel;
  // column n = g: head hh = g >> 1, block jj = g & 1 of the pair
  const int jj = g & 1, hh = g >> 1;
  float fh = f[0];
#pragma unroll
  for (int h = 1; h < CSA2_INDEXER_HEADS; ++h) fh = hh == h ? f[h] : fh;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // b0: block 2p (jj == 0), b1: block 2p+1 (jj == 1)
        const int c = 64 * p + 32 * half + 8 * t4 + 2 * kq;
        const bool live = jj == half;
        float x0 = 0.f, x1 = 0.f;
        if (live) {
          x0 = load_elem(a.q_idx, a.q_dtype, qb + hh * 128 + c) * fh;
          x1 = load_elem(a.q_idx, a.q_dtype, qb + hh * 128 + c + 1) * fh;
        }
        const float h0v = __half2float(__float2half_rn(x0)), h1v = __half2float(__float2half_rn(x1));
        bf[p][kq][0][half] = f16x2_bits(h0v, h1v);
        if constexpr (NPART == 2) bf[p][kq][NPART - 1][half] = f16x2_bits(x0 - h0v, x1 - h1v);
      }
    }
  }
}

// The four E8M0 bytes of w as floats (2^(e-127), exact; 0xFF gives NaN).
__device__ __forceinline__ void e8m0x4_decode(uint32_t w, float (&sc)[4]) {
  uint32_t s01, s23;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n"
      " cvt.rn.bf16x2.ue8m0x2 %0, lo;\n cvt.rn.bf16x2.ue8m0x2 %1, hi;\n}\n"
      : "=r"(s01), "=r"(s23)
      : "r"(w));
  sc[0] = __uint_as_float(s01 << 16);
  sc[1] = __uint_as_float(s01 & 0xFFFF0000u);
  sc[2] = __uint_as_float(s23 << 16);
  sc[3] = __uint_as_float(s23 & 0xFFFF0000u);
}

// One m16 row tile: rows g (words wl, scale word sl) and g+8 (wh, sh) of a
// 16-entry group. Returns the score of row g in lanes with even t4 and of row g+8
// in lanes with odd t4.
template <int NPART>
__device__ __forceinline__ float scan_m16(const uint32_t (&wl)[4], const uint32_t (&wh)[4], uint32_t sl, uint32_t sh,
                                          const uint32_t (&bf)[2][4][NPART][2], float wsel, int t4) {
  float acc[2][NPART][4];
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int nt = 0; nt < NPART; ++nt) acc[p][nt][0] = acc[p][nt][1] = acc[p][nt][2] = acc[p][nt][3] = 0.f;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    uint32_t lo0[4], lo1[4], hi0[4], hi1[4];
    e2m1x8_to_f16x2(wl[2 * p], lo0);
    e2m1x8_to_f16x2(wl[2 * p + 1], lo1);
    e2m1x8_to_f16x2(wh[2 * p], hi0);
    e2m1x8_to_f16x2(wh[2 * p + 1], hi1);
#pragma unroll
    for (int kq = 0; kq < 4; ++kq)
#pragma unroll
      for (int nt = 0; nt < NPART; ++nt)
        mma_16816(acc[p][nt], lo0[kq], hi0[kq], lo1[kq], hi1[kq], bf[p][kq][nt][0], bf[p][kq][nt][1]);
  }
  // acc[p][.][2 rr + jj]: row g + 8 rr, column 2 t4 + jj = head t4, block 2p + jj
  float part[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    float sc[4];
    e8m0x4_decode(rr ? sh : sl, sc);
    float d[4];
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        d[2 * p + jj] = acc[p][0][2 * rr + jj];
        if constexpr (NPART == 2) d[2 * p + jj] += acc[p][1][2 * rr + jj];
      }
    const float v = fmaf(d[3], sc[3], fmaf(d[2], sc[2], fmaf(d[1], sc[1], d[0] * sc[0])));
    part[rr] = wsel * fmaxf(v, 0.f);
  }
  // heads: lanes t4 and t4^1 trade the row the other one keeps, then t4 ^ 2
  const bool odd = (t4 & 1) != 0;
  float keep = odd ? part[1] : part[0];
  keep += __shfl_xor_sync(0xffffffffu, odd ? part[0] : part[1], 1);
  keep += __shfl_xor_sync(0xffffffffu, keep, 2);
  return keep;
}

// ---------------------------------------------------------------- gather form
// Scores a list of candidate positions (the hierarchical pool): rows are
// gathered, so each lane loads its words straight from global memory, one
// 32-entry tile ahead.
template <int NPART>
__global__ void __launch_bounds__(kScanThreads, 2) k_indexer_scan_gather(const ScanArgs a) {
  pdl_wait_and_release();
  const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int64_t gw = (int64_t)blockIdx.x * kScanWarps + (threadIdx.x >> 5);
  const int64_t nw = (int64_t)gridDim.x * kScanWarps;
  const int64_t t_begin = gw * a.total_tiles / nw, t_end = (gw + 1) * a.total_tiles / nw;
  if (t_begin >= t_end) return;
  const uint64_t pol = l2_evict_first_policy();
  const uint64_t spol = l2_scores_policy(a.scratch);

  uint32_t bf[2][4][NPART][2];
  float wsel = 0.f;
  int setup_b = -1;

  ScanTile cur, nxt;
  scan_load_tile(cur, t_begin, a, g, t4, pol);
  for (int64_t t = t_begin; t < t_end; ++t) {
    if (t + 1 < t_end) scan_load_tile(nxt, t + 1, a, g, t4, pol);
    if (cur.b != setup_b) {
      scan_setup<NPART>(cur.b, a, lane, g, t4, bf, wsel);
      setup_b = cur.b;
    }
#pragma unroll
    for (int st = 0; st < 2; ++st) {  // rows (2st, 2st+1) = entries g + 16st (+8)
      const int rl = 2 * st, rh = 2 * st + 1;
      const float sc = scan_m16<NPART>(cur.w[rl], cur.w[rh], cur.s[rl], cur.s[rh], bf, wsel, t4);
      if (t4 < 2) {  // lane t4 == 0 stores row rl, lane t4 == 1 row rh
        const int r = t4 ? rh : rl;
        if ((cur.flags >> r) & 1u) {
          const int64_t e = cur.e0 + g + 8 * r;
          st_score(a.scores + (size_t)cur.b * a.stride + e, ((cur.flags >> (4 + r)) & 1u) ? sc : -INFINITY, spol);
        }
      }
    }
    cur = nxt;
  }
}

// ---------------------------------------------------------------- streaming form
// Scores every entry of every sequence. A producer warp streams 512-entry stages
// -- four TMA boxes of 128 rows x 64 bytes of codes (64-byte swizzle) and one bulk
// copy of their E8M0 bytes -- into a ring of three shared-memory stages; eight
// consumer warps take 64 rows (four m16 tiles) each per stage, so one wait and
// one release cover four independent tiles. Two blocks share an SM (209 KB of
// stages in flight per SM). Full/empty mbarriers hand the stages back and forth;
// every wait gives up after about a second, records CSA2_ERR_TIMEOUT and stops
// the block. (Measured on B300 at 32 x 131,072 entries: 16-row warp tiles and
// 128-row stages ran at 3.8 TB/s, 32-row tiles at 4.6, 64-row tiles at 5.2.)
//
// With the 64-byte swizzle the 16-byte chunk j of row r sits at chunk
// j ^ ((r >> 1) & 3), which makes the consumers' 32-bit loads (word t4 of each
// chunk, rows g + 8r) free of bank conflicts.
#ifndef CSA2_SCAN_CONSUMERS
#define CSA2_SCAN_CONSUMERS 8
#endif
constexpr int kTmaConsumers = CSA2_SCAN_CONSUMERS;
constexpr int kTmaThreads = (kTmaConsumers + 1) * 32;
#ifndef CSA2_SCAN_STAGE_ROWS
#define CSA2_SCAN_STAGE_ROWS 512
#endif
#ifndef CSA2_SCAN_STAGES
#define CSA2_SCAN_STAGES 3
#endif
#ifndef CSA2_SCAN_BLOCKS_PER_SM
#define CSA2_SCAN_BLOCKS_PER_SM 2
#endif
constexpr int kTmaRows = 128;                           // rows of one TMA box
constexpr int kTmaStageRows = CSA2_SCAN_STAGE_ROWS;     // rows of one stage (whole boxes)
constexpr int kTmaWarpRows = kTmaStageRows / kTmaConsumers;
constexpr int kTmaWarpM16 = kTmaWarpRows / 16;          // m16 tiles per consumer warp per stage
constexpr int kTmaStages = CSA2_SCAN_STAGES;
constexpr int kTmaBlocksPerSM = CSA2_SCAN_BLOCKS_PER_SM;
constexpr int kTmaStageBytes = kTmaStageRows * 68;      // codes, then the E8M0 bytes
constexpr int kTmaSmem = kTmaStages * kTmaStageBytes + 2 * kTmaStages * 8 + 64 + 1024;
static_assert(kTmaStageRows % kTmaRows == 0 && kTmaWarpRows % 16 == 0, "stage shape");
static_assert(kTmaStageBytes % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled boxes");

struct TmaScanArgs {
  const void* q_idx;
  int q_dtype;
  const float* w;
  const uint8_t* codes;
  const uint8_t* scales;
  int64_t cap;
  const int32_t* len;
  float* scores;
  int scratch;  // the scores are a decode step's scratch (see l2_scores_policy)
  int64_t tiles_per_seq;  // ceil(cap / tile rows): 256-row stages (mma.sync form), 128 (tcgen05 form)
  int64_t total_tiles;
};

template <int NPART>
__global__ void __launch_bounds__(kTmaThreads, kTmaBlocksPerSM)
k_indexer_scan_tma(const __grid_constant__ CUtensorMap tmap, const TmaScanArgs a) {
  pdl_wait();  // (the next kernel may launch once every thread has released it, at its end)
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32addr(smem);
  const uint32_t bar_full = sbase + kTmaStages * kTmaStageBytes;
  const uint32_t bar_empty = bar_full + 8 * kTmaStages;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kTmaStages * kTmaStageBytes + 16 * kTmaStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTmaStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kTmaConsumers);
    }
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  const int64_t t_begin = (int64_t)blockIdx.x * a.total_tiles / gridDim.x;
  const int64_t t_end = (int64_t)(blockIdx.x + 1) * a.total_tiles / gridDim.x;
  int b0 = (int)(t_begin / a.tiles_per_seq);
  int64_t e00 = (t_begin - (int64_t)b0 * a.tiles_per_seq) * kTmaStageRows;
  const int64_t seq_rows = a.tiles_per_seq * kTmaStageRows;

  if (warp == kTmaConsumers) {
    // ---------------- producer (one lane)
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      asm volatile("prefetch.tensormap [%0];\n" ::"l"(&tmap) : "memory");
      uint32_t it = 0;
      int b = b0;
      int64_t e0 = e00;
      int64_t n_b = min((int64_t)__ldg(a.len + b), a.cap);
      for (int64_t t = t_begin; t < t_end; ++t) {
        if (e0 < n_b) {
          const uint32_t s = it % kTmaStages, ph = (it / kTmaStages) & 1u;
          if (!mbar_wait_bounded(bar_empty + 8 * s, ph ^ 1u, abort)) break;
          const uint32_t st = sbase + s * kTmaStageBytes;
          const int64_t row = (int64_t)b * a.cap + e0;
          // the last stage of a sequence holds fewer boxes when cap is not a multiple of
          // the stage rows (cap is a multiple of 128)
          const int64_t left = a.cap - e0;
          const uint32_t rows = left >= kTmaStageRows ? (uint32_t)kTmaStageRows : (uint32_t)left;
          mbar_arrive_expect_tx(bar_full + 8 * s, rows * 68);
          for (uint32_t q = 0; q < rows / kTmaRows; ++q)
            tma_load_rows(st + q * kTmaRows * 64, &tmap, 0, (int32_t)(row + q * kTmaRows), bar_full + 8 * s, pol);
          bulk_load(st + kTmaStageRows * 64, a.scales + row * 4, rows * 4, bar_full + 8 * s, pol);
          ++it;
        }
        e0 += kTmaStageRows;
        if (e0 >= seq_rows && t + 1 < t_end) {
          e0 = 0;
          ++b;
          n_b = min((int64_t)__ldg(a.len + b), a.cap);
        }
      }
      // drain: every issued stage must land before the block exits
      for (uint32_t j = (it > kTmaStages ? it - kTmaStages : 0); j < it; ++j) {
        volatile int no_abort = 0;
        mbar_wait_bounded(bar_full + 8 * (j % kTmaStages), (j / kTmaStages) & 1u, &no_abort);
      }
    }
  } else {
    // ---------------- consumers: warp w owns rows kTmaWarpRows * w + g + 8r of every stage
    // (kTmaWarpM16 m16 tiles)
    const int g = lane >> 2, t4 = lane & 3;
    const int r0 = kTmaWarpRows * warp + g;
    const uint32_t swz = (uint32_t)((g >> 1) & 3);  // the same for every row r0 + 8r
    const uint64_t spol = l2_scores_policy(a.scratch);
    ScanArgs sa;
    sa.q_idx = a.q_idx;
    sa.q_dtype = a.q_dtype;
    sa.w = a.w;
    uint32_t bf[2][4][NPART][2];
    float wsel = 0.f;
    int setup_b = -1;
    uint32_t it = 0;
    int b = b0;
    int64_t e0 = e00;
    int64_t n_b = min((int64_t)__ldg(a.len + b), a.cap);
    for (int64_t t = t_begin; t < t_end; ++t) {
      if (e0 < n_b) {
        if (b != setup_b) {
          scan_setup<NPART>(b, sa, lane, g, t4, bf, wsel);
          setup_b = b;
        }
        const uint32_t s = it % kTmaStages, ph = (it / kTmaStages) & 1u;
        if (!mbar_wait_bounded(bar_full + 8 * s, ph, abort)) break;
        const unsigned char* st = smem + s * kTmaStageBytes;
        uint32_t w[2 * kTmaWarpM16][4], sw[2 * kTmaWarpM16];
#pragma unroll
        for (int r = 0; r < 2 * kTmaWarpM16; ++r) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            w[r][j] = *reinterpret_cast<const uint32_t*>(st + 64 * (r0 + 8 * r) + 16u * ((uint32_t)j ^ swz) + 4u * t4);
          sw[r] = *reinterpret_cast<const uint32_t*>(st + kTmaStageRows * 64 + 4 * (r0 + 8 * r));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        ++it;
        // lanes t4 and t4 + 2 hold the same row: even t4 row r0 + 16 m, odd t4 that + 8
        const int64_t erow = e0 + r0 + 8 * (t4 & 1);
        float* sp = a.scores + (size_t)b * a.cap + erow;
        if (NPART == 1 && e0 + kTmaStageRows <= n_b) {  // every row of the stage is valid
#pragma unroll
          for (int m = 0; m < kTmaWarpM16; ++m) {
            const float sc = scan_m16<NPART>(w[2 * m], w[2 * m + 1], sw[2 * m], sw[2 * m + 1], bf, wsel, t4);
            if (t4 < 2) st_score(sp + 16 * m, sc, spol);
          }
        } else {  // the last stage of the sequence (and every stage of fp32 queries)
#pragma unroll
          for (int m = 0; m < kTmaWarpM16; ++m) {
            const float sc = scan_m16<NPART>(w[2 * m], w[2 * m + 1], sw[2 * m], sw[2 * m + 1], bf, wsel, t4);
            if (t4 < 2 && erow + 16 * m < n_b) st_score(sp + 16 * m, sc, spol);
          }
        }
      }
      e0 += kTmaStageRows;
      if (e0 >= seq_rows && t + 1 < t_end) {
        e0 = 0;
        ++b;
        n_b = min((int64_t)__ldg(a.len + b), a.cap);
      }
    }
  }
  // one thread of a block releasing the next kernel counts for the whole block, and the
  // producer warp's idle lanes get here at once: release only when every thread has
  __syncthreads();
  pdl_release();
}

}  // namespace csa2
