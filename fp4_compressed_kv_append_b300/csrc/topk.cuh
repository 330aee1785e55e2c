// topk_select: exact Top-k per row, ties to the lower position, output ascending.
//
// Pages: "890 octets de cache KV par token", section "L'architecture",
// "Deuxiemement" (each Full layer selects new Top-512 indices; the hierarchical
// indexer keeps 16,384 candidate positions).
//
// Every candidate i gets the 64-bit key (order(score_i) << 32) | (2^32-1 - pos_i):
// keys are distinct, and "larger key" is exactly "higher score, then lower
// position". One 1024-thread block per row runs an MSB-first radix select over
// 12-bit digits to find tau, the k-th largest key: each pass histograms the digit of
// the candidates that share the prefix found so far (shared-memory atomics) and a
// block scan picks the digit holding the k-th key. Once those candidates fit in
// shared memory they are copied there and the remaining passes read shared memory.
// A last ordered compaction pass writes every position whose key is >= tau, in
// position order, so the output is ascending by construction.
#pragma once

#include "common.cuh"

namespace csa2 {

constexpr int kTopkThreads = 1024;
constexpr int kTopkBins = 4096;  // 12-bit digits
constexpr int kTopkCap = 4096;   // candidates kept in shared memory

struct TopkShared {
  uint32_t hist[kTopkBins];
  unsigned long long cand[kTopkCap];
  uint32_t warp_sums[32];
  uint32_t n_cand;
  uint32_t sel_digit, sel_above, sel_count;
};

__device__ __forceinline__ unsigned long long topk_key(float s, uint32_t pos) {
  return ((unsigned long long)float_order_key(s) << 32) | (unsigned long long)(0xFFFFFFFFu - pos);
}

// Exclusive scan of one value per thread over the block (1024 threads); returns
// the exclusive prefix and writes the block total to *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const uint32_t before = wid ? warp_sums[wid - 1] : 0u;
  *total = warp_sums[31];
  const uint32_t r = before + x - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kTopkThreads)
k_topk(const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ nvec,
       const int32_t* __restrict__ cand, int k, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkShared& sh = *reinterpret_cast<TopkShared*>(smem_raw);
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  int64_t n = nvec ? (int64_t)__ldg(nvec + b) : stride;
  n = n < 0 ? 0 : (n > stride ? stride : n);
  const float* row = scores + (size_t)b * stride;
  const int32_t* crow = cand ? cand + (size_t)b * stride : nullptr;
  int32_t* orow = out + (size_t)b * k;

  // ---- number of valid candidates
  uint32_t m = (uint32_t)n;
  if (crow) {
    uint32_t c = 0;
    for (int64_t i = tid; i < n; i += kTopkThreads) c += __ldg(crow + i) >= 0;
    uint32_t tot;
    block_exclusive_scan(c, sh.warp_sums, &tot);
    m = tot;
  }

  unsigned long long tau = 0;  // every valid key is >= 0: with m <= k all are kept
  if (m > (uint32_t)k) {
    unsigned long long prefix = 0;
    int consumed = 0;          // high key bits fixed so far
    uint32_t krem = (uint32_t)k;
    uint32_t cnt_eq = m;
    bool in_smem = false;
    while (true) {
      if (!in_smem && cnt_eq <= (uint32_t)kTopkCap) {
        if (tid == 0) sh.n_cand = 0;
        __syncthreads();
        for (int64_t i = tid; i < n; i += kTopkThreads) {
          const int32_t pos = crow ? __ldg(crow + i) : (int32_t)i;
          if (pos < 0) continue;
          const unsigned long long key = topk_key(__ldg(row + i), (uint32_t)pos);
          if (consumed == 0 || (key >> (64 - consumed)) == (prefix >> (64 - consumed))) {
            const uint32_t slot = atomicAdd(&sh.n_cand, 1u);
            if (slot < (uint32_t)kTopkCap) sh.cand[slot] = key;
          }
        }
        __syncthreads();
        in_smem = true;
      }
      if (consumed == 64) break;
      const int dbits = (64 - consumed) < 12 ? (64 - consumed) : 12;
      const int shift = 64 - consumed - dbits;
      const uint32_t dmask = (1u << dbits) - 1u;
      for (int i = tid; i < kTopkBins; i += kTopkThreads) sh.hist[i] = 0;
      __syncthreads();
      if (in_smem) {
        const uint32_t nc = sh.n_cand < (uint32_t)kTopkCap ? sh.n_cand : (uint32_t)kTopkCap;
        for (uint32_t i = tid; i < nc; i += kTopkThreads) {
          const unsigned long long key = sh.cand[i];
          if (consumed == 0 || (key >> (64 - consumed)) == (prefix >> (64 - consumed)))
            atomicAdd(&sh.hist[(uint32_t)(key >> shift) & dmask], 1u);
        }
      } else {
        for (int64_t i = tid; i < n; i += kTopkThreads) {
          const int32_t pos = crow ? __ldg(crow + i) : (int32_t)i;
          if (pos < 0) continue;
          const unsigned long long key = topk_key(__ldg(row + i), (uint32_t)pos);
          if (consumed == 0 || (key >> (64 - consumed)) == (prefix >> (64 - consumed)))
            atomicAdd(&sh.hist[(uint32_t)(key >> shift) & dmask], 1u);
        }
      }
      __syncthreads();
      // thread t owns bins [4096-4(t+1), 4096-4t), scanned from the highest bin down
      const int hi_bin = kTopkBins - 4 * tid - 1;
      uint32_t own = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) own += sh.hist[hi_bin - j];
      uint32_t tot;
      const uint32_t above = block_exclusive_scan(own, sh.warp_sums, &tot);
      if (above < krem && above + own >= krem) {
        uint32_t acc = above;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t h = sh.hist[hi_bin - j];
          if (acc + h >= krem) {
            sh.sel_digit = (uint32_t)(hi_bin - j);
            sh.sel_above = acc;
            sh.sel_count = h;
            break;
          }
          acc += h;
        }
      }
      __syncthreads();
      prefix |= (unsigned long long)sh.sel_digit << shift;
      krem -= sh.sel_above;
      cnt_eq = sh.sel_count;
      consumed += dbits;
      __syncthreads();
    }
    tau = prefix;
  }

  // ---- ordered compaction: positions with key >= tau, ascending
  uint32_t written = 0;
  for (int64_t t0 = 0; t0 < n; t0 += kTopkThreads) {
    const int64_t i = t0 + tid;
    bool take = false;
    int32_t pos = -1;
    if (i < n) {
      pos = crow ? __ldg(crow + i) : (int32_t)i;
      if (pos >= 0) take = topk_key(__ldg(row + i), (uint32_t)pos) >= tau;
    }
    uint32_t tot;
    const uint32_t r = block_exclusive_scan(take ? 1u : 0u, sh.warp_sums, &tot);
    if (take && written + r < (uint32_t)k) orow[written + r] = pos;
    written += tot;
    if (written >= (uint32_t)k) break;
  }
  for (uint32_t j = written + tid; j < (uint32_t)k; j += kTopkThreads) orow[j] = -1;
}

}  // namespace csa2
