// Top-k of a decode step fused with the indexer scan (k <= kFusedMaxK).
//
// Pages: "890 octets de cache KV par token", "Deuxiemement" (each Full layer
// scores the cache with its indexer and keeps new Top-512 indices).
//
// Three launches replace "scan every entry, then select over every score":
//  1. k_row_threshold: per row, tau = a lower bound of the key of rank
//     ceil(T * samples / len) among 1024 evenly spaced scored samples
//     (T = 4k + 256 keys expected >= tau); resets the row's count;
//  2. the streaming scan writes every score and appends every key >= tau to the
//     row's candidate list (kFusedCap keys);
//  3. k_select_candidates: with c candidates, min(k, len) <= c <= kFusedCap means
//     the list holds the k largest keys; the exact k-th largest K comes from the
//     range radix over the list and the keys >= K are emitted in position order.
//     Otherwise (an unlucky sample) the block repeats the filter on the row's
//     stored scores with a fresh threshold from 4096 samples (topk_row), and
//     selects over the whole row only if that misses too: slower, same result.
#pragma once

#include "indexer_scan.cuh"
#include "topk.cuh"

namespace csa2 {

constexpr int kFusedMaxK = 1024;
constexpr int kFusedCap = 8192;

// Keys wanted >= tau per row: 4k + 256 (2,304 for k = 512); the candidate list
// holds kFusedCap, so an overflow needs the threshold sample off by several
// standard deviations.
__host__ __device__ constexpr unsigned long long fused_target(int k) { return 4ull * (unsigned)k + 256ull; }

struct FusedSelectArgs {
  unsigned long long* tau;         // [batch]
  uint32_t* cand_count;            // [batch]
  unsigned long long* cand_keys;   // [batch][kFusedCap]
};

// A lower bound of the key of rank r among buf[0..n) (two range-radix rounds).
struct TauSelect {
  TopkCtl* sh;
  __device__ unsigned long long operator()(const unsigned long long* buf, uint32_t n, uint32_t r) const {
    return block_select(BufSrc{buf}, n, r, *sh, 2);
  }
};

template <int NPART>
__global__ void __launch_bounds__(kTopkThreads)
k_row_threshold(const ScanArgs a, int k, FusedSelectArgs f) {
  __shared__ TopkCtl sh;
  __shared__ unsigned long long keys[kThreshSamples];
  const int b = blockIdx.x;
  if (threadIdx.x == 0) f.cand_count[b] = 0;
  scan_threshold_row<NPART>(a, b, fused_target(k), keys, TauSelect{&sh}, f.tau + b);
}

__global__ void __launch_bounds__(kTopkThreads)
k_select_candidates(const float* __restrict__ scores, int64_t cap, const int32_t* __restrict__ len, int k,
                    FusedSelectArgs f, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkCtl& sh = *reinterpret_cast<TopkCtl*>(smem_raw);
  unsigned long long* buf = reinterpret_cast<unsigned long long*>(smem_raw + sizeof(TopkCtl));
  const int b = blockIdx.x, tid = threadIdx.x;
  const uint32_t n = (uint32_t)min((int64_t)__ldg(len + b), cap);
  const uint32_t c = __ldg(f.cand_count + b);
  int32_t* orow = out + (size_t)b * k;
  const uint32_t need = n < (uint32_t)k ? n : (uint32_t)k;
  if (c <= (uint32_t)kFusedCap && c >= need) {
    const unsigned long long* src = f.cand_keys + (size_t)b * kFusedCap;
    for (uint32_t j = tid; j < c; j += kTopkThreads) buf[j] = __ldg(src + j);
    __syncthreads();
    const unsigned long long K = c > (uint32_t)k ? block_select(BufSrc{buf}, c, (uint32_t)k, sh) : 0ull;
    topk_emit_sorted(buf, c, K, k, nullptr, orow, sh);
    return;
  }
  topk_row(scores + (size_t)b * cap, n, k, fused_target(k), buf, kFusedCap, orow, sh);
}

}  // namespace csa2
