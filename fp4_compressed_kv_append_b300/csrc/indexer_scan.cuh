// indexer_score: score_t = sum_h w_h * max(0, q_h . k_t) over the 4 indexer heads,
// k_t the MXFP4 key (E2M1 codes times the E8M0 scale of each 32-channel block).
//
// Pages: "Le cache KV en FP4", section "Les ingredients", item 2 (the 128-channel
// indexer key scores positions) and section "Cles d'indexeur" (eq. 68: E2M1 with an
// E8M0 scale per 32 channels).
//
// CUDA-core form: one thread per entry. The 64 code bytes of an entry are read as
// four 16-byte vectors, the queries live in shared memory as float. Each block of
// 32 channels is summed unscaled (the codes are exact small numbers), then scaled by
// its power of two, in float32.
#pragma once

#include "common.cuh"

namespace csa2 {

constexpr int kScanThreads = 256;

__global__ void __launch_bounds__(kScanThreads)
k_indexer_scan_simple(const void* __restrict__ q_idx, int q_dtype, const float* __restrict__ w,
                      const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                      int64_t cap, const int32_t* __restrict__ len,
                      const int32_t* __restrict__ cand, int P, float* __restrict__ scores,
                      int64_t stride) {
  __shared__ float qs[CSA2_INDEXER_HEADS][CSA2_INDEXER_DIM];
  __shared__ float ws[CSA2_INDEXER_HEADS];
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < CSA2_INDEXER_HEADS * CSA2_INDEXER_DIM; i += blockDim.x)
    qs[i / CSA2_INDEXER_DIM][i % CSA2_INDEXER_DIM] =
        load_elem(q_idx, q_dtype, (size_t)b * CSA2_INDEXER_HEADS * CSA2_INDEXER_DIM + i);
  if (threadIdx.x < CSA2_INDEXER_HEADS) ws[threadIdx.x] = w[b * CSA2_INDEXER_HEADS + threadIdx.x];
  __syncthreads();

  const int n_b = min((int64_t)__ldg(len + b), cap);  // never past the capacity
  const int n = cand ? P : n_b;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  int64_t pos = i;
  if (cand) {
    pos = __ldg(cand + (size_t)b * P + i);
    if (pos < 0 || pos >= n_b) {
      if (pos >= n_b) set_dev_error(CSA2_ERR_BOUNDS);
      scores[(size_t)b * stride + i] = -INFINITY;
      return;
    }
  }
  const size_t row = (size_t)b * cap + pos;
  const uint4* cp = reinterpret_cast<const uint4*>(codes + row * 64);
  const uint32_t sc = __ldg(reinterpret_cast<const uint32_t*>(scales + row * 4));
  float acc[CSA2_INDEXER_HEADS] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int blk = 0; blk < 4; ++blk) {
    const uint4 v = __ldg(cp + blk);
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    float part[CSA2_INDEXER_HEADS] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 32; ++j) {  // channel 32*blk + j, nibble j of the block's 16 bytes
      const uint32_t c = (wd[j >> 3] >> (4 * (j & 7))) & 15u;
      float val = e2m1_magnitude(c & 7u);
      val = (c & 8u) ? -val : val;
#pragma unroll
      for (int h = 0; h < CSA2_INDEXER_HEADS; ++h) part[h] = fmaf(qs[h][32 * blk + j], val, part[h]);
    }
    const float s = e8m0_decode((sc >> (8 * blk)) & 0xFFu);
#pragma unroll
    for (int h = 0; h < CSA2_INDEXER_HEADS; ++h) acc[h] = fmaf(part[h], s, acc[h]);
  }
  float score = 0.f;
#pragma unroll
  for (int h = 0; h < CSA2_INDEXER_HEADS; ++h) score = fmaf(ws[h], fmaxf(acc[h], 0.f), score);
  scores[(size_t)b * stride + i] = score;
}

}  // namespace csa2
