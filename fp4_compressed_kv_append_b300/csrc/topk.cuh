// topk_select: exact Top-k per row, ties to the lower position, output ascending.
//
// Pages: "890 octets de cache KV par token", section "L'architecture",
// "Deuxiemement" (each Full layer selects new Top-512 indices; the hierarchical
// indexer keeps 16,384 candidate positions).
//
// Every candidate slot i gets the 64-bit key (order(score_i) << 32) | (2^32-1 - i):
// keys are distinct, and "larger key" is exactly "higher score, then lower slot"
// (slots are positions, or indices into an ascending candidate list). One
// 1024-thread block per row:
//  1. sample: the keys of S evenly spaced slots; tau = the r-th largest sample,
//     r chosen so that about (k + CAP)/2 keys of the row are expected >= tau;
//  2. filter: every valid key >= tau is appended to a shared-memory buffer of CAP
//     keys (warp ballot + one atomic per warp);
//  3. exact select of the k-th largest key K among them (below); the k keys >= K,
//     compacted in place and bitonic-sorted by slot, give the output.
// If fewer than k or more than CAP keys pass the filter (an unlucky sample), the
// block selects K over the whole row instead and writes the keys >= K by an
// ordered compaction over the row -- slower, same result.
//
// Exact select ("range radix"): among the active keys (those in [lo, hi]) find
// min and max; histogram (key - min) >> shift into at most 2048 bins, shift
// chosen so the bins span exactly [min, max]; the bin holding the wanted rank
// (counted from the top) becomes the new [lo, hi]. Fitting the bins to the
// occupied range spreads even tightly clustered scores over many bins, so the
// shared-memory atomics do not pile onto a few addresses. Stops when min == max.
#pragma once

#include "common.cuh"

namespace csa2 {

constexpr int kTopkThreads = 1024;
constexpr int kSelBits = 11;
constexpr int kSelBins = 1 << kSelBits;

struct TopkCtl {
  uint32_t hist[kSelBins];
  uint32_t warp_u32[32];
  unsigned long long warp_a[32], warp_b[32];
  unsigned long long bc_a, bc_b;
  uint32_t bc_u32[4];
  uint32_t count;
};

// Candidate-buffer capacity (keys) for a given k; the shared memory is
// sizeof(TopkCtl) + 8 * cap bytes.
__host__ __device__ constexpr uint32_t topk_cap(int k) {
  return k <= 1024 ? 4096u
                   : ((3u * (uint32_t)k / 2u + 2048u + 1023u) / 1024u * 1024u < 16384u
                          ? 16384u
                          : ((3u * (uint32_t)k / 2u + 2048u + 1023u) / 1024u * 1024u > 24576u
                                 ? 24576u
                                 : (3u * (uint32_t)k / 2u + 2048u + 1023u) / 1024u * 1024u));
}

// Sample size of step 1 (never above topk_cap(k)).
__host__ __device__ constexpr uint32_t topk_sample(int k) { return k <= 1024 ? 4096u : 16384u; }

__device__ __forceinline__ unsigned long long topk_key(float s, uint32_t slot) {
  return ((unsigned long long)float_order_key(s) << 32) | (unsigned long long)(0xFFFFFFFFu - slot);
}

// Exclusive scan over the block of one value per thread; *total gets the sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, TopkCtl& sh, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh.warp_u32[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t s = sh.warp_u32[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sh.warp_u32[lane] = s;
  }
  __syncthreads();
  const uint32_t before = wid ? sh.warp_u32[wid - 1] : 0u;
  *total = sh.warp_u32[31];
  __syncthreads();
  return before + x - v;
}

__device__ __forceinline__ uint32_t block_sum(uint32_t v, TopkCtl& sh) {
  uint32_t t;
  block_excl_scan(v, sh, &t);
  return t;
}

// Block-wide min and max of 64-bit values; every thread gets both.
__device__ __forceinline__ void block_minmax(unsigned long long& mn, unsigned long long& mx, TopkCtl& sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long a = __shfl_xor_sync(0xffffffffu, mn, o);
    const unsigned long long b = __shfl_xor_sync(0xffffffffu, mx, o);
    mn = a < mn ? a : mn;
    mx = b > mx ? b : mx;
  }
  if (lane == 0) {
    sh.warp_a[wid] = mn;
    sh.warp_b[wid] = mx;
  }
  __syncthreads();
  if (wid == 0) {
    mn = sh.warp_a[lane];
    mx = sh.warp_b[lane];
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const unsigned long long a = __shfl_xor_sync(0xffffffffu, mn, o);
      const unsigned long long b = __shfl_xor_sync(0xffffffffu, mx, o);
      mn = a < mn ? a : mn;
      mx = b > mx ? b : mx;
    }
    if (lane == 0) {
      sh.bc_a = mn;
      sh.bc_b = mx;
    }
  }
  __syncthreads();
  mn = sh.bc_a;
  mx = sh.bc_b;
  __syncthreads();
}

// The rank-th largest (1-based) key among those >= 1 produced by src(i), i < n.
// Requires 1 <= rank <= number of such keys. Keys are distinct.
template <class Src>
__device__ unsigned long long block_select(const Src& src, uint32_t n, uint32_t rank, TopkCtl& sh) {
  const int tid = threadIdx.x;
  unsigned long long lo = 1, hi = ~0ull;
  uint32_t krem = rank;
  for (int iter = 0; iter < 64; ++iter) {
    unsigned long long mn = ~0ull, mx = 0;
    for (uint32_t i = tid; i < n; i += kTopkThreads) {
      const unsigned long long x = src(i);
      if (x >= lo && x <= hi) {
        mn = x < mn ? x : mn;
        mx = x > mx ? x : mx;
      }
    }
    block_minmax(mn, mx, sh);
    if (mn >= mx) return mx == 0 ? mn : mx;  // one key left (or, defensively, none)
    const unsigned long long d = mx - mn;
    const int bits = 64 - __clzll((long long)d);
    const int shift = bits > kSelBits ? bits - kSelBits : 0;
    const uint32_t nb = (uint32_t)(d >> shift) + 1u;
    for (uint32_t j = tid; j < nb; j += kTopkThreads) sh.hist[j] = 0;
    __syncthreads();
    for (uint32_t i = tid; i < n; i += kTopkThreads) {
      const unsigned long long x = src(i);
      if (x >= mn && x <= mx) atomicAdd(&sh.hist[(uint32_t)((x - mn) >> shift)], 1u);
    }
    __syncthreads();
    // thread t owns bins nb-1-2t and nb-2-2t (scanned from the top)
    const int b0 = (int)nb - 1 - 2 * tid, b1 = b0 - 1;
    const uint32_t h0 = b0 >= 0 ? sh.hist[b0] : 0u, h1 = b1 >= 0 ? sh.hist[b1] : 0u;
    uint32_t tot;
    const uint32_t above = block_excl_scan(h0 + h1, sh, &tot);
    if (above < krem && above + h0 + h1 >= krem) {
      if (above + h0 >= krem) {
        sh.bc_u32[0] = (uint32_t)b0;
        sh.bc_u32[1] = above;
      } else {
        sh.bc_u32[0] = (uint32_t)b1;
        sh.bc_u32[1] = above + h0;
      }
    }
    __syncthreads();
    const uint32_t bin = sh.bc_u32[0];
    krem -= sh.bc_u32[1];
    lo = mn + ((unsigned long long)bin << shift);
    const unsigned long long span = (1ull << shift) - 1ull;
    hi = (mx - lo) < span ? mx : lo + span;
    __syncthreads();
  }
  return lo;
}

struct RowSrc {  // keys straight from the score row (invalid slots -> 0)
  const float* row;
  const int32_t* crow;
  __device__ unsigned long long operator()(uint32_t i) const {
    if (crow && __ldg(crow + i) < 0) return 0ull;
    return topk_key(__ldg(row + i), i);
  }
};

struct BufSrc {  // keys in shared memory
  const unsigned long long* buf;
  __device__ unsigned long long operator()(uint32_t i) const { return buf[i]; }
};

__global__ void __launch_bounds__(kTopkThreads, 1)
k_topk(const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ nvec,
       const int32_t* __restrict__ cand, int k, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkCtl& sh = *reinterpret_cast<TopkCtl*>(smem_raw);
  unsigned long long* buf = reinterpret_cast<unsigned long long*>(smem_raw + sizeof(TopkCtl));
  const uint32_t CAP = topk_cap(k);
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  int64_t n64 = nvec ? (int64_t)__ldg(nvec + b) : stride;
  n64 = n64 < 0 ? 0 : (n64 > stride ? stride : n64);
  const uint32_t n = (uint32_t)n64;
  const float* row = scores + (size_t)b * stride;
  const int32_t* crow = cand ? cand + (size_t)b * stride : nullptr;
  int32_t* orow = out + (size_t)b * k;
  const RowSrc rsrc{row, crow};

  // ---- number of valid slots
  uint32_t m = n;
  if (crow) {
    uint32_t c = 0;
    for (uint32_t i = tid; i < n; i += kTopkThreads) c += __ldg(crow + i) >= 0;
    m = block_sum(c, sh);
  }

  if (m <= (uint32_t)k) {  // every valid slot is selected, in slot order
    uint32_t written = 0;
    for (uint32_t t0 = 0; t0 < n; t0 += kTopkThreads) {
      const uint32_t i = t0 + tid;
      const int32_t pos = i < n ? (crow ? __ldg(crow + i) : (int32_t)i) : -1;
      uint32_t tot;
      const uint32_t r = block_excl_scan(pos >= 0 ? 1u : 0u, sh, &tot);
      if (pos >= 0) orow[written + r] = pos;
      written += tot;
    }
    for (uint32_t j = written + tid; j < (uint32_t)k; j += kTopkThreads) orow[j] = -1;
    return;
  }

  // ---- 1. sample -> tau
  const uint32_t S_target = topk_sample(k);
  const uint32_t S = n < S_target ? n : S_target;
  uint32_t sv = 0;
  for (uint32_t s = tid; s < S; s += kTopkThreads) {
    const uint32_t i = (uint32_t)(((unsigned long long)s * n) / S);
    const unsigned long long key = rsrc(i);
    buf[s] = key;
    sv += key != 0ull;
  }
  sv = block_sum(sv, sh);  // (also a barrier for buf)
  unsigned long long tau = 1ull;  // no valid sample: every valid key passes
  if (sv > 0) {
    const unsigned long long target = ((unsigned long long)k + CAP) / 2;
    unsigned long long r = (target * sv + m - 1) / m;
    r = r < 1 ? 1 : (r > sv ? sv : r);
    tau = block_select(BufSrc{buf}, S, (uint32_t)r, sh);
  }
  const uint32_t thi = (uint32_t)(tau >> 32), tlo = (uint32_t)tau;

  // ---- 2. filter (keys >= tau; a valid key's high word is never 0)
  if (tid == 0) sh.count = 0;
  __syncthreads();
  const bool vec = (((uintptr_t)row | (uintptr_t)crow) & 15u) == 0;
  for (uint32_t t0 = 0; t0 < n; t0 += 4 * kTopkThreads) {
    const uint32_t i0 = t0 + 4 * tid;
    float sc[4];
    int32_t cv[4] = {0, 0, 0, 0};
    if (vec && i0 + 3 < n) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(row + i0));
      sc[0] = v.x; sc[1] = v.y; sc[2] = v.z; sc[3] = v.w;
      if (crow) {
        const int4 cc = __ldg(reinterpret_cast<const int4*>(crow + i0));
        cv[0] = cc.x; cv[1] = cc.y; cv[2] = cc.z; cv[3] = cc.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        sc[u] = i0 + u < n ? __ldg(row + i0 + u) : 0.f;
        cv[u] = i0 + u < n ? (crow ? __ldg(crow + i0 + u) : 0) : -1;
      }
    }
    bool pass[4];
    bool any = false;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t kh = float_order_key(sc[u]);
      pass[u] = cv[u] >= 0 && (kh > thi || (kh == thi && 0xFFFFFFFFu - (i0 + u) >= tlo));
      any |= pass[u];
    }
    if (__any_sync(0xffffffffu, any)) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const unsigned mask = __ballot_sync(0xffffffffu, pass[u]);
        if (mask) {
          const int leader = __ffs(mask) - 1;
          uint32_t base = 0;
          if (lane == leader) base = atomicAdd(&sh.count, (uint32_t)__popc(mask));
          base = __shfl_sync(0xffffffffu, base, leader);
          if (pass[u]) {
            const uint32_t at = base + __popc(mask & ((1u << lane) - 1u));
            if (at < CAP) buf[at] = topk_key(sc[u], i0 + u);
          }
        }
      }
    }
  }
  __syncthreads();
  const uint32_t c = sh.count;
  __syncthreads();

  if (c >= (uint32_t)k && c <= CAP) {
    // ---- 3. exact select among the candidates, compact, sort by slot
    const unsigned long long K = block_select(BufSrc{buf}, c, (uint32_t)k, sh);
    // ordered in-place compaction of the slots of keys >= K into the front of buf (as u32)
    uint32_t* slots = reinterpret_cast<uint32_t*>(buf);
    uint32_t written = 0;
    for (uint32_t t0 = 0; t0 < c; t0 += kTopkThreads) {
      const uint32_t i = t0 + tid;
      const unsigned long long key = i < c ? buf[i] : 0ull;
      const bool take = i < c && key >= K;
      uint32_t tot;
      const uint32_t rr = block_excl_scan(take ? 1u : 0u, sh, &tot);  // every read of this chunk precedes
      if (take) slots[written + rr] = 0xFFFFFFFFu - (uint32_t)key;     // writes, which stay below it
      written += tot;
      __syncthreads();
    }
    uint32_t kp = 1;
    while (kp < (uint32_t)k) kp <<= 1;
    for (uint32_t j = (uint32_t)k + tid; j < kp; j += kTopkThreads) slots[j] = 0xFFFFFFFFu;
    __syncthreads();
    for (uint32_t size = 2; size <= kp; size <<= 1) {
      for (uint32_t half = size >> 1; half > 0; half >>= 1) {
        for (uint32_t i = tid; i < kp / 2; i += kTopkThreads) {
          const uint32_t lo_i = 2 * half * (i / half) + (i % half), hi_i = lo_i + half;
          const uint32_t x = slots[lo_i], y = slots[hi_i];
          const bool asc = (lo_i & size) == 0;
          if ((x > y) == asc) {
            slots[lo_i] = y;
            slots[hi_i] = x;
          }
        }
        __syncthreads();
      }
    }
    for (uint32_t j = tid; j < (uint32_t)k; j += kTopkThreads) {
      const uint32_t sl = slots[j];
      orow[j] = crow ? __ldg(crow + sl) : (int32_t)sl;
    }
    return;
  }

  // ---- fallback: select over the whole row, ordered compaction over the row
  const unsigned long long K = block_select(rsrc, n, (uint32_t)k, sh);
  uint32_t written = 0;
  for (uint32_t t0 = 0; t0 < n && written < (uint32_t)k; t0 += kTopkThreads) {
    const uint32_t i = t0 + tid;
    const unsigned long long key = i < n ? rsrc(i) : 0ull;
    const bool take = key != 0ull && key >= K;
    uint32_t tot;
    const uint32_t rr = block_excl_scan(take ? 1u : 0u, sh, &tot);
    if (take && written + rr < (uint32_t)k) orow[written + rr] = crow ? __ldg(crow + i) : (int32_t)i;
    written += tot;
  }
  for (uint32_t j = written + tid; j < (uint32_t)k; j += kTopkThreads) orow[j] = -1;
}

}  // namespace csa2
