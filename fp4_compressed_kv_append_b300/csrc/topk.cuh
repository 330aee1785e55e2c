// topk_select: exact Top-k per row, ties to the lower position, output ascending.
//
// Pages: "890 octets de cache KV par token", section "L'architecture",
// "Deuxiemement" (each Full layer selects new Top-512 indices; the hierarchical
// indexer keeps 16,384 candidate positions).
//
// Every slot i of a row gets the 64-bit key (order(score_i) << 32) | (2^32-1 - i):
// keys are distinct, and "larger key" is exactly "higher score, then lower slot"
// (slots are positions, or indices into an ascending candidate list). Invalid
// slots get key 0.
//
// One cluster of kTopkCluster blocks per row; block r owns slice r of the row.
// Small k (<= 1024):
//  A. block r samples its slice and takes tau_r, the smallest key sharing its
//     12-bit prefix (sign, exponent, 3 mantissa bits) with the sample key of rank
//     ceil(T_r * samples / valid_r), T_r = 3k / blocks;
//  B. block r appends its keys >= tau_r to a local buffer, reserves room in block
//     0's buffer (one remote atomic) and copies them there; after this cluster
//     barrier only block 0 goes on;
//  C. block 0: if the candidates number at least k, K is the k-th largest; they
//     hold every key >= K when K >= max_r tau_r, and the k keys >= K are
//     written in slot order through a slot bitmap (rows of up to kBitmapSlots;
//     longer rows: compacted and bitonic-sorted). With fewer than k candidates, all of
//     them when every tau_r was 1 (fewer than k valid slots). Otherwise (an
//     unlucky sample) block 0 selects over the whole row: slower, same result.
// Large k (the hierarchical pool): every block sends samples to block 0, which
// takes one tau for the row; each block counts its keys >= tau, reserves room
// and writes them into block 0's buffer; block 0 finds K (the whole row when
// fewer than k or more than CAP passed); then each block writes its slots with
// key >= K in slot order (32-slot words, one block scan) at the offset given by
// the counts of the blocks before it; the last block pads -1.
// Every cluster barrier is reached by every thread of every block, and no block
// touches another block's shared memory after the last one.
//
// Range radix (exact select): among the active keys (those in [lo, hi]) find min
// and max; histogram (key - min) >> shift into at most 2048 bins, shift chosen so
// the bins span exactly [min, max]; the bin holding the wanted rank (counted from
// the top) becomes the new [lo, hi]. Fitting the bins to the occupied range
// spreads even tightly clustered scores over many bins, so the shared-memory
// atomics do not pile onto a few addresses. Once the bin holds at most 32 keys,
// one warp ranks them directly.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace csa2 {

constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkCluster = 8;
constexpr int kSelBits = 11;
constexpr int kSelBins = 1 << kSelBits;

// Block 0's candidate buffer (keys), a block's local buffer (keys; none for large
// k) and the row's sample count, by k. Shared memory per block: sizeof(TopkCtl)
// + 8 (cap + local).
__host__ __device__ constexpr uint32_t topk_cap(int k) { return k <= 1024 ? 6144u : 24576u; }
__host__ __device__ constexpr uint32_t topk_local_cap(int k) { return k <= 1024 ? 2048u : 0u; }
__host__ __device__ constexpr uint32_t topk_samples(int k) { return k <= 1024 ? 2048u : 16384u; }

constexpr int kPrefixBins = 4096;        // 12-bit key prefixes (sign, exponent, 3 mantissa bits)
constexpr uint32_t kBitmapSlots = 131072; // ordered output through a slot bitmap up to this row length

struct TopkCtl {
  uint32_t hist[kPrefixBins];
  unsigned long long small[32];
  uint32_t warp_u32[32];
  unsigned long long warp_a[32], warp_b[32];
  unsigned long long bc_a, bc_b;
  uint32_t bc_u32[4];
  uint32_t nsmall;
  uint32_t lcount;             // this block: local candidates
  // block 0 only (written remotely by the others)
  uint32_t count;              // candidates reserved in block 0's buffer
  uint32_t valid;              // valid slots of the row (candidate lists)
  uint32_t whole_row;          // K came from the whole row: output by re-reading
  uint32_t over_of[kTopkCluster];  // block r's local buffer overflowed
  unsigned long long tau_of[kTopkCluster];  // block r's threshold (small k)
  unsigned long long tau, K;
  uint32_t sel[kTopkCluster];  // selected slots per block
};

__host__ __device__ constexpr size_t topk_smem_bytes(int k) {
  return sizeof(TopkCtl) + 8u * ((size_t)topk_cap(k) + topk_local_cap(k)) + (k <= 1024 ? kBitmapSlots / 8 : 0);
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
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kTopkWarps; ++w) {
    const uint32_t s = sh.warp_u32[w];
    before += w < wid ? s : 0u;
    tot += s;
  }
  *total = tot;
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
  mn = sh.warp_a[0];
  mx = sh.warp_b[0];
#pragma unroll
  for (int w = 1; w < kTopkWarps; ++w) {
    const unsigned long long a = sh.warp_a[w], b = sh.warp_b[w];
    mn = a < mn ? a : mn;
    mx = b > mx ? b : mx;
  }
  __syncthreads();
}

// The rank-th largest (1-based) of the keys >= 1 produced by src(i), i < n; keys
// are distinct and 1 <= rank <= their number. With max_iters rounds only, returns
// a key <= the answer (the lower end of the range reached).
template <class Src>
__device__ unsigned long long block_select(const Src& src, uint32_t n, uint32_t rank, TopkCtl& sh,
                                           int max_iters = 64) {
  const int tid = threadIdx.x, lane = tid & 31;
  unsigned long long lo = 1, hi = ~0ull;
  uint32_t krem = rank;
  for (int iter = 0; iter < max_iters; ++iter) {
    unsigned long long mn = ~0ull, mx = 0;
    for (uint32_t i = tid; i < n; i += kTopkThreads) {
      const unsigned long long x = src(i);
      if (x >= lo && x <= hi) {
        mn = x < mn ? x : mn;
        mx = x > mx ? x : mx;
      }
    }
    block_minmax(mn, mx, sh);
    if (mn >= mx) return mx == 0 ? lo : mx;  // one key left (none: defensive)
    const unsigned long long d = mx - mn;
    const int bits = 64 - __clzll((long long)d);
    const int shift = bits > kSelBits ? bits - kSelBits : 0;
    const uint32_t nb = (uint32_t)(d >> shift) + 1u;
    for (uint32_t j = tid; j < nb; j += kTopkThreads) sh.hist[j] = 0;
    if (tid == 0) sh.nsmall = 0;
    __syncthreads();
    for (uint32_t i = tid; i < n; i += kTopkThreads) {
      const unsigned long long x = src(i);
      if (x >= mn && x <= mx) atomicAdd(&sh.hist[(uint32_t)((x - mn) >> shift)], 1u);
    }
    __syncthreads();
    // thread t owns bins nb-1-P*t .. nb-P*(t+1), scanned from the top
    constexpr int P = kSelBins / kTopkThreads;
    const int btop = (int)nb - 1 - P * tid;
    uint32_t own = 0;
#pragma unroll
    for (int j = 0; j < P; ++j) own += btop - j >= 0 ? sh.hist[btop - j] : 0u;
    uint32_t tot;
    const uint32_t above = block_excl_scan(own, sh, &tot);
    if (above < krem && above + own >= krem) {
      uint32_t acc = above;
#pragma unroll
      for (int j = 0; j < P; ++j) {
        const uint32_t h = btop - j >= 0 ? sh.hist[btop - j] : 0u;
        if (acc < krem && acc + h >= krem) {
          sh.bc_u32[0] = (uint32_t)(btop - j);
          sh.bc_u32[1] = acc;
          sh.bc_u32[2] = h;
        }
        acc += h;
      }
    }
    __syncthreads();
    const uint32_t bin = sh.bc_u32[0], in_bin = sh.bc_u32[2];
    krem -= sh.bc_u32[1];
    lo = mn + ((unsigned long long)bin << shift);
    const unsigned long long span = (1ull << shift) - 1ull;
    hi = (mx - lo) < span ? mx : lo + span;
    if (in_bin <= 32) {  // finish by ranking the bin's keys in one warp
      for (uint32_t i = tid; i < n; i += kTopkThreads) {
        const unsigned long long x = src(i);
        if (x >= lo && x <= hi) sh.small[atomicAdd(&sh.nsmall, 1u)] = x;
      }
      __syncthreads();
      if (tid < 32) {
        const unsigned long long mine = lane < (int)in_bin ? sh.small[lane] : 0ull;
        uint32_t greater = 0;
        for (uint32_t j = 0; j < in_bin; ++j) greater += sh.small[j] > mine;
        if (lane < (int)in_bin && greater + 1 == krem) sh.bc_a = mine;
      }
      __syncthreads();
      const unsigned long long r = sh.bc_a;
      __syncthreads();
      return r;
    }
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

// Bit j of the result: slot base+j (< end) is valid and its key is >= (hi:lo).
// The 32 slots are read as 8 independent 16-byte loads when vec (base % 4 == 0).
__device__ __forceinline__ uint32_t topk_word_mask(const float* row, const int32_t* crow, uint32_t base,
                                                   uint32_t end, uint32_t khi, uint32_t klo, bool vec) {
  float sc[32];
  int32_t cv[32];
  if (vec && base + 32 <= end) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(row + base) + q);
      sc[4 * q] = v.x; sc[4 * q + 1] = v.y; sc[4 * q + 2] = v.z; sc[4 * q + 3] = v.w;
    }
    if (crow) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int4 c = __ldg(reinterpret_cast<const int4*>(crow + base) + q);
        cv[4 * q] = c.x; cv[4 * q + 1] = c.y; cv[4 * q + 2] = c.z; cv[4 * q + 3] = c.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) cv[j] = 0;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const bool in = base + j < end;
      sc[j] = in ? __ldg(row + base + j) : 0.f;
      cv[j] = in ? (crow ? __ldg(crow + base + j) : 0) : -1;
    }
  }
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t kh = float_order_key(sc[j]);
    const bool take = cv[j] >= 0 && (kh > khi || (kh == khi && 0xFFFFFFFFu - (base + j) >= klo));
    m |= (take ? 1u : 0u) << j;
  }
  return m;
}

// 16 slots of one filter round: t0 + 4*(tid + q*threads) + u (q, u < 4), read as
// four independent 16-byte loads; bit j of vmask: slot j valid.
struct TopkRound {
  float sc[16];
  uint32_t vmask;
};

__device__ __forceinline__ void topk_load_round(TopkRound& R, const float* row, const int32_t* crow, uint32_t t0,
                                                uint32_t hi_slot, bool vec) {
  R.vmask = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t i0 = t0 + 4 * (threadIdx.x + q * kTopkThreads);
    if (vec && i0 + 3 < hi_slot) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(row + i0));
      R.sc[4 * q] = v.x; R.sc[4 * q + 1] = v.y; R.sc[4 * q + 2] = v.z; R.sc[4 * q + 3] = v.w;
      if (crow) {
        const int4 cc = __ldg(reinterpret_cast<const int4*>(crow + i0));
        R.vmask |= ((cc.x >= 0) | (cc.y >= 0) << 1 | (cc.z >= 0) << 2 | (uint32_t)(cc.w >= 0) << 3) << (4 * q);
      } else {
        R.vmask |= 0xFu << (4 * q);
      }
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool in = i0 + u < hi_slot;
        R.sc[4 * q + u] = in ? __ldg(row + i0 + u) : 0.f;
        const bool ok = in && (!crow || __ldg(crow + i0 + u) >= 0);
        R.vmask |= (ok ? 1u : 0u) << (4 * q + u);
      }
    }
  }
}

__device__ __forceinline__ uint32_t topk_round_pass(const TopkRound& R, uint32_t t0, uint32_t thi, uint32_t tlo) {
  uint32_t pm = 0;
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const uint32_t slot = t0 + 4 * (threadIdx.x + (u >> 2) * kTopkThreads) + (u & 3);
    const uint32_t kh = float_order_key(R.sc[u]);
    const bool p = (kh > thi || (kh == thi && 0xFFFFFFFFu - slot >= tlo));
    pm |= (p ? 1u : 0u) << u;
  }
  return pm & R.vmask;
}

// Append this thread's passing keys of a round at dst[*counter ...] (one atomic per warp).
__device__ __forceinline__ void topk_round_emit(const TopkRound& R, uint32_t t0, uint32_t pm,
                                                unsigned long long* dst, uint32_t* counter, uint32_t limit) {
  const int lane = threadIdx.x & 31;
  const uint32_t cnt = __popc(pm);
  uint32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
  uint32_t base = 0;
  if (lane == 31 && wtot) base = atomicAdd(counter, wtot);
  base = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    if ((pm >> u) & 1u) {
      const uint32_t slot = t0 + 4 * (threadIdx.x + (u >> 2) * kTopkThreads) + (u & 3);
      if (base < limit) dst[base] = topk_key(R.sc[u], slot);
      ++base;
    }
  }
}

// All keys of [lo_slot, hi_slot) >= (thi:tlo) appended at dst via counter; the
// next round's loads are in flight while a round is tested.
__device__ __forceinline__ void topk_filter(const float* row, const int32_t* crow, uint32_t lo_slot,
                                            uint32_t hi_slot, bool vec, uint32_t thi, uint32_t tlo,
                                            unsigned long long* dst, uint32_t* counter, uint32_t limit) {
  if (lo_slot >= hi_slot) return;
  TopkRound cur, nxt;
  topk_load_round(cur, row, crow, lo_slot, hi_slot, vec);
  for (uint32_t t0 = lo_slot; t0 < hi_slot; t0 += 16 * kTopkThreads) {
    const bool more = t0 + 16 * kTopkThreads < hi_slot;
    if (more) topk_load_round(nxt, row, crow, t0 + 16 * kTopkThreads, hi_slot, vec);
    const uint32_t pm = topk_round_pass(cur, t0, thi, tlo);
    if (__any_sync(0xffffffffu, pm != 0)) topk_round_emit(cur, t0, pm, dst, counter, limit);
    if (more) cur = nxt;
  }
}

// Lower bound of the rank-th largest of the nonzero keys src(i), i < n: the
// smallest key whose 12-bit prefix is that of the rank-th largest (one histogram
// of prefixes, one scan from the top). 1 <= rank <= number of nonzero keys.
template <class Src>
__device__ unsigned long long block_prefix_bound(const Src& src, uint32_t n, uint32_t rank, TopkCtl& sh) {
  const int tid = threadIdx.x;
  for (int j = tid; j < kPrefixBins; j += kTopkThreads) sh.hist[j] = 0;
  __syncthreads();
  for (uint32_t i = tid; i < n; i += kTopkThreads) {
    const unsigned long long x = src(i);
    if (x) atomicAdd(&sh.hist[(uint32_t)(x >> 52)], 1u);
  }
  __syncthreads();
  constexpr int P = kPrefixBins / kTopkThreads;
  const int btop = kPrefixBins - 1 - P * tid;
  uint32_t own = 0;
#pragma unroll
  for (int j = 0; j < P; ++j) own += sh.hist[btop - j];
  uint32_t tot;
  const uint32_t above = block_excl_scan(own, sh, &tot);
  if (above < rank && above + own >= rank) {
    uint32_t acc = above;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      const uint32_t h = sh.hist[btop - j];
      if (acc < rank && acc + h >= rank) sh.bc_u32[0] = (uint32_t)(btop - j);
      acc += h;
    }
  }
  __syncthreads();
  const unsigned long long r = (unsigned long long)sh.bc_u32[0] << 52;
  __syncthreads();
  return r < 1ull ? 1ull : r;
}

// Block 0, rows of at most kBitmapSlots slots: mark the slots of the keys >= K
// among buf[0..c) in a bitmap, then write them in slot order (one block scan over
// the words), padded with -1 up to k.
__device__ void topk_emit_bitmap(const unsigned long long* buf, uint32_t c, unsigned long long K, uint32_t n,
                                 int k, const int32_t* crow, int32_t* orow, uint32_t* bits, TopkCtl& sh) {
  const int tid = threadIdx.x;
  const uint32_t nw = (n + 31) / 32;
  for (uint32_t j = tid; j < nw; j += kTopkThreads) bits[j] = 0;
  __syncthreads();
  for (uint32_t j = tid; j < c; j += kTopkThreads) {
    const unsigned long long x = buf[j];
    if (x >= K) {
      const uint32_t slot = 0xFFFFFFFFu - (uint32_t)x;
      atomicOr(bits + (slot >> 5), 1u << (slot & 31));
    }
  }
  __syncthreads();
  const uint32_t wpt = (nw + kTopkThreads - 1) / kTopkThreads;
  const uint32_t w0 = tid * wpt < nw ? tid * wpt : nw, w1 = w0 + wpt < nw ? w0 + wpt : nw;
  uint32_t mine = 0;
  for (uint32_t w = w0; w < w1; ++w) mine += __popc(bits[w]);
  uint32_t total;
  uint32_t at = block_excl_scan(mine, sh, &total);
  for (uint32_t w = w0; w < w1 && at < (uint32_t)k; ++w) {
    uint32_t m = bits[w];
    while (m && at < (uint32_t)k) {
      const uint32_t slot = 32 * w + (__ffs(m) - 1);
      m &= m - 1;
      orow[at++] = crow ? __ldg(crow + slot) : (int32_t)slot;
    }
  }
  for (uint32_t j = total + tid; j < (uint32_t)k; j += kTopkThreads) orow[j] = -1;
}

// Block 0: write the slots of the keys >= K among buf[0..c) (all when K is 0) in
// ascending slot order as positions, padded with -1 up to k (in-place ordered
// compaction, then a bitonic sort).
__device__ void topk_emit_sorted(unsigned long long* buf, uint32_t c, unsigned long long K, int k,
                                 const int32_t* crow, int32_t* orow, TopkCtl& sh) {
  const int tid = threadIdx.x;
  uint32_t* slots = reinterpret_cast<uint32_t*>(buf);
  uint32_t written = 0;
  for (uint32_t t0 = 0; t0 < c; t0 += kTopkThreads) {
    const uint32_t i = t0 + tid;
    const unsigned long long key = i < c ? buf[i] : 0ull;
    const bool take = i < c && key >= K;
    uint32_t tot;
    const uint32_t rr = block_excl_scan(take ? 1u : 0u, sh, &tot);  // every read of the chunk comes first;
    if (take) slots[written + rr] = 0xFFFFFFFFu - (uint32_t)key;     // the writes stay below the chunk
    written += tot;
    __syncthreads();
  }
  uint32_t kp = 1;
  while (kp < written) kp <<= 1;
  for (uint32_t j = written + tid; j < kp; j += kTopkThreads) slots[j] = 0xFFFFFFFFu;
  __syncthreads();
  for (uint32_t size = 2; size <= kp; size <<= 1) {
    for (uint32_t half = size >> 1; half > 0; half >>= 1) {
      for (uint32_t i = tid; i < kp / 2; i += kTopkThreads) {
        const uint32_t lo_i = 2 * half * (i / half) + (i % half), hi_i = lo_i + half;
        const uint32_t x = slots[lo_i], y = slots[hi_i];
        if ((x > y) == ((lo_i & size) == 0)) {
          slots[lo_i] = y;
          slots[hi_i] = x;
        }
      }
      __syncthreads();
    }
  }
  for (uint32_t j = tid; j < (uint32_t)k; j += kTopkThreads) {
    int32_t pos = -1;
    if (j < written) pos = crow ? __ldg(crow + slots[j]) : (int32_t)slots[j];
    orow[j] = pos;
  }
}

// Block 0 alone, exact over the whole row: K, then the keys >= K by an ordered
// compaction over the row.
__device__ void topk_whole_row(const RowSrc& rsrc, uint32_t n, int k, int32_t* orow, TopkCtl& sh) {
  const int tid = threadIdx.x;
  uint32_t m = 0;
  for (uint32_t i = tid; i < n; i += kTopkThreads) m += rsrc(i) != 0ull;
  m = block_sum(m, sh);
  const unsigned long long K = m <= (uint32_t)k ? 1ull : block_select(rsrc, n, (uint32_t)k, sh);
  uint32_t written = 0;
  for (uint32_t t0 = 0; t0 < n && written < (uint32_t)k; t0 += kTopkThreads) {
    const uint32_t i = t0 + tid;
    const unsigned long long key = i < n ? rsrc(i) : 0ull;
    const bool take = key != 0ull && key >= K;
    uint32_t tot;
    const uint32_t rr = block_excl_scan(take ? 1u : 0u, sh, &tot);
    if (take && written + rr < (uint32_t)k) orow[written + rr] = rsrc.crow ? __ldg(rsrc.crow + i) : (int32_t)i;
    written += tot;
  }
  for (uint32_t j = written + tid; j < (uint32_t)k; j += kTopkThreads) orow[j] = -1;
}

__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkThreads)
k_topk(const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ nvec,
       const int32_t* __restrict__ cand, int k, int32_t* __restrict__ out) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkCtl& sh = *reinterpret_cast<TopkCtl*>(smem_raw);
  unsigned long long* gbuf = reinterpret_cast<unsigned long long*>(smem_raw + sizeof(TopkCtl));
  const uint32_t CAP = topk_cap(k), LCAP = topk_local_cap(k);
  unsigned long long* lbuf = gbuf + CAP;
  uint32_t* bits = reinterpret_cast<uint32_t*>(lbuf + LCAP);  // small k, block 0: slot bitmap
  const uint32_t rank = cluster.block_rank();
  TopkCtl& sh0 = *cluster.map_shared_rank(&sh, 0);
  unsigned long long* gbuf0 = cluster.map_shared_rank(gbuf, 0);

  const int b = blockIdx.y, tid = threadIdx.x;
  int64_t n64 = nvec ? (int64_t)__ldg(nvec + b) : stride;
  n64 = n64 < 0 ? 0 : (n64 > stride ? stride : n64);
  const uint32_t n = (uint32_t)n64;
  const float* row = scores + (size_t)b * stride;
  const int32_t* crow = cand ? cand + (size_t)b * stride : nullptr;
  int32_t* orow = out + (size_t)b * k;
  const RowSrc rsrc{row, crow};
  const bool vec = (((uintptr_t)row | (uintptr_t)crow) & 15u) == 0;
  // slice of this block: boundaries rounded up to multiples of 4 (16-byte loads)
  auto slice_start = [n](uint32_t r) -> uint32_t {
    const uint32_t x = (uint32_t)(((unsigned long long)n * r / kTopkCluster + 3) & ~3ull);
    return x < n ? x : n;
  };
  const uint32_t lo_slot = slice_start(rank);
  const uint32_t hi_slot = rank + 1 == kTopkCluster ? n : slice_start(rank + 1);
  const uint32_t slen = hi_slot - lo_slot;
  const unsigned long long T = ((unsigned long long)k + CAP) / 2;  // candidates wanted per row

  if (tid == 0) {
    sh.lcount = 0;
    if (rank == 0) {
      sh.count = 0;
      sh.valid = 0;
    }
  }
  cluster.sync();

  if (LCAP > 0) {
    // ================= small k: local thresholds, block 0 finishes alone
    // A. tau_r: about T/clusters keys of this slice are expected >= tau_r (T = 3k)
    const uint32_t S0 = topk_samples(k);  // a power of two
    const uint32_t S = slen < S0 ? slen : S0;
    uint32_t sv = 0;
    for (uint32_t s = tid; s < S; s += kTopkThreads) {
      const uint32_t i = lo_slot + (S == slen ? s : (uint32_t)(((unsigned long long)s * slen) >> (__ffs(S0) - 1)));
      const unsigned long long key = rsrc(i);
      lbuf[s] = key;
      sv += key != 0ull;
    }
    sv = block_sum(sv, sh);
    unsigned long long tau = 1ull;
    uint32_t mr = slen;  // valid slots of the slice, estimated from the sample for candidate lists
    if (crow && S > 0) mr = (uint32_t)(((unsigned long long)sv * slen + S - 1) / S);
    const unsigned long long Tr = (3ull * (unsigned long long)k + kTopkCluster - 1) / kTopkCluster;
    if (sv > 0 && mr > Tr) {
      unsigned long long r = (Tr * sv + mr - 1) / mr;
      r = r < 1 ? 1 : (r > sv ? sv : r);
      tau = block_prefix_bound(BufSrc{lbuf}, S, (uint32_t)r, sh);
    }
    // B. keys >= tau_r into the local buffer, then block 0's buffer
    topk_filter(row, crow, lo_slot, hi_slot, vec, (uint32_t)(tau >> 32), (uint32_t)tau, lbuf, &sh.lcount, LCAP);
    __syncthreads();
    const uint32_t cr = sh.lcount;
    if (tid == 0) {
      sh.bc_u32[3] = atomicAdd(&sh0.count, cr);
      sh0.tau_of[rank] = tau;
      sh0.over_of[rank] = cr > LCAP ? 1u : 0u;
    }
    __syncthreads();
    const uint32_t off = sh.bc_u32[3];
    if (cr <= LCAP && off + cr <= CAP)
      for (uint32_t j = tid; j < cr; j += kTopkThreads) gbuf0[off + j] = lbuf[j];
    cluster.sync();  // the last cluster barrier: only block 0 goes on
    if (rank != 0) return;
    // C. block 0: the candidates hold every key >= K when K >= max tau_r
    const uint32_t c = sh.count;
    unsigned long long taumax = 0ull;
    uint32_t bad = 0;
    for (int r = 0; r < kTopkCluster; ++r) {
      taumax = sh.tau_of[r] > taumax ? sh.tau_of[r] : taumax;
      bad |= sh.over_of[r];
    }
    if (!bad && c <= CAP) {
      if (c >= (uint32_t)k) {
        const unsigned long long K = block_select(BufSrc{gbuf}, c, (uint32_t)k, sh);
        if (K >= taumax) {
          if (n <= kBitmapSlots) topk_emit_bitmap(gbuf, c, K, n, k, crow, orow, bits, sh);
          else topk_emit_sorted(gbuf, c, K, k, crow, orow, sh);
          return;
        }
      } else if (taumax == 1ull) {  // every valid slot passed: fewer than k valid
        if (n <= kBitmapSlots) topk_emit_bitmap(gbuf, c, 1ull, n, k, crow, orow, bits, sh);
        else topk_emit_sorted(gbuf, c, 0ull, k, crow, orow, sh);
        return;
      }
    }
    topk_whole_row(rsrc, n, k, orow, sh);
    return;
  }

  // ================= large k: one threshold for the row, output by every block
  // valid slots of the row (a candidate list may hold -1)
  uint32_t m = n;
  if (crow) {
    uint32_t c = 0;
    for (uint32_t i = lo_slot + tid; i < hi_slot; i += kTopkThreads) c += __ldg(crow + i) >= 0;
    c = block_sum(c, sh);
    if (tid == 0 && c) atomicAdd(&sh0.valid, c);
  }
  // A. samples into block 0, tau
  const uint32_t S0 = topk_samples(k);
  const uint32_t S = n < S0 ? n : S0;
  for (uint32_t s = rank * kTopkThreads + tid; s < S; s += kTopkCluster * kTopkThreads) {
    const uint32_t i = S == n ? s : (uint32_t)(((unsigned long long)s * n) / S);
    gbuf0[s] = rsrc(i);
  }
  cluster.sync();
  if (crow) m = sh0.valid;
  if (rank == 0) {
    unsigned long long tau = 1ull;  // every valid key
    if (m > (uint32_t)k) {
      uint32_t sv = 0;
      for (uint32_t s = tid; s < S; s += kTopkThreads) sv += gbuf[s] != 0ull;
      sv = block_sum(sv, sh);
      if (sv > 0) {
        unsigned long long r = (T * sv + m - 1) / m;
        r = r < 1 ? 1 : (r > sv ? sv : r);
        tau = block_select(BufSrc{gbuf}, S, (uint32_t)r, sh, 2);
      }
    }
    if (tid == 0) sh.tau = tau;
  }
  cluster.sync();
  {
    // B. count, reserve, write
    const unsigned long long tau = sh0.tau;
    const uint32_t thi = (uint32_t)(tau >> 32), tlo = (uint32_t)tau;
    uint32_t mine = 0;
    for (uint32_t t0 = lo_slot; t0 < hi_slot; t0 += 16 * kTopkThreads) {
      TopkRound R;
      topk_load_round(R, row, crow, t0, hi_slot, vec);
      mine += __popc(topk_round_pass(R, t0, thi, tlo));
    }
    mine = block_sum(mine, sh);
    if (tid == 0) sh.bc_u32[3] = atomicAdd(&sh0.count, mine);
    __syncthreads();
    const uint32_t off = sh.bc_u32[3];
    if (off + mine <= CAP) topk_filter(row, crow, lo_slot, hi_slot, vec, thi, tlo, gbuf0 + off, &sh.lcount, mine);
  }
  cluster.sync();
  // C. K (block 0)
  if (rank == 0) {
    const uint32_t c = sh.count;
    unsigned long long K = 1ull;
    if (m > (uint32_t)k)
      K = (c >= (uint32_t)k && c <= CAP) ? block_select(BufSrc{gbuf}, c, (uint32_t)k, sh)
                                         : block_select(rsrc, n, (uint32_t)k, sh);
    if (tid == 0) sh.K = K;
  }
  cluster.sync();
  // D. ordered output: thread t owns a contiguous run of 32-slot words of the slice
  const unsigned long long K = sh0.K;
  const uint32_t khi = (uint32_t)(K >> 32), klo = (uint32_t)K;
  const uint32_t nwords = (slen + 31) / 32;
  const uint32_t wpt = (nwords + kTopkThreads - 1) / kTopkThreads;
  const uint32_t w0 = tid * wpt < nwords ? tid * wpt : nwords;
  const uint32_t w1 = w0 + wpt < nwords ? w0 + wpt : nwords;
  uint32_t mine = 0;
  for (uint32_t w = w0; w < w1; ++w)
    mine += __popc(topk_word_mask(row, crow, lo_slot + 32 * w, hi_slot, khi, klo, vec));
  uint32_t block_tot;
  const uint32_t before_me = block_excl_scan(mine, sh, &block_tot);
  if (tid == 0) sh0.sel[rank] = block_tot;
  cluster.sync();
  uint32_t offset = 0, total = 0;
  for (uint32_t r = 0; r < kTopkCluster; ++r) {
    const uint32_t v = sh0.sel[r];
    offset += r < rank ? v : 0u;
    total += v;
  }
  cluster.sync();  // no block touches another block's shared memory after this point
  if (mine) {
    uint32_t at = offset + before_me;
    for (uint32_t w = w0; w < w1 && at < (uint32_t)k; ++w) {
      const uint32_t base = lo_slot + 32 * w;
      uint32_t msk = topk_word_mask(row, crow, base, hi_slot, khi, klo, vec);
      while (msk && at < (uint32_t)k) {
        const uint32_t j = __ffs(msk) - 1;
        msk &= msk - 1;
        orow[at++] = crow ? __ldg(crow + base + j) : (int32_t)(base + j);
      }
    }
  }
  if (rank + 1 == kTopkCluster)
    for (uint32_t j = total + tid; j < (uint32_t)k; j += kTopkThreads) orow[j] = -1;
}

}  // namespace csa2
