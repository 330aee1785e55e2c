// topk_select: exact Top-k per row, ties to the lower position, output ascending.
//
// Pages: "890 octets de cache KV par token", section "L'architecture",
// "Deuxiemement" (each Full layer selects new Top-512 indices; the hierarchical
// indexer keeps 16,384 candidate positions).
//
// Order: slot i of a row has the 32-bit key order(score_i) (a float order that
// puts every float, -0 = +0, in the order of its value). A larger key wins; among
// equal keys the lower slot wins. Slots past the row's length, and candidate
// slots holding -1, are invalid and never selected.
//
// One cluster of CLUSTER blocks of THREADS threads per row (the shape is a template
// parameter; the launcher picks it by row length); block r owns slice r of the row
// and each of its threads a contiguous run of the slice. Radix select over the
// cluster:
//  0. every block reads its slice once (kept as keys in shared memory when the
//     slice has at most kRxSliceCap = 36 x THREADS slots, else re-read from global
//     memory by each pass: coalesced 16-byte chunks for the passes whose order does
//     not matter, rounds of four consecutive chunks a thread for the ordered ones)
//     and publishes its valid count and key range to every block;
//  1. if the row has at most k valid slots they are all selected. Otherwise:
//  1a. a bound first: every thread also keeps the largest key it read, and block r
//     finds lb_r, the lower edge of the bin (one fitted histogram level over its
//     thread maxima) where m = ceil(k / 8) maxima are reached from the top. The
//     maxima are keys of distinct slots, so at least 8 m >= k keys of the row are at
//     or above L = min_r lb_r (lb_r travels with the count and key range). Each
//     block writes its keys >= L, in slot order, into its own region of block 0's
//     list (kRxListCap / 8 entries; about 75 each for k = 512 over 131,072 i.i.d.
//     scores) and its count to every block. After that one barrier, if every region
//     held its keys, block 0's first four warps line the regions up and finish
//     (rx_finish_small): the k-th key from one fitted histogram of the list and a
//     rank inside its bin, then the list walked in slot order gives the output.
//     Otherwise (heavy ties, say) the levels below run instead;
//  1b. per level: each block histograms the keys of the current range [lo, hi] into
//     kRxBins bins of width 2^shift (the smallest width that covers the range, so
//     the bins follow the occupied keys); block r sums bins [256 r, 256 r + 256)
//     over the cluster (distributed shared memory) and publishes the segment
//     total; every block then finds the segment, and inside it the bin, where the
//     count from the top reaches the wanted rank. That bin is the next range; the
//     search ends at a bin of one key T (or early, at a bin taken whole);
//     as soon as the keys at or above the chosen bin number at most kRxListCap
//     (usually after the first level), every block appends those keys, in slot
//     order, to block 0's list (one remote atomic reserves its run) and block 0
//     finishes alone: block-local histogram levels over the list give T, and the
//     list walked in block order gives the ordered output;
//  2. otherwise the selection is every key > T plus the first (k - count(key > T)) slots
//     with key T; each block counts its part (one block scan), publishes it, and
//     writes its selected slots in slot order at the offset the earlier blocks'
//     counts give (an ordered compaction, so no sort). The last block pads -1.
// Every cluster barrier is reached by every thread of every block, and no block
// touches another block's shared memory after the last one.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace csa2 {

constexpr int kRxBins = 2048;                          // bins per level
constexpr uint32_t kRxRunCap = 36;                     // slots per thread kept in shared memory
constexpr uint32_t kRxListCap = 2048;                  // keys block 0 finishes alone
static_assert(kRxRunCap % 4 == 0 && kRxRunCap < 64, "runs of whole chunks; valid bits in one 64-bit word");

// Control block of one cluster shape: THREADS threads per block, CLUSTER blocks per
// row. The shape's constants live here so every helper that takes the control block
// knows them.
template <int THREADS, int CLUSTER>
struct alignas(16) TopkCtl {
  static constexpr int kThreads = THREADS;
  static constexpr int kWarps = THREADS / 32;
  static constexpr int kCluster = CLUSTER;
  static constexpr int kSegBins = kRxBins / CLUSTER;            // bins summed by each block
  static constexpr uint32_t kSliceCap = kRxRunCap * THREADS;    // slots a block keeps
  static_assert(kSegBins <= THREADS, "one thread per segment bin");

  uint32_t hist[2][kRxBins];          // this block's histogram; levels alternate
  uint32_t seg[2][CLUSTER];           // segment totals of the cluster histogram, by block
  uint32_t cnt[CLUSTER];              // valid slots, by block
  uint32_t kmin[CLUSTER], kmax[CLUSTER];  // key range of the valid slots, by block
  uint32_t gt[CLUSTER], eq[CLUSTER];      // selected counts (key > T, key == T), by block
  uint32_t lb[CLUSTER], lbok[CLUSTER];    // bound of each block's thread maxima, and whether it holds
  uint32_t lcnt[CLUSTER];                 // keys at or above the row bound, by block
  uint32_t fcnt[3][4];                    // block 0's finish: per-warp partials (scan; two bits in flight)
  uint32_t fsum[4];                       // block 0's finish: per-warp totals of the output scan
  unsigned long long warp_u64[THREADS / 32];
  uint32_t warp_u32[THREADS / 32];
  uint32_t warp_a[THREADS / 32], warp_b[THREADS / 32];
  uint32_t warp_c[THREADS / 32], warp_d[THREADS / 32], warp_e[THREADS / 32];
  uint32_t bc[4];
  // block 0 only, written by every block: the gathered list
  uint32_t list_n;                        // entries reserved
  uint32_t seg_off[CLUSTER], seg_cnt[CLUSTER];  // block r's run of the list
};

// Shared memory of a shape: the control block, the kept keys (kSliceCap), their
// valid bits (one 64-bit word per thread) and block 0's gathered list (keys, slots):
// 109 KB for 512 threads (two blocks per SM), 186 KB for 1,024 (one).
template <int THREADS, int CLUSTER>
constexpr size_t topk_smem() {
  static_assert(sizeof(TopkCtl<THREADS, CLUSTER>) % 16 == 0,
                "the kept keys after the control block are read 16 bytes at a time");
  return sizeof(TopkCtl<THREADS, CLUSTER>) + 4u * kRxRunCap * THREADS + 8u * THREADS + 8u * kRxListCap;
}

// Kept keys: chunk j (4 keys) of thread t's run. The XOR keeps both the run
// owner's 16-byte reads (fixed j) and the coalesced filing (8 consecutive chunks
// of a run per 8 lanes) free of bank conflicts.
template <int THREADS>
__device__ __forceinline__ uint32_t rx_kidx(uint32_t j, uint32_t t) { return j * THREADS + (t ^ j); }

// The shape's constants under the names the code below uses.
#define CSA2_TOPK_SHAPE(Ctl)                                   \
  constexpr int kTopkThreads = Ctl::kThreads;                  \
  constexpr int kTopkWarps = Ctl::kWarps;                      \
  constexpr int kTopkCluster = Ctl::kCluster;                  \
  constexpr int kRxSegBins = Ctl::kSegBins;                    \
  constexpr uint32_t kRxSliceCap = Ctl::kSliceCap;             \
  (void)kTopkThreads; (void)kTopkWarps; (void)kTopkCluster; (void)kRxSegBins; (void)kRxSliceCap

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory"); }

// Exclusive scan over the block of one value per thread; *total gets the sum.
template <class Ctl>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, Ctl& sh, uint32_t* total) {
  CSA2_TOPK_SHAPE(Ctl);
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

// The same for 64-bit values (two 32-bit counts packed high:low).
template <class Ctl>
__device__ __forceinline__ unsigned long long block_excl_scan64(unsigned long long v, Ctl& sh,
                                                                unsigned long long* total) {
  CSA2_TOPK_SHAPE(Ctl);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh.warp_u64[wid] = x;
  __syncthreads();
  unsigned long long before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kTopkWarps; ++w) {
    const unsigned long long s = sh.warp_u64[w];
    before += w < wid ? s : 0ull;
    tot += s;
  }
  *total = tot;
  __syncthreads();
  return before + x - v;
}

// Block-wide sums of c and cv, and min / max of the keys (mn, mx) and of the
// thread maxima (tmn, tmx); every thread gets all six.
template <class Ctl>
__device__ __forceinline__ void block_load_stats(uint32_t& c, uint32_t& mn, uint32_t& mx, uint32_t& cv,
                                                 uint32_t& tmn, uint32_t& tmx, Ctl& sh) {
  CSA2_TOPK_SHAPE(Ctl);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    c += __shfl_xor_sync(0xffffffffu, c, o);
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    cv += __shfl_xor_sync(0xffffffffu, cv, o);
    tmn = min(tmn, __shfl_xor_sync(0xffffffffu, tmn, o));
    tmx = max(tmx, __shfl_xor_sync(0xffffffffu, tmx, o));
  }
  if (lane == 0) {
    sh.warp_u32[wid] = c;
    sh.warp_a[wid] = mn;
    sh.warp_b[wid] = mx;
    sh.warp_c[wid] = cv;
    sh.warp_d[wid] = tmn;
    sh.warp_e[wid] = tmx;
  }
  __syncthreads();
  c = 0;
  mn = 0xFFFFFFFFu;
  mx = 0;
  cv = 0;
  tmn = 0xFFFFFFFFu;
  tmx = 0;
#pragma unroll
  for (int w = 0; w < kTopkWarps; ++w) {
    c += sh.warp_u32[w];
    mn = min(mn, sh.warp_a[w]);
    mx = max(mx, sh.warp_b[w]);
    cv += sh.warp_c[w];
    tmn = min(tmn, sh.warp_d[w]);
    tmx = max(tmx, sh.warp_e[w]);
  }
  __syncthreads();
}

// A row as seen by one thread: its run [s_begin, s_end) of slots, read either from
// the block's kept keys (chunk j of thread t at keys4[j * threads + t], so the
// 16-byte reads of a warp are contiguous) or from global memory.
struct RxRow {
  const float* row;
  const int32_t* crow;
  uint32_t s_begin, s_end;  // this thread's run
  uint32_t lo, hi;          // the block's slice
  bool kept, vec;
};

// Scores and validity of slots s0 .. s0+3 of the thread's run (s0 < R.s_end).
__device__ __forceinline__ void rx_load4(const RxRow& R, uint32_t s0, float (&x)[4], bool (&ok)[4]) {
  if (R.vec && s0 + 4 <= R.s_end) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(R.row + s0));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
#pragma unroll
    for (int u = 0; u < 4; ++u) ok[u] = true;
  } else {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ok[u] = s0 + u < R.s_end;
      x[u] = ok[u] ? __ldg(R.row + s0 + u) : 0.f;
    }
  }
  if (R.crow) {
#pragma unroll
    for (int u = 0; u < 4; ++u) ok[u] = ok[u] && __ldg(R.crow + s0 + u) >= 0;
  }
}

// Scores and validity of slots s0 .. s0+3 below `end` (s0 < end, s0 a multiple of 4
// from the slice start).
__device__ __forceinline__ void rx_load4_to(const RxRow& R, uint32_t s0, uint32_t end, float (&x)[4],
                                            bool (&ok)[4]) {
  if (R.vec && s0 + 4 <= end) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(R.row + s0));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
#pragma unroll
    for (int u = 0; u < 4; ++u) ok[u] = true;
  } else {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ok[u] = s0 + u < end;
      x[u] = ok[u] ? __ldg(R.row + s0 + u) : 0.f;
    }
  }
  if (R.crow) {
#pragma unroll
    for (int u = 0; u < 4; ++u) ok[u] = ok[u] && __ldg(R.crow + s0 + u) >= 0;
  }
}

// f(slot, key) for every valid slot of the thread's run, in slot order.
template <int kTopkThreads, int kBatch, class F>
__device__ __forceinline__ void rx_visit(const RxRow& R, const uint4* keys4, const unsigned long long* vbits,
                                         F&& f) {
  if (R.kept) {
    const unsigned long long vb = vbits[threadIdx.x];
    const uint32_t L = R.s_end - R.s_begin;
    if ((L & 3u) == 0 && vb == (1ull << L) - 1ull) {  // whole chunks of valid slots: no per-slot test
#pragma unroll
      for (uint32_t j = 0; j < kRxRunCap / 4; ++j) {
        if (4 * j < L) {
          const uint4 k4 = keys4[rx_kidx<kTopkThreads>(j, threadIdx.x)];
          f(R.s_begin + 4 * j, k4.x);
          f(R.s_begin + 4 * j + 1, k4.y);
          f(R.s_begin + 4 * j + 2, k4.z);
          f(R.s_begin + 4 * j + 3, k4.w);
        }
      }
      return;
    }
#pragma unroll
    for (uint32_t j = 0; j < kRxRunCap / 4; ++j) {
      const uint32_t s0 = R.s_begin + 4 * j;
      if (s0 >= R.s_end) break;
      const uint4 k4 = keys4[rx_kidx<kTopkThreads>(j, threadIdx.x)];
      const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if ((vb >> (4 * j + u)) & 1ull) f(s0 + u, kk[u]);
    }
    return;
  }
  // re-read from global memory: kBatch chunks of the run in flight before any is used
  // (shapes whose rows are normally kept use 1, which keeps their registers free)
  if constexpr (kBatch == 1) {
#pragma unroll 4
    for (uint32_t s0 = R.s_begin; s0 < R.s_end; s0 += 4) {
      float x[4];
      bool ok[4];
      rx_load4(R, s0, x, ok);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (ok[u]) f(s0 + u, float_order_key(x[u]));
    }
  } else {
    for (uint32_t s0 = R.s_begin; s0 < R.s_end; s0 += 4 * kBatch) {
      float x[kBatch][4];
      bool ok[kBatch][4];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (s0 + 4 * i < R.s_end) {
          rx_load4(R, s0 + 4 * i, x[i], ok[i]);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) ok[i][u] = false;
        }
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (ok[i][u]) f(s0 + 4 * i + u, float_order_key(x[i][u]));
    }
  }
}

// f(slot, key) for every valid slot of the block's slice, in no particular order. A
// slice kept in shared memory is visited as by rx_visit; otherwise the block reads it
// in coalesced 16-byte chunks (chunk g by thread g mod threads), kBatch chunks a
// thread in flight.
template <int kTopkThreads, int kBatch, class F>
__device__ __forceinline__ void rx_visit_any(const RxRow& R, const uint4* keys4, const unsigned long long* vbits,
                                             F&& f) {
  if (R.kept) {
    rx_visit<kTopkThreads, 1>(R, keys4, vbits, f);
    return;
  }
  const uint32_t nch = (R.hi - R.lo + 3) / 4;
  for (uint32_t g0 = 0; g0 < nch; g0 += kTopkThreads * kBatch) {
    float x[kBatch][4];
    bool ok[kBatch][4];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const uint32_t g = g0 + (uint32_t)(i * kTopkThreads) + threadIdx.x;
      if (g < nch) {
        rx_load4_to(R, R.lo + 4 * g, R.hi, x[i], ok[i]);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) ok[i][u] = false;
      }
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const uint32_t s0 = R.lo + 4 * (g0 + (uint32_t)(i * kTopkThreads) + threadIdx.x);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (ok[i][u]) f(s0 + u, float_order_key(x[i][u]));
    }
  }
}

// Smallest shift with (span >> shift) < kRxBins.
__device__ __forceinline__ uint32_t rx_shift(uint32_t span) {
  if (span < (uint32_t)kRxBins) return 0;
  return (uint32_t)(32 - __clz(span)) - 11u;  // bit length of span, less 11
}

// Block 0 of the cluster, after the gather: the rank `need` (from the top) among
// the list keys in [lo, hi] (every list key above hi is selected already), by
// block-local histogram levels. Returns the tie key T in *T and how many keys
// equal to T are selected in *take_eq; or *T = bin start - 1 and *take_eq = 0 when
// a bin is taken whole.
template <class Ctl>
__device__ void rx_list_select(const uint32_t* lkey, uint32_t c, uint32_t need, uint32_t lo, uint32_t hi,
                               Ctl& sh, long long* T, uint32_t* take_eq) {
  CSA2_TOPK_SHAPE(Ctl);
  const int tid = threadIdx.x;
  constexpr int BPT = kRxBins / kTopkThreads;  // bins per thread, highest first
  for (;;) {
    const uint32_t shift = rx_shift(hi - lo);
    for (int j = tid; j < kRxBins; j += kTopkThreads) sh.hist[1][j] = 0;
    __syncthreads();
    for (uint32_t i = tid; i < c; i += kTopkThreads) {
      const uint32_t key = lkey[i];
      if (key - lo <= hi - lo) atomicAdd(&sh.hist[1][(key - lo) >> shift], 1u);
    }
    __syncthreads();
    const int btop = kRxBins - 1 - BPT * tid;
    uint32_t own = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) own += sh.hist[1][btop - j];
    uint32_t tot;
    const uint32_t above = block_excl_scan(own, sh, &tot);
    if (above < need && above + own >= need) {
      uint32_t acc = above;
#pragma unroll
      for (int j = 0; j < BPT; ++j) {
        const uint32_t h = sh.hist[1][btop - j];
        if (acc < need && acc + h >= need) {
          sh.bc[0] = (uint32_t)(btop - j);
          sh.bc[1] = acc;
          sh.bc[2] = h;
        }
        acc += h;
      }
    }
    __syncthreads();
    const uint32_t B = sh.bc[0], above_b = sh.bc[1], cnt_b = sh.bc[2];
    __syncthreads();
    const uint32_t blo = lo + (B << shift);
    if (above_b + cnt_b == need) {
      *T = (long long)blo - 1;
      *take_eq = 0;
      return;
    }
    if (shift == 0) {
      *T = (long long)blo;
      *take_eq = need - above_b;
      return;
    }
    need -= above_b;
    lo = blo;
    hi = min(hi, blo + ((1u << shift) - 1u));
  }
}

// Block 0 after a gather: the list (keys, slots) holds every key >= lo of the row in
// cl entries, block r's run at seg_off[r] (seg_cnt[r] entries, slot order); keys above
// hi are selected already, and `need` more come from [lo, hi]. Selects them
// (rx_list_select) and writes the k positions in ascending slot order.
template <class Ctl>
__device__ void rx_finish_list(const uint32_t* lkey, const uint32_t* lslot, uint32_t cl, uint32_t need,
                               uint32_t lo, uint32_t hi, Ctl& sh, int k, const int32_t* crow, int32_t* orow) {
  CSA2_TOPK_SHAPE(Ctl);
  const int tid = threadIdx.x;
  long long T;
  uint32_t teq;
  rx_list_select(lkey, cl, need, lo, hi, sh, &T, &teq);
  // ordered output: walk the list in block order (EPT entries per thread)
  uint32_t voff[kTopkCluster], poff[kTopkCluster];
  uint32_t acc = 0;
#pragma unroll
  for (int q = 0; q < kTopkCluster; ++q) {
    voff[q] = acc;
    poff[q] = sh.seg_off[q];
    acc += sh.seg_cnt[q];
  }
  constexpr uint32_t EPT = kRxListCap / kTopkThreads;
  uint32_t pk[EPT], ps[EPT];
  uint32_t gt = 0, eq = 0;
#pragma unroll
  for (uint32_t e = 0; e < EPT; ++e) {
    const uint32_t p = EPT * tid + e;  // position in block order
    pk[e] = 0;
    ps[e] = 0;
    if (p < cl) {
      uint32_t phys = p;
#pragma unroll
      for (int q = 0; q < kTopkCluster; ++q)
        if (p >= voff[q] && p < voff[q] + sh.seg_cnt[q]) phys = poff[q] + (p - voff[q]);
      pk[e] = lkey[phys];
      ps[e] = lslot[phys];
      gt += (long long)pk[e] > T;
      eq += (long long)pk[e] == T;
    }
  }
  unsigned long long tot64;
  const unsigned long long ex64 = block_excl_scan64(((unsigned long long)gt << 32) | eq, sh, &tot64);
  uint32_t eqi = (uint32_t)ex64;
  uint32_t pos = (uint32_t)(ex64 >> 32) + min(teq, eqi);
#pragma unroll
  for (uint32_t e = 0; e < EPT; ++e) {
    if (EPT * tid + e < cl) {
      bool take = (long long)pk[e] > T;
      if ((long long)pk[e] == T) take = eqi++ < teq;
      if (take && pos < (uint32_t)k) orow[pos++] = crow ? __ldg(crow + ps[e]) : (int32_t)ps[e];
    }
  }
}

// Block 0 after the bound path's gather, threads 0 .. kFinThreads - 1 only (the other
// warps have left): the list (keys, slots) holds, in slot order, every key >= lo of
// the row in n <= kRxListCap entries, all <= hi, and the `need` largest are selected.
// Thread t keeps list entries [KPT t, KPT t + KPT) in registers.
//  * the need-th largest key T: one histogram of the list over kRxBins bins fitted to
//    [lo, hi] finds the bin B where the count from the top reaches need; when B holds
//    at most 32 keys (the usual case), one warp ranks them against each other and
//    picks T; otherwise the bits of T below the bin width are found one by one (the
//    entries of B that match the bits chosen so far and have the next bit set are
//    counted: if they reach the rank still wanted the bit is 1, else 0);
//  * every key > T and the first (need - count(key > T)) entries with key T are
//    written in list order, at offsets from one scan of the counts.
constexpr int kFinThreads = 128;
constexpr int kFinWarps = kFinThreads / 32;
static_assert(kFinWarps == 4 && kRxListCap % kFinThreads == 0 && kRxListCap <= 65535, "finish shape");
static_assert(kRxBins % kFinThreads == 0, "whole bins per finishing thread");

__device__ __forceinline__ void fin_bar() { asm volatile("bar.sync 1, %0;\n" ::"n"(kFinThreads) : "memory"); }

// Exclusive scan over the kFinThreads finishing threads (slot: 4 words of shared memory).
__device__ __forceinline__ uint32_t fin_excl_scan(uint32_t v, uint32_t* slot, uint32_t* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) slot[w] = inc;
  fin_bar();
  uint32_t ex = inc - v, tot = 0;
#pragma unroll
  for (int q = 0; q < kFinWarps; ++q) {
    ex += q < w ? slot[q] : 0u;
    tot += slot[q];
  }
  *total = tot;
  return ex;
}

template <class Ctl>
__device__ void rx_finish_small(const uint32_t* lkey, const uint32_t* lslot, uint32_t n, uint32_t need, uint32_t lo,
                                uint32_t hi, Ctl& sh, int k, const int32_t* crow, int32_t* orow) {
  CSA2_TOPK_SHAPE(Ctl);
  constexpr int KPT = kRxListCap / kFinThreads;   // list entries per thread
  constexpr int BPT = kRxBins / kFinThreads;      // bins per thread, highest first
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint32_t base = KPT * tid;
  uint32_t key[KPT];
  uint32_t valid = 0;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    const bool v = base + e < n;
    key[e] = v ? lkey[base + e] : 0u;
    valid |= (v ? 1u : 0u) << e;
  }
  // ---- the bin of rank `need`
  const uint32_t shift = rx_shift(hi - lo);
  uint32_t* hist = sh.hist[1];
#pragma unroll
  for (int j = 0; j < BPT; ++j) hist[BPT * tid + j] = 0;
  fin_bar();
#pragma unroll
  for (int e = 0; e < KPT; ++e)
    if ((valid >> e) & 1u) atomicAdd(&hist[(key[e] - lo) >> shift], 1u);
  fin_bar();
  const int btop = kRxBins - 1 - BPT * tid;
  uint32_t own = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) own += hist[btop - j];
  uint32_t tot;
  const uint32_t above = fin_excl_scan(own, sh.fcnt[0], &tot);
  if (above < need && above + own >= need) {
    uint32_t acc = above;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      const uint32_t h = hist[btop - j];
      if (acc < need && acc + h >= need) {
        sh.bc[0] = (uint32_t)(btop - j);
        sh.bc[1] = acc;
        sh.bc[2] = h;
      }
      acc += h;
    }
  }
  if (tid == 0) sh.bc[3] = 0;  // keys of bin B collected so far
  fin_bar();
  const uint32_t B = sh.bc[0], above_b = sh.bc[1], cnt_b = sh.bc[2];
  const uint32_t blo = lo + (B << shift);
  const uint32_t r = need - above_b;  // rank wanted inside bin B (1-based)
  auto in_b = [&](int e) { return ((valid >> e) & 1u) && ((key[e] - lo) >> shift) == B; };
  uint32_t T;
  if (above_b + cnt_b == need) {  // bin B is taken whole
    // every key >= blo: T is the smallest key of B, and all keys equal to it are taken
    uint32_t m = 0xFFFFFFFFu;
#pragma unroll
    for (int e = 0; e < KPT; ++e)
      if (in_b(e)) m = min(m, key[e]);
    m = __reduce_min_sync(0xffffffffu, m);
    if (lane == 0) sh.fcnt[1][w] = m;
    fin_bar();
    T = min(min(sh.fcnt[1][0], sh.fcnt[1][1]), min(sh.fcnt[1][2], sh.fcnt[1][3]));
  } else if (cnt_b <= 32) {
    // collect the keys of B and rank them in one warp
    uint32_t* bk = sh.hist[0];  // (free in this path)
#pragma unroll
    for (int e = 0; e < KPT; ++e)
      if (in_b(e)) bk[atomicAdd(&sh.bc[3], 1u)] = key[e];
    fin_bar();
    if (w == 0) {
      const uint32_t mine = lane < (int)cnt_b ? bk[lane] : 0u;
      uint32_t gt = 0, ge = 0;
      for (int j = 0; j < (int)cnt_b; ++j) {
        const uint32_t o = __shfl_sync(0xffffffffu, mine, j);
        gt += o > mine ? 1u : 0u;
        ge += o >= mine ? 1u : 0u;
      }
      if (lane < (int)cnt_b && gt < r && r <= ge) sh.bc[3] = mine;  // every such lane holds the same key
    }
    fin_bar();
    T = sh.bc[3];
  } else {
    // bit by bit over the offsets key - blo (< 2^shift) of the entries of B
    uint32_t mask = 0, prefix = 0, rem = r;
    for (int bit = (int)shift - 1; bit >= 0; --bit) {
      const uint32_t m2 = mask | (1u << bit), p2 = prefix | (1u << bit);
      uint32_t c = 0;
#pragma unroll
      for (int e = 0; e < KPT; ++e) c += (in_b(e) && ((key[e] - blo) & m2) == p2) ? 1u : 0u;
      c = __reduce_add_sync(0xffffffffu, c);
      if (lane == 0) sh.fcnt[1 + (bit & 1)][w] = c;
      fin_bar();
      c = sh.fcnt[1 + (bit & 1)][0] + sh.fcnt[1 + (bit & 1)][1] + sh.fcnt[1 + (bit & 1)][2] +
          sh.fcnt[1 + (bit & 1)][3];
      if (c >= rem) prefix = p2;
      else rem -= c;
      mask = m2;
    }
    T = blo + prefix;
  }
  // ---- ordered output: (count > T) << 16 | (count == T) per thread, scanned
  uint32_t gt = 0, eq = 0;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    if ((valid >> e) & 1u) {
      gt += key[e] > T ? 1u : 0u;
      eq += key[e] == T ? 1u : 0u;
    }
  }
  uint32_t both;
  const uint32_t ex = fin_excl_scan((gt << 16) | eq, sh.fsum, &both);
  const uint32_t take_eq = need - (both >> 16);  // ties taken, in list order
  uint32_t eqi = ex & 0xFFFFu;
  uint32_t pos = (ex >> 16) + min(take_eq, eqi);
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    if ((valid >> e) & 1u) {
      bool take = key[e] > T;
      if (key[e] == T) take = eqi++ < take_eq;
      if (take && pos < (uint32_t)k) {
        const uint32_t sl = lslot[base + e];
        orow[pos++] = crow ? __ldg(crow + sl) : (int32_t)sl;
      }
    }
  }
}

template <int THREADS, int CLUSTER>
__global__ void __cluster_dims__(CLUSTER, 1, 1) __launch_bounds__(THREADS, THREADS >= 1024 ? 1 : 2)
k_topk(const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ nvec,
       const int32_t* __restrict__ cand, int k, int32_t* __restrict__ out, int discard) {
  using TopkCtlT = TopkCtl<THREADS, CLUSTER>;
  CSA2_TOPK_SHAPE(TopkCtlT);
  pdl_wait_and_release();
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkCtlT& sh = *reinterpret_cast<TopkCtlT*>(smem_raw);
  uint4* keys4 = reinterpret_cast<uint4*>(smem_raw + sizeof(TopkCtlT));
  unsigned long long* vbits = reinterpret_cast<unsigned long long*>(smem_raw + sizeof(TopkCtlT) + 4u * kRxSliceCap);
  uint32_t* lkey = reinterpret_cast<uint32_t*>(vbits + kTopkThreads);  // block 0: the gathered list (keys, then slots)
  uint32_t* lslot = lkey + kRxListCap;
  const uint32_t rank = cluster.block_rank();
  const int b = blockIdx.y, tid = threadIdx.x;

  cluster_arrive_relaxed();  // every block has started once the matching wait returns
  if (tid == 0) sh.list_n = 0;

  int64_t n64 = nvec ? (int64_t)__ldg(nvec + b) : stride;
  n64 = n64 < 0 ? 0 : (n64 > stride ? stride : n64);
  const uint32_t n = (uint32_t)n64;
  const float* row = scores + (size_t)b * stride;
  const int32_t* crow = cand ? cand + (size_t)b * stride : nullptr;
  int32_t* orow = out + (size_t)b * k;
  // slice of this block: boundaries rounded up to multiples of 4 (16-byte loads)
  auto slice_start = [n](uint32_t r) -> uint32_t {
    const uint32_t x = (uint32_t)(((unsigned long long)n * r / kTopkCluster + 3) & ~3ull);
    return x < n ? x : n;
  };
  const uint32_t lo_slot = slice_start(rank);
  const uint32_t hi_slot = rank + 1 == kTopkCluster ? n : slice_start(rank + 1);
  const uint32_t slen = hi_slot - lo_slot;
  // runs of a multiple of 4 slots per thread
  const uint32_t run = (((slen + kTopkThreads - 1) / kTopkThreads) + 3) & ~3u;
  RxRow R;
  R.row = row;
  R.crow = crow;
  R.s_begin = min(lo_slot + run * (uint32_t)tid, hi_slot);
  R.s_end = min(R.s_begin + run, hi_slot);
  R.lo = lo_slot;
  R.hi = hi_slot;
  R.vec = (((uintptr_t)row | (uintptr_t)crow) & 15u) == 0;
  R.kept = slen <= kRxSliceCap;

  // ---- 0. read the slice (kept in shared memory when it fits), count, key range;
  // every thread also keeps the largest key it read (tkey; tv: it read a valid slot)
  uint32_t c = 0, mn = 0xFFFFFFFFu, mx = 0, tkey = 0, tv = 0;
  if (R.kept && R.vec && !crow) {
    // plain scores: the block reads the slice in coalesced 16-byte chunks (chunk g
    // by thread g % threads) and files chunk g under its run owner g / cpr
    const uint32_t cpr = run / 4, nch = (slen + 3) / 4;
    float4 v[kRxRunCap / 4];
#pragma unroll
    for (uint32_t i = 0; i < kRxRunCap / 4; ++i) {
      const uint32_t g = i * kTopkThreads + tid;
      const uint32_t s0 = lo_slot + 4 * g;
      if (g < nch && s0 + 4 <= hi_slot) {
        v[i] = __ldg(reinterpret_cast<const float4*>(row + s0));
      } else if (g < nch) {  // the ragged end of the row
        v[i].x = __ldg(row + s0);
        v[i].y = s0 + 1 < hi_slot ? __ldg(row + s0 + 1) : 0.f;
        v[i].z = s0 + 2 < hi_slot ? __ldg(row + s0 + 2) : 0.f;
        v[i].w = s0 + 3 < hi_slot ? __ldg(row + s0 + 3) : 0.f;
      }
    }
#pragma unroll
    for (uint32_t i = 0; i < kRxRunCap / 4; ++i) {
      const uint32_t g = i * kTopkThreads + tid;
      if (g < nch) {
        const uint32_t s0 = lo_slot + 4 * g;
        uint32_t kk[4] = {float_order_key(v[i].x), float_order_key(v[i].y), float_order_key(v[i].z),
                          float_order_key(v[i].w)};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (s0 + u < hi_slot) {
            ++c;
            mn = min(mn, kk[u]);
            mx = max(mx, kk[u]);
            tkey = max(tkey, kk[u]);
            tv = 1;
          } else {
            kk[u] = 0u;
          }
        }
        const uint32_t t = g / cpr, jj = g - t * cpr;
        keys4[rx_kidx<kTopkThreads>(jj, t)] = make_uint4(kk[0], kk[1], kk[2], kk[3]);
      }
    }
    const uint32_t L = R.s_end - R.s_begin;  // valid slots of this thread's run
    vbits[tid] = (1ull << L) - 1ull;          // L <= kRxRunCap < 64
  } else if (R.kept) {
    unsigned long long vb = 0;
#pragma unroll
    for (uint32_t j = 0; j < kRxRunCap / 4; ++j) {
      const uint32_t s0 = R.s_begin + 4 * j;
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      bool ok[4] = {false, false, false, false};
      if (s0 < R.s_end) rx_load4(R, s0, x, ok);
      uint32_t kk[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        kk[u] = ok[u] ? float_order_key(x[u]) : 0u;
        if (ok[u]) {
          vb |= 1ull << (4 * j + u);
          ++c;
          mn = min(mn, kk[u]);
          mx = max(mx, kk[u]);
          tkey = max(tkey, kk[u]);
          tv = 1;
        }
      }
      if (s0 < R.s_end) keys4[rx_kidx<kTopkThreads>(j, tid)] = make_uint4(kk[0], kk[1], kk[2], kk[3]);
    }
    vbits[tid] = vb;
  } else {
    rx_visit_any<kTopkThreads, (kTopkCluster > 8 && kTopkThreads < 1024 ? 8 : 1)>(R, nullptr, nullptr, [&](uint32_t, uint32_t key) {
      ++c;
      mn = min(mn, key);
      mx = max(mx, key);
      tkey = max(tkey, key);
      tv = 1;
    });
  }
  for (int j = tid; j < kRxBins; j += kTopkThreads) {
    sh.hist[0][j] = 0;
    sh.hist[1][j] = 0;
  }
  uint32_t cv = tv, tmn = tv ? tkey : 0xFFFFFFFFu, tmx = tkey;
  block_load_stats(c, mn, mx, cv, tmn, tmx, sh);  // (its barriers also order the kept keys and hist[])
  if (discard && R.kept) {
    // the scores are a decode step's scratch, now held as keys: drop the slice's whole
    // 128-byte lines from L2 without writing them back (lines shared with a
    // neighbouring slice stay)
    const uintptr_t a0 = ((uintptr_t)(row + lo_slot) + 127u) & ~(uintptr_t)127u;
    const uintptr_t a1 = (uintptr_t)(row + hi_slot) & ~(uintptr_t)127u;
    for (uintptr_t ad = a0 + 128u * (uintptr_t)tid; ad < a1; ad += 128u * kTopkThreads)
      asm volatile("discard.global.L2 [%0], 128;\n" ::"l"(ad) : "memory");
  }

  // ---- 0b. a lower bound of the row's k-th key. The threads' largest keys sit in
  // distinct slots, so if every block has m = ceil(k / clusters) thread maxima at or
  // above its bound lb, at least k keys of the row are at or above the smallest lb.
  // lb: the lower edge of the bin (one fitted histogram level over the block's thread
  // maxima) where the count from the top reaches m.
  const uint32_t m_th = ((uint32_t)k + kTopkCluster - 1) / kTopkCluster;
  // (R.kept can differ between blocks; every block must hold for the bound to be used)
  const bool lb_ok = R.kept && cv >= m_th && (uint32_t)k <= kRxListCap;
  uint32_t lb = 0;
  if (lb_ok) {
    const uint32_t tshift = rx_shift(tmx - tmn);
    if (tv) atomicAdd(&sh.hist[1][(tkey - tmn) >> tshift], 1u);
    __syncthreads();
    constexpr int BPT = kRxBins / kTopkThreads;  // bins per thread, highest first
    const int btop = kRxBins - 1 - BPT * tid;
    uint32_t own = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) own += sh.hist[1][btop - j];
    uint32_t tot;
    const uint32_t above = block_excl_scan(own, sh, &tot);
    if (above < m_th && above + own >= m_th) {
      uint32_t acc = above;
#pragma unroll
      for (int j = 0; j < BPT; ++j) {
        const uint32_t h = sh.hist[1][btop - j];
        if (acc < m_th && acc + h >= m_th) sh.bc[0] = (uint32_t)(btop - j);
        acc += h;
      }
    }
    __syncthreads();
    lb = tmn + (sh.bc[0] << tshift);
    for (int j = tid; j < kRxBins; j += kTopkThreads) sh.hist[1][j] = 0;  // (levels start from zeroed bins)
  }

  cluster_wait();
  if (tid < kTopkCluster) {
    TopkCtlT& dst = *cluster.map_shared_rank(&sh, (unsigned)tid);
    dst.cnt[rank] = c;
    dst.kmin[rank] = mn;
    dst.kmax[rank] = mx;
    dst.lb[rank] = lb;
    dst.lbok[rank] = lb_ok ? 1u : 0u;
  }
  cluster.sync();
  uint32_t V = 0, klo = 0xFFFFFFFFu, khi = 0, L = 0xFFFFFFFFu;
  bool bound = true;
  for (int q = 0; q < kTopkCluster; ++q) {
    V += sh.cnt[q];
    if (sh.cnt[q]) {
      klo = min(klo, sh.kmin[q]);
      khi = max(khi, sh.kmax[q]);
    }
    bound = bound && sh.lbok[q] != 0;
    L = min(L, sh.lb[q]);
  }
  // ---- 1. the threshold: select key > Tc, and the first take_eq slots with key == Tc
  long long Tc = -1;       // every valid key is > -1
  uint32_t take_eq = 0;
  if (V > (uint32_t)k && bound) {
    // ---- 1a. every key >= L goes to block 0's list: block r writes its keys >= L, in
    // slot order, into region r of the list (kRxListCap / clusters entries) and its
    // count to every block; after one barrier every block knows whether all regions
    // held their keys. If so block 0 lines the regions up in slot order and finishes
    // alone; otherwise (heavy ties, say) the histogram levels below run instead
    constexpr uint32_t kSeg = kRxListCap / kTopkCluster;
    uint32_t own = 0;
    unsigned long long qmask = 0;  // the run's slots that qualify
    rx_visit<kTopkThreads, (kTopkCluster > 8 && kTopkThreads < 1024 ? 8 : 1)>(R, keys4, vbits, [&](uint32_t sl, uint32_t key) {
      if (key >= L) {
        ++own;
        qmask |= 1ull << (sl - R.s_begin);
      }
    });
    uint32_t cnt_r;
    uint32_t at = block_excl_scan(own, sh, &cnt_r);
    {
      uint32_t* lkey0 = cluster.map_shared_rank(lkey, 0u) + kSeg * rank;
      uint32_t* lslot0 = cluster.map_shared_rank(lslot, 0u) + kSeg * rank;
      while (qmask && at < kSeg) {
        const int bi = __ffsll((long long)qmask) - 1;
        qmask &= qmask - 1;
        lkey0[at] = reinterpret_cast<const uint32_t*>(keys4 + rx_kidx<kTopkThreads>((uint32_t)bi >> 2, tid))[bi & 3];
        lslot0[at] = R.s_begin + (uint32_t)bi;
        ++at;
      }
    }
    if (tid < kTopkCluster) cluster.map_shared_rank(&sh, (unsigned)tid)->lcnt[rank] = cnt_r;
    cluster.sync();  // counts everywhere; regions complete where they held their keys
    bool fits = true;
    for (int q = 0; q < kTopkCluster; ++q) fits = fits && sh.lcnt[q] <= kSeg;
    if (fits) {
      if (rank != 0 || tid >= kFinThreads) return;  // only block 0's first four warps go on
      // line the regions up, in block (= slot) order, over the kept keys (free now)
      uint32_t* ck = reinterpret_cast<uint32_t*>(keys4);
      uint32_t* cs = ck + kRxListCap;
      uint32_t total = 0;
      for (int q = 0; q < kTopkCluster; ++q) {
        const uint32_t cq = sh.lcnt[q];
        for (uint32_t e = tid; e < cq; e += kFinThreads) {
          ck[total + e] = lkey[kSeg * q + e];
          cs[total + e] = lslot[kSeg * q + e];
        }
        total += cq;
      }
      fin_bar();
      rx_finish_small(ck, cs, total, (uint32_t)k, L, khi, sh, k, crow, orow);
      return;  // exactly k selected: no padding
    }
    // too many keys reach the bound (heavy ties, say): the histogram levels below
  }
  if (V > (uint32_t)k) {
    uint32_t need = (uint32_t)k;  // still to select inside [klo, khi]
    for (int level = 0;; ++level) {
      const int hb = level & 1;
      const uint32_t shift = rx_shift(khi - klo);
      const uint32_t lo = klo, hi = khi;
      rx_visit_any<kTopkThreads, (kTopkCluster > 8 && kTopkThreads < 1024 ? 8 : 1)>(R, keys4, vbits, [&](uint32_t, uint32_t key) {
        if (key - lo <= hi - lo) atomicAdd(&sh.hist[hb][(key - lo) >> shift], 1u);
      });
      cluster.sync();  // every block's histogram of this level is complete
      // block r: segment r of the cluster histogram
      uint32_t v = 0;
      if (tid < kRxSegBins) {
#pragma unroll
        for (int q = 0; q < kTopkCluster; ++q)
          v += cluster.map_shared_rank(&sh.hist[hb][0], (unsigned)q)[kRxSegBins * rank + tid];
      }
      uint32_t segtot;
      block_excl_scan(v, sh, &segtot);
      if (tid < kTopkCluster) cluster.map_shared_rank(&sh, (unsigned)tid)->seg[hb][rank] = segtot;
      cluster.sync();  // segment totals everywhere
      // segment holding rank `need` counted from the top
      uint32_t above = 0;
      int sstar = 0;
      for (int s = kTopkCluster - 1; s >= 0; --s) {
        const uint32_t t = sh.seg[hb][s];
        if (above + t >= need) {
          sstar = s;
          break;
        }
        above += t;
      }
      // its bins, highest first: thread i holds bin 256 s* + 255 - i
      uint32_t cb = 0;
      const int bin = kRxSegBins * sstar + (kRxSegBins - 1 - tid);
      if (tid < kRxSegBins) {
#pragma unroll
        for (int q = 0; q < kTopkCluster; ++q) cb += cluster.map_shared_rank(&sh.hist[hb][0], (unsigned)q)[bin];
      }
      uint32_t tot;
      const uint32_t ex = block_excl_scan(cb, sh, &tot);
      if (tid < kRxSegBins && above + ex < need && above + ex + cb >= need) {
        sh.bc[0] = (uint32_t)bin;
        sh.bc[1] = above + ex;  // keys of this level's range above the bin
        sh.bc[2] = cb;
      }
      __syncthreads();
      const uint32_t B = sh.bc[0], above_b = sh.bc[1], cnt_b = sh.bc[2];
      const uint32_t blo = lo + (B << shift);
      if (above_b + cnt_b == need) {  // the bin is taken whole: every key >= blo
        Tc = (long long)blo - 1;
        take_eq = 0;
        break;
      }
      if (shift == 0) {  // a bin of one key
        Tc = (long long)blo;
        take_eq = need - above_b;
        break;
      }
      if ((uint32_t)k - need + above_b + cnt_b <= kRxListCap) {
        // ---- 1b. few keys reach the bin: gather every key >= blo into block 0,
        // which finishes alone (each block reserves its run of the list with one
        // remote atomic and writes it in slot order)
        uint32_t own = 0;
        unsigned long long qmask = 0;  // kept runs: the run's slots that qualify
        rx_visit_any<kTopkThreads, (kTopkCluster > 8 && kTopkThreads < 1024 ? 8 : 1)>(R, keys4, vbits, [&](uint32_t sl, uint32_t key) {
          if (key >= blo) {
            ++own;
            if (R.kept) qmask |= 1ull << (sl - R.s_begin);
          }
        });
        uint32_t cnt_r;
        const uint32_t at0 = block_excl_scan(own, sh, &cnt_r);
        if (tid == 0) {
          TopkCtlT& sh0 = *cluster.map_shared_rank(&sh, 0u);
          const uint32_t off = atomicAdd(&sh0.list_n, cnt_r);
          sh0.seg_off[rank] = off;
          sh0.seg_cnt[rank] = cnt_r;
          sh.bc[3] = off;
        }
        __syncthreads();
        uint32_t at = sh.bc[3] + at0;
        uint32_t* lkey0 = cluster.map_shared_rank(lkey, 0u);
        uint32_t* lslot0 = cluster.map_shared_rank(lslot, 0u);
        if (R.kept) {  // only the qualifying slots, in slot order
          while (qmask) {
            const int bi = __ffsll((long long)qmask) - 1;
            qmask &= qmask - 1;
            lkey0[at] = reinterpret_cast<const uint32_t*>(keys4 + rx_kidx<kTopkThreads>((uint32_t)bi >> 2, tid))[bi & 3];
            lslot0[at] = R.s_begin + (uint32_t)bi;
            ++at;
          }
        } else {
          // not kept: in rounds of one chunk per thread (slot order = chunk order =
          // thread order within a round), each placed by one block scan
          constexpr uint32_t kQ = 4;  // consecutive chunks a thread per round
          uint32_t at_run = sh.bc[3];
          const uint32_t nch = (R.hi - R.lo + 3) / 4;
          for (uint32_t g0 = 0; g0 < nch; g0 += kTopkThreads * kQ) {
            float x[kQ][4];
            bool ok[kQ][4];
#pragma unroll
            for (uint32_t i = 0; i < kQ; ++i) {
              const uint32_t g = g0 + kQ * tid + i;
#pragma unroll
              for (int u = 0; u < 4; ++u) ok[i][u] = false;
              if (g < nch) rx_load4_to(R, R.lo + 4 * g, R.hi, x[i], ok[i]);
            }
            uint32_t q = 0;
#pragma unroll
            for (uint32_t i = 0; i < kQ; ++i)
#pragma unroll
              for (int u = 0; u < 4; ++u) q += (ok[i][u] && float_order_key(x[i][u]) >= blo) ? 1u : 0u;
            uint32_t rt;
            uint32_t a = at_run + block_excl_scan(q, sh, &rt);
#pragma unroll
            for (uint32_t i = 0; i < kQ; ++i)
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t key = float_order_key(x[i][u]);
                if (ok[i][u] && key >= blo) {
                  lkey0[a] = key;
                  lslot0[a] = R.lo + 4 * (g0 + kQ * tid + i) + (uint32_t)u;
                  ++a;
                }
              }
            at_run += rt;
          }
        }
        cluster.sync();  // the last cluster barrier: only block 0 goes on
        if (rank != 0) return;
        rx_finish_list(lkey, lslot, sh.list_n, need - above_b, blo, min(hi, blo + ((1u << shift) - 1u)), sh, k,
                       crow, orow);
        return;  // exactly k selected: no padding
      }
      need -= above_b;
      klo = blo;
      khi = min(hi, blo + ((1u << shift) - 1u));
      __syncthreads();
      // the next level's histogram: no block reads this buffer any more (every
      // block passed the barrier after its last reads of it)
      for (int j = tid; j < kRxBins; j += kTopkThreads) sh.hist[hb ^ 1][j] = 0;
      __syncthreads();
    }
  }

  // ---- 2. ordered output
  uint32_t gt = 0, eq = 0;
  rx_visit_any<kTopkThreads, (kTopkCluster > 8 && kTopkThreads < 1024 ? 8 : 1)>(R, keys4, vbits, [&](uint32_t, uint32_t key) {
    gt += (long long)key > Tc;
    eq += (long long)key == Tc;
  });
  unsigned long long tot64;
  const unsigned long long ex64 =
      block_excl_scan64(((unsigned long long)gt << 32) | eq, sh, &tot64);
  if (tid < kTopkCluster) {
    TopkCtlT& dst = *cluster.map_shared_rank(&sh, (unsigned)tid);
    dst.gt[rank] = (uint32_t)(tot64 >> 32);
    dst.eq[rank] = (uint32_t)tot64;
  }
  cluster.sync();  // the last cluster barrier: from here on, local memory only
  long long sel_before = 0, eq_before = 0, gt_before = 0, total = 0;
  for (int q = 0; q < kTopkCluster; ++q) {
    const long long g = sh.gt[q], e = sh.eq[q];
    const long long te = min(max((long long)take_eq - eq_before, 0ll), e);  // ties block q takes
    if (q < (int)rank) sel_before += g + te;
    if (q < (int)rank) gt_before += g;
    total += g + te;
    if (q < (int)rank) eq_before += e;
  }
  if (!R.kept) {
    // not kept: in rounds of one chunk per thread, each placed by one block scan; a
    // taken slot with G keys > T and E ties before it in the row goes to G + min(E,
    // take_eq)
    // (kQ consecutive chunks a thread per round: kQ loads in flight, thread order = slot
    // order)
    constexpr uint32_t kQ = 4;
    long long G0 = gt_before, E0 = eq_before;
    const uint32_t nch = (R.hi - R.lo + 3) / 4;
    for (uint32_t g0 = 0; g0 < nch; g0 += kTopkThreads * kQ) {
      float x[kQ][4];
      bool ok[kQ][4];
#pragma unroll
      for (uint32_t i = 0; i < kQ; ++i) {
        const uint32_t g = g0 + kQ * tid + i;
#pragma unroll
        for (int u = 0; u < 4; ++u) ok[i][u] = false;
        if (g < nch) rx_load4_to(R, R.lo + 4 * g, R.hi, x[i], ok[i]);
      }
      uint32_t cg = 0, ce = 0;
#pragma unroll
      for (uint32_t i = 0; i < kQ; ++i)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (ok[i][u]) {
            const uint32_t kk = float_order_key(x[i][u]);
            cg += (long long)kk > Tc ? 1u : 0u;
            ce += (long long)kk == Tc ? 1u : 0u;
          }
        }
      unsigned long long rt;
      const unsigned long long rex = block_excl_scan64(((unsigned long long)cg << 32) | ce, sh, &rt);
      long long G = G0 + (long long)(rex >> 32), E = E0 + (long long)(uint32_t)rex;
#pragma unroll
      for (uint32_t i = 0; i < kQ; ++i)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (!ok[i][u]) continue;
          const uint32_t kk = float_order_key(x[i][u]);
          const uint32_t sl = R.lo + 4 * (g0 + kQ * tid + i) + (uint32_t)u;
          if ((long long)kk > Tc) {
            const long long p = G + min(E, (long long)take_eq);
            if (p < k) orow[p] = crow ? __ldg(crow + sl) : (int32_t)sl;
            ++G;
          } else if ((long long)kk == Tc) {
            if (E < (long long)take_eq && G + E < k) orow[G + E] = crow ? __ldg(crow + sl) : (int32_t)sl;
            ++E;
          }
        }
      G0 += (long long)(rt >> 32);
      E0 += (long long)(uint32_t)rt;
    }
    if (rank + 1 == kTopkCluster)
      for (long long j = total + tid; j < k; j += kTopkThreads) orow[j] = -1;
    return;
  }
  const long long eq_t = eq_before + (long long)(uint32_t)ex64;  // ties before this thread's run
  long long pos = sel_before + (long long)(ex64 >> 32) +
                  min(max((long long)take_eq - eq_before, 0ll), (long long)(uint32_t)ex64);
  long long eqi = eq_t;
  rx_visit<kTopkThreads, (kTopkCluster > 8 && kTopkThreads < 1024 ? 8 : 1)>(R, keys4, vbits, [&](uint32_t s, uint32_t key) {
    bool take = (long long)key > Tc;
    if ((long long)key == Tc) {
      take = eqi < (long long)take_eq;
      ++eqi;
    }
    if (take && pos < k) orow[pos++] = crow ? __ldg(crow + s) : (int32_t)s;
  });
  if (rank + 1 == kTopkCluster)
    for (long long j = total + tid; j < k; j += kTopkThreads) orow[j] = -1;
}

}  // namespace csa2
