// libcsa2: host side of the C ABI declared in include/csa2.h. Validates
// arguments, sizes grids and launches the kernels of this directory on the
// caller's stream. The library allocates no device memory.
#include <atomic>
#include <cstring>
#include <mutex>

#include <cuda.h>

#include "common.cuh"
#include "quant_append.cuh"
#include "indexer_scan.cuh"
#include "indexer_scan_tc.cuh"
#include "topk.cuh"
#include "attention.cuh"
#include "attention_cl.cuh"

namespace csa2 {
namespace {

std::atomic<uint64_t> g_launches{0};

// Measurement hook (csa2_set_scan_events): event pairs recorded around the streaming
// indexer scans, the i-th launch since the hook was set taking pair i mod n.
constexpr int kMaxScanEvents = 64;
thread_local cudaEvent_t g_scan_ev_before[kMaxScanEvents], g_scan_ev_after[kMaxScanEvents];
thread_local int g_scan_ev_n = 0, g_scan_ev_next = 0;

void record_hook_event(cudaEvent_t ev, cudaStream_t s) {
  if (!ev) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  cudaEventRecordWithFlags(ev, s, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0u);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Kernels may launch while the kernel before them in the stream finishes (each
// kernel waits for it with griddepcontrol.wait before touching global memory);
// CSA2_PDL=0 launches them one after another instead (read once).
bool pdl_enabled() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("CSA2_PDL");
    v = (e && strcmp(e, "0") == 0) ? 0 : 1;
  }
  return v == 1;
}

// Launch `kern` on `s` with programmatic stream serialization (when enabled) and,
// when cluster_x > 0, a cluster of cluster_x blocks along x.
template <typename... KArgs, typename... Args>
void launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, unsigned cluster_x,
              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  unsigned n = 0;
  if (pdl_enabled()) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 0) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

inline csa2_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

csa2_status check_cache(const csa2_cache_view* c) {
  if (!c || !c->lat_codes || !c->lat_scales || !c->idx_codes || !c->idx_scales || !c->len)
    return CSA2_ERR_ARG;
  if (c->cap <= 0 || (c->cap % 128) != 0 || c->batch <= 0 || c->batch > 65535) return CSA2_ERR_ARG;
  if (c->cap > (int64_t)INT32_MAX) return CSA2_ERR_UNSUPPORTED;
  if (!aligned16(c->lat_codes) || !aligned16(c->lat_scales) || !aligned16(c->idx_codes) ||
      !aligned16(c->idx_scales))
    return CSA2_ERR_ALIGN;
  return CSA2_OK;
}

// ------------------------------------------------------------ launchers (no validation)
template <auto Kern>
void ensure_max_smem(int bytes);

void launch_append(const void* lat, const void* ikey, csa2_dtype dt, int T, int ratio, const float* w0l,
                   const float* w1l, const float* w0i, const float* w1i, const csa2_cache_view& c,
                   cudaStream_t s) {
  const int n_new = T / ratio;
  const dim3 grid((n_new + kAppendBlockEntries - 1) / kAppendBlockEntries, c.batch);
  if (dt == CSA2_F32) {
    ensure_max_smem<k_quant_append<float>>((int)append_stage_bytes<float>(2));
    launch_k(k_quant_append<float>, grid, dim3(kAppendWarps * 32), append_stage_bytes<float>(ratio), s, 0u,
             (const float*)lat, (const float*)ikey, T, ratio, w0l, w1l, w0i, w1i, c.lat_codes, c.lat_scales,
             c.idx_codes, c.idx_scales, c.len, c.cap, n_new);
  } else {
    ensure_max_smem<k_quant_append<uint16_t>>((int)append_stage_bytes<uint16_t>(2));
    launch_k(k_quant_append<uint16_t>, grid, dim3(kAppendWarps * 32), append_stage_bytes<uint16_t>(ratio), s, 0u,
             (const uint16_t*)lat, (const uint16_t*)ikey, T, ratio, w0l, w1l, w0i, w1i, c.lat_codes, c.lat_scales,
             c.idx_codes, c.idx_scales, c.len, c.cap, n_new);
  }
  g_launches += 1;
  if (grid.x > 1) {  // several blocks per sequence: advance len once they are all done
    launch_k(k_bump_len, dim3((c.batch + 255) / 256), dim3(256), 0, s, 0u, c.len, c.batch, c.cap, n_new);
    g_launches += 1;
  }
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

constexpr int kMaxDevices = 64;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  return dev;
}

// Raise Kern's dynamic shared-memory limit to `bytes`, once per device (function
// attributes belong to the device's context).
template <auto Kern>
void ensure_max_smem(int bytes) {
  static std::atomic<int> done[kMaxDevices];
  const int dev = current_device();
  if (done[dev].load(std::memory_order_acquire)) return;
  cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  done[dev].store(1, std::memory_order_release);
}

template <int NPART>
void launch_scan_gather(const ScanArgs& a, cudaStream_t s) {
  static std::atomic<int> per_sm_of[kMaxDevices];  // resident blocks per SM, per device
  const int dev = current_device();
  int per_sm = per_sm_of[dev].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_indexer_scan_gather<NPART>, kScanThreads, 0);
    per_sm = occ > 0 ? occ : 1;
    per_sm_of[dev].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t want = (a.total_tiles + kScanWarps - 1) / kScanWarps;  // >= 1 tile per warp
  const int64_t full = (int64_t)sm_count() * per_sm;
  const int grid = (int)(want < full ? want : full);
  launch_k(k_indexer_scan_gather<NPART>, dim3(grid), dim3(kScanThreads), 0, s, 0u, a);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Tensor map of the key codes viewed as rows x 64 bytes; box 128 rows, 64-byte swizzle.
bool make_codes_map(CUtensorMap* m, const uint8_t* codes, int64_t rows) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc || rows <= 0 || rows >= ((int64_t)1 << 31)) return false;
  const cuuint64_t gdim[2] = {64, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {64};
  const cuuint32_t box[2] = {64, (cuuint32_t)kTmaRows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), gdim, gstride, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NPART>
void launch_scan_tma(const CUtensorMap& m, const TmaScanArgs& a, cudaStream_t s) {
  ensure_max_smem<k_indexer_scan_tma<NPART>>(kTmaSmem);
  const int64_t full = (int64_t)sm_count() * kTmaBlocksPerSM;
  const int grid = (int)(a.total_tiles < full ? a.total_tiles : full);
  launch_k(k_indexer_scan_tma<NPART>, dim3(grid), dim3(kTmaThreads), kTmaSmem, s, 0u, m, a);
}

template <int NPART>
void launch_scan_tc(const CUtensorMap& m, const TmaScanArgs& a, cudaStream_t s) {
  using S = TcShape<NPART>;
  ensure_max_smem<k_indexer_scan_tc<NPART>>(S::Smem);
  // two blocks per SM: their 256-column tensor-memory allocations fill the SM's 512
  // columns, and registers (96 x 320 per block) and shared memory allow two
  static std::atomic<int> per_sm_of[kMaxDevices];
  const int dev = current_device();
  int per_sm = per_sm_of[dev].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    int smem_sm = 0;
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    per_sm = smem_sm >= 2 * (S::Smem + 1024) ? 2 : 1;
    per_sm_of[dev].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t full = (int64_t)sm_count() * per_sm;
  const int grid = (int)(a.total_tiles < full ? a.total_tiles : full);
  launch_k(k_indexer_scan_tc<NPART>, dim3(grid), dim3(kTcThreads), S::Smem, s, 0u, m, a);
}

// Which streaming scan runs: the mma.sync form unless CSA2_SCAN_KERNEL=tc asks for
// the tcgen05 form (read once).
bool scan_uses_tcgen05() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("CSA2_SCAN_KERNEL");
    v = (e && strcmp(e, "tc") == 0) ? 1 : 0;
  }
  return v == 1;
}

void launch_scan(const void* q_idx, csa2_dtype dt, const float* w, const uint8_t* codes, const uint8_t* scales,
                 int64_t cap, const int32_t* len, const int32_t* cand, int P, float* scores, int batch,
                 cudaStream_t s, int scratch = 0) {
  g_launches += 1;
  CUtensorMap m;
  if (!cand && cap % kTmaRows == 0 && make_codes_map(&m, codes, (int64_t)batch * cap)) {
    TmaScanArgs t;
    t.q_idx = q_idx;
    t.q_dtype = (int)dt;
    t.w = w;
    t.codes = codes;
    t.scales = scales;
    t.cap = cap;
    t.len = len;
    t.scores = scores;
    t.scratch = scratch;
    const int64_t tile_rows = scan_uses_tcgen05() ? kTmaRows : kTmaStageRows;
    t.tiles_per_seq = (cap + tile_rows - 1) / tile_rows;
    t.total_tiles = t.tiles_per_seq * batch;
    const int ev = g_scan_ev_n > 0 ? g_scan_ev_next++ % g_scan_ev_n : -1;
    if (ev >= 0) record_hook_event(g_scan_ev_before[ev], s);
    if (scan_uses_tcgen05()) {
      if (dt == CSA2_F32) launch_scan_tc<2>(m, t, s);
      else launch_scan_tc<1>(m, t, s);
    } else {
      if (dt == CSA2_F32) launch_scan_tma<2>(m, t, s);
      else launch_scan_tma<1>(m, t, s);
    }
    if (ev >= 0) record_hook_event(g_scan_ev_after[ev], s);
    return;
  }
  ScanArgs a;
  a.q_idx = q_idx;
  a.q_dtype = (int)dt;
  a.w = w;
  a.codes = codes;
  a.scales = scales;
  a.cap = cap;
  a.len = len;
  a.cand = cand;
  a.P = P;
  a.scores = scores;
  a.scratch = scratch;
  a.stride = cand ? P : cap;
  a.tiles_per_seq = (a.stride + kScanTile - 1) / kScanTile;
  a.total_tiles = a.tiles_per_seq * batch;
  if (dt == CSA2_F32) launch_scan_gather<2>(a, s);
  else launch_scan_gather<1>(a, s);
}

template <int THREADS, int CLUSTER>
void launch_topk_shape(const float* scores, const int32_t* n, int64_t stride, int k, const int32_t* cand,
                       int32_t* out, int batch, cudaStream_t s, int discard) {
  constexpr size_t smem = topk_smem<THREADS, CLUSTER>();
  if (CLUSTER > 8) {  // beyond the portable cluster size (set once per device)
    static std::atomic<int> done[kMaxDevices];
    const int dev = current_device();
    if (!done[dev].load(std::memory_order_acquire)) {
      cudaFuncSetAttribute(k_topk<THREADS, CLUSTER>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      done[dev].store(1, std::memory_order_release);
    }
  }
  ensure_max_smem<k_topk<THREADS, CLUSTER>>((int)smem);
  launch_k(k_topk<THREADS, CLUSTER>, dim3(CLUSTER, batch), dim3(THREADS), smem, s, 0u, scores, stride, n, cand, k,
           out, discard);
}

// One cluster per row, every block keeping its slice in shared memory where it can:
// four 512-thread blocks up to 73,728 slots (71 clusters at once on B300, so a 64-row
// batch is one wave), eight up to 147,456 (33 at once), sixteen 1,024-thread blocks
// (one per SM) up to 589,824 (7 at once); beyond that, sixteen 512-thread blocks that
// re-read their slices from global memory at each pass.
void launch_topk(const float* scores, const int32_t* n, int64_t stride, int k, const int32_t* cand,
                 int32_t* out, int batch, cudaStream_t s, int discard = 0) {
  if ((uint64_t)stride <= 4ull * TopkCtl<512, 4>::kSliceCap)
    launch_topk_shape<512, 4>(scores, n, stride, k, cand, out, batch, s, discard);
  else if ((uint64_t)stride <= 8ull * TopkCtl<512, 8>::kSliceCap)
    launch_topk_shape<512, 8>(scores, n, stride, k, cand, out, batch, s, discard);
  else if ((uint64_t)stride <= 16ull * TopkCtl<1024, 16>::kSliceCap)
    launch_topk_shape<1024, 16>(scores, n, stride, k, cand, out, batch, s, discard);
  else
    launch_topk_shape<512, 16>(scores, n, stride, k, cand, out, batch, s, discard);
  g_launches += 1;
}

// Sliding-window rows of an attention launch: bf16 rows, or FP8 rows (E4M3 codes and
// E8M0 scales), W of them per sequence.
struct Window {
  const uint16_t* bf16;
  const uint8_t* codes;
  const uint8_t* scales;
  int W;
};

template <int NPART>
void launch_attn_t(const void* q, csa2_dtype dt, int H, float scale, const csa2_cache_view& c, const int32_t* idx,
                   int k, const Window& win, float* out, cudaStream_t s) {
  ensure_max_smem<k_sparse_attn<NPART>>(kAttnSmem);
  launch_k(k_sparse_attn<NPART>, dim3(2 * (H / kAttnHeads), c.batch), dim3(kAttnThreads), kAttnSmem, s, 0u, q,
           (int)dt, scale, c.lat_codes, c.lat_scales, c.len, c.cap, idx, k, win.bf16, win.codes, win.scales, win.W,
           H, out);
}

// One attention layer of a launch: its queries, selection, window rows and output.
struct AttnLayer {
  const void* q;
  const int32_t* idx;
  Window win;
  float* out;
};

// Key-split form: one cluster of ceil((k + W) / 128) blocks per (sequence, 64 heads,
// layer); the layers of one launch share the cache, k, W, H and the query type.
template <int NPART>
void launch_attn_cl(const AttnLayer* L, int nl, csa2_dtype dt, int H, float scale, const csa2_cache_view& c, int k,
                    int W, int q_early, cudaStream_t s) {
  ensure_max_smem<k_sparse_attn_cl<NPART>>(kAclSmem);
  AclLayers t = {};
  for (int i = 0; i < nl; ++i) {
    t.q[i] = L[i].q;
    t.idx[i] = L[i].idx;
    t.swa[i] = L[i].win.bf16;
    t.swa_codes[i] = L[i].win.codes;
    t.swa_scales[i] = L[i].win.scales;
    t.out[i] = L[i].out;
  }
  // C blocks per (sequence, 64 heads, layer): one 128-key chunk each while the rows fill
  // fewer than one block per SM, else fewer blocks with several chunks each (down to one
  // block a row: no merge). fp32 queries keep one chunk per block.
  const int c_full = (k + W + kAclKeys - 1) / kAclKeys;
  int C = c_full;
  if (NPART == 1) {
    const int64_t rows = (int64_t)(H / kAclHeads) * c.batch * nl;
    const int64_t per = (int64_t)sm_count() / (rows > 0 ? rows : 1);
    C = (int)(per < 1 ? 1 : per < c_full ? per : c_full);
  }
  launch_k(k_sparse_attn_cl<NPART>, dim3((unsigned)(C * (H / kAclHeads)), (unsigned)c.batch, (unsigned)nl),
           dim3(kAclThreads), kAclSmem, s, C > 1 ? (unsigned)C : 0u, t, (int)dt, scale, c.lat_codes, c.lat_scales,
           c.len, c.cap, k, W, H, q_early, C);
}

// The key-split form covers 64-head groups and up to 1,024 keys per row; the
// chunked form everything else. CSA2_ATTN_KERNEL=chunked forces the chunked form
// (read once).
bool attn_key_split(int H, int k, int W) {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("CSA2_ATTN_KERNEL");
    v = (e && strcmp(e, "chunked") == 0) ? 0 : 1;
  }
  return v == 1 && H % kAclHeads == 0 && k + W >= 1 && k + W <= kAclKeys * kAclMaxBlocks;
}

// Attention for nl layers (at most kAclMaxLayers, all with the same W) over cache c:
// one key-split launch covering every layer, or one chunked launch per layer. q_early:
// the kernel before this launch on `s` is this library's Top-k, which does not write
// q; the queries may then be read before waiting for it.
void launch_attn(const AttnLayer* L, int nl, csa2_dtype dt, int H, float scale, const csa2_cache_view& c, int k,
                 cudaStream_t s, int q_early = 0) {
  const int W = L[0].win.W;
  if (attn_key_split(H, k, W)) {
    if (dt == CSA2_F32) launch_attn_cl<2>(L, nl, dt, H, scale, c, k, W, q_early, s);
    else launch_attn_cl<1>(L, nl, dt, H, scale, c, k, W, q_early, s);
    g_launches += 1;
    return;
  }
  for (int i = 0; i < nl; ++i) {
    if (dt == CSA2_F32) launch_attn_t<2>(L[i].q, dt, H, scale, c, L[i].idx, k, L[i].win, L[i].out, s);
    else launch_attn_t<1>(L[i].q, dt, H, scale, c, L[i].idx, k, L[i].win, L[i].out, s);
    g_launches += 1;
  }
}

// One thread waits, with the kernels' bounded wait and the given budget, on an
// mbarrier that nothing ever arrives at: the wait runs out, records
// CSA2_ERR_TIMEOUT in the device status word and the kernel returns.
__global__ void k_selftest_wait(uint64_t budget_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32addr(&bar);
  mbar_init(b, 1);
  abort_flag = 0;
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  mbar_wait_bounded_ns(b, 0u, &abort_flag, budget_ns);
}

// A window is either bf16 rows or FP8 rows (codes and scales together), never both;
// W > 0 needs rows.
csa2_status check_window(const uint16_t* swa, const uint8_t* codes, const uint8_t* scales, int W) {
  if (W < 0 || W > CSA2_MAX_WINDOW || (codes == nullptr) != (scales == nullptr) || (swa && codes))
    return CSA2_ERR_ARG;
  if (W > 0 && !swa && !codes) return CSA2_ERR_ARG;
  if ((swa && !aligned16(swa)) || (codes && (!aligned16(codes) || !aligned16(scales)))) return CSA2_ERR_ALIGN;
  return CSA2_OK;
}

template <typename Tin>
void launch_store(const StoreArgs& a, int batch, int blocks, cudaStream_t s) {
  int rmax = 1;
  for (int i = 0; i < a.n_layers; ++i) rmax = a.L[i].ratio > rmax ? a.L[i].ratio : rmax;
  ensure_max_smem<k_store_append<Tin>>((int)append_stage_bytes<Tin>(2));
  launch_k(k_store_append<Tin>, dim3((unsigned)blocks, (unsigned)batch), dim3(kAppendWarps * 32),
           append_stage_bytes<Tin>(rmax), s, 0u, a);
  launch_k(k_store_bump, dim3((unsigned)a.n_layers), dim3(256), 0, s, 0u, a, batch);
  g_launches += 2;
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" {

csa2_status csa2_selftest_wait_timeout(uint64_t budget_ns, csa2_stream_t stream) {
  if (budget_ns > 1000000000ull) return CSA2_ERR_ARG;
  k_selftest_wait<<<1, 32, 0, (cudaStream_t)stream>>>(budget_ns);
  return cudaGetLastError() == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

csa2_status kv_quant_append(const void* lat, const void* ikey, csa2_dtype in_dtype, int32_t T, int32_t ratio,
                            const float* w0_lat, const float* w1_lat, const float* w0_idx, const float* w1_idx,
                            const csa2_cache_view* cache, csa2_stream_t stream) {
  const csa2_status cs = check_cache(cache);
  if (cs != CSA2_OK) return cs;
  if (in_dtype != CSA2_F32 && in_dtype != CSA2_BF16) return CSA2_ERR_ARG;
  if (T < 0 || (ratio != 1 && ratio != 2)) return CSA2_ERR_ARG;
  if (ratio == 2 && ((T & 1) || !w0_lat || !w1_lat || !w0_idx || !w1_idx)) return CSA2_ERR_ARG;
  if (ratio == 2 && (!aligned16(w0_lat) || !aligned16(w1_lat) || !aligned16(w0_idx) || !aligned16(w1_idx)))
    return CSA2_ERR_ALIGN;
  if (T == 0) return CSA2_OK;
  if (!lat || !ikey) return CSA2_ERR_ARG;
  if (!aligned16(lat) || !aligned16(ikey)) return CSA2_ERR_ALIGN;
  launch_append(lat, ikey, in_dtype, T, ratio, w0_lat, w1_lat, w0_idx, w1_idx, *cache, (cudaStream_t)stream);
  return launch_status();
}

csa2_status indexer_score(const void* q_idx, csa2_dtype q_dtype, const float* w, const uint8_t* idx_codes,
                          const uint8_t* idx_scales, int64_t cap, const int32_t* len, const int32_t* cand,
                          int32_t P, float* scores, int32_t batch, csa2_stream_t stream) {
  if (!q_idx || !w || !idx_codes || !idx_scales || !len || !scores) return CSA2_ERR_ARG;
  if (q_dtype != CSA2_F32 && q_dtype != CSA2_BF16) return CSA2_ERR_ARG;
  if (cap <= 0 || cap % 128 || cap > INT32_MAX || batch <= 0 || batch > 65535) return CSA2_ERR_ARG;
  if (cand && (P <= 0 || P > CSA2_MAX_TOPK)) return CSA2_ERR_ARG;
  if (!aligned16(idx_codes) || !aligned16(idx_scales)) return CSA2_ERR_ALIGN;
  launch_scan(q_idx, q_dtype, w, idx_codes, idx_scales, cap, len, cand, P, scores, batch, (cudaStream_t)stream);
  return launch_status();
}

csa2_status topk_select(const float* scores, const int32_t* n, int64_t stride, int32_t k, const int32_t* cand,
                        int32_t* out_idx, int32_t batch, csa2_stream_t stream) {
  if (!scores || !out_idx) return CSA2_ERR_ARG;
  if (stride <= 0 || stride > INT32_MAX || k < 1 || k > CSA2_MAX_TOPK || batch <= 0) return CSA2_ERR_ARG;
  launch_topk(scores, n, stride, k, cand, out_idx, batch, (cudaStream_t)stream);
  return launch_status();
}

csa2_status sparse_latent_attn(const void* q, csa2_dtype q_dtype, int32_t H, float scale,
                               const csa2_cache_view* cache, const int32_t* idx, int32_t k, const uint16_t* swa,
                               const uint8_t* swa_codes, const uint8_t* swa_scales, int32_t W, float* out,
                               csa2_stream_t stream) {
  const csa2_status cs = check_cache(cache);
  if (cs != CSA2_OK) return cs;
  if (!q || !out || (q_dtype != CSA2_F32 && q_dtype != CSA2_BF16)) return CSA2_ERR_ARG;
  if (H != 16 && H != 32 && H != 64) return CSA2_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || k < 0 || k > CSA2_MAX_TOPK) return CSA2_ERR_ARG;
  if (k > 0 && !idx) return CSA2_ERR_ARG;
  const csa2_status ws = check_window(swa, swa_codes, swa_scales, W);
  if (ws != CSA2_OK) return ws;
  if (!aligned16(q) || !aligned16(out)) return CSA2_ERR_ALIGN;
  const AttnLayer L{q, idx, Window{swa, swa_codes, swa_scales, W}, out};
  launch_attn(&L, 1, q_dtype, H, scale, *cache, k, (cudaStream_t)stream);
  return launch_status();
}

csa2_status csa2_swa_quant(const void* rows, csa2_dtype in_dtype, int64_t n_rows, uint8_t* codes, uint8_t* scales,
                           csa2_stream_t stream) {
  if (in_dtype != CSA2_F32 && in_dtype != CSA2_BF16) return CSA2_ERR_ARG;
  if (n_rows < 0 || n_rows > ((int64_t)INT32_MAX) * kSwaWarps) return CSA2_ERR_ARG;
  if (n_rows == 0) return CSA2_OK;
  if (!rows || !codes || !scales) return CSA2_ERR_ARG;
  if (!aligned16(rows) || !aligned16(codes) || !aligned16(scales)) return CSA2_ERR_ALIGN;
  const dim3 grid((unsigned)((n_rows + kSwaWarps - 1) / kSwaWarps));
  if (in_dtype == CSA2_F32)
    launch_k(k_swa_quant<float>, grid, dim3(kSwaWarps * 32), 0, (cudaStream_t)stream, 0u, (const float*)rows,
             n_rows, codes, scales);
  else
    launch_k(k_swa_quant<uint16_t>, grid, dim3(kSwaWarps * 32), 0, (cudaStream_t)stream, 0u, (const uint16_t*)rows,
             n_rows, codes, scales);
  g_launches += 1;
  return launch_status();
}

csa2_status csa2_store_append(const csa2_store_layer* layers, int32_t n_layers, csa2_dtype in_dtype, int32_t T,
                              csa2_stream_t stream) {
  if (!layers || n_layers < 1 || n_layers > kStoreMaxLayers) return CSA2_ERR_ARG;
  if (in_dtype != CSA2_F32 && in_dtype != CSA2_BF16) return CSA2_ERR_ARG;
  if (T < 0) return CSA2_ERR_ARG;
  StoreArgs a{};
  a.n_layers = n_layers;
  a.T = T;
  int batch = -1, blocks = 0;
  for (int i = 0; i < n_layers; ++i) {
    const csa2_store_layer& L = layers[i];
    const csa2_status cs = check_cache(L.cache);
    if (cs != CSA2_OK) return cs;
    if (batch >= 0 && L.cache->batch != batch) return CSA2_ERR_ARG;
    batch = L.cache->batch;
    if (L.ratio != 1 && L.ratio != 2) return CSA2_ERR_ARG;
    if (L.ratio == 2 && ((T & 1) || !L.w0_lat || !L.w1_lat || !L.w0_idx || !L.w1_idx)) return CSA2_ERR_ARG;
    if (L.ratio == 2 && (!aligned16(L.w0_lat) || !aligned16(L.w1_lat) || !aligned16(L.w0_idx) ||
                         !aligned16(L.w1_idx)))
      return CSA2_ERR_ALIGN;
    if (T > 0 && (!L.lat || !L.ikey)) return CSA2_ERR_ARG;
    if (T > 0 && (!aligned16(L.lat) || !aligned16(L.ikey))) return CSA2_ERR_ALIGN;
    StoreLayer& S = a.L[i];
    S.lat = L.lat;
    S.ikey = L.ikey;
    S.w0l = L.w0_lat;
    S.w1l = L.w1_lat;
    S.w0i = L.w0_idx;
    S.w1i = L.w1_idx;
    S.lat_codes = L.cache->lat_codes;
    S.lat_scales = L.cache->lat_scales;
    S.idx_codes = L.cache->idx_codes;
    S.idx_scales = L.cache->idx_scales;
    S.len = L.cache->len;
    S.cap = L.cache->cap;
    S.ratio = L.ratio;
    S.n_new = T / L.ratio;
    S.block0 = blocks;
    blocks += (S.n_new + kAppendBlockEntries - 1) / kAppendBlockEntries;
  }
  if (T == 0) return CSA2_OK;
  if (in_dtype == CSA2_F32) launch_store<float>(a, batch, blocks, (cudaStream_t)stream);
  else launch_store<uint16_t>(a, batch, blocks, (cudaStream_t)stream);
  return launch_status();
}

namespace {
struct StepLayout {
  size_t scores, pool, pscores, sel, total;
};

StepLayout step_layout(int32_t batch, int64_t max_entries, int32_t H, int32_t k, int32_t pool, int32_t W) {
  StepLayout L{};
  size_t off = 0;
  L.scores = off;
  off += round_up((size_t)batch * (size_t)max_entries * sizeof(float), 256);
  L.pool = off;
  off += round_up((size_t)batch * (size_t)pool * sizeof(int32_t), 256);
  L.pscores = off;
  off += round_up((size_t)batch * (size_t)pool * sizeof(float), 256);
  L.sel = off;  // two selections: a layer's attention can wait for a later layer's
  off += 2 * round_up((size_t)batch * (size_t)k * sizeof(int32_t), 256);
  L.total = off;
  (void)H;
  (void)W;
  return L;
}
}  // namespace

size_t csa2_workspace_size(int32_t batch, int64_t max_entries, int32_t H, int32_t k, int32_t pool, int32_t W) {
  return step_layout(batch, max_entries, H, k, pool, W).total;
}

csa2_status csa2_decode_step(const csa2_layer_desc* layers, int32_t n_layers, int32_t batch, int32_t H, int32_t k,
                             csa2_dtype dtype, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  if (!layers || n_layers < 1 || batch <= 0 || batch > 65535) return CSA2_ERR_ARG;
  if (dtype != CSA2_F32 && dtype != CSA2_BF16) return CSA2_ERR_ARG;
  if (H != 16 && H != 32 && H != 64) return CSA2_ERR_UNSUPPORTED;
  if (k < 1 || k > CSA2_MAX_TOPK) return CSA2_ERR_ARG;
  if (layers[0].mode != CSA2_FULL) return CSA2_ERR_ARG;
  // validate every layer and find the workspace sizes
  int64_t max_cap = 0;
  int32_t max_pool = 0, max_W = 0;
  for (int i = 0; i < n_layers; ++i) {
    const csa2_layer_desc& L = layers[i];
    if (L.mode != CSA2_FULL && L.mode != CSA2_REINDEX && L.mode != CSA2_REUSE) return CSA2_ERR_ARG;
    if (!L.q || !L.out) return CSA2_ERR_ARG;
    const csa2_status wst = check_window(L.swa, L.swa_codes, L.swa_scales, L.W);
    if (wst != CSA2_OK) return wst;
    if (!aligned16(L.q) || !aligned16(L.out)) return CSA2_ERR_ALIGN;
    if (L.mode == CSA2_FULL) {
      const csa2_status cs = check_cache(L.cache);
      if (cs != CSA2_OK) return cs;
      if (L.cache->batch != batch) return CSA2_ERR_ARG;
      if (L.pool < 0 || L.pool > CSA2_MAX_TOPK || (L.pool > 0 && (L.pool <= k || !L.q_idx2 || !L.w_idx2)))
        return CSA2_ERR_ARG;
      max_cap = L.cache->cap > max_cap ? L.cache->cap : max_cap;
      max_pool = L.pool > max_pool ? L.pool : max_pool;
    }
    if (L.mode != CSA2_REUSE && (!L.q_idx || !L.w_idx)) return CSA2_ERR_ARG;
    if (L.mode == CSA2_REINDEX && ((L.own_idx_codes == nullptr) != (L.own_idx_scales == nullptr)))
      return CSA2_ERR_ARG;
    if (L.mode == CSA2_REINDEX && L.own_idx_codes && (!aligned16(L.own_idx_codes) || !aligned16(L.own_idx_scales)))
      return CSA2_ERR_ALIGN;
    max_W = L.W > max_W ? L.W : max_W;
  }
  const StepLayout SL = step_layout(batch, max_cap, H, k, max_pool, max_W);
  if (!ws || ws_bytes < SL.total) return CSA2_ERR_WORKSPACE;
  if (!aligned16(ws)) return CSA2_ERR_ALIGN;
  char* base = static_cast<char*>(ws);
  float* scores = reinterpret_cast<float*>(base + SL.scores);
  int32_t* pool_idx = reinterpret_cast<int32_t*>(base + SL.pool);
  float* pscores = reinterpret_cast<float*>(base + SL.pscores);
  int32_t* sel[2] = {reinterpret_cast<int32_t*>(base + SL.sel),
                     reinterpret_cast<int32_t*>(base + SL.sel + round_up((size_t)batch * (size_t)k * sizeof(int32_t), 256))};
  cudaStream_t s = (cudaStream_t)stream;
  // Top-k of every entry of a cache: scores, then the cluster select
  auto scan_and_select = [&](const void* qi, const float* wi, const uint8_t* kc, const uint8_t* ksc,
                             const csa2_cache_view* c, int32_t* out_idx) {
    launch_scan(qi, dtype, wi, kc, ksc, c->cap, c->len, nullptr, 0, scores, batch, s, 1);
    launch_topk(scores, c->len, c->cap, k, nullptr, out_idx, batch, s, 1);
  };

  // Each layer's attention is deferred and launched together with the following
  // layers' (one launch, one grid layer each) while they share the cache and the
  // window length: a layer's attention waits at most until a later Top-k would
  // overwrite the selection it reads, the cache changes, or the group is full.
  const float scale = 1.0f / sqrtf((float)CSA2_LATENT_DIM);
  AttnLayer pend[kAclMaxLayers];
  int np = 0;
  const csa2_cache_view* pend_cache = nullptr;
  auto pending_reads = [&](const int32_t* p) {
    for (int j = 0; j < np; ++j)
      if (pend[j].idx == p) return true;
    return false;
  };
  auto flush = [&]() {
    if (np > 0) launch_attn(pend, np, dtype, H, scale, *pend_cache, k, s, 1);
    np = 0;
  };

  const csa2_cache_view* main = nullptr;
  const int32_t* last = nullptr;
  int pool = 0;
  for (int i = 0; i < n_layers; ++i) {
    const csa2_layer_desc& L = layers[i];
    if (L.mode == CSA2_FULL || L.mode == CSA2_REINDEX) {
      // this layer's selection: its own output array, else a workspace selection that
      // no deferred attention reads
      int32_t* dst = L.idx_out;
      if (!dst) {
        dst = !pending_reads(sel[0]) ? sel[0] : !pending_reads(sel[1]) ? sel[1] : nullptr;
        if (!dst) {
          flush();
          dst = sel[0];
        }
      } else if (pending_reads(dst)) {
        flush();
      }
      if (L.mode == CSA2_FULL) {
        main = L.cache;
        pool = L.pool;
        if (pool > 0) {
          launch_scan(L.q_idx, dtype, L.w_idx, main->idx_codes, main->idx_scales, main->cap, main->len, nullptr, 0,
                      scores, batch, s, 1);
          launch_topk(scores, main->len, main->cap, pool, nullptr, pool_idx, batch, s, 1);
          launch_scan(L.q_idx2, dtype, L.w_idx2, main->idx_codes, main->idx_scales, main->cap, main->len, pool_idx,
                      pool, pscores, batch, s, 1);
          launch_topk(pscores, nullptr, pool, k, pool_idx, dst, batch, s, 1);
        } else {
          scan_and_select(L.q_idx, L.w_idx, main->idx_codes, main->idx_scales, main, dst);
        }
      } else {
        const uint8_t* kc = L.own_idx_codes ? L.own_idx_codes : main->idx_codes;
        const uint8_t* ksc = L.own_idx_scales ? L.own_idx_scales : main->idx_scales;
        if (pool > 0) {
          launch_scan(L.q_idx, dtype, L.w_idx, kc, ksc, main->cap, main->len, pool_idx, pool, pscores, batch, s, 1);
          launch_topk(pscores, nullptr, pool, k, pool_idx, dst, batch, s, 1);
        } else {
          scan_and_select(L.q_idx, L.w_idx, kc, ksc, main, dst);
        }
      }
      last = dst;
    } else if (L.idx_out) {
      if (cudaMemcpyAsync(L.idx_out, last, (size_t)batch * k * sizeof(int32_t), cudaMemcpyDeviceToDevice, s) !=
          cudaSuccess)
        return CSA2_ERR_CUDA;
    }
    if (np > 0 && (pend_cache != main || pend[0].win.W != L.W || np == kAclMaxLayers)) flush();
    pend[np++] = AttnLayer{L.q, last, Window{L.swa, L.swa_codes, L.swa_scales, L.W}, L.out};
    pend_cache = main;
  }
  flush();
  return launch_status();
}

csa2_status csa2_sync_status(csa2_stream_t stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CSA2_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_dev_error, sizeof(int)) != cudaSuccess) return CSA2_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(int)) != cudaSuccess) return CSA2_ERR_CUDA;
  }
  return (csa2_status)v;
}

const char* csa2_status_str(csa2_status st) {
  switch (st) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_ARG: return "invalid argument";
    case CSA2_ERR_ALIGN: return "pointer not 16-byte aligned";
    case CSA2_ERR_UNSUPPORTED: return "unsupported shape";
    case CSA2_ERR_CUDA: return "CUDA runtime error";
    case CSA2_ERR_TIMEOUT: return "device wait timed out";
    case CSA2_ERR_BOUNDS: return "index or append outside the cache";
    case CSA2_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

uint64_t csa2_launch_count(void) { return g_launches.load(); }

csa2_status csa2_set_scan_events(void* const* before, void* const* after, int32_t n) {
  if (n < 0 || n > kMaxScanEvents || (n > 0 && (!before || !after))) return CSA2_ERR_ARG;
  for (int i = 0; i < n; ++i)
    if (!before[i] || !after[i]) return CSA2_ERR_ARG;
  for (int i = 0; i < n; ++i) {
    g_scan_ev_before[i] = static_cast<cudaEvent_t>(before[i]);
    g_scan_ev_after[i] = static_cast<cudaEvent_t>(after[i]);
  }
  g_scan_ev_n = n;
  g_scan_ev_next = 0;
  return CSA2_OK;
}

// ---------------------------------------------------------------- allocation-free decode step
// Scratch of csa2_decode_step_static: one file-scope device array, present on every
// device that loads this library until the process exits. Host code only ever uses
// its per-device address from cudaGetSymbolAddress (the symbol itself is a host-side
// stand-in there).
static __device__ __align__(256) unsigned char g_static_ws[CSA2_STATIC_WS_BYTES];

namespace {
std::mutex g_static_ws_mutex;
void* g_static_ws_ptr[64] = {nullptr};
}  // namespace

csa2_status csa2_decode_step_static(const csa2_layer_desc* layers, int32_t n_layers, int32_t batch, int32_t H,
                                    int32_t k, csa2_dtype dtype, csa2_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CSA2_ERR_CUDA;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_ws_mutex);
    if (!g_static_ws_ptr[dev]) {  // first call on this device: look the array up (device is current)
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return CSA2_ERR_CUDA;
      g_static_ws_ptr[dev] = p;
    }
    ws = g_static_ws_ptr[dev];
  }
  return csa2_decode_step(layers, n_layers, batch, H, k, dtype, ws, (size_t)CSA2_STATIC_WS_BYTES, stream);
}

}  // extern "C"
