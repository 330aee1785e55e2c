/*
 * csa2.h -- C ABI of the CSA2 FP4 compressed-KV decode path (libcsa2.so).
 *
 * The operations follow the pages on DeepSeek-V4.1-Flash's KV cache:
 *   "Le cache KV en FP4 -- les 890 octets, verifies" (cache record: eq. 288 and
 *     eq. 68, section "D'ou viennent ces deux reglages", "Le compte par couche");
 *   "DeepSeek V4.1 Flash : 890 octets de cache KV par token", section
 *     "L'architecture", paragraphs "Deuxiemement" (Full/Reindex/Reuse, Top-512,
 *     16,384-position hierarchical indexer) and "Troisiemement" (E2M1 + E4M3 per
 *     16 channels, 128-token sliding window);
 *   "DeepSeek-V4.1 Flash compresse le KV-Cache de 4 fois", section "Mecanismes
 *     de compression du KV-Cache", items 1-3 (shared 512-d latent for keys and
 *     values, ratio-2 merge with per-channel weights, cross-layer modes).
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is a DEVICE pointer unless the comment says "host".
 *    The caller owns all memory; the library allocates nothing.
 *  - Every call is asynchronous on the caller's stream ``stream`` (0 = legacy
 *    default stream). Arguments are validated on the host before any launch;
 *    a failed check returns a non-zero csa2_status and launches nothing.
 *  - Device-side errors (an index out of range, a wait that ran out) are
 *    recorded in a per-process device status word; csa2_sync_status() reads
 *    and clears it. No C++ exception crosses this boundary.
 *  - Cache layout is struct-of-arrays per layer, row = entry:
 *      lat_codes  [batch][cap][256] u8  E2M1 codes, channel 2j in the low nibble
 *      lat_scales [batch][cap][32]  u8  E4M3 (fn) scale of channels 16i..16i+15
 *      idx_codes  [batch][cap][64]  u8  E2M1 codes of the 128-channel indexer key
 *      idx_scales [batch][cap][4]   u8  E8M0 scale of channels 32i..32i+31
 *      len        [batch]           i32 number of valid entries per sequence
 *    288 + 68 bytes per entry, as on the pages. ``cap`` must be a multiple of
 *    128 and every array 16-byte aligned.
 *  - bf16 tensors are passed as raw 16-bit patterns (uint16_t).
 *  - Environment switches, read once per process (for measurements):
 *    CSA2_SCAN_KERNEL=tc runs the streaming indexer scan on the tcgen05 form
 *    instead of the mma.sync form; CSA2_ATTN_KERNEL=chunked runs attention on
 *    the chunked form for every shape; CSA2_PDL=0 launches kernels without
 *    programmatic dependent launch. The forms agree within the parity
 *    tolerances (fp32 rounding order differs; packed bytes are identical).
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSA2_API __attribute__((visibility("default")))
#else
#define CSA2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* csa2_stream_t; /* a cudaStream_t */

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_ARG = 1,         /* null pointer, bad size, bad enum value */
  CSA2_ERR_ALIGN = 2,       /* a pointer is not 16-byte aligned */
  CSA2_ERR_UNSUPPORTED = 3, /* a valid but unsupported shape (e.g. head count) */
  CSA2_ERR_CUDA = 4,        /* a CUDA runtime call failed */
  CSA2_ERR_TIMEOUT = 5,     /* a bounded device wait ran out (device word) */
  CSA2_ERR_BOUNDS = 6,      /* an index or an append fell outside the cache (device word) */
  CSA2_ERR_WORKSPACE = 7    /* the workspace is smaller than csa2_workspace_size() */
} csa2_status;

typedef enum { CSA2_F32 = 0, CSA2_BF16 = 1 } csa2_dtype;

typedef enum { CSA2_FULL = 0, CSA2_REINDEX = 1, CSA2_REUSE = 2 } csa2_mode;

enum {
  CSA2_LATENT_DIM = 512,  /* main-KV latent channels */
  CSA2_INDEXER_DIM = 128, /* indexer-key channels */
  CSA2_INDEXER_HEADS = 4, /* indexer query heads */
  CSA2_MAX_TOPK = 16384,  /* largest k of topk_select (the hierarchical pool size) */
  CSA2_MAX_WINDOW = 1024  /* largest sliding window */
};

/* Size of the device scratch built into the library for csa2_decode_step_static. */
#define CSA2_STATIC_WS_BYTES (24u << 20) /* 24 MiB */

/* One layer's global cache (host struct holding device pointers). */
typedef struct {
  uint8_t* lat_codes;  /* [batch][cap][256] */
  uint8_t* lat_scales; /* [batch][cap][32]  */
  uint8_t* idx_codes;  /* [batch][cap][64]  */
  uint8_t* idx_scales; /* [batch][cap][4]   */
  int32_t* len;        /* [batch] */
  int64_t cap;         /* entries per sequence, multiple of 128 */
  int32_t batch;
} csa2_cache_view;

/*
 * kv_quant_append -- write T source tokens per sequence into the cache.
 *
 * "Le cache KV en FP4", sections "Cache principal" (eq. 288) and "Cles
 * d'indexeur" (eq. 68); "compresse le KV-Cache de 4 fois", item 2 (ratio-2
 * merge with learned per-channel weights).
 *   lat   [batch][T][512], ikey [batch][T][128], dtype ``in_dtype`` (f32 or bf16).
 *   ratio 1: each token becomes an entry. ratio 2: entry i merges tokens 2i and
 *     2i+1 as e = w0*x_{2i} + w1*x_{2i+1} per channel in float32 (two rounded
 *     products, one rounded sum); T must be even. w0_lat/w1_lat [512] and
 *     w0_idx/w1_idx [128] f32, 16-byte aligned, ignored (may be NULL) for ratio 1.
 *   Latent: per 16 channels s = E4M3(amax/6) (nearest-even, saturating at 448),
 *     code = E2M1(x/s) (float32 division, nearest-even, saturating at 6); s = 0
 *     gives all-zero codes. Indexer key: per 32 channels X = floor(log2 amax)-2
 *     clamped to [-127,127], E8M0 byte X+127, code = E2M1(x * 2^-X).
 *   Entries are written at rows len[b] .. len[b]+T/ratio-1, then len[b] grows by
 *   T/ratio. An append past ``cap`` writes nothing for that sequence and records
 *   CSA2_ERR_BOUNDS in the device status word.
 */
CSA2_API csa2_status kv_quant_append(const void* lat, const void* ikey, csa2_dtype in_dtype, int32_t T,
                            int32_t ratio, const float* w0_lat, const float* w1_lat,
                            const float* w0_idx, const float* w1_idx,
                            const csa2_cache_view* cache /* host struct */, csa2_stream_t stream);

/* One source layer of csa2_store_append (host struct holding device pointers). */
typedef struct {
  const void* lat;               /* [batch][T][512] */
  const void* ikey;              /* [batch][T][128] */
  int32_t ratio;                 /* 1 or 2 */
  const float* w0_lat;           /* ratio 2: merge weights as in kv_quant_append */
  const float* w1_lat;
  const float* w0_idx;
  const float* w1_idx;
  const csa2_cache_view* cache;  /* host ptr: this layer's cache */
} csa2_store_layer;

/*
 * csa2_store_append -- write T source tokens into each of up to 8 layers' caches in
 * one launch.
 *
 * "Le cache KV en FP4", section "Le compte par couche" (table and eq. 890): the
 * global cache holds four source layers, 2, 8 and 14 at ratio 2 (178 B per token)
 * and 20 at ratio 1 (356 B per token), 890 B per token in all; "Ce que cela donne
 * aux echelles reelles": 0.87 GiB at 1,048,576 tokens.
 *   layers: host array of n_layers (1..8) descriptors; every cache has the same
 *     batch. Each layer packs exactly as kv_quant_append does with its own ratio
 *     and weights (T even when any layer has ratio 2) and appends T/ratio entries
 *     at its len[b]; an append past a layer's cap writes nothing for that layer and
 *     sequence and records CSA2_ERR_BOUNDS.
 *   Sources and weights 16-byte aligned (CSA2_ERR_ALIGN otherwise).
 */
CSA2_API csa2_status csa2_store_append(const csa2_store_layer* layers, int32_t n_layers, csa2_dtype in_dtype,
                                       int32_t T, csa2_stream_t stream);

/*
 * csa2_swa_quant -- pack sliding-window rows as FP8.
 *
 * "Le cache KV en FP4", section "La contrepartie : la fenetre glissante": each
 * layer keeps its 128-token window in FP8, 512 values plus 512/16 scale bytes per
 * token (40 x 128 x (512 + 512/16) = 2,66 MiB per sequence). The page leaves the
 * scale format open; this library reads it as a power-of-two (E8M0) scale per 16
 * values: X = floor(log2 amax) - 8 clamped to [-127, 127], scale byte X + 127,
 * value codes E4M3(x * 2^-X) (nearest-even, saturating at 448; amax = 0 gives
 * X = -127 and +0 codes).
 *   rows [n_rows][512] (in_dtype f32 or bf16); codes [n_rows][512] u8 (E4M3 fn);
 *   scales [n_rows][32] u8 (E8M0). All 16-byte aligned.
 */
CSA2_API csa2_status csa2_swa_quant(const void* rows, csa2_dtype in_dtype, int64_t n_rows, uint8_t* codes,
                                    uint8_t* scales, csa2_stream_t stream);

/*
 * indexer_score -- score cached entries with the 4-head indexer.
 *
 * "Le cache KV en FP4", section "Les ingredients", item 2 (the 128-channel key
 * scores positions). score_t = sum_h w_h * max(0, q_h . k_t), k_t the
 * dequantised MXFP4 key, accumulated in float32.
 *   q_idx [batch][4][128] (q_dtype), w [batch][4] f32.
 *   idx_codes [batch][cap][64], idx_scales [batch][cap][4], len [batch].
 *   cand == NULL: scores[b][t] for t < len[b] (row stride ``cap``).
 *   cand != NULL: [batch][P] cache positions (-1 = empty slot); scores[b][i] for
 *     i < P (row stride P); empty slots get -inf. A position >= len[b] records
 *     CSA2_ERR_BOUNDS and scores -inf.
 *   scores: f32 output.
 */
CSA2_API csa2_status indexer_score(const void* q_idx, csa2_dtype q_dtype, const float* w,
                          const uint8_t* idx_codes, const uint8_t* idx_scales, int64_t cap,
                          const int32_t* len, const int32_t* cand, int32_t P, float* scores,
                          int32_t batch, csa2_stream_t stream);

/*
 * topk_select -- exact Top-k per sequence.
 *
 * "890 octets de cache KV par token", "Deuxiemement" (new Top-512 indices; a
 * 16,384-position candidate pool). The k largest scores of row b, ties to the
 * lower position (-0 equals +0); with fewer than k valid candidates all are
 * kept. Output positions ascending, padded with -1.
 *   scores [batch][stride] f32; n [batch] valid count per row (NULL: stride).
 *   cand == NULL: candidate i is position i. cand != NULL: [batch][stride]
 *     positions (ascending; -1 = empty slot, skipped).
 *   out_idx [batch][k] i32. 1 <= k <= CSA2_MAX_TOPK.
 *   The selection keeps its state in shared memory: no scratch.
 */
CSA2_API csa2_status topk_select(const float* scores, const int32_t* n, int64_t stride, int32_t k,
                        const int32_t* cand, int32_t* out_idx, int32_t batch, csa2_stream_t stream);

/*
 * sparse_latent_attn -- gather the selected entries, dequantise, attend.
 *
 * "compresse le KV-Cache de 4 fois", item 1: keys and values share one 512-d
 * latent. l_hj = (q_h . v_j) * scale, softmax over the selected entries and the
 * window rows together, o_h = sum_j p_hj v_j, written in float32.
 *   q [batch][H][512] (q_dtype), H in {16, 32, 64}; scale > 0 (1/sqrt(512)).
 *   cache: the main KV (only lat_codes/lat_scales/len/cap are read).
 *   idx [batch][k] positions, -1 skipped; 0 <= k <= CSA2_MAX_TOPK. A position
 *     >= len[b] is skipped and records CSA2_ERR_BOUNDS.
 *   The window ("La contrepartie : la fenetre glissante"; "Troisiemement": 128
 *     tokens): W rows per sequence, either bf16 rows swa [batch][W][512] or FP8
 *     rows swa_codes [batch][W][512] + swa_scales [batch][W][32] (the csa2_swa_quant
 *     format); NULL pointers with W = 0. Window values enter the tensor cores as
 *     fp16: they must lie within its range (|x| <= 65504), and magnitudes below
 *     about 2^-21 are rounded to its grid.
 *   out [batch][H][512] f32. With no key at all the output row is zero.
 *   The partial results of a row stay on chip: no scratch.
 */
CSA2_API csa2_status sparse_latent_attn(const void* q, csa2_dtype q_dtype, int32_t H, float scale,
                               const csa2_cache_view* cache /* host struct */,
                               const int32_t* idx, int32_t k, const uint16_t* swa,
                               const uint8_t* swa_codes, const uint8_t* swa_scales, int32_t W,
                               float* out, csa2_stream_t stream);

/* One layer of a decode step (host struct holding device pointers). */
typedef struct {
  csa2_mode mode;
  const csa2_cache_view* cache;  /* host ptr; FULL: this layer's cache (others: ignored) */
  const uint8_t* own_idx_codes;  /* REINDEX: its own keys [batch][cap][64]; NULL = cache's */
  const uint8_t* own_idx_scales; /* REINDEX: [batch][cap][4] */
  const void* q_idx;             /* FULL/REINDEX: [batch][4][128] */
  const float* w_idx;            /* FULL/REINDEX: [batch][4] */
  int32_t pool;                  /* FULL: 0, or the hierarchical pool size (k < pool) */
  const void* q_idx2;            /* FULL with pool: second indexer [batch][4][128] */
  const float* w_idx2;           /* FULL with pool: [batch][4] */
  const void* q;                 /* [batch][H][512] */
  const uint16_t* swa;           /* [batch][W][512] bf16 window rows, or NULL */
  const uint8_t* swa_codes;      /* or FP8 window rows: [batch][W][512] E4M3 ... */
  const uint8_t* swa_scales;     /* ... and [batch][W][32] E8M0 (csa2_swa_quant); NULL for bf16 */
  int32_t W;                     /* window rows (0 without a window) */
  float* out;                    /* [batch][H][512] f32 */
  int32_t* idx_out;              /* optional [batch][k]: receives the positions attended with */
} csa2_layer_desc;

/*
 * csa2_decode_step -- one decode step through a group of layers.
 *
 * "890 octets de cache KV par token", "Deuxiemement": each layer is Full (own
 * main KV, own indexer, new Top-k), Reindex (external main KV, own rescoring)
 * or Reuse (main KV and indices taken over); the first Full layer may build a
 * hierarchical pool of candidates that deeper indexing scores alone.
 *   FULL: scores all entries of its cache (or, with pool > 0, takes the Top-pool
 *     of that scan and rescores the pool with q_idx2/w_idx2), selects Top-k,
 *     attends over its cache.
 *   REINDEX: scores the keys own_idx_* (or the Full cache's) with its q_idx over
 *     all entries, or over the pool when the Full layer built one; selects
 *     Top-k; attends over the main KV of the latest Full layer.
 *   REUSE: attends with the indices of the latest Full/Reindex layer.
 * The first layer must be FULL. layers is a host array of n_layers descriptors.
 * q, q_idx, q_idx2 share ``dtype``. ws: at least csa2_workspace_size(...) bytes,
 * caller-owned, any contents (every part is written before it is read).
 * Launches only; no host synchronisation inside. The attention of consecutive
 * layers that share the main KV and the window length W is launched together
 * (one launch for up to four layers), so a layer's attention may run after later
 * layers' scans and selections; until then its selection stays in its idx_out or
 * in one of the workspace's two selections. The step reads a layer's q while the
 * Top-k before its attention may still run, so q must not overlap any layer's
 * idx_out or the workspace (inputs and outputs are distinct buffers anyway).
 */
CSA2_API csa2_status csa2_decode_step(const csa2_layer_desc* layers, int32_t n_layers, int32_t batch,
                             int32_t H, int32_t k, csa2_dtype dtype, void* ws, size_t ws_bytes,
                             csa2_stream_t stream);

/*
 * csa2_decode_step_static -- csa2_decode_step without a caller-provided workspace.
 *
 * The pages have no counterpart to this call: it is a convenience of the library.
 * Some callers cannot allocate device memory at the point where they run a decode
 * step: a host program without a device allocator of its own, a plug-in that
 * must not touch the allocator of the framework that hosts it, or a serving loop
 * that forbids allocation after start-up. This entry point runs the same step
 * (same arguments and results as csa2_decode_step) with its scratch in an array
 * of CSA2_STATIC_WS_BYTES (24 MiB) compiled into the library; it allocates and
 * frees nothing. The caller still owns every input and output.
 *   - A step that needs more than CSA2_STATIC_WS_BYTES of scratch
 *     (csa2_workspace_size() > CSA2_STATIC_WS_BYTES; for instance more than
 *     about six million cached entries over the batch) is rejected with
 *     CSA2_ERR_WORKSPACE and launches nothing.
 *   - Every device that loads the library keeps the array until the process
 *     exits. The first call on a device (with that device current) looks the
 *     array up with cudaGetSymbolAddress; make that first call before any stream
 *     capture on the device.
 *   - All calls share the one array: calls that may overlap on the GPU (other
 *     streams, other host threads) race on it and must be serialised by the
 *     caller. Nothing in it needs to start at zero; it keeps the last call's
 *     contents.
 *   - The array's address is looked up once per device ordinal and kept: after
 *     cudaDeviceReset (or any other teardown of the device's primary context) in
 *     the same process that address is stale, so this call is not supported
 *     after such a reset.
 */
CSA2_API csa2_status csa2_decode_step_static(const csa2_layer_desc* layers, int32_t n_layers, int32_t batch,
                                             int32_t H, int32_t k, csa2_dtype dtype, csa2_stream_t stream);

/* Scratch bytes of csa2_decode_step for these sizes (max_entries = cap): scores
 * [batch][max_entries] f32, pool positions and scores [batch][pool], two
 * selections [batch][k]. */
CSA2_API size_t csa2_workspace_size(int32_t batch, int64_t max_entries, int32_t H, int32_t k, int32_t pool,
                           int32_t W);

/* Synchronise ``stream``, return and clear the device status word
 * (CSA2_OK, CSA2_ERR_BOUNDS, CSA2_ERR_TIMEOUT), or CSA2_ERR_CUDA. */
CSA2_API csa2_status csa2_sync_status(csa2_stream_t stream);

/* Static description of a status code (never NULL). */
CSA2_API const char* csa2_status_str(csa2_status status);

/* Number of kernels this library launched since load (host counter). */
CSA2_API uint64_t csa2_launch_count(void);

/*
 * csa2_set_scan_events -- measurement hook for the dominant kernel.
 *
 * Not an operation of the method: lets a benchmark time the streaming indexer
 * scans inside indexer_score and csa2_decode_step. ``before``/``after`` are host
 * arrays of n cudaEvent_t handles (0 <= n <= 64; n = 0 turns the hook off). Later
 * calls made from this host thread record, around the i-th streaming scan launch
 * since the hook was set, before[i mod n] right before it and after[i mod n] right
 * after it, on the launch's stream (as external event nodes while the stream is
 * being captured into a CUDA graph). The caller owns the events and keeps them
 * alive while the hook is set. CSA2_ERR_ARG for n out of range or a NULL handle.
 */
CSA2_API csa2_status csa2_set_scan_events(void* const* before, void* const* after, int32_t n);

/*
 * csa2_selftest_wait_timeout -- test hook for the failure detection.
 *
 * Not an operation of the method (the pages have no counterpart). Launches one
 * block on ``stream`` in which one thread waits, with the same bounded mbarrier
 * wait as the streaming kernels but a limit of ``budget_ns`` nanoseconds, on a
 * barrier that nothing ever arrives at. The wait runs out, records
 * CSA2_ERR_TIMEOUT in the device status word and the kernel returns; the next
 * csa2_sync_status() on that stream reports it (and clears it). Nothing faults,
 * traps or hangs. budget_ns <= 1e9, else CSA2_ERR_ARG; CSA2_ERR_CUDA if the
 * launch fails.
 */
CSA2_API csa2_status csa2_selftest_wait_timeout(uint64_t budget_ns, csa2_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H */
