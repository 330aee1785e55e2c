"""CPU oracle of the CSA2 FP4 compressed-KV decode path.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``
(its ``cpu_baseline`` leg and its ``--impl reference`` arm) may import this
module. It shares no code with the CUDA path and imports nothing from it.

Each function states the passage of the pages it follows. Pages are cited by
title and section:

* [FP4]   "Le cache KV en FP4 -- les 890 octets, verifies" (mkdocs.reaper.mx),
          sections "Les ingredients", "Cache principal" (eq. 288),
          "Cles d'indexeur" (eq. 68), "D'ou viennent ces deux reglages",
          "Le compte par couche" (table and eq. 890), "Ce que cela donne aux
          echelles reelles" (table), "La contrepartie : la fenetre glissante".
* [CTX]   "DeepSeek V4.1 Flash : 890 octets de cache KV par token"
          (contextstudios.ai), section "L'architecture : trois leviers",
          paragraphs "Deuxiemement" (CSA2 modes, Top-512, 16,384-candidate HSI)
          and "Troisiemement" (E2M1 with E4M3 per 16 channels, 128-token window).
* [TF24]  "DeepSeek-V4.1 Flash compresse le KV-Cache de 4 fois" (techfi24.com),
          section "Mecanismes de compression", items 1-3.
* [F24]   "KV cache da 890 byte per token" (flash24.org), section
          "Tre meccanismi", second and third paragraphs.

The pages give no formula for the indexer score, the attention scale, the
tie rule or the merge arithmetic. Each function states the reading it takes
where the pages are silent: the merge is two rounded float32 products and one
rounded sum; the score is sum_h w_h * max(0, q_h . k) over 4 indexer heads; ties
in the Top-k go to the lower position and the output is ascending; attention
is scaled by 1/sqrt(512) and the window rows join the selected entries in one
softmax.

Floating point: quantisation decisions are taken in IEEE float32, the precision
of the quantiser's inputs (numpy float32 arithmetic rounds each operation to
nearest, with no fused multiply-add). Scores and attention are computed in
float64.
"""
from __future__ import annotations

import math

import numpy as np

from . import formats as F

LATENT_DIM = 512          # [FP4] "Les ingredients", item 1: 512-channel latent
INDEXER_DIM = 128         # [FP4] "Les ingredients", item 2: 128-channel indexer key
MAIN_BLOCK = 16           # [FP4] "Cache principal": one E4M3 scale per 16 channels
INDEXER_BLOCK = 32        # [FP4] "Cles d'indexeur": one E8M0 scale per 32 channels
MAIN_CODE_BYTES = LATENT_DIM // 2                  # 256
MAIN_SCALE_BYTES = LATENT_DIM // MAIN_BLOCK        # 32
IDX_CODE_BYTES = INDEXER_DIM // 2                  # 64
IDX_SCALE_BYTES = INDEXER_DIM // INDEXER_BLOCK     # 4
TOPK = 512                # [CTX] "Deuxiemement": new Top-512 indices
HSI_POOL = 16384          # [CTX] "Deuxiemement": candidates limited to 16,384 positions
SWA_WINDOW = 128          # [CTX] "Troisiemement": 128-token sliding window
SWA_BLOCK = 16            # [FP4] "La contrepartie": 512/16 scale bytes per FP8 window token
E4M3_EMAX = 8             # largest E4M3 exponent: 448 = 1.75 * 2**8


# =========================================================== a1: ratio-2 merge
def merge_ratio2(x_even: np.ndarray, x_odd: np.ndarray, w0: np.ndarray, w1: np.ndarray) -> np.ndarray:
    """Merge two consecutive positions into one cache entry with per-channel weights.

    [TF24] item 2 and [FP4] "Le compte par couche": a ratio-m layer stores one
    entry per m tokens; the encoder merges two consecutive positions with learned
    per-channel weights. Reading: e[c] = w0[c]*x_{2i}[c] + w1[c]*x_{2i+1}[c],
    evaluated in float32 as two rounded products and one rounded sum.
    """
    x0 = np.asarray(x_even, dtype=np.float32)
    x1 = np.asarray(x_odd, dtype=np.float32)
    p0 = np.multiply(x0, np.asarray(w0, dtype=np.float32), dtype=np.float32)
    p1 = np.multiply(x1, np.asarray(w1, dtype=np.float32), dtype=np.float32)
    return np.add(p0, p1, dtype=np.float32)


# ===================================================== a2: main-KV quantisation
def quantize_main(x: np.ndarray):
    """Quantise latents [n, 512] to E2M1 codes with one E4M3 scale per 16 channels.

    [FP4] "Cache principal" (eq. 288) and "D'ou viennent ces deux reglages" (the
    quantiser is called with block 16 and an E4M3 scale dtype); [CTX]
    "Troisiemement" (E2M1, one E4M3 scale per 16 channels).
    Reading, per 16-channel block, in float32:
      amax = max |x|;  s = E4M3(amax / 6) (nearest, ties even, saturating at 448);
      if s == 0 every code is +0, else code_c = E2M1(x_c / s) (float32 division).
    Returns (codes [n, 512] uint8 0..15, scale codes [n, 32] uint8).
    """
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[0]
    blocks = x.reshape(n, LATENT_DIM // MAIN_BLOCK, MAIN_BLOCK)
    amax = np.abs(blocks).max(axis=-1)                                   # float32
    ratio = np.divide(amax, np.float32(6.0), dtype=np.float32)          # fl32(amax/6)
    s_code = F.e4m3_encode(ratio)
    s_val = F.e4m3_decode(s_code).astype(np.float32)                     # exact
    safe = np.where(s_val == 0, np.float32(1.0), s_val).astype(np.float32)
    q = np.divide(blocks, safe[..., None], dtype=np.float32)            # fl32(x/s)
    codes = F.e2m1_encode(q)
    codes = np.where((s_val == 0)[..., None], np.uint8(0), codes).astype(np.uint8)
    return codes.reshape(n, LATENT_DIM), s_code


def dequantize_main(codes: np.ndarray, s_code: np.ndarray) -> np.ndarray:
    """E2M1 codes [n, 512] and E4M3 scales [n, 32] -> float64 latents (exact)."""
    n = codes.shape[0]
    v = F.e2m1_decode(codes).reshape(n, LATENT_DIM // MAIN_BLOCK, MAIN_BLOCK)
    s = F.e4m3_decode(s_code)
    return (v * s[..., None]).reshape(n, LATENT_DIM)


# ================================================ a3: indexer-key quantisation
def indexer_shared_exponent(amax: np.ndarray) -> np.ndarray:
    """MX shared exponent X of a 32-channel block: floor(log2 amax) - 2, clamped to [-127, 127].

    [FP4] "Cles d'indexeur": 128 channels, E2M1, one E8M0 scale per 32 channels,
    "le MXFP4 standard". Reading: the OCP MX conversion, whose shared exponent is
    floor(log2(amax)) minus the largest exponent of E2M1 (2). amax = 0 gives -127.
    """
    amax = np.asarray(amax, dtype=np.float64)
    pos = amax > 0
    x = np.where(pos, F.floor_log2(np.where(pos, amax, 1.0)) - 2, -127)
    return np.clip(x, -127, 127).astype(np.int64)


def quantize_indexer(x: np.ndarray):
    """Quantise indexer keys [n, 128] to MXFP4: E2M1 codes, one E8M0 scale per 32 channels.

    Per block: X = indexer_shared_exponent(amax), e8m0 = X + 127,
    code_c = E2M1(x_c * 2**-X) (the scaling by a power of two is exact; values
    above 6 saturate, as in the MX conversion).
    Returns (codes [n, 128] uint8, e8m0 [n, 4] uint8).
    """
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[0]
    blocks = x.reshape(n, INDEXER_DIM // INDEXER_BLOCK, INDEXER_BLOCK).astype(np.float64)
    amax = np.abs(blocks).max(axis=-1)
    X = indexer_shared_exponent(amax)
    scaled = np.ldexp(blocks, -X[..., None])
    codes = F.e2m1_encode(scaled).reshape(n, INDEXER_DIM)
    return codes, (X + 127).astype(np.uint8)


def dequantize_indexer(codes: np.ndarray, e8m0: np.ndarray) -> np.ndarray:
    """MXFP4 codes [n, 128] and E8M0 scales [n, 4] -> float64 keys (exact)."""
    n = codes.shape[0]
    v = F.e2m1_decode(codes).reshape(n, INDEXER_DIM // INDEXER_BLOCK, INDEXER_BLOCK)
    return (v * F.e8m0_decode(e8m0)[..., None]).reshape(n, INDEXER_DIM)


# ===================================================== packing (two codes/byte)
def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Pack 4-bit codes two per byte: channel 2j in the low nibble, 2j+1 in the high one.

    The pages fix 4 bits per channel ([FP4] eq. 288: 512 x 4/8 bytes) but not the
    nibble order; the reading is low nibble first.
    """
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 15
    out[..., 1::2] = p >> 4
    return out


# ============================================== the cache and the append step
class Cache:
    """One layer's global cache for a batch of sequences, in host memory.

    [FP4] "Les ingredients": the global cache holds the main KV (512-channel
    latent) and the indexer keys (128 channels), nothing else. Per entry:
    256 B of latent codes + 32 B of E4M3 scales (eq. 288) and 64 B of indexer
    codes + 4 B of E8M0 scales (eq. 68). Struct-of-arrays, one row per entry.
    """

    def __init__(self, batch: int, cap: int):
        self.batch, self.cap = batch, cap
        self.lat_codes = np.zeros((batch, cap, MAIN_CODE_BYTES), np.uint8)
        self.lat_scales = np.zeros((batch, cap, MAIN_SCALE_BYTES), np.uint8)
        self.idx_codes = np.zeros((batch, cap, IDX_CODE_BYTES), np.uint8)
        self.idx_scales = np.zeros((batch, cap, IDX_SCALE_BYTES), np.uint8)
        self.len = np.zeros(batch, np.int64)


def encode_entries(lat: np.ndarray, ikey: np.ndarray, ratio: int,
                   w0_lat=None, w1_lat=None, w0_idx=None, w1_idx=None):
    """Turn T source tokens [T, 512] / [T, 128] into T/ratio packed entries.

    ratio 1: every token is an entry. ratio 2: consecutive pairs are merged first
    (merge_ratio2, separate weight vectors for the latent and the indexer key).
    Reading: T must be even for ratio 2 (a lone trailing token is not cached).
    Returns (lat_codes [n,256], lat_scales [n,32], idx_codes [n,64], idx_scales [n,4]).
    """
    lat = np.asarray(lat, dtype=np.float32)
    ikey = np.asarray(ikey, dtype=np.float32)
    if ratio == 2:
        if lat.shape[0] % 2:
            raise ValueError("ratio 2 needs an even number of tokens")
        lat = merge_ratio2(lat[0::2], lat[1::2], w0_lat, w1_lat)
        ikey = merge_ratio2(ikey[0::2], ikey[1::2], w0_idx, w1_idx)
    elif ratio != 1:
        raise ValueError("ratio must be 1 or 2")
    lc, ls = quantize_main(lat)
    ic, iscale = quantize_indexer(ikey)
    return pack_nibbles(lc), ls, pack_nibbles(ic), iscale


def append(cache: Cache, lat: np.ndarray, ikey: np.ndarray, ratio: int,
           w0_lat=None, w1_lat=None, w0_idx=None, w1_idx=None) -> None:
    """Append T tokens per sequence (lat [B, T, 512], ikey [B, T, 128]) at each len[b]."""
    for b in range(cache.batch):
        lc, ls, ic, isc = encode_entries(lat[b], ikey[b], ratio, w0_lat, w1_lat, w0_idx, w1_idx)
        n0, n = int(cache.len[b]), lc.shape[0]
        if n0 + n > cache.cap:
            raise ValueError("append past capacity")
        cache.lat_codes[b, n0:n0 + n] = lc
        cache.lat_scales[b, n0:n0 + n] = ls
        cache.idx_codes[b, n0:n0 + n] = ic
        cache.idx_scales[b, n0:n0 + n] = isc
        cache.len[b] = n0 + n


def entry_latents(lat_codes: np.ndarray, lat_scales: np.ndarray) -> np.ndarray:
    """Packed latent rows [n,256] + scales [n,32] -> float64 [n, 512]."""
    return dequantize_main(unpack_nibbles(lat_codes), lat_scales)


def entry_keys(idx_codes: np.ndarray, idx_scales: np.ndarray) -> np.ndarray:
    """Packed indexer rows [n,64] + scales [n,4] -> float64 [n, 128]."""
    return dequantize_indexer(unpack_nibbles(idx_codes), idx_scales)


# ===================================================== b1: indexer scoring
def indexer_scores(q_idx: np.ndarray, w: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """Score cached entries with the multi-head indexer, in float64.

    [FP4] "Les ingredients", item 2: the 128-channel indexer key is used to score
    positions. The score formula is not on the pages; the reading is
    score_t = sum_h w_h * max(0, q_h . k_t) over 4 indexer heads.
    q_idx [H_idx, 128], w [H_idx], keys [n, 128] (float64) -> scores [n].
    """
    q = np.asarray(q_idx, dtype=np.float64)
    dots = keys @ q.T                                   # [n, H_idx]
    return np.maximum(dots, 0.0) @ np.asarray(w, dtype=np.float64)


# ===================================================== c1: Top-k selection
def topk_positions(scores: np.ndarray, k: int, positions: np.ndarray | None = None) -> np.ndarray:
    """Exact Top-k: the k largest scores, ties to the lower position, output ascending.

    [CTX] "Deuxiemement": each Full layer selects new Top-512 indices. Readings:
    ties go to the lower position; with fewer than k candidates all of them are
    kept; the output lists positions in ascending order, padded with -1 to k.
    ``positions`` maps candidate i to its cache position (default: i).
    """
    s = np.asarray(scores, dtype=np.float64)
    pos = np.arange(s.shape[0]) if positions is None else np.asarray(positions, dtype=np.int64)
    order = np.lexsort((pos, -s))                        # score desc, then position asc
    chosen = np.sort(pos[order[:k]])
    out = np.full(k, -1, dtype=np.int64)
    out[:chosen.shape[0]] = chosen
    return out


# ===================================================== b2: hierarchical indexer
def hsi_select(keys: np.ndarray, q1: np.ndarray, w1: np.ndarray, q2: np.ndarray, w2: np.ndarray,
               pool: int = HSI_POOL, k: int = TOPK):
    """Hierarchical Sparse Indexer: pool by the first indexer, then rescore the pool.

    [CTX] "Deuxiemement" and [F24] second paragraph: the first Full layer builds a
    pool of 16,384 candidate positions; deeper indexing scores only the pool.
    Reading: the pool is the exact Top-16,384 of indexer 1 over all entries; a
    second indexer (own query and weights, the same keys) rescores the pool; the
    Top-512 of those scores, ties to the lower position, is the selection.
    Returns (selection [k], pool [pool]) as positions, -1 padded.
    """
    s1 = indexer_scores(q1, w1, keys)
    pool_pos = topk_positions(s1, pool)
    valid = pool_pos[pool_pos >= 0]
    s2 = indexer_scores(q2, w2, keys[valid])
    return topk_positions(s2, k, positions=valid), pool_pos


# ===================================================== d1/d2: sparse attention
def sparse_attention(q: np.ndarray, values: np.ndarray, scale: float | None = None) -> np.ndarray:
    """Multi-head attention in which each key is also its value, in float64.

    [TF24] item 1: one 512-dimensional latent is shared by keys and values.
    Reading: logits l_hj = (q_h . v_j) * scale with scale = 1/sqrt(512), softmax
    over j (maximum subtracted), o_h = sum_j p_hj v_j. No keys -> zeros.
    q [H, 512], values [m, 512] -> o [H, 512].
    """
    q = np.asarray(q, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(LATENT_DIM)
    if v.shape[0] == 0:
        return np.zeros((q.shape[0], v.shape[1] if v.ndim == 2 else LATENT_DIM))
    logits = (q @ v.T) * scale
    logits = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    return (p @ v) / p.sum(axis=1, keepdims=True)


def attend(q: np.ndarray, lat_codes: np.ndarray, lat_scales: np.ndarray, idx: np.ndarray,
           swa: np.ndarray | None = None, scale: float | None = None) -> np.ndarray:
    """Gather the selected entries of one sequence, dequantise, attend.

    idx [k] positions (-1 entries skipped). swa: optional [W, 512] float values of
    the sliding window ([FP4] "La contrepartie"; [CTX] "Troisiemement": a
    128-token window kept outside the global cache). Reading: the window rows are
    extra keys/values in the same softmax as the selected entries.
    """
    sel = np.asarray(idx)
    sel = sel[sel >= 0]
    v = entry_latents(lat_codes[sel], lat_scales[sel])
    if swa is not None and len(swa):
        v = np.concatenate([v, np.asarray(swa, dtype=np.float64)], axis=0)
    return sparse_attention(q, v, scale)


# ===================================================== e1: one decode step
FULL, REINDEX, REUSE = 0, 1, 2


def decode_step(layers, k: int = TOPK):
    """Run a group of layers for every sequence of a batch.

    [CTX] "Deuxiemement": each CSA2 layer is statically Full (own main KV, own
    indexer, new Top-512), Reindex (external main KV, own rescoring) or Reuse
    (main KV and indices taken over). [F24]: layers share the main KV and the
    indexer key, and sparse indices are reused.

    ``layers`` is a list of dicts with keys:
      mode (FULL/REINDEX/REUSE); cache (Cache: main KV, and for FULL the keys);
      keys_codes/keys_scales ([B,cap,64]/[B,cap,4], optional for REINDEX: its own
      keys; default the cache's); q_idx [B,Hi,128]; w_idx [B,Hi];
      pool (0 or pool size, FULL only), q_idx2/w_idx2 (second indexer, when pool);
      q [B,H,512]; swa [B,W,512] or None.
    Readings: REUSE takes the indices of the most recent FULL/REINDEX layer; a
    REINDEX layer attends over the main KV of the most recent FULL layer; when a
    FULL layer built a pool, a later REINDEX layer scores only that pool.
    Returns (outputs: list of [B,H,512], indices: list of [B,k]).
    """
    outs, idxs = [], []
    last_idx = None
    main = None
    pool = None
    for L in layers:
        mode = L["mode"]
        if mode == FULL:
            main = L["cache"]
        elif main is None:
            raise ValueError("the first layer of a group must be FULL")
        B = main.batch
        if mode in (FULL, REINDEX):
            kc = L.get("keys_codes")
            ks = L.get("keys_scales")
            if kc is None:
                kc, ks = main.idx_codes, main.idx_scales
            sel = np.full((B, k), -1, np.int64)
            new_pool = []
            for b in range(B):
                n = int(main.len[b])
                keys = entry_keys(kc[b, :n], ks[b, :n])
                if mode == FULL and L.get("pool", 0):
                    s_b, p_b = hsi_select(keys, L["q_idx"][b], L["w_idx"][b],
                                          L["q_idx2"][b], L["w_idx2"][b], L["pool"], k)
                    sel[b] = s_b
                    new_pool.append(p_b)
                elif mode == REINDEX and pool is not None:
                    pv = pool[b][pool[b] >= 0]
                    s = indexer_scores(L["q_idx"][b], L["w_idx"][b], keys[pv])
                    sel[b] = topk_positions(s, k, positions=pv)
                else:
                    s = indexer_scores(L["q_idx"][b], L["w_idx"][b], keys)
                    sel[b] = topk_positions(s, k)
            if mode == FULL:
                pool = new_pool if new_pool else None
            last_idx = sel
        if last_idx is None:
            raise ValueError("REUSE needs an earlier FULL or REINDEX layer")
        H = L["q"].shape[1]
        out = np.zeros((B, H, LATENT_DIM))
        for b in range(B):
            swa = None if L.get("swa") is None else L["swa"][b]
            out[b] = attend(L["q"][b], main.lat_codes[b], main.lat_scales[b], last_idx[b], swa)
        outs.append(out)
        idxs.append(last_idx.copy())
    return outs, idxs


# ===================================================== FP8 sliding-window rows
def quantize_swa(x: np.ndarray):
    """Quantise window rows [n, 512] to FP8: E4M3 values with one scale byte per 16.

    [FP4] "La contrepartie : la fenetre glissante": every layer keeps its 128-token
    window in FP8, 512 values plus 512/16 scale bytes per token (eq. 2,66 Mio). The
    page leaves the scale format open. Reading: a power-of-two E8M0 scale per 16
    values, as in the MX conversion: X = floor(log2 amax) - 8 (the largest E4M3
    exponent), clamped to [-127, 127]; byte X + 127; value code = E4M3(x * 2**-X),
    nearest-even, saturating at 448. amax = 0 gives X = -127 and +0 codes.
    Returns (codes [n, 512] uint8, e8m0 [n, 32] uint8).
    """
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[0]
    blocks = x.reshape(n, LATENT_DIM // SWA_BLOCK, SWA_BLOCK).astype(np.float64)
    amax = np.abs(blocks).max(axis=-1)
    pos = amax > 0
    X = np.where(pos, F.floor_log2(np.where(pos, amax, 1.0)) - E4M3_EMAX, -127)
    X = np.clip(X, -127, 127).astype(np.int64)
    codes = F.e4m3_encode(np.ldexp(blocks, -X[..., None])).reshape(n, LATENT_DIM)
    return codes.astype(np.uint8), (X + 127).astype(np.uint8)


def dequantize_swa(codes: np.ndarray, e8m0: np.ndarray) -> np.ndarray:
    """FP8 window rows (E4M3 codes [n, 512], E8M0 scales [n, 32]) -> float64 [n, 512] (exact)."""
    n = codes.shape[0]
    v = F.e4m3_decode(codes).reshape(n, LATENT_DIM // SWA_BLOCK, SWA_BLOCK)
    return (v * F.e8m0_decode(e8m0)[..., None]).reshape(n, LATENT_DIM)


# ===================================================== multi-layer store
def store_entries(layer_sources, layers=None, weights=None):
    """Pack T source tokens into the global cache of every source layer.

    [FP4] "Le compte par couche": the global cache holds four source layers, 2, 8 and
    14 at ratio 2 and 20 at ratio 1; a ratio-m layer stores one entry per m tokens.
    ``layer_sources`` is a list of (lat [T, 512], ikey [T, 128]) per layer, ``layers``
    the (number, zone, ratio) rows (default SOURCE_LAYERS) and ``weights`` the merge
    weights (w0_lat, w1_lat, w0_idx, w1_idx) of each ratio-2 layer (None for ratio 1).
    Returns one (lat_codes, lat_scales, idx_codes, idx_scales) tuple per layer.
    """
    layers = SOURCE_LAYERS if layers is None else layers
    weights = [None] * len(layers) if weights is None else weights
    out = []
    for (lat, ikey), (_, _, ratio), w in zip(layer_sources, layers, weights):
        out.append(encode_entries(lat, ikey, ratio, *(w if w is not None else [None] * 4)))
    return out


# ===================================================== footprint arithmetic
def entry_bytes(channels: int, block: int, bits: int = 4, scale_bytes: int = 1) -> float:
    """Bytes of one cache entry: channels*bits/8 of codes + one scale per block.

    [FP4] eq. 288 (512 ch, block 16, E4M3 scale) and eq. 68 (128 ch, block 32, E8M0).
    block=None means no scales.
    """
    data = channels * bits / 8
    return data + (0 if block is None else channels / block * scale_bytes)


#: [FP4] "Le compte par couche": the four source layers of the global cache
SOURCE_LAYERS = ((2, "encodeur", 2), (8, "encodeur", 2), (14, "encodeur", 2), (20, "decodeur", 1))


def bytes_per_token(main_block=MAIN_BLOCK, idx_block=INDEXER_BLOCK, layers=SOURCE_LAYERS) -> float:
    """Global-cache bytes per token: sum over source layers of (main + indexer) / ratio.

    [FP4] "Le compte par couche": a ratio-m layer stores one entry per m tokens.
    """
    per_entry = entry_bytes(LATENT_DIM, main_block) + entry_bytes(INDEXER_DIM, idx_block)
    return sum(per_entry / ratio for _, _, ratio in layers)


def swa_bytes_per_sequence(layers: int = 40, window: int = SWA_WINDOW, dim: int = LATENT_DIM,
                           block: int = 16) -> float:
    """[FP4] "La contrepartie": each of 40 layers keeps 128 tokens of 512 FP8 values
    plus one 1-byte scale per 16 values."""
    return layers * window * (dim + dim / block)
