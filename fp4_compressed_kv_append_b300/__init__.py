"""CSA2 FP4 compressed-KV decode path on B300 (sm_103a).

Thin torch-facing binding of the C ABI in ``include/csa2.h`` (libcsa2.so). Every
function here only marshals arguments (device pointers, sizes, the current CUDA
stream) and calls the library of the same name; all computation runs in the
library's CUDA kernels. torch provides device memory and streams.
"""
from __future__ import annotations

import ctypes as C
import math

import torch

from . import _abi as A
from ._abi import Csa2Error, FULL, REINDEX, REUSE  # noqa: F401

LATENT_DIM, INDEXER_DIM, INDEXER_HEADS = A.LATENT_DIM, A.INDEXER_DIM, A.INDEXER_HEADS
DEFAULT_SCALE = 1.0 / math.sqrt(LATENT_DIM)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return A.F32
    if t.dtype == torch.bfloat16:
        return A.BF16
    raise TypeError(f"expected float32 or bfloat16, got {t.dtype}")


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


class Cache:
    """One layer's global cache: SoA device arrays (see include/csa2.h).

    lat_codes [B, cap, 256] u8, lat_scales [B, cap, 32] u8, idx_codes [B, cap, 64] u8,
    idx_scales [B, cap, 4] u8, len [B] int32. ``cap`` is a multiple of 128.
    """

    def __init__(self, batch: int, cap: int, device="cuda"):
        if cap % 128:
            raise ValueError("cap must be a multiple of 128")
        self.batch, self.cap = batch, cap
        u8 = dict(dtype=torch.uint8, device=device)
        self.lat_codes = torch.zeros(batch, cap, 256, **u8)
        self.lat_scales = torch.zeros(batch, cap, 32, **u8)
        self.idx_codes = torch.zeros(batch, cap, 64, **u8)
        self.idx_scales = torch.zeros(batch, cap, 4, **u8)
        self.len = torch.zeros(batch, dtype=torch.int32, device=device)
        self._view = None

    def view(self) -> A.CacheView:
        if self._view is None:
            self._view = A.CacheView(self.lat_codes.data_ptr(), self.lat_scales.data_ptr(),
                                     self.idx_codes.data_ptr(), self.idx_scales.data_ptr(),
                                     self.len.data_ptr(), self.cap, self.batch)
        return self._view


def kv_quant_append(lat, ikey, ratio: int, cache: Cache, w0_lat=None, w1_lat=None, w0_idx=None, w1_idx=None,
                    stream=None) -> None:
    """Append T tokens per sequence (lat [B,T,512], ikey [B,T,128]; f32 or bf16)."""
    _contig(lat, ikey, w0_lat, w1_lat, w0_idx, w1_idx)
    A.check(A.lib().kv_quant_append(_ptr(lat), _ptr(ikey), _dt(lat), lat.shape[1], ratio, _ptr(w0_lat),
                                    _ptr(w1_lat), _ptr(w0_idx), _ptr(w1_idx), C.byref(cache.view()),
                                    _stream(stream)), "kv_quant_append")


def indexer_score(q_idx, w, idx_codes, idx_scales, length, scores=None, cand=None, stream=None):
    """scores [B, cap] (or [B, P] with cand [B, P]) of the 4-head indexer."""
    _contig(q_idx, w, idx_codes, idx_scales, length, cand)
    B, cap = idx_codes.shape[0], idx_codes.shape[1]
    P = 0 if cand is None else cand.shape[1]
    if scores is None:
        scores = torch.empty(B, P if cand is not None else cap, dtype=torch.float32, device=idx_codes.device)
    A.check(A.lib().indexer_score(_ptr(q_idx), _dt(q_idx), _ptr(w), _ptr(idx_codes), _ptr(idx_scales), cap,
                                  _ptr(length), _ptr(cand), P, _ptr(scores), B, _stream(stream)), "indexer_score")
    return scores


def topk_select(scores, k: int, n=None, out=None, cand=None, stream=None):
    """Exact Top-k positions per row, ascending, -1 padded: out [B, k] int32."""
    _contig(scores, n, cand)
    B, stride = scores.shape
    if out is None:
        out = torch.empty(B, k, dtype=torch.int32, device=scores.device)
    A.check(A.lib().topk_select(_ptr(scores), _ptr(n), stride, k, _ptr(cand), _ptr(out), B, _stream(stream)),
            "topk_select")
    return out


def _window(swa):
    """(bf16 rows, FP8 codes, FP8 scales, W) of a window: a bf16 tensor [B, W, 512], or the
    (codes [B, W, 512], scales [B, W, 32]) uint8 pair of swa_quant, or None."""
    if swa is None:
        return None, None, None, 0
    if isinstance(swa, (tuple, list)):
        codes, scales = swa
        _contig(codes, scales)
        return None, codes, scales, codes.shape[1]
    _contig(swa)
    return swa, None, None, swa.shape[1]


def swa_quant(rows, stream=None):
    """FP8 window rows of rows [..., 512] (f32 or bf16): (codes [..., 512], scales [..., 32]) uint8."""
    _contig(rows)
    n = rows.numel() // LATENT_DIM
    codes = torch.empty(rows.shape, dtype=torch.uint8, device=rows.device)
    scales = torch.empty(rows.shape[:-1] + (LATENT_DIM // 16,), dtype=torch.uint8, device=rows.device)
    A.check(A.lib().csa2_swa_quant(_ptr(rows), _dt(rows), n, _ptr(codes), _ptr(scales), _stream(stream)),
            "csa2_swa_quant")
    return codes, scales


def store_append(layers, stream=None) -> None:
    """Append T tokens to every layer of a store in one launch. ``layers`` is a list of
    (lat [B,T,512], ikey [B,T,128], ratio, cache, weights) with weights (w0_lat, w1_lat,
    w0_idx, w1_idx) for ratio 2 (None for ratio 1); sources share one dtype."""
    descs = (A.StoreLayer * len(layers))()
    keep = []
    for d, (lat, ikey, ratio, cache, w) in zip(descs, layers):
        w = w or (None,) * 4
        _contig(lat, ikey, *w)
        view = cache.view()
        keep.append(view)
        d.lat, d.ikey, d.ratio = _ptr(lat), _ptr(ikey), ratio
        d.w0_lat, d.w1_lat, d.w0_idx, d.w1_idx = (_ptr(x) for x in w)
        d.cache = C.pointer(view)
    lat0 = layers[0][0]
    A.check(A.lib().csa2_store_append(descs, len(layers), _dt(lat0), lat0.shape[1], _stream(stream)),
            "csa2_store_append")


def sparse_latent_attn(q, cache: Cache, idx, out=None, swa=None, scale: float = DEFAULT_SCALE, stream=None):
    """o [B, H, 512] f32 from q [B, H, 512], selected positions idx [B, k] and the window
    swa (bf16 rows [B, W, 512] or the FP8 (codes, scales) pair of swa_quant)."""
    _contig(q, idx, out)
    B, H, _ = q.shape
    k = 0 if idx is None else idx.shape[1]
    bf, codes, scales, W = _window(swa)
    if out is None:
        out = torch.empty(B, H, LATENT_DIM, dtype=torch.float32, device=q.device)
    A.check(A.lib().sparse_latent_attn(_ptr(q), _dt(q), H, scale, C.byref(cache.view()), _ptr(idx), k, _ptr(bf),
                                       _ptr(codes), _ptr(scales), W, _ptr(out), _stream(stream)),
            "sparse_latent_attn")
    return out


class Layer:
    """One layer of a decode step (fields as in csa2_layer_desc)."""

    def __init__(self, mode, q, out, cache: Cache | None = None, q_idx=None, w_idx=None, own_idx_codes=None,
                 own_idx_scales=None, pool: int = 0, q_idx2=None, w_idx2=None, swa=None, idx_out=None):
        self.mode, self.q, self.out, self.cache = mode, q, out, cache
        self.q_idx, self.w_idx = q_idx, w_idx
        self.own_idx_codes, self.own_idx_scales = own_idx_codes, own_idx_scales
        self.pool, self.q_idx2, self.w_idx2, self.swa = pool, q_idx2, w_idx2, swa
        self.idx_out = idx_out

    def desc(self) -> A.LayerDesc:
        _contig(self.q, self.out, self.q_idx, self.w_idx, self.q_idx2, self.w_idx2)
        cache_ptr = C.pointer(self.cache.view()) if self.cache is not None else None
        bf, codes, scales, W = _window(self.swa)
        return A.LayerDesc(self.mode, cache_ptr, _ptr(self.own_idx_codes), _ptr(self.own_idx_scales),
                           _ptr(self.q_idx), _ptr(self.w_idx), self.pool, _ptr(self.q_idx2), _ptr(self.w_idx2),
                           _ptr(self.q), _ptr(bf), _ptr(codes), _ptr(scales), W, _ptr(self.out), _ptr(self.idx_out))


def workspace_size(batch: int, max_entries: int, H: int, k: int = 512, pool: int = 0, W: int = 0) -> int:
    return A.lib().csa2_workspace_size(batch, max_entries, H, k, pool, W)


class DecodeStep:
    """A prepared decode step: the layer descriptors are built once, each call only launches."""

    def __init__(self, layers, k: int = 512, ws=None):
        self.layers = list(layers)
        self.k = k
        first = self.layers[0]
        B, H = first.q.shape[0], first.q.shape[1]
        self.B, self.H, self.dtype = B, H, _dt(first.q)
        cap = max(L.cache.cap for L in self.layers if L.cache is not None)
        pool = max(L.pool for L in self.layers)
        W = max(_window(L.swa)[3] for L in self.layers)
        need = workspace_size(B, cap, H, k, pool, W)
        self.ws = ws if ws is not None and ws.numel() >= need else torch.empty(need, dtype=torch.uint8,
                                                                               device=first.q.device)
        self._descs = (A.LayerDesc * len(self.layers))(*[L.desc() for L in self.layers])

    def __call__(self, stream=None) -> None:
        A.check(A.lib().csa2_decode_step(self._descs, len(self.layers), self.B, self.H, self.k, self.dtype,
                                         _ptr(self.ws), self.ws.numel(), _stream(stream)), "csa2_decode_step")


def csa2_decode_step(layers, k: int = 512, ws=None, stream=None) -> None:
    """Run one decode step through ``layers`` (a list of Layer)."""
    DecodeStep(layers, k, ws)(stream)


def sync_status(stream=None) -> int:
    """Synchronise and return (and clear) the device status word; 0 = no device error."""
    return A.lib().csa2_sync_status(_stream(stream))


def launch_count() -> int:
    return A.lib().csa2_launch_count()


def set_scan_events(pairs=None) -> None:
    """Measurement hook: ``pairs`` is a list of (before, after) torch.cuda.Events; the
    i-th streaming indexer-scan launch made by later calls from this thread records
    pair i mod len(pairs) around itself (None or []: off). The events must already
    exist on the device (record them once first)."""
    pairs = list(pairs or [])
    n = len(pairs)
    before = (C.c_void_p * max(n, 1))(*[a.cuda_event for a, _ in pairs])
    after = (C.c_void_p * max(n, 1))(*[b.cuda_event for _, b in pairs])
    A.check(A.lib().csa2_set_scan_events(before, after, n), "csa2_set_scan_events")
