"""The five workloads of the CSA2 FP4 decode path, built on the device through the
public API (kv_quant_append to fill the caches, then one prepared DecodeStep).

  0 tiny ratio-1 layer (1 x 4,096 entries, 16 heads, fp32 queries)
  1 cache write (65,536 bf16 tokens, ratio-2 merge) -- append only
  2 batched decode at 128K (32 x 131,072 entries, 64 heads, bf16 queries)
  3 1M-token ratio-2 layer (8 x 524,288 entries) with a 16,384-candidate pool
  4 decoder group Full/Reindex/Reuse/Reuse (64 x 65,536 entries, 128-token window)
  5 prefill store: 1,048,576 bf16 tokens into the four source layers of the global
    cache (layers 2, 8 and 14 at ratio 2, layer 20 at ratio 1) -- append only

A Reindex layer scores its own indexer-key array (``reindex_keys="own"``, the
default) or the Full layer's keys with its own query (``reindex_keys="shared"``).
Window rows are bf16 (``window="bf16"``, the default) or packed as FP8 from the
same bf16 rows (``window="fp8"``).

Sizes can be reduced (batch, tokens) for tests; the structure stays the same.
All inputs come from ``workloads`` (seeded, synthetic).
"""
from __future__ import annotations

import torch

from . import Cache, DecodeStep, Layer, kv_quant_append, FULL, REINDEX, REUSE
from . import swa_quant, store_append
from . import workloads as WL

CONFIGS = {
    0: dict(name="tiny ratio-1 layer", B=1, tokens=4096, ratio=1, H=16, dtype=torch.float32, src="lognormal",
            seed=0, modes=(FULL,), pool=0, W=0),
    1: dict(name="cache write, ratio-2 merge", B=1, tokens=65536, ratio=2, src="outlier", seed=0),
    2: dict(name="batched decode, ratio-1 layer, 128K context", B=32, tokens=131072, ratio=1, H=64,
            dtype=torch.bfloat16, src="lognormal", seed=1, modes=(FULL,), pool=0, W=0),
    3: dict(name="1M-token ratio-2 layer, hierarchical indexer", B=8, tokens=1048576, ratio=2, H=64,
            dtype=torch.bfloat16, src="lognormal", seed=2, modes=(FULL,), pool=16384, W=0),
    4: dict(name="decoder group Full/Reindex/Reuse/Reuse", B=64, tokens=65536, ratio=1, H=64,
            dtype=torch.bfloat16, src="lognormal", seed=3, modes=(FULL, REINDEX, REUSE, REUSE), pool=0, W=128,
            reindex_keys="own"),
    5: dict(name="prefill store, four source layers", B=1, tokens=1048576, src="outlier", seed=0,
            layers=((2, 2), (8, 2), (14, 2), (20, 1))),
}
TOPK = 512


def config(cfg_id: int, **override) -> dict:
    c = dict(CONFIGS[cfg_id])
    c.update({k: v for k, v in override.items() if v is not None})
    c["id"] = cfg_id
    return c


def source_tokens(c: dict, b: int, device="cuda", stream: str = "tokens"):
    if c["src"] == "outlier":
        return WL.outlier_tokens(c["seed"], b, c["tokens"], device=device)
    return WL.lognormal_tokens(c["seed"], b, c["tokens"], device=device, stream=stream)


def _sub(cache: Cache, b: int) -> Cache:
    v = Cache.__new__(Cache)
    v.batch, v.cap = 1, cache.cap
    v.lat_codes, v.lat_scales = cache.lat_codes[b:b + 1], cache.lat_scales[b:b + 1]
    v.idx_codes, v.idx_scales = cache.idx_codes[b:b + 1], cache.idx_scales[b:b + 1]
    v.len = cache.len[b:b + 1]
    v._view = None
    return v


def fill_cache(c: dict, extra: int = 0, stream: str = "tokens") -> Cache:
    """Append every sequence's source tokens (one sequence per call)."""
    entries = c["tokens"] // c["ratio"]
    cap = (entries + extra + 127) // 128 * 128
    cache = Cache(c["B"], cap)
    w = WL.merge_weights(c["seed"], device="cuda") if c["ratio"] == 2 else (None,) * 4
    for b in range(c["B"]):
        lat, ikey = source_tokens(c, b, stream=stream)
        kv_quant_append(lat[None], ikey[None], c["ratio"], _sub(cache, b), *w)
        del lat, ikey
    return cache


class DecodeWorkload:
    """Caches, per-layer queries/windows/outputs and a prepared DecodeStep for config c."""

    def __init__(self, c: dict, extra: int = 0):
        self.c = c
        B, H, dt = c["B"], c["H"], c["dtype"]
        self.cache = fill_cache(c, extra)
        self.reindex_keys = None
        if REINDEX in c["modes"] and c.get("reindex_keys", "own") == "own":
            self.reindex_keys = fill_cache(c, extra, stream="reindex-keys")  # only its indexer keys are read
        self.layers, self.inputs = [], []
        for li, mode in enumerate(c["modes"]):
            q, q_idx, w_idx = WL.queries(c["seed"], li, B, H, dtype=dt, device="cuda")
            q_idx2 = w_idx2 = None
            if mode == FULL and c["pool"]:
                _, q_idx2, w_idx2 = WL.queries(c["seed"], li, B, H, dtype=dt, device="cuda", tag="q2")
            swa = WL.window(c["seed"], li, B, c["W"], device="cuda") if c["W"] else None
            swa_arg = swa_quant(swa) if swa is not None and c.get("window", "bf16") == "fp8" else swa
            out = torch.empty(B, H, 512, dtype=torch.float32, device="cuda")
            idx_out = torch.empty(B, TOPK, dtype=torch.int32, device="cuda")
            own = ((self.reindex_keys.idx_codes, self.reindex_keys.idx_scales)
                   if mode == REINDEX and self.reindex_keys is not None else (None, None))
            self.layers.append(Layer(mode, q, out, cache=self.cache if mode == FULL else None,
                                     q_idx=None if mode == REUSE else q_idx, w_idx=None if mode == REUSE else w_idx,
                                     own_idx_codes=own[0], own_idx_scales=own[1], pool=c["pool"] if mode == FULL else 0,
                                     q_idx2=q_idx2, w_idx2=w_idx2, swa=swa_arg, idx_out=idx_out))
            self.inputs.append(dict(q=q, q_idx=q_idx, w_idx=w_idx, q_idx2=q_idx2, w_idx2=w_idx2, swa=swa,
                                    swa_fp8=swa_arg if swa_arg is not swa else None))
        self.step = DecodeStep(self.layers, TOPK)

    def __call__(self, stream=None):
        self.step(stream)

    @property
    def outputs(self):
        return [L.out for L in self.layers]

    @property
    def indices(self):
        return [L.idx_out for L in self.layers]


class StoreWorkload:
    """The multi-layer store of config c: per layer, its bf16 sources (drawn with the
    layer number as the sequence tag), its merge weights (ratio 2) and its cache."""

    def __init__(self, c: dict, T: int = None):
        self.c = c
        T = c["tokens"] if T is None else T
        self.T = T
        self.sources, self.weights, self.caches = [], [], []
        for layer, ratio in c["layers"]:
            lat, ikey = WL.outlier_tokens(c["seed"], layer, T, device="cuda")
            self.sources.append((lat[None], ikey[None]))
            self.weights.append(WL.merge_weights(c["seed"], device="cuda", layer=layer) if ratio == 2 else None)
            self.caches.append(Cache(c["B"], (T // ratio + 127) // 128 * 128))

    def layers(self):
        return [(lat, ikey, ratio, cache, w) for (lat, ikey), (_, ratio), cache, w
                in zip(self.sources, self.c["layers"], self.caches, self.weights)]

    def __call__(self, stream=None):
        store_append(self.layers(), stream)

    def stored_bytes(self):
        """Bytes the caches hold for the appended entries (288 + 68 per entry)."""
        return sum(int(c.len.sum()) * (256 + 32 + 64 + 4) for c in self.caches)
