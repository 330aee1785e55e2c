"""Shared test helpers: build the five workloads on the GPU through the C ABI,
build the same inputs for the CPU oracle, and compare under the stated rules.

Comparison rules (stated by the method's acceptance criteria):
  * packed codes, scales and lengths: bit-exact;
  * Top-k index sets: equal, except positions whose oracle score lies within
    1e-6 relative of the oracle's k-th score (near-ties);
  * attention output: per (sequence, head) row, max |o_gpu - o_ref| / max |o_ref|
    <= 2e-3.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import fp4_compressed_kv_append_b300 as K
from fp4_compressed_kv_append_b300 import workloads as WL
from oracle import csa2 as O

ATTN_TOL = 2e-3
TIE_REL = 1e-6


def np_(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy()
    return t.numpy()


def sub_view(cache: K.Cache, b: int) -> K.Cache:
    """A one-sequence view of sequence b of a device cache (shares memory)."""
    v = K.Cache.__new__(K.Cache)
    v.batch, v.cap = 1, cache.cap
    v.lat_codes, v.lat_scales = cache.lat_codes[b:b + 1], cache.lat_scales[b:b + 1]
    v.idx_codes, v.idx_scales = cache.idx_codes[b:b + 1], cache.idx_scales[b:b + 1]
    v.len = cache.len[b:b + 1]
    v._view = None
    return v


# ------------------------------------------------------------------ sources
def sources(cfg: str, seed: int, b: int, T: int, device):
    """Source tokens of sequence b: (lat, ikey) on ``device``."""
    if cfg == "outlier":
        return WL.outlier_tokens(seed, b, T, device=device)
    return WL.lognormal_tokens(seed, b, T, device=device)


def build_gpu_cache(cfg, seed, B, T, ratio, cap, weights=None, stream_tag="tokens"):
    """Append T tokens per sequence, one sequence at a time, through kv_quant_append."""
    cache = K.Cache(B, cap)
    for b in range(B):
        if cfg == "outlier":
            lat, ikey = WL.outlier_tokens(seed, b, T, device="cuda")
        else:
            lat, ikey = WL.lognormal_tokens(seed, b, T, device="cuda", stream=stream_tag)
        w = weights or (None, None, None, None)
        K.kv_quant_append(lat[None], ikey[None], ratio, sub_view(cache, b), *w)
        del lat, ikey
    return cache


def oracle_cache_rows(cfg, seed, b, T, ratio, weights=None, stream_tag="tokens"):
    """The oracle's packed rows of sequence b (sources drawn on the GPU generator, copied)."""
    if cfg == "outlier":
        lat, ikey = WL.outlier_tokens(seed, b, T, device="cuda")
    else:
        lat, ikey = WL.lognormal_tokens(seed, b, T, device="cuda", stream=stream_tag)
    w = [None] * 4 if weights is None else [np_(x) for x in weights]
    return O.encode_entries(np_(lat), np_(ikey), ratio, *w)


def host_cache_from_rows(rows_per_seq, cap):
    """An oracle Cache from per-sequence packed rows."""
    B = len(rows_per_seq)
    c = O.Cache(B, cap)
    for b, (lc, ls, ic, isc) in enumerate(rows_per_seq):
        n = lc.shape[0]
        c.lat_codes[b, :n], c.lat_scales[b, :n] = lc, ls
        c.idx_codes[b, :n], c.idx_scales[b, :n] = ic, isc
        c.len[b] = n
    return c


def assert_rows_equal(gpu: K.Cache, b: int, rows):
    lc, ls, ic, isc = rows
    n = lc.shape[0]
    assert int(gpu.len[b]) == n
    for name, ref in (("lat_codes", lc), ("lat_scales", ls), ("idx_codes", ic), ("idx_scales", isc)):
        got = np_(getattr(gpu, name)[b, :n])
        bad = np.argwhere(got != ref)
        assert bad.size == 0, f"{name} differs at {bad[:5].tolist()} (seq {b})"


# ------------------------------------------------------------------ comparisons
def score_tolerance(q_idx, w, keys):
    """|fp32 score - exact score| bound for 128-term fp32 dot products (plus the head sum)."""
    absdot = np.abs(keys) @ np.abs(np.asarray(q_idx, np.float64)).T         # [n, 4]
    return 64 * 2.0 ** -24 * (absdot @ np.abs(np.asarray(w, np.float64))) + 1e-37


def assert_topk_match(got_idx, ref_idx, ref_scores, positions=None, where=""):
    """Sets equal except near-ties around the oracle's k-th score; both sorted, -1 padded."""
    got = np.asarray(got_idx)
    ref = np.asarray(ref_idx)
    vg = got[got >= 0]
    vr = ref[ref >= 0]
    assert np.all(np.diff(vg) > 0), f"{where}: output not strictly ascending"
    assert np.all(got[len(vg):] == -1) and np.all(got[:len(vg)] >= 0), f"{where}: padding not at the end"
    assert len(vg) == len(vr), f"{where}: {len(vg)} selected, oracle {len(vr)}"
    diff = set(vg.tolist()) ^ set(vr.tolist())
    if not diff:
        return 0
    s = np.asarray(ref_scores, np.float64)
    pos = np.arange(len(s)) if positions is None else np.asarray(positions)
    score_of = dict(zip(pos.tolist(), s.tolist()))
    tau = min(score_of[p] for p in vr.tolist())
    for p in diff:
        assert p in score_of, f"{where}: position {p} is not among the candidates"
        assert abs(score_of[p] - tau) <= TIE_REL * abs(tau), \
            f"{where}: position {p} (score {score_of[p]}) differs, kth score {tau}"
    return len(diff)


def attn_rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.abs(got - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    return float(np.max(num / np.where(den == 0, 1.0, den)))


def seed_everything(seed=0):
    torch.manual_seed(seed)
    np.random.seed(seed)


__all__ = ["K", "WL", "O", "np_", "sub_view", "build_gpu_cache", "oracle_cache_rows", "host_cache_from_rows",
           "assert_rows_equal", "score_tolerance", "assert_topk_match", "attn_rel_err", "ATTN_TOL", "math"]
