"""Per-kernel timing of the CSA2 FP4 decode path on random (valid) cache bytes.

    python -m fp4_compressed_kv_append_b300.kernel_bench --kernel scan --batch 32 --entries 131072
    python -m fp4_compressed_kv_append_b300.kernel_bench --kernel all

Kernels: scan (indexer_score over every entry), topk (topk_select, k = 512),
attn (sparse_latent_attn over 512 selected entries), append (kv_quant_append of
one token per sequence), write (kv_quant_append of 2 x --entries bf16 tokens of one
sequence at ratio 2, the cache length reset before each launch), step (one
Full-layer csa2_decode_step). The launches are
captured in a CUDA graph, each between two CUDA events; with --flush a 256 MB
buffer is written between launches so that L2 holds nothing of the inputs. Prints one JSON
line per kernel: average microseconds per launch, algorithmic bytes per launch
(68 per scanned entry, 288 per gathered entry, 4 per score read by Top-k, 2,560
in + 356 out per written entry) and
the resulting GB/s.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import Cache, DecodeStep, Layer, FULL, indexer_score, kv_quant_append, \
    sparse_latent_attn, topk_select
from . import workloads as WL


def make_cache(B, N, seed=0):
    cap = (N + 127) // 128 * 128 + 128
    c = Cache(B, cap)
    lc, ls, ic, isc = WL.random_cache_bytes(seed, B, cap, device="cuda")
    c.lat_codes.copy_(lc)
    c.lat_scales.copy_(ls)
    c.idx_codes.copy_(ic)
    c.idx_scales.copy_(isc)
    c.len.fill_(N)
    del lc, ls, ic, isc
    return c


def time_launches(fn, iters, warmup, flush):
    """Average device time of fn's launches. The launches are captured in a CUDA
    graph with an event pair around each one, so host-side submission time is
    not counted."""
    buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if flush else None
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
          for _ in range(iters)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for a, b in ev:
            if buf is not None:
                buf.fill_(1)
            a.record()
            fn()
            b.record()
    g.replay()  # warm
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / iters * 1e3


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--kernel", default="all", choices=["all", "scan", "topk", "attn", "append", "write", "step"])
    p.add_argument("--batch", type=int, default=32)
    p.add_argument("--entries", type=int, default=131072)
    p.add_argument("--heads", type=int, default=64)
    p.add_argument("--k", type=int, default=512)
    p.add_argument("--iters", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--flush", action="store_true")
    a = p.parse_args()
    B, N, H, k = a.batch, a.entries, a.heads, a.k
    cache = make_cache(B, N)
    q, q_idx, w = WL.queries(0, 0, B, H, dtype=torch.bfloat16, device="cuda")
    scores = torch.empty(B, cache.cap, dtype=torch.float32, device="cuda")
    sel = torch.empty(B, k, dtype=torch.int32, device="cuda")
    out = torch.empty(B, H, 512, dtype=torch.float32, device="cuda")
    indexer_score(q_idx, w, cache.idx_codes, cache.idx_scales, cache.len, scores=scores)
    topk_select(scores, k, n=cache.len, out=sel)
    tok = WL.new_token(0, 0, B, device="cuda")
    runs = {
        "scan": (lambda: indexer_score(q_idx, w, cache.idx_codes, cache.idx_scales, cache.len, scores=scores),
                 68 * B * N),
        "topk": (lambda: topk_select(scores, k, n=cache.len, out=sel), 4 * B * N),
        "attn": (lambda: sparse_latent_attn(q, cache, sel, out=out), 288 * B * k),
    }
    if a.kernel in ("append", "all"):
        cache.len.fill_(N - 1)  # the appended token rewrites the last row each launch
        runs["append"] = (lambda: (cache.len.fill_(N - 1), kv_quant_append(tok[0], tok[1], 1, cache)),
                          (2048 + 512 + 356) * B)
    if a.kernel == "write":  # one ratio-2 bulk append (bf16 sources with outlier channels)
        lat, ikey = WL.outlier_tokens(0, 0, 2 * N, device="cuda")
        wcache = Cache(1, (N + 127) // 128 * 128)
        mw = WL.merge_weights(0, device="cuda")
        zero = torch.zeros_like(wcache.len)
        runs = {"write": (lambda: (wcache.len.copy_(zero),
                                   kv_quant_append(lat[None], ikey[None], 2, wcache, *mw)),
                          (2560 + 356) * N)}
    if a.kernel in ("step", "all"):
        step = DecodeStep([Layer(FULL, q, out, cache=cache, q_idx=q_idx, w_idx=w)], k)
        runs["step"] = (step, 68 * B * N + 288 * B * k)
    for name, (fn, nbytes) in runs.items():
        if a.kernel not in ("all", name):
            continue
        us = time_launches(fn, a.iters, a.warmup, a.flush)
        print(json.dumps({"kernel": name, "batch": B, "entries": N, "heads": H, "k": k, "us": us,
                          "algorithmic_bytes": nbytes, "gbs": nbytes / us / 1e3, "flush": a.flush}), flush=True)


if __name__ == "__main__":
    main()
