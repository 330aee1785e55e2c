"""Seeded synthetic inputs for the five workloads of the CSA2 FP4 decode path.

This module only draws random numbers (torch generators, seeded) and casts them
to the input dtypes; it holds none of the method's arithmetic. Both the CUDA
path and the CPU oracle consume what it returns.

Workloads (the shapes, sizes and value distributions of the method's stated
problem; every value is synthetic):

  0 tiny ratio-1 layer: 1 sequence x 4,096 entries; fp32 latents N(0,1) times a
    per-channel LogNormal(0,1) magnitude (512 + 128 channels); 16 query heads,
    q ~ N(0, 1/512); 4 indexer heads, q_idx ~ N(0, 1/128), w ~ U(0,1); seed 0.
  1 cache write: 65,536 bf16 tokens, latent 512 + key 128 channels ~ N(0,1),
    round(0.01*C) channels scaled x20 as outliers; ratio-2 merge weights
    w0, w1 ~ U(0,1) per channel; seed 0.
  2 batched decode: 32 sequences x 131,072 entries, ratio 1, latents as in 0,
    64 heads, bf16 q and q_idx; seed 1.
  3 1M-token ratio-2 layer: 8 sequences x 1,048,576 tokens (524,288 entries),
    latents as in 0 merged with U(0,1) weights; two indexers; pool 16,384;
    64 heads; seed 2.
  4 decoder group Full/Reindex/Reuse/Reuse over one ratio-1 cache: 64 sequences x
    65,536 entries; the Reindex layer has its own indexer keys; a 128-token bf16
    window N(0,1) per layer; 64 heads; seed 3.

Variances: N(0, 1/512) means variance 1/512.
"""
from __future__ import annotations

import hashlib

import torch

LAT, IDX = 512, 128


def generator(seed: int, *tags, device="cpu") -> torch.Generator:
    """A torch generator on ``device`` seeded from (seed, tags) by SHA-256."""
    h = hashlib.sha256(repr((int(seed),) + tuple(tags)).encode()).digest()
    g = torch.Generator(device=device)
    g.manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))
    return g


def channel_magnitudes(seed: int, device="cpu"):
    """Per-channel LogNormal(0,1) magnitudes: (m_lat [512], m_idx [128]) fp32."""
    g = generator(seed, "magnitudes", device=device)
    m = torch.randn(LAT + IDX, generator=g, device=device).exp_()
    return m[:LAT], m[LAT:]


def lognormal_tokens(seed: int, seq: int, T: int, device="cpu", stream: str = "tokens"):
    """fp32 sources of one sequence: N(0,1) * per-channel magnitude.

    Returns (lat [T, 512], ikey [T, 128]) float32.
    """
    m_lat, m_idx = channel_magnitudes(seed, device)
    g = generator(seed, stream, seq, device=device)
    lat = torch.randn(T, LAT, generator=g, device=device).mul_(m_lat)
    ikey = torch.randn(T, IDX, generator=g, device=device).mul_(m_idx)
    return lat, ikey


def outlier_tokens(seed: int, seq: int, T: int, device="cpu"):
    """bf16 sources N(0,1) with round(0.01*C) rng-chosen channels scaled x20.

    Returns (lat [T, 512], ikey [T, 128]) bfloat16.
    """
    g = generator(seed, "outlier-channels", device="cpu")
    o_lat = torch.randperm(LAT, generator=g)[: round(0.01 * LAT)]
    o_idx = torch.randperm(IDX, generator=g)[: round(0.01 * IDX)]
    s_lat = torch.ones(LAT)
    s_lat[o_lat] = 20.0
    s_idx = torch.ones(IDX)
    s_idx[o_idx] = 20.0
    g2 = generator(seed, "tokens", seq, device=device)
    lat = torch.randn(T, LAT, generator=g2, device=device).mul_(s_lat.to(device))
    ikey = torch.randn(T, IDX, generator=g2, device=device).mul_(s_idx.to(device))
    return lat.to(torch.bfloat16), ikey.to(torch.bfloat16)


def merge_weights(seed: int, device="cpu", layer=None):
    """U(0,1) per-channel merge weights: (w0_lat, w1_lat [512], w0_idx, w1_idx [128]) fp32
    (``layer``: the weights of one source layer of a multi-layer store)."""
    g = generator(seed, "merge-weights", device=device) if layer is None else \
        generator(seed, "merge-weights", layer, device=device)
    w = torch.rand(2 * (LAT + IDX), generator=g, device=device)
    return w[:LAT], w[LAT:2 * LAT], w[2 * LAT:2 * LAT + IDX], w[2 * LAT + IDX:]


def queries(seed: int, layer, B: int, H: int, dtype=torch.bfloat16, n_idx_heads: int = 4,
            device="cpu", tag: str = "q"):
    """Decode-step queries of one layer.

    Returns q [B, H, 512] ~ N(0, 1/512), q_idx [B, n_idx_heads, 128] ~ N(0, 1/128)
    (both cast to ``dtype``), w_idx [B, n_idx_heads] ~ U(0,1) fp32.
    """
    g = generator(seed, tag, layer, device=device)
    q = torch.randn(B, H, LAT, generator=g, device=device).mul_(LAT ** -0.5).to(dtype)
    q_idx = torch.randn(B, n_idx_heads, IDX, generator=g, device=device).mul_(IDX ** -0.5).to(dtype)
    w_idx = torch.rand(B, n_idx_heads, generator=g, device=device)
    return q, q_idx, w_idx


def window(seed: int, layer, B: int, W: int = 128, device="cpu"):
    """Sliding-window rows of one layer: [B, W, 512] bf16 ~ N(0,1)."""
    g = generator(seed, "window", layer, device=device)
    return torch.randn(B, W, LAT, generator=g, device=device).to(torch.bfloat16)


def new_token(seed: int, step: int, B: int, device="cpu"):
    """The token appended by one decode step, per sequence: fp32 (lat [B,1,512], ikey [B,1,128])."""
    m_lat, m_idx = channel_magnitudes(seed, device)
    g = generator(seed, "decode-token", step, device=device)
    lat = torch.randn(B, 1, LAT, generator=g, device=device).mul_(m_lat)
    ikey = torch.randn(B, 1, IDX, generator=g, device=device).mul_(m_idx)
    return lat, ikey


def scores(seed: int, B: int, n: int, device="cpu", ties: int = 0):
    """fp32 score rows [B, n] >= 0 for stand-alone Top-k cases.

    ``ties`` > 0 quantises the draws to that many distinct levels, so equal scores
    occur often and the tie rule decides.
    """
    g = generator(seed, "scores", device=device)
    s = torch.rand(B, n, generator=g, device=device)
    if ties:
        s = torch.floor(s * ties) / ties
    return s


def random_cache_bytes(seed: int, B: int, cap: int, device="cpu", scale_lo: int = 120, scale_hi: int = 135):
    """Uniformly random packed cache bytes for kernel timing (every byte pattern is a
    valid pair of E2M1 codes). Scales: E8M0 bytes in [scale_lo, scale_hi) for the keys,
    E4M3 bytes 0x30..0x4F (about 0.5 to 16) for the latent.

    Returns (lat_codes [B,cap,256], lat_scales [B,cap,32], idx_codes [B,cap,64],
    idx_scales [B,cap,4]) uint8.
    """
    g = generator(seed, "random-cache", device=device)
    u8 = dict(dtype=torch.uint8, device=device, generator=g)
    lat_codes = torch.randint(0, 256, (B, cap, 256), **u8)
    lat_scales = torch.randint(0x30, 0x50, (B, cap, 32), **u8)
    idx_codes = torch.randint(0, 256, (B, cap, 64), **u8)
    idx_scales = torch.randint(scale_lo, scale_hi, (B, cap, 4), **u8)
    return lat_codes, lat_scales, idx_codes, idx_scales
