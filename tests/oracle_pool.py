"""Oracle encodes of long sequences in worker processes (test infrastructure).

Packing the rows of one full-size sequence (131,072 to 524,288 cache entries)
takes the numpy oracle tens of seconds. The tests split a sequence's source
tokens into chunks and encode the chunks in a pool of worker processes. The
pool is started with ``spawn`` (a worker never inherits a process that has
touched the GPU), and workers import only numpy and the oracle.
"""
from __future__ import annotations

import atexit
import multiprocessing as mp
import os

import numpy as np

CHUNK_ENTRIES = 4096
_POOL = None


def _encode(args):
    from oracle import csa2 as O
    lat, ikey, ratio, w = args
    return O.encode_entries(lat, ikey, ratio, *w)


def _pool():
    global _POOL
    if _POOL is None:
        n = max(1, min(32, os.cpu_count() or 1))
        _POOL = mp.get_context("spawn").Pool(n)
        atexit.register(_POOL.terminate)
    return _POOL


def encode_rows(lat: np.ndarray, ikey: np.ndarray, ratio: int, weights=None):
    """oracle.csa2.encode_entries of [T, 512] / [T, 128] sources, chunk by chunk in
    the worker pool; returns the concatenated (lat_codes, lat_scales, idx_codes,
    idx_scales) rows. A chunk boundary falls on an even token, so a ratio-2 merge
    pairs the same tokens as a single call would."""
    w = [None] * 4 if weights is None else list(weights)
    step = CHUNK_ENTRIES * ratio
    jobs = [(lat[i:i + step], ikey[i:i + step], ratio, w) for i in range(0, len(lat), step)]
    if len(jobs) <= 2:
        parts = [_encode(j) for j in jobs]
    else:
        parts = _pool().map(_encode, jobs, chunksize=1)
    return tuple(np.concatenate([p[j] for p in parts]) for j in range(4))
