"""The C-ABI library without a GPU: it loads, exports every declared entry point,
and rejects bad arguments on the host before any CUDA call."""
import ctypes as C
import os
import re

import pytest

from fp4_compressed_kv_append_b300 import _abi as A

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_functions():
    names = []
    for f in sorted(os.listdir(HEADER)):
        if f.endswith(".h"):
            text = open(os.path.join(HEADER, f)).read()
            names += re.findall(r"CSA2_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert {"kv_quant_append", "indexer_score", "topk_select", "sparse_latent_attn",
            "csa2_decode_step"} <= set(names)
    lib = A.lib()
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    for s in range(8):
        assert A.status_str(s) and A.status_str(s) != "unknown status"
    assert A.status_str(99) == "unknown status"


def test_workspace_sizes():
    L = A.lib()
    # the decode step needs the scores, the pool and the selection
    total = L.csa2_workspace_size(32, 131072, 64, 512, 0, 0)
    assert total >= 32 * 131072 * 4 + 2 * 32 * 512 * 4  # scores, two selections
    pooled = L.csa2_workspace_size(8, 524288, 64, 512, 16384, 0)
    assert pooled >= 8 * 524288 * 4 + 2 * 8 * 16384 * 4 + 2 * 8 * 512 * 4


def _fake_cache(cap=256, batch=2, base=0x10000):
    return A.CacheView(base, base + 0x1000, base + 0x2000, base + 0x3000, base + 0x4000, cap, batch)


def test_host_validation_rejects_before_any_launch():
    L = A.lib()
    cv = _fake_cache()
    # null cache, bad ratio, odd T at ratio 2
    assert L.kv_quant_append(0x100, 0x200, A.BF16, 4, 1, None, None, None, None, None, None) == A.ERR_ARG
    assert L.kv_quant_append(0x100, 0x200, A.BF16, 4, 3, None, None, None, None, C.byref(cv), None) == A.ERR_ARG
    assert L.kv_quant_append(0x100, 0x200, A.BF16, 3, 2, 1, 1, 1, 1, C.byref(cv), None) == A.ERR_ARG
    # capacity not a multiple of 128; misaligned source
    bad = _fake_cache(cap=200)
    assert L.kv_quant_append(0x100, 0x200, A.BF16, 4, 1, None, None, None, None, C.byref(bad), None) == A.ERR_ARG
    assert L.kv_quant_append(0x101, 0x200, A.BF16, 4, 1, None, None, None, None, C.byref(cv), None) == A.ERR_ALIGN
    # T = 0 is a no-op
    assert L.kv_quant_append(None, None, A.BF16, 0, 1, None, None, None, None, C.byref(cv), None) == A.OK
    # indexer: null scores, pool too large
    assert L.indexer_score(0x100, A.BF16, 0x200, 0x1000, 0x2000, 256, 0x300, None, 0, None, 2, None) == A.ERR_ARG
    assert L.indexer_score(0x100, A.BF16, 0x200, 0x1000, 0x2000, 256, 0x300, 0x400, 20000, 0x500, 2,
                           None) == A.ERR_ARG
    # top-k: k out of range
    assert L.topk_select(0x100, None, 1000, 0, None, 0x200, 1, None) == A.ERR_ARG
    assert L.topk_select(0x100, None, 1000, 16385, None, 0x200, 1, None) == A.ERR_ARG
    # attention: head count, a window without rows
    assert L.sparse_latent_attn(0x100, A.BF16, 48, 0.04, C.byref(cv), 0x200, 512, None, None, None, 0, 0x300,
                                None) == A.ERR_UNSUPPORTED
    assert L.sparse_latent_attn(0x100, A.BF16, 64, 0.04, C.byref(cv), 0x200, 512, None, None, None, 5, 0x300,
                                None) == A.ERR_ARG
    # bounded-wait self-test: a limit over one second is refused before any launch
    assert L.csa2_selftest_wait_timeout(1_000_000_001, None) == A.ERR_ARG


def test_decode_step_validation():
    L = A.lib()
    cv = _fake_cache()
    lay = (A.LayerDesc * 2)()
    for d in lay:
        d.q, d.out, d.q_idx, d.w_idx = 0x100, 0x200, 0x300, 0x400
    lay[0].mode, lay[0].cache = A.REUSE, C.pointer(cv)
    lay[1].mode = A.REUSE
    assert L.csa2_decode_step(lay, 2, 2, 64, 512, A.BF16, 0x1000, 1 << 40, None) == A.ERR_ARG  # first not FULL
    lay[0].mode = A.FULL
    lay[0].pool = 400                                                                          # pool <= k
    assert L.csa2_decode_step(lay, 2, 2, 64, 512, A.BF16, 0x1000, 1 << 40, None) == A.ERR_ARG
    lay[0].pool = 0
    assert L.csa2_decode_step(lay, 2, 2, 64, 512, A.BF16, 0x1000, 16, None) == A.ERR_WORKSPACE
    assert L.csa2_decode_step(lay, 2, 2, 24, 512, A.BF16, 0x1000, 1 << 40, None) == A.ERR_UNSUPPORTED
    assert L.csa2_decode_step(lay, 2, 3, 64, 512, A.BF16, 0x1000, 1 << 40, None) == A.ERR_ARG  # batch mismatch


def test_launch_counter_starts_at_zero_without_gpu_work():
    assert A.lib().csa2_launch_count() == 0


def test_store_append_and_window_validation():
    L = A.lib()
    cv, cv3 = _fake_cache(), _fake_cache(batch=3)
    lay = (A.StoreLayer * 2)()
    for d in lay:
        d.lat, d.ikey, d.ratio, d.cache = 0x1000, 0x2000, 1, C.pointer(cv)
    assert L.csa2_store_append(lay, 0, A.BF16, 4, None) == A.ERR_ARG        # no layer
    assert L.csa2_store_append(lay, 9, A.BF16, 4, None) == A.ERR_ARG        # more than 8
    lay[1].ratio = 2                                                        # ratio 2 without weights
    assert L.csa2_store_append(lay, 2, A.BF16, 4, None) == A.ERR_ARG
    lay[1].w0_lat = lay[1].w1_lat = lay[1].w0_idx = lay[1].w1_idx = 0x3000
    assert L.csa2_store_append(lay, 2, A.BF16, 5, None) == A.ERR_ARG        # odd T at ratio 2
    lay[1].w1_idx = 0x3004
    assert L.csa2_store_append(lay, 2, A.BF16, 4, None) == A.ERR_ALIGN      # unaligned weights
    lay[1].w1_idx = 0x3000
    lay[1].cache = C.pointer(cv3)
    assert L.csa2_store_append(lay, 2, A.BF16, 4, None) == A.ERR_ARG        # batch mismatch
    lay[1].cache = C.pointer(cv)
    assert L.csa2_store_append(lay, 2, A.BF16, 0, None) == A.OK             # T = 0: nothing to do
    # FP8 window rows: null outputs, unaligned rows, bad dtype
    assert L.csa2_swa_quant(0x100, A.BF16, 4, None, 0x300, None) == A.ERR_ARG
    assert L.csa2_swa_quant(0x101, A.BF16, 4, 0x200, 0x300, None) == A.ERR_ALIGN
    assert L.csa2_swa_quant(0x100, 7, 4, 0x200, 0x300, None) == A.ERR_ARG
    assert L.csa2_swa_quant(None, A.BF16, 0, None, None, None) == A.OK
    # attention: a window given both as bf16 and FP8 rows, or FP8 codes without scales
    assert L.sparse_latent_attn(0x100, A.BF16, 64, 0.04, C.byref(cv), 0x200, 512, 0x400, 0x500, 0x600, 8, 0x300,
                                None) == A.ERR_ARG
    assert L.sparse_latent_attn(0x100, A.BF16, 64, 0.04, C.byref(cv), 0x200, 512, None, 0x500, None, 8, 0x300,
                                None) == A.ERR_ARG
