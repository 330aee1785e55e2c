"""Whole decode steps of the five workloads against the oracle.

Reduced sizes (several tiles and a ragged tail) are checked on every sequence;
the full sizes are checked on sampled sequences, plus properties on all of them.
"""
import numpy as np
import pytest
import torch

from fp4_compressed_kv_append_b300 import configs as CF
from oracle import csa2 as O
from tests import harness as Hh
from tests import oracle_pool as OP
from tests.harness import np_

pytestmark = pytest.mark.gpu


def _oracle_rows(c, b, stream="tokens"):
    lat, ikey = CF.source_tokens(c, b, stream=stream)
    w = [np_(x) for x in CF.WL.merge_weights(c["seed"], device="cuda")] if c["ratio"] == 2 else None
    return OP.encode_rows(np_(lat), np_(ikey), c["ratio"], w)


def _window_ref(inp, b):
    """The oracle's window rows of sequence b, [1, W, 512] float64: the bf16 rows, or
    their FP8 packing by the oracle (the GPU's packed bytes must equal it)."""
    if inp["swa"] is None:
        return None
    rows = np_(inp["swa"][b])
    if inp.get("swa_fp8") is None:
        return rows[None].astype(np.float64)
    codes, scales = O.quantize_swa(rows)
    gc, gs = inp["swa_fp8"]
    assert np.array_equal(np_(gc[b]), codes) and np.array_equal(np_(gs[b]), scales), "FP8 window bytes"
    return O.dequantize_swa(codes, scales)[None]


def _check_sequence(wl: CF.DecodeWorkload, b: int):
    """Sequence b of a decode step against the oracle: the packed cache rows
    bit-exact; every Full/Reindex selection equal to the oracle's up to near-ties
    (1e-6 of the k-th score); every layer's attention output within 2e-3 of the
    oracle's attention over the GPU's own selection, which the previous check has
    validated (so a legal near-tie swap never skips the attention check)."""
    c = wl.c
    rows = _oracle_rows(c, b)
    Hh.assert_rows_equal(wl.cache, b, rows)
    host = Hh.host_cache_from_rows([rows], wl.cache.cap)
    n = int(host.len[0])
    own = None
    if wl.reindex_keys is not None:
        r2 = _oracle_rows(c, b, stream="reindex-keys")
        Hh.assert_rows_equal(wl.reindex_keys, b, r2)
        own = Hh.host_cache_from_rows([r2], wl.cache.cap)
    f64 = lambda t: None if t is None else np_(t[b:b + 1]).astype(np.float64)  # noqa: E731
    layers = []
    for li, mode in enumerate(c["modes"]):
        inp = wl.inputs[li]
        L = dict(mode=mode, q=f64(inp["q"]), swa=_window_ref(inp, b))
        if mode == O.FULL:
            L.update(cache=host, q_idx=f64(inp["q_idx"]), w_idx=f64(inp["w_idx"]), pool=c["pool"],
                     q_idx2=f64(inp["q_idx2"]), w_idx2=f64(inp["w_idx2"]))
        elif mode == O.REINDEX:
            L.update(q_idx=f64(inp["q_idx"]), w_idx=f64(inp["w_idx"]),
                     keys_codes=own.idx_codes if own else None, keys_scales=own.idx_scales if own else None)
        layers.append(L)
    _, idxs = O.decode_step(layers, CF.TOPK)
    keys_main = O.entry_keys(host.idx_codes[0, :n], host.idx_scales[0, :n])
    keys_own = keys_main if own is None else O.entry_keys(own.idx_codes[0, :n], own.idx_scales[0, :n])
    pool_pos = None
    swaps = 0
    for li, mode in enumerate(c["modes"]):
        got_idx = np_(wl.indices[li][b])
        inp = wl.inputs[li]
        where = f"seq {b} layer {li}"
        qi, wi = f64(inp["q_idx"]), f64(inp["w_idx"])
        if mode == O.FULL:
            if c["pool"]:
                pool = O.topk_positions(O.indexer_scores(qi[0], wi[0], keys_main), c["pool"])
                pool_pos = pool[pool >= 0]
                s2 = O.indexer_scores(f64(inp["q_idx2"])[0], f64(inp["w_idx2"])[0], keys_main[pool_pos])
                swaps += Hh.assert_topk_match(got_idx, idxs[li][0], s2, positions=pool_pos, where=where)
            else:
                pool_pos = None
                s = O.indexer_scores(qi[0], wi[0], keys_main)
                swaps += Hh.assert_topk_match(got_idx, idxs[li][0], s, where=where)
        elif mode == O.REINDEX:
            if pool_pos is not None:
                s = O.indexer_scores(qi[0], wi[0], keys_own[pool_pos])
                swaps += Hh.assert_topk_match(got_idx, idxs[li][0], s, positions=pool_pos, where=where)
            else:
                s = O.indexer_scores(qi[0], wi[0], keys_own)
                swaps += Hh.assert_topk_match(got_idx, idxs[li][0], s, where=where)
        else:
            assert np.array_equal(got_idx, np_(wl.indices[li - 1][b])), where
        swa = _window_ref(inp, b)
        ref = O.attend(f64(inp["q"])[0], host.lat_codes[0], host.lat_scales[0], got_idx,
                       None if swa is None else swa[0])
        err = Hh.attn_rel_err(np_(wl.outputs[li][b]), ref)
        assert err <= Hh.ATTN_TOL, f"{where}: attention error {err:.3g} ({swaps} near-tie swaps so far)"
    return swaps


def _run(cfg_id, sample=None, **override):
    c = CF.config(cfg_id, **override)
    wl = CF.DecodeWorkload(c)
    wl()
    torch.cuda.synchronize()
    assert Hh.K.sync_status() == 0
    B = c["B"]
    n = int(wl.cache.len[0])
    for li in range(len(c["modes"])):  # properties on every sequence
        idx = wl.indices[li].cpu().numpy()
        for b in range(B):
            v = idx[b][idx[b] >= 0]
            assert len(v) == min(CF.TOPK, n) and np.all(np.diff(v) > 0) and v.max() < n
        assert torch.isfinite(wl.outputs[li]).all()
    for b in (range(B) if sample is None else sample):
        _check_sequence(wl, b)


def test_config0_tiny_ratio1_full_size():
    _run(0)


def test_config2_reduced():
    _run(2, B=3, tokens=2600)


def test_config3_reduced_hierarchical_pool():
    _run(3, B=2, tokens=2 * 20000)


def test_config4_reduced_group_with_window():
    _run(4, B=3, tokens=3000)


def test_fewer_entries_than_k():
    _run(2, B=2, tokens=300)


def test_pool_then_reindex_own_keys_then_reuse():
    """A Full layer builds the 16,384-candidate pool; the Reindex layer after it
    scores only the pool, with its own key array; Reuse takes its selection."""
    _run(3, B=2, tokens=2 * 20000, modes=(CF.FULL, CF.REINDEX, CF.REUSE), W=24, reindex_keys="own")


def test_pool_then_reindex_shared_keys_then_reuse():
    _run(3, B=2, tokens=2 * 20000, modes=(CF.FULL, CF.REINDEX, CF.REUSE), W=0, reindex_keys="shared")


def test_config4_reduced_fp8_window():
    """The decoder group with its windows packed as FP8 (E4M3, one E8M0 scale per 16)."""
    _run(4, B=3, tokens=3000, window="fp8")


def test_reindex_with_the_full_layers_keys():
    """The pages' reading of Reindex: the same indexer keys as the Full layer,
    rescored with the layer's own query."""
    _run(4, B=3, tokens=3000, reindex_keys="shared")


@pytest.mark.slow
def test_config2_full_size_sampled():
    _run(2, sample=[0, 4, 9, 13, 18, 22, 27, 31])


@pytest.mark.slow
def test_config3_full_size_sampled():
    _run(3, sample=list(range(8)))


@pytest.mark.slow
def test_config4_full_size_sampled():
    _run(4, sample=[0, 9, 18, 27, 36, 45, 54, 63])


def test_decode_step_misleading_sample_falls_back_exactly():
    """Top-k takes its candidate threshold from evenly spaced samples of each slice.
    Giving every 128th entry (a subset of the samples) much larger keys puts the
    thresholds inside that group, so too few candidates pass and the exact
    whole-row selection runs; the result must still equal the exact Top-512."""
    import torch
    import fp4_compressed_kv_append_b300 as K
    from fp4_compressed_kv_append_b300 import workloads as WL
    B, N, k = 2, 131072, 512
    cap = N + 128
    cache = K.Cache(B, cap)
    lc, ls, ic, isc = WL.random_cache_bytes(7, B, cap, device="cuda", scale_lo=118, scale_hi=122)
    sampled = (torch.arange(1024, device="cuda") * N) // 1024
    isc[:, sampled] = 134                                  # 2^7 larger key scales at the sampled positions
    for name, t in zip(("lat_codes", "lat_scales", "idx_codes", "idx_scales"), (lc, ls, ic, isc)):
        getattr(cache, name).copy_(t)
    cache.len.fill_(N)
    q, q_idx, w = WL.queries(7, 0, B, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(B, 64, 512, dtype=torch.float32, device="cuda")
    idx = torch.empty(B, k, dtype=torch.int32, device="cuda")
    K.DecodeStep([K.Layer(K.FULL, q, out, cache=cache, q_idx=q_idx, w_idx=w, idx_out=idx)], k)()
    torch.cuda.synchronize()
    assert K.sync_status() == 0
    for b in range(B):
        keys = O.entry_keys(np_(cache.idx_codes[b, :N]), np_(cache.idx_scales[b, :N]))
        s = O.indexer_scores(np_(q_idx[b]).astype(np.float64), np_(w[b]), keys)
        ref = O.topk_positions(s, k)
        Hh.assert_topk_match(np_(idx[b]), ref, s, where=f"seq {b}")


def test_selections_kept_in_the_workspace():
    """Eight layers (Full, Reindex, Reuse, Reindex, then four Reuse) whose selections
    stay in the workspace (no idx_out): the deferred attention then uses both
    workspace selections, is flushed when neither is free (before the second
    Reindex), and is split at four layers per launch. Every output equals, bit for
    bit, that of the same step with each selection in its own array, whose outputs
    are compared with the oracle first."""
    from fp4_compressed_kv_append_b300 import DecodeStep, Layer
    modes = (CF.FULL, CF.REINDEX, CF.REUSE, CF.REINDEX, CF.REUSE, CF.REUSE, CF.REUSE, CF.REUSE)
    c = CF.config(4, B=2, tokens=3000, modes=modes)
    wl = CF.DecodeWorkload(c)
    wl()
    torch.cuda.synchronize()
    assert Hh.K.sync_status() == 0
    for b in range(c["B"]):
        _check_sequence(wl, b)
    layers = [Layer(L.mode, L.q, torch.full_like(L.out, float("nan")), cache=L.cache, q_idx=L.q_idx, w_idx=L.w_idx,
                    own_idx_codes=L.own_idx_codes, own_idx_scales=L.own_idx_scales, pool=L.pool, q_idx2=L.q_idx2,
                    w_idx2=L.w_idx2, swa=L.swa) for L in wl.layers]
    DecodeStep(layers, CF.TOPK)()
    torch.cuda.synchronize()
    assert Hh.K.sync_status() == 0
    for li, (ref, L) in enumerate(zip(wl.outputs, layers)):
        assert torch.equal(ref, L.out), f"layer {li}"
