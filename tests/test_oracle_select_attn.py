"""Oracle pins: indexer scores, Top-k, the hierarchical pool, attention, window, modes."""
import math

import numpy as np
import torch

from oracle import csa2
from tests import oracle_pins as P


def test_scores_vs_brute_force():
    P.check_scores(csa2.indexer_scores)


def test_topk_vs_brute_force_with_ties():
    P.check_topk(csa2.topk_positions)


def test_hsi_special_cases():
    P.check_hsi(csa2.hsi_select, csa2.indexer_scores, csa2.topk_positions)


def test_attention_vs_library_sdpa_and_closed_forms():
    P.check_attention(csa2.sparse_attention)


def _cache(rng, B=2, n=700):
    lat = (rng.standard_normal((B, n, 512)) * np.exp(rng.standard_normal(512))).astype(np.float32)
    key = (rng.standard_normal((B, n, 128)) * np.exp(rng.standard_normal(128))).astype(np.float32)
    c = csa2.Cache(B, n + 4)
    csa2.append(c, lat, key, 1)
    return c


def test_attend_with_all_entries_equals_dense_attention():
    rng = np.random.default_rng(5)
    c = _cache(rng, 1, 300)
    q = rng.standard_normal((4, 512)) / math.sqrt(512)
    idx = np.concatenate([np.arange(300), -np.ones(212, np.int64)])
    v = csa2.entry_latents(c.lat_codes[0, :300], c.lat_scales[0, :300])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(v)[None], torch.from_numpy(v)[None],
        scale=1 / math.sqrt(512))[0].numpy()
    assert np.allclose(csa2.attend(q, c.lat_codes[0], c.lat_scales[0], idx), ref, rtol=1e-12, atol=1e-12)


def test_window_special_cases():
    rng = np.random.default_rng(6)
    c = _cache(rng, 1, 200)
    q = rng.standard_normal((4, 512)) / math.sqrt(512)
    idx = np.arange(50)
    no_win = csa2.attend(q, c.lat_codes[0], c.lat_scales[0], idx)
    assert np.array_equal(csa2.attend(q, c.lat_codes[0], c.lat_scales[0], idx, np.zeros((0, 512))), no_win)
    win = rng.standard_normal((16, 512))
    only_win = csa2.attend(q, c.lat_codes[0], c.lat_scales[0], -np.ones(8, np.int64), win)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(win)[None], torch.from_numpy(win)[None],
        scale=1 / math.sqrt(512))[0].numpy()
    assert np.allclose(only_win, ref, rtol=1e-12, atol=1e-12)


def test_modes_reuse_and_reindex():
    rng = np.random.default_rng(8)
    B, n, H, k = 2, 700, 4, 64
    c = _cache(rng, B, n)
    q = rng.standard_normal((B, H, 512)) / math.sqrt(512)
    q2 = rng.standard_normal((B, H, 512)) / math.sqrt(512)
    qi = rng.standard_normal((B, 4, 128)) / math.sqrt(128)
    wi = rng.uniform(0, 1, (B, 4))
    layers = [dict(mode=csa2.FULL, cache=c, q_idx=qi, w_idx=wi, q=q),
              dict(mode=csa2.REINDEX, q_idx=qi, w_idx=wi, q=q2),
              dict(mode=csa2.REUSE, q=q)]
    outs, idxs = csa2.decode_step(layers, k)
    # Reindex with the same keys and query selects what Full selected
    assert np.array_equal(idxs[1], idxs[0])
    # Reuse attends with the indices of the previous layer: same query -> same output as Full
    assert np.array_equal(outs[2], outs[0])
    for b in range(B):
        s = csa2.indexer_scores(qi[b], wi[b], csa2.entry_keys(c.idx_codes[b, :n], c.idx_scales[b, :n]))
        assert np.array_equal(idxs[0][b], csa2.topk_positions(s, k))
        assert np.allclose(outs[1][b], csa2.attend(q2[b], c.lat_codes[b], c.lat_scales[b], idxs[0][b]))


def test_attend_window_is_one_joint_softmax_with_the_entries():
    P.check_attend_window(csa2.attend)


def test_decode_modes_reindex_own_keys_pool_and_reuse():
    P.check_decode_modes(csa2.decode_step, csa2.FULL, csa2.REINDEX, csa2.REUSE)
