"""Planted mistakes: each test hands a pin a deliberately broken copy of an oracle
function (on the CPU, in the oracle only) and checks that the pin rejects it.
This shows the pins would catch a dropped term, a wrong sign, rounding rule,
index or operand order in the oracle itself."""
import math

import numpy as np
import pytest

from oracle import csa2, formats as F
from tests import oracle_pins as P


def _fails(check, *args):
    with pytest.raises((AssertionError, ValueError, IndexError)):
        check(*args)


def test_e2m1_ties_away_from_zero_is_caught():
    def bad(v):
        v = np.asarray(v, np.float64)
        a = np.abs(v)
        d = np.abs(a[..., None] - F.E2M1_MAGNITUDES)
        code = (d.shape[-1] - 1 - np.argmin(d[..., ::-1], axis=-1)).astype(np.uint8)  # ties upward
        return code | (np.signbit(v).astype(np.uint8) << 3)
    _fails(P.check_e2m1_encode, bad)


def test_e2m1_dropped_sign_is_caught():
    _fails(P.check_e2m1_encode, lambda v: F.e2m1_encode(np.abs(np.asarray(v))))


def test_e4m3_without_saturation_is_caught():
    def bad(v):
        v = np.asarray(v, np.float64)
        out = F.e4m3_encode(np.minimum(v, 448.0))
        return np.where(v > 448, np.uint8(0x7F), out)
    _fails(P.check_e4m3_encode, bad)


def test_scale_amax_over_4_is_caught():
    orig = F.e4m3_encode

    def bad_quant(x):
        x = np.asarray(x, np.float32)
        return csa2.quantize_main(x * np.float32(1.5))
    _fails(P.check_quantize_main_brute, bad_quant)
    assert F.e4m3_encode is orig


def test_indexer_exponent_off_by_one_is_caught(monkeypatch):
    real = csa2.indexer_shared_exponent
    monkeypatch.setattr(csa2, "indexer_shared_exponent", lambda a: np.clip(real(a) + 1, -127, 127))
    _fails(P.check_quantize_indexer, csa2.quantize_indexer, csa2.dequantize_indexer)


def test_swapped_nibbles_are_caught():
    bad = lambda c: (np.asarray(c)[..., 1::2] | (np.asarray(c)[..., 0::2] << 4)).astype(np.uint8)  # noqa: E731
    _fails(P.check_pack, bad, csa2.unpack_nibbles)


def test_merge_with_one_rounding_is_caught():
    def fused(x0, x1, w0, w1):
        return (np.asarray(x0, np.float64) * w0 + np.asarray(x1, np.float64) * w1).astype(np.float32)
    _fails(P.check_merge, fused)


def test_merge_with_swapped_weights_is_caught():
    _fails(P.check_merge, lambda x0, x1, w0, w1: csa2.merge_ratio2(x0, x1, w1, w0))


def test_scores_without_relu_or_with_a_dropped_head_are_caught():
    _fails(P.check_scores, lambda q, w, k: (k @ np.asarray(q).T) @ w)
    _fails(P.check_scores, lambda q, w, k: np.maximum(k @ np.asarray(q)[:3].T, 0) @ np.asarray(w)[:3])


def test_topk_wrong_tie_rule_or_order_is_caught():
    def ties_high(s, k, positions=None):
        s = np.asarray(s, np.float64)
        pos = np.arange(len(s)) if positions is None else np.asarray(positions)
        order = np.lexsort((-pos, -s))
        out = np.full(k, -1)
        ch = np.sort(pos[order[:k]])
        out[:len(ch)] = ch
        return out
    _fails(P.check_topk, ties_high)

    def descending(s, k, positions=None):
        out = csa2.topk_positions(s, k, positions)
        v = out[out >= 0][::-1]
        return np.concatenate([v, out[out < 0]])
    _fails(P.check_topk, descending)


def test_attention_missing_scale_or_transposed_softmax_is_caught():
    _fails(P.check_attention, lambda q, v, scale=None: csa2.sparse_attention(q, v, 1.0))

    def wrong_axis(q, v, scale=None):
        logits = (np.asarray(q) @ np.asarray(v).T) / math.sqrt(512)
        p = np.exp(logits - logits.max(0, keepdims=True))
        return (p / p.sum(0, keepdims=True)) @ v
    _fails(P.check_attention, wrong_axis)


def test_hsi_rescoring_with_the_wrong_indexer_is_caught():
    def bad(keys, q1, w1, q2, w2, pool=16384, k=512):
        return csa2.hsi_select(keys, q1, w1, q1, w1, pool, k)
    _fails(P.check_hsi, bad, csa2.indexer_scores, csa2.topk_positions)


def test_window_as_a_second_softmax_is_caught():
    def averaged(q, lc, ls, idx, swa=None, scale=None):  # two softmaxes, averaged
        a = csa2.attend(q, lc, ls, idx, None, scale)
        return a if swa is None or not len(swa) else 0.5 * (a + csa2.attend(q, lc, ls, -np.ones(1, int), swa, scale))
    _fails(P.check_attend_window, averaged)

    def summed(q, lc, ls, idx, swa=None, scale=None):  # two softmaxes, summed
        a = csa2.attend(q, lc, ls, idx, None, scale)
        return a if swa is None or not len(swa) else a + csa2.attend(q, lc, ls, -np.ones(1, int), swa, scale)
    _fails(P.check_attend_window, summed)

    _fails(P.check_attend_window, lambda q, lc, ls, idx, swa=None, scale=None: csa2.attend(q, lc, ls, idx))


def _modes(fn):
    P.check_decode_modes(fn, csa2.FULL, csa2.REINDEX, csa2.REUSE)


def test_reindex_scoring_the_full_layers_keys_is_caught():
    def full_keys(layers, k):
        return csa2.decode_step([{a: v for a, v in L.items() if a not in ("keys_codes", "keys_scales")}
                                 for L in layers], k)
    _fails(_modes, full_keys)


def test_reindex_ignoring_the_pool_is_caught():
    def no_pool(layers, k):
        outs, idxs = csa2.decode_step(layers, k)
        flat = [dict(L, pool=0) if L["mode"] == csa2.FULL else L for L in layers]
        outs2, idxs2 = csa2.decode_step(flat, k)  # later layers as if no pool had been built
        return outs[:1] + outs2[1:], idxs[:1] + idxs2[1:]
    _fails(_modes, no_pool)


def test_reuse_of_the_full_selection_instead_of_the_latest_is_caught():
    def reuse_full(layers, k):
        outs, idxs = csa2.decode_step(layers, k)
        first = [layers[0]] + [dict(mode=csa2.REUSE, q=L["q"], swa=L.get("swa")) for L in layers[1:]]
        outs2, idxs2 = csa2.decode_step(first, k)
        return ([o2 if L["mode"] == csa2.REUSE else o for L, o, o2 in zip(layers, outs, outs2)],
                [i2 if L["mode"] == csa2.REUSE else i for L, i, i2 in zip(layers, idxs, idxs2)])
    _fails(_modes, reuse_full)


def test_fp8_window_exponent_or_block_mistakes_are_caught(monkeypatch):
    real = csa2.quantize_swa

    def emax7(x):  # the scale exponent off by one
        x = np.asarray(x, np.float32)
        c, s = real(x * np.float32(2.0))
        return c, (s.astype(np.int64) - 1).astype(np.uint8)
    _fails(P.check_quantize_swa, emax7, csa2.dequantize_swa)

    def block32(x):  # one scale per 32 values
        x = np.asarray(x, np.float32)
        n = x.shape[0]
        b = x.reshape(n, 16, 32)
        amax = np.repeat(np.abs(b).max(-1, keepdims=True), 32, -1).reshape(n, 512)
        c, s = real(np.where(np.arange(512) % 16 == 0, amax * np.sign(x + 1e-30), x).astype(np.float32))
        return c, s
    _fails(P.check_quantize_swa, block32, csa2.dequantize_swa)
