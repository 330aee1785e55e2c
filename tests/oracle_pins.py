"""Pins of the CPU oracle: checks against page numbers, format definitions,
library routines, closed forms and brute force. Each ``check_*`` takes the
oracle function(s) it pins as arguments, so that ``test_oracle_mutations.py``
can hand it a deliberately broken copy and see the pin fail.

The brute-force references here are written independently of the oracle:
exact rational arithmetic (fractions.Fraction) and plain Python loops.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------ exact helpers
def round_f32(fr: Fraction) -> Fraction:
    """Exact round-to-nearest-even of a rational to IEEE binary32 (finite range)."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    q, r = divmod(a, ulp)
    if r > ulp / 2 or (r == ulp / 2 and q % 2 == 1):
        q += 1
    return sign * q * ulp


def e2m1_brute(v: Fraction, negative: bool | None = None) -> int:
    """Nearest E2M1 code by exhaustive search, ties to even mantissa, saturating.

    ``negative`` carries the sign of a zero input (a Fraction has no -0)."""
    mags = []
    for e in range(4):
        for m in range(2):
            val = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
            mags.append((val, e * 2 + m))
    a = abs(v)
    best = None
    for val, code in mags:
        d = abs(a - val)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    neg = (v < 0) if negative is None else negative
    return best[1] | (8 if neg else 0)


def e4m3_values():
    out = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            val = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
            out.append((val, e * 8 + m))
    return out


E4M3_TABLE = e4m3_values()


def e4m3_brute(v: Fraction) -> int:
    a = min(abs(v), Fraction(448))
    best = None
    for val, code in E4M3_TABLE:
        d = abs(a - val)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    return best[1] | (0x80 if v < 0 else 0)


def e2m1_test_values():
    """Tie points, their float32 neighbours, the grid itself, and random values."""
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 7.0, 100.0, 1e30, 3.0e38]
    vals = []
    for t in ties + grid:
        t32 = np.float32(t)
        vals += [t32, np.nextafter(t32, np.float32(np.inf)), np.nextafter(t32, np.float32(0))]
    rng = np.random.default_rng(123)
    vals += list(rng.uniform(0, 8, 400).astype(np.float32))
    vals = np.array(vals, dtype=np.float32)
    return np.concatenate([vals, -vals])


# ------------------------------------------------------------ format pins
def check_e2m1_decode(decode):
    ref = golden("e2m1_e8m0.json")["e2m1_values_by_code"]
    got = decode(np.arange(16))
    assert np.array_equal(got, np.array(ref)), got
    assert np.array_equal(np.signbit(got[8:]), np.ones(8, bool))


def check_e2m1_encode(encode):
    vals = e2m1_test_values()
    got = encode(vals)
    ref = [e2m1_brute(Fraction(float(x)), bool(np.signbit(x))) for x in vals]
    assert list(got) == ref
    # every code round-trips (the negative zero keeps its sign)
    codes = np.arange(16)
    from_defn = np.array(golden("e2m1_e8m0.json")["e2m1_values_by_code"])
    assert list(encode(from_defn)) == list(codes)


def check_e4m3_decode(decode):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = decode(np.arange(256))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def check_e4m3_encode(encode):
    rng = np.random.default_rng(7)
    finite = np.array([v for v, _ in E4M3_TABLE], dtype=np.float64)
    mids = (finite[1:] + finite[:-1]) / 2
    vals = [np.float32(x) for x in np.concatenate([finite, mids])]
    vals += [np.nextafter(np.float32(x), np.float32(np.inf)) for x in mids]
    vals += [np.nextafter(np.float32(x), np.float32(0)) for x in mids]
    vals += list(rng.uniform(0, 448, 500).astype(np.float32))
    vals += list(np.exp2(rng.uniform(-14, 9, 500)).astype(np.float32))
    vals = np.array(vals, dtype=np.float32)
    vals = vals[vals <= 448]
    vals = np.concatenate([vals, -vals])
    got = encode(vals)
    lib = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, lib)
    # saturation above the largest finite value (the library cast gives NaN there)
    big = np.array([448.0, 449.0, 464.0, 480.0, 1e6, 3e38], dtype=np.float32)
    assert list(encode(big)) == [0x7E] * 6
    for x in [0.3, 1e-3, 2.0 ** -10, 2.0 ** -10 * 1.0000001, 100.25]:
        assert encode(np.array([x], np.float32))[0] == e4m3_brute(Fraction(float(np.float32(x))))


def check_e8m0(decode, floor_log2):
    g = golden("e2m1_e8m0.json")
    assert decode(np.array([g["e8m0_bias"]]))[0] == 1.0
    assert math.isnan(decode(np.array([g["e8m0_nan_code"]]))[0])
    for c in (0, 1, 100, 127, 128, 254):
        assert decode(np.array([c]))[0] == 2.0 ** (c - 127)
    rng = np.random.default_rng(3)
    a = np.exp2(rng.uniform(-140, 120, 1000))
    a = np.concatenate([a, np.exp2(np.arange(-140, 120).astype(np.float64))])
    got = floor_log2(a)
    for x, e in zip(a, got):
        m, ex = math.frexp(float(x))
        assert e == ex - 1


# ------------------------------------------------------------ quantiser pins
def quant_main_brute(block):
    """Independent exact-rational restatement of the 16-channel block quantiser."""
    xs = [Fraction(float(x)) for x in block]
    amax = max(abs(x) for x in xs)
    ratio = round_f32(amax / 6)
    s_code = e4m3_brute(ratio)
    s_val = dict((c, v) for v, c in E4M3_TABLE)[s_code & 0x7F]
    if s_val == 0:
        return [0] * len(xs), s_code
    return [e2m1_brute(round_f32(x / s_val)) for x in xs], s_code


def check_quantize_main_brute(quantize_main):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((6, 512)) * np.exp(rng.standard_normal(512))).astype(np.float32)
    x[0, :16] = 0.0                       # all-zero block: scale 0
    x[1, 16:32] *= 1e-4                   # tiny block: subnormal scale
    x[2, 32:48] *= 1e4                    # huge block: saturated scale
    codes, scales = quantize_main(x)
    for n in range(x.shape[0]):
        for b in range(32):
            c_ref, s_ref = quant_main_brute(x[n, 16 * b:16 * b + 16])
            assert scales[n, b] == s_ref, (n, b)
            assert list(codes[n, 16 * b:16 * b + 16]) == c_ref, (n, b)


def check_quantize_main_invariants(quantize_main, dequantize_main):
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((64, 512)) * np.exp(rng.standard_normal(512))).astype(np.float32)
    codes, scales = quantize_main(x)
    xd = dequantize_main(codes, scales)
    # idempotence: Q(D(Q(x))) = Q(x) for normal-range scales
    c2, s2 = quantize_main(xd.astype(np.float32))
    sv = scales.astype(np.int64)
    normal = ((sv >> 3) & 15) >= 1
    blk_codes = codes.reshape(64, 32, 16)
    blk_c2 = c2.reshape(64, 32, 16)
    assert np.array_equal(blk_codes[normal], blk_c2[normal])
    assert np.array_equal(scales[normal], s2[normal])
    # the largest element of a normal-scale block encodes to +-6 (code 7)
    blocks = x.reshape(64, 32, 16)
    arg = np.abs(blocks).argmax(axis=-1)
    top = np.take_along_axis(blk_codes, arg[..., None], axis=-1)[..., 0] & 7
    assert np.all(top[normal] == 7)
    # reconstruction error at most half the local E2M1 gap (times the scale)
    from fractions import Fraction as Fr  # noqa: F401
    s = np.array([[float(dict((c, v) for v, c in E4M3_TABLE)[int(c) & 0x7F]) for c in row] for row in scales])
    err = np.abs(blocks.astype(np.float64) - xd.reshape(64, 32, 16)) / np.where(s == 0, 1, s)[..., None]
    mag = np.abs(blocks) / np.where(s == 0, 1, s)[..., None]
    half_gap = np.where(mag < 2, 0.25, np.where(mag < 4, 0.5, 1.0))
    assert np.all(err[normal] <= half_gap[normal] + 1e-12)


def quant_idx_brute(block):
    xs = [Fraction(float(x)) for x in block]
    amax = max(abs(x) for x in xs)
    if amax == 0:
        X = -127
    else:
        X = amax.numerator.bit_length() - amax.denominator.bit_length()
        if Fraction(2) ** X > amax:
            X -= 1
        X = max(-127, min(127, X - 2))
    return [e2m1_brute(x * Fraction(2) ** -X) for x in xs], X + 127


def check_quantize_indexer(quantize_indexer, dequantize_indexer):
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((40, 128)) * np.exp(rng.standard_normal(128))).astype(np.float32)
    x[0, :32] = 0.0
    x[1, 32:64] = 2.0 ** -140
    codes, e8 = quantize_indexer(x)
    for n in range(x.shape[0]):
        for b in range(4):
            c_ref, e_ref = quant_idx_brute(x[n, 32 * b:32 * b + 32])
            assert e8[n, b] == e_ref, (n, b)
            assert list(codes[n, 32 * b:32 * b + 32]) == c_ref, (n, b)
    xd = dequantize_indexer(codes, e8)
    c2, e2 = quantize_indexer(xd.astype(np.float32))
    assert np.array_equal(c2[2:], codes[2:]) and np.array_equal(e2[2:], e8[2:])
    # amax * 2**-X lies in [4, 8) for every non-degenerate block
    blocks = np.abs(x[2:].reshape(-1, 4, 32)).max(-1)
    scaled = blocks / np.exp2(e8[2:].astype(np.float64) - 127)
    assert np.all((scaled >= 4) & (scaled < 8))


def check_pack(pack_nibbles, unpack_nibbles):
    codes = np.array([[1, 2, 3, 4, 15, 0, 8, 7]], np.uint8)
    packed = pack_nibbles(codes)
    assert list(packed[0]) == [0x21, 0x43, 0x0F, 0x78]       # channel 2j in the low nibble
    assert np.array_equal(unpack_nibbles(packed), codes)


def check_merge(merge_ratio2):
    rng = np.random.default_rng(14)
    x0 = rng.standard_normal(300).astype(np.float32) * 10
    x1 = rng.standard_normal(300).astype(np.float32) * 10
    w0 = rng.uniform(0, 1, 300).astype(np.float32)
    w1 = rng.uniform(0, 1, 300).astype(np.float32)
    got = merge_ratio2(x0, x1, w0, w1)
    for i in range(300):
        p0 = round_f32(Fraction(float(w0[i])) * Fraction(float(x0[i])))
        p1 = round_f32(Fraction(float(w1[i])) * Fraction(float(x1[i])))
        assert Fraction(float(got[i])) == round_f32(p0 + p1), i
    one, zero = np.ones(300, np.float32), np.zeros(300, np.float32)
    assert np.array_equal(merge_ratio2(x0, x1, one, zero), x0)


# ------------------------------------------------------------ scoring / selection pins
def scores_brute(q, w, keys):
    out = []
    for t in range(keys.shape[0]):
        s = 0.0
        for h in range(q.shape[0]):
            d = math.fsum(float(q[h, c]) * float(keys[t, c]) for c in range(keys.shape[1]))
            s += float(w[h]) * max(0.0, d)
        out.append(s)
    return np.array(out)


def check_scores(indexer_scores):
    rng = np.random.default_rng(15)
    q = rng.standard_normal((4, 128)) / math.sqrt(128)
    w = rng.uniform(0, 1, 4)
    keys = rng.standard_normal((24, 128))
    got = indexer_scores(q, w, keys)
    assert np.allclose(got, scores_brute(q, w, keys), rtol=1e-12, atol=1e-12)
    assert np.all(got >= 0)
    onehot = np.array([0.0, 0.0, 1.0, 0.0])
    assert np.allclose(indexer_scores(q, onehot, keys), np.maximum(keys @ q[2], 0), rtol=1e-12, atol=1e-15)


def topk_brute(scores, k, positions=None):
    pos = list(range(len(scores))) if positions is None else [int(p) for p in positions]
    order = sorted(range(len(scores)), key=lambda i: (-float(scores[i]), pos[i]))
    chosen = sorted(pos[i] for i in order[:k])
    return chosen + [-1] * (k - len(chosen))


def check_topk(topk_positions):
    rng = np.random.default_rng(16)
    for n, k, levels in [(40, 7, 0), (40, 7, 3), (9, 12, 0), (64, 64, 2), (1, 1, 0), (0, 4, 0), (100, 30, 5)]:
        s = rng.uniform(0, 1, n)
        if levels:
            s = np.floor(s * levels) / levels
        assert list(topk_positions(s, k)) == topk_brute(s, k), (n, k, levels)
    s = np.zeros(20)
    assert list(topk_positions(s, 5)) == [0, 1, 2, 3, 4]
    s = rng.uniform(0, 1, 30)
    pos = np.sort(rng.choice(1000, 30, replace=False))
    assert list(topk_positions(s, 8, positions=pos)) == topk_brute(s, 8, pos)


def check_hsi(hsi_select, indexer_scores, topk_positions):
    rng = np.random.default_rng(17)
    keys = rng.standard_normal((300, 128))
    q1, q2 = rng.standard_normal((4, 128)), rng.standard_normal((4, 128))
    w1, w2 = rng.uniform(0, 1, 4), rng.uniform(0, 1, 4)
    flat = topk_positions(indexer_scores(q1, w1, keys), 20)
    sel, pool = hsi_select(keys, q1, w1, q1, w1, pool=64, k=20)
    assert np.array_equal(sel, flat)                               # same indexer twice
    sel2, pool2 = hsi_select(keys, q1, w1, q2, w2, pool=400, k=20)
    assert np.array_equal(sel2, topk_positions(indexer_scores(q2, w2, keys), 20))  # pool >= n
    sel3, pool3 = hsi_select(keys, q1, w1, q2, w2, pool=50, k=20)
    assert set(sel3[sel3 >= 0]) <= set(pool3[pool3 >= 0])            # result within the pool


def check_attention(sparse_attention):
    rng = np.random.default_rng(18)
    q = rng.standard_normal((5, 512)) / math.sqrt(512) * 30
    v = rng.standard_normal((37, 512))
    got = sparse_attention(q, v)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(v)[None], torch.from_numpy(v)[None],
        scale=1 / math.sqrt(512))[0].numpy()
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(sparse_attention(q, v[3:4]), np.repeat(v[3:4], 5, 0), rtol=0, atol=1e-15)
    assert np.allclose(sparse_attention(np.zeros((2, 512)), v), np.repeat(v.mean(0, keepdims=True), 2, 0),
                       rtol=1e-12, atol=1e-14)
    perm = rng.permutation(37)
    assert np.allclose(sparse_attention(q, v[perm]), got, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------ window and layer-mode pins
# Independent decoders of the packed cache bytes: the E2M1 value table of the golden
# file, torch's float8_e4m3fn cast for the main scales and 2^(e-127) for E8M0; nibbles
# split with plain integer arithmetic (channel 2j low, 2j+1 high).
def _nibbles_ref(packed):
    p = np.asarray(packed, np.int64)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.int64)
    out[..., 0::2] = p % 16
    out[..., 1::2] = p // 16
    return out


def latents_ref(lat_codes, lat_scales):
    """[n, 256] packed codes + [n, 32] E4M3 scale bytes -> float64 [n, 512]."""
    table = np.array(golden("e2m1_e8m0.json")["e2m1_values_by_code"], np.float64)
    vals = table[_nibbles_ref(lat_codes)]
    sc = torch.from_numpy(np.ascontiguousarray(lat_scales, np.uint8)).view(torch.float8_e4m3fn)
    sc = sc.to(torch.float64).numpy()
    return vals * np.repeat(sc, 16, axis=-1)


def keys_ref(idx_codes, idx_scales):
    """[n, 64] packed codes + [n, 4] E8M0 bytes -> float64 [n, 128]."""
    table = np.array(golden("e2m1_e8m0.json")["e2m1_values_by_code"], np.float64)
    vals = table[_nibbles_ref(idx_codes)]
    sc = np.exp2(np.asarray(idx_scales, np.float64) - golden("e2m1_e8m0.json")["e8m0_bias"])
    return vals * np.repeat(sc, 32, axis=-1)


def sdpa_ref(q, rows):
    """Dense float64 softmax attention of q [H, 512] over rows [m, 512] with K = V = rows,
    scale 1/sqrt(512) (torch's library routine)."""
    t = torch.from_numpy(np.ascontiguousarray(rows, np.float64))[None]
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(np.ascontiguousarray(q, np.float64))[None], t, t, scale=1 / math.sqrt(512))[0].numpy()


def random_cache_rows(rng, n):
    """Packed rows of n entries: every byte is a valid pair of E2M1 codes; E4M3 scale
    bytes 0x28..0x4F (about 0.25 to 15), E8M0 bytes 120..134."""
    return (rng.integers(0, 256, (n, 256), dtype=np.uint8), rng.integers(0x28, 0x50, (n, 32), dtype=np.uint8),
            rng.integers(0, 256, (n, 64), dtype=np.uint8), rng.integers(120, 135, (n, 4), dtype=np.uint8))


def check_attend_window(attend):
    """Selected entries and window rows share one softmax: attend over k > 0 entries
    and W > 0 window rows equals dense attention over the concatenation of the
    dequantised selected rows and the window rows ("Le cache KV en FP4", "La
    contrepartie : la fenetre glissante"; "890 octets", "Troisiemement")."""
    rng = np.random.default_rng(21)
    lc, ls, _, _ = random_cache_rows(rng, 400)
    lat = latents_ref(lc, ls)
    for k_sel, W, wscale in [(37, 5, 1.0), (200, 128, 3.0), (1, 1, 0.3), (300, 64, 8.0)]:
        q = rng.standard_normal((6, 512)) / math.sqrt(512) * 4
        sel = np.sort(rng.choice(400, k_sel, replace=False))
        idx = np.concatenate([sel, -np.ones(9, np.int64)])
        rng.shuffle(idx)
        win = rng.standard_normal((W, 512)) * wscale
        got = attend(q, lc, ls, idx, win)
        ref = sdpa_ref(q, np.concatenate([lat[sel], win]))
        assert np.allclose(got, ref, rtol=1e-11, atol=1e-12), (k_sel, W)
        # both halves carry weight: the joint result is neither part alone
        assert not np.allclose(got, sdpa_ref(q, lat[sel]), rtol=1e-6, atol=1e-9)
        assert not np.allclose(got, sdpa_ref(q, win), rtol=1e-6, atol=1e-9)


class _HostCache:
    """A plain container with the oracle cache's fields (no oracle code)."""

    def __init__(self, rows_per_seq):
        B, cap = len(rows_per_seq), max(r[0].shape[0] for r in rows_per_seq) + 8
        self.batch, self.cap = B, cap
        self.lat_codes = np.zeros((B, cap, 256), np.uint8)
        self.lat_scales = np.zeros((B, cap, 32), np.uint8)
        self.idx_codes = np.zeros((B, cap, 64), np.uint8)
        self.idx_scales = np.zeros((B, cap, 4), np.uint8)
        self.len = np.zeros(B, np.int64)
        for b, (lc, ls, ic, isc) in enumerate(rows_per_seq):
            n = lc.shape[0]
            self.lat_codes[b, :n], self.lat_scales[b, :n] = lc, ls
            self.idx_codes[b, :n], self.idx_scales[b, :n] = ic, isc
            self.len[b] = n


def check_decode_modes(decode_step, FULL, REINDEX, REUSE):
    """Layer modes ("890 octets de cache KV par token", "Deuxiemement"):
      * a Reindex layer with its own key array selects the Top-k of its own query
        scored against THOSE keys and attends over the Full layer's main KV;
      * after a Full layer that built a hierarchical pool, a Reindex layer (own keys
        or the shared ones) ranks only the pool's positions;
      * Reuse attends, with its own query, over the latest Full/Reindex selection.
    References: brute-force scores (math.fsum) and Top-k (sorted), dense attention
    by the library routine, keys and latents decoded by the independent decoders."""
    rng = np.random.default_rng(22)
    B, n, H, k, P = 2, 300, 4, 8, 40
    rows = [random_cache_rows(rng, n) for _ in range(B)]
    own = [random_cache_rows(rng, n) for _ in range(B)]
    main, own_c = _HostCache(rows), _HostCache(own)
    q = [rng.standard_normal((B, H, 512)) / math.sqrt(512) * 4 for _ in range(3)]
    qi = [rng.standard_normal((B, 4, 128)) / math.sqrt(128) for _ in range(3)]
    wi = [rng.uniform(0, 1, (B, 4)) for _ in range(3)]

    def brute_sel(b, qq, ww, keys, positions):
        s = scores_brute(qq, ww, keys[positions])
        return topk_brute(s, k, positions)

    # --- Full -> Reindex (own keys) -> Reuse, no pool
    layers = [dict(mode=FULL, cache=main, q_idx=qi[0], w_idx=wi[0], q=q[0]),
              dict(mode=REINDEX, keys_codes=own_c.idx_codes, keys_scales=own_c.idx_scales, q_idx=qi[1],
                   w_idx=wi[1], q=q[1]),
              dict(mode=REUSE, q=q[2])]
    outs, idxs = decode_step(layers, k)
    for b in range(B):
        km, ko = keys_ref(rows[b][2], rows[b][3]), keys_ref(own[b][2], own[b][3])
        lat = latents_ref(rows[b][0], rows[b][1])
        allpos = list(range(n))
        e0 = brute_sel(b, qi[0][b], wi[0][b], km, allpos)
        e1 = brute_sel(b, qi[1][b], wi[1][b], ko, allpos)
        assert e1 != brute_sel(b, qi[1][b], wi[1][b], km, allpos)  # own keys decide
        assert list(idxs[0][b]) == e0 and list(idxs[1][b]) == e1 and list(idxs[2][b]) == e1
        assert np.allclose(outs[0][b], sdpa_ref(q[0][b], lat[e0]), rtol=1e-11, atol=1e-12)
        assert np.allclose(outs[1][b], sdpa_ref(q[1][b], lat[e1]), rtol=1e-11, atol=1e-12)
        assert np.allclose(outs[2][b], sdpa_ref(q[2][b], lat[e1]), rtol=1e-11, atol=1e-12)

    # --- Full with a pool -> Reindex (shared keys) -> Reindex (own keys) -> Reuse
    qp, wp = rng.standard_normal((B, 4, 128)) / math.sqrt(128), rng.uniform(0, 1, (B, 4))
    layers = [dict(mode=FULL, cache=main, q_idx=qi[0], w_idx=wi[0], pool=P, q_idx2=qp, w_idx2=wp, q=q[0]),
              dict(mode=REINDEX, q_idx=qi[1], w_idx=wi[1], q=q[1]),
              dict(mode=REINDEX, keys_codes=own_c.idx_codes, keys_scales=own_c.idx_scales, q_idx=qi[2],
                   w_idx=wi[2], q=q[2]),
              dict(mode=REUSE, q=q[1])]
    outs, idxs = decode_step(layers, k)
    for b in range(B):
        km, ko = keys_ref(rows[b][2], rows[b][3]), keys_ref(own[b][2], own[b][3])
        lat = latents_ref(rows[b][0], rows[b][1])
        pool = [p for p in topk_brute(scores_brute(qi[0][b], wi[0][b], km), P) if p >= 0]
        e0 = brute_sel(b, qp[b], wp[b], km, pool)
        e1 = brute_sel(b, qi[1][b], wi[1][b], km, pool)
        e2 = brute_sel(b, qi[2][b], wi[2][b], ko, pool)
        assert e1 != brute_sel(b, qi[1][b], wi[1][b], km, list(range(n)))  # the pool decides
        assert e2 != brute_sel(b, qi[2][b], wi[2][b], ko, list(range(n)))
        assert [list(idxs[i][b]) for i in range(4)] == [e0, e1, e2, e2]
        for i, (qq, sel) in enumerate([(q[0], e0), (q[1], e1), (q[2], e2), (q[1], e2)]):
            assert np.allclose(outs[i][b], sdpa_ref(qq[b], lat[sel]), rtol=1e-11, atol=1e-12), i


# ------------------------------------------------------------ FP8 window pins
def swa_block_brute(block):
    """Exact restatement of one 16-value FP8 window block: X = floor(log2 amax) - 8
    (by exact rational comparison), E4M3 of x * 2^-X by exhaustive nearest search."""
    xs = [Fraction(float(x)) for x in block]
    amax = max(abs(x) for x in xs)
    if amax == 0:
        return [0x80 if np.signbit(np.float32(x)) else 0 for x in block], 0
    e = 0
    while Fraction(2) ** (e + 1) <= amax:
        e += 1
    while Fraction(2) ** e > amax:
        e -= 1
    X = max(min(e - 8, 127), -127)
    codes = []
    for x, xf in zip(block, xs):
        v = xf * Fraction(2) ** -X
        c = e4m3_brute(v)
        if v == 0 and np.signbit(np.float32(x)):
            c |= 0x80
        codes.append(c)
    return codes, X + 127


def check_quantize_swa(quantize_swa, dequantize_swa):
    rng = np.random.default_rng(31)
    x = (rng.standard_normal((6, 512)) * np.exp(rng.uniform(-6, 6, (6, 1)))).astype(np.float32)
    x[0, :16] = 0.0
    x[0, 16:32] = -0.0
    x[1, 32:48] *= 1e-30
    x[2, 48:64] = np.float32(1e30)
    codes, scales = quantize_swa(x)
    assert codes.shape == (6, 512) and scales.shape == (6, 32)
    assert codes.nbytes / 6 + scales.nbytes / 6 == 512 + 32  # 544 bytes per window token
    for r in range(6):
        for blk in range(32):
            c, s = swa_block_brute(x[r, 16 * blk:16 * blk + 16])
            assert list(codes[r, 16 * blk:16 * blk + 16]) == c and scales[r, blk] == s, (r, blk)
    d = dequantize_swa(codes, scales)
    c2, s2 = quantize_swa(d.astype(np.float32))
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)  # idempotent
    # the E4M3 decode of the codes times 2^(e - 127) is the dequantised value
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(d, ref * np.repeat(np.exp2(scales.astype(np.float64) - 127), 16, axis=1))
