"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Every case is seeded and synthetic (fp4_compressed_kv_append_b300.workloads);
both sides consume the same source values; no expected value comes from the
CUDA path.
"""
import math

import numpy as np
import pytest
import torch

from tests import harness as Hh
from tests.harness import K, O, WL, np_

pytestmark = pytest.mark.gpu


def _rows_chunked(lat, ikey, ratio, w=None, chunk=4096):
    """Oracle rows of one sequence, in chunks of whole entries (entries are independent)."""
    step = chunk * ratio
    parts = [O.encode_entries(lat[i:i + step], ikey[i:i + step], ratio, *(w or [None] * 4))
             for i in range(0, lat.shape[0], step)]
    return tuple(np.concatenate([p[j] for p in parts]) for j in range(4))


# ============================================================== append
@pytest.mark.parametrize("T,ratio,kind", [(4096, 1, "lognormal"), (1337, 1, "lognormal"), (2 * 677, 2, "outlier"),
                                          (2 * 300, 2, "lognormal"), (1, 1, "outlier")])
def test_append_bit_exact(T, ratio, kind):
    seed = 0
    cap = ((T // ratio + 127) // 128) * 128 + 128
    w = WL.merge_weights(seed, device="cuda") if ratio == 2 else None
    B = 2
    cache = K.Cache(B, cap)
    for b in range(B):
        lat, ikey = Hh.sources(kind, seed, b, T, "cuda")
        K.kv_quant_append(lat[None], ikey[None], ratio, Hh.sub_view(cache, b), *(w or [None] * 4))
        rows = _rows_chunked(np_(lat), np_(ikey), ratio, None if w is None else [np_(x) for x in w])
        torch.cuda.synchronize()
        Hh.assert_rows_equal(cache, b, rows)
    assert K.sync_status() == 0


def test_append_full_cache_write_workload():
    """65,536 bf16 tokens with outlier channels, ratio 2 -> 32,768 entries, bit-exact."""
    seed, T = 0, 65536
    w = WL.merge_weights(seed, device="cuda")
    lat, ikey = WL.outlier_tokens(seed, 0, T, device="cuda")
    cache = K.Cache(1, 32768)
    K.kv_quant_append(lat[None], ikey[None], 2, cache, *w)
    rows = _rows_chunked(np_(lat), np_(ikey), 2, [np_(x) for x in w])
    torch.cuda.synchronize()
    Hh.assert_rows_equal(cache, 0, rows)


def test_append_in_two_calls_and_edge_values():
    """Appends land at len; zero, negative-zero, tiny, huge and saturating blocks."""
    rng = np.random.default_rng(5)
    lat = (rng.standard_normal((2, 40, 512)) * 3).astype(np.float32)
    key = (rng.standard_normal((2, 40, 128)) * 3).astype(np.float32)
    lat[0, 0, :16] = 0.0
    lat[0, 1, :16] = -0.0
    lat[0, 2, 16:32] *= 1e-6
    lat[0, 3, 32:48] *= 1e5
    lat[0, 4, 48:64] = 3e38
    key[0, 0, :32] = 0.0
    key[0, 1, :32] = -0.0
    key[0, 2, 32:64] = 2.0 ** -140
    key[0, 3, 64:96] = 3e38
    cache = K.Cache(2, 128)
    tl, tk = torch.from_numpy(lat).cuda(), torch.from_numpy(key).cuda()
    K.kv_quant_append(tl[:, :25].contiguous(), tk[:, :25].contiguous(), 1, cache)
    K.kv_quant_append(tl[:, 25:].contiguous(), tk[:, 25:].contiguous(), 1, cache)
    torch.cuda.synchronize()
    for b in range(2):
        Hh.assert_rows_equal(cache, b, O.encode_entries(lat[b], key[b], 1))


def _tie_rows(n_rows, rng):
    """Latent rows whose 16-channel blocks have amax = 6 s for an E4M3 scale s, so
    x / s lands exactly on every E2M1 tie point (0.25, 0.75, ..., 5), on the float32
    neighbours of the products t s, and on the grid; key rows whose 32-channel blocks
    have amax = 6 * 2^X, so x * 2^-X does the same for the MXFP4 codes."""
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 0.0],
                    np.float32)
    lat = np.zeros((n_rows, 512), np.float32)
    key = np.zeros((n_rows, 128), np.float32)
    for r in range(n_rows):
        for blk in range(32):
            e, m = int(rng.integers(-6, 7)), int(rng.integers(0, 8))
            sc = np.float32((1 + m / 8) * 2.0 ** e)
            v = (ties[rng.permutation(15)] * sc).astype(np.float32)
            way = rng.integers(0, 3, 15)  # exact product, next float up, next float down
            v = np.where(way == 1, np.nextafter(v, np.float32(np.inf)), v)
            v = np.where(way == 2, np.nextafter(v, np.float32(0)), v).astype(np.float32)
            v *= np.where(rng.integers(0, 2, 15) == 1, np.float32(-1), np.float32(1))
            lat[r, 16 * blk:16 * blk + 16] = np.concatenate([[np.float32(6) * sc], v])
        for blk in range(4):
            X = int(rng.integers(-20, 20))
            v = (np.concatenate([ties, ties[:15], [0.1, 0.2]]).astype(np.float32)[rng.permutation(32)] *
                 np.float32(2.0 ** X)).astype(np.float32)
            way = rng.integers(0, 3, 32)
            v = np.where(way == 1, np.nextafter(v, np.float32(np.inf)), v)
            v = np.where(way == 2, np.nextafter(v, np.float32(0)), v).astype(np.float32)
            v *= np.where(rng.integers(0, 2, 32) == 1, np.float32(-1), np.float32(1))
            v[0] = np.float32(6 * 2.0 ** X)
            key[r, 32 * blk:32 * blk + 32] = v
    return lat, key


def test_append_every_e2m1_tie_point_bit_exact():
    """The packing rounds x / s (and x * 2^-X) onto E2M1 with ties to the even code,
    saturating, keeping the sign of zero: every tie point, its float32 neighbours and
    the grid, with E4M3 scales of every mantissa, against the oracle."""
    rng = np.random.default_rng(11)
    lat, key = _tie_rows(96, rng)
    cache = K.Cache(1, 128)
    K.kv_quant_append(torch.from_numpy(lat)[None].cuda(), torch.from_numpy(key)[None].cuda(), 1, cache)
    torch.cuda.synchronize()
    Hh.assert_rows_equal(cache, 0, O.encode_entries(lat, key, 1))
    assert K.sync_status() == 0


def test_append_past_capacity_is_refused_on_device():
    cache = K.Cache(1, 128)
    lat, ikey = WL.lognormal_tokens(0, 0, 100, device="cuda")
    K.kv_quant_append(lat[None], ikey[None], 1, cache)
    K.kv_quant_append(lat[None], ikey[None], 1, cache)  # 200 > 128: refused
    assert K.sync_status() == K.A.ERR_BOUNDS
    assert int(cache.len[0]) == 100
    assert K.sync_status() == 0


def test_append_argument_errors():
    cache = K.Cache(1, 128)
    lat, ikey = WL.lognormal_tokens(0, 0, 3, device="cuda")
    with pytest.raises(K.Csa2Error) as e:
        K.kv_quant_append(lat[None], ikey[None], 2, cache, *WL.merge_weights(0, device="cuda"))
    assert e.value.status == K.A.ERR_ARG
    with pytest.raises(K.Csa2Error):
        K.kv_quant_append(lat[None], ikey[None], 3, cache)


# ============================================================== FP8 window rows
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_swa_quant_bit_exact(dtype):
    """FP8 window rows (E4M3 values, one E8M0 scale per 16) equal the oracle's, with
    zero, negative-zero, tiny, huge and saturating blocks."""
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((300, 512)) * np.exp(rng.uniform(-8, 8, (300, 1)))).astype(np.float32)
    x[0, :16], x[0, 16:32], x[1, 32:48] = 0.0, -0.0, 2.0 ** -140
    x[2, 48:64] = np.float32(3e38)
    x[3, 64:80] = np.float32(500.0) * (1 + np.arange(16) / 64)  # above 448 times 2^X: saturates
    t = torch.from_numpy(x).to(dtype).cuda()
    codes, scales = K.swa_quant(t)
    torch.cuda.synchronize()
    rc, rs = O.quantize_swa(np_(t))
    assert np.array_equal(np_(codes), rc) and np.array_equal(np_(scales), rs)
    assert K.sync_status() == 0


# ============================================================== indexer scores
def _small_cache(B, N, seed=1, cap=None):
    cap = cap or ((N + 127) // 128) * 128
    cache = Hh.build_gpu_cache("lognormal", seed, B, N, 1, cap)
    host = Hh.host_cache_from_rows([Hh.oracle_cache_rows("lognormal", seed, b, N, 1) for b in range(B)], cap)
    return cache, host


@pytest.mark.parametrize("cap", [2560, 2688])  # an even and an odd multiple of 128 rows
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_indexer_scores_within_fp32_bound(dtype, cap):
    B, N = 3, 2500
    cache, host = _small_cache(B, N, cap=cap)
    _, q_idx, w = WL.queries(1, "scan", B, 16, dtype=dtype, device="cuda")
    scores = K.indexer_score(q_idx, w, cache.idx_codes, cache.idx_scales, cache.len)
    torch.cuda.synchronize()
    for b in range(B):
        keys = O.entry_keys(host.idx_codes[b, :N], host.idx_scales[b, :N])
        ref = O.indexer_scores(np_(q_idx[b]).astype(np.float64), np_(w[b]), keys)
        tol = Hh.score_tolerance(np_(q_idx[b]), np_(w[b]), keys)
        err = np.abs(np_(scores[b, :N]).astype(np.float64) - ref)
        assert np.all(err <= tol), (b, float((err / tol).max()))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_indexer_scores_long_rows_ragged_lengths(dtype):
    # many 128-entry tiles per block, sequences that end inside a tile, an empty
    # sequence and a one-entry sequence; keys are uniformly random bytes
    B, cap = 5, 65536
    lens = [cap, 0, 1, 40001, cap - 1]
    _, _, ic, isc = WL.random_cache_bytes(11, B, cap, device="cuda", scale_lo=118, scale_hi=136)
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    _, q_idx, w = WL.queries(2, "scan", B, 16, dtype=dtype, device="cuda")
    scores = K.indexer_score(q_idx, w, ic, isc, ln)
    torch.cuda.synchronize()
    assert K.sync_status() == 0
    ic_h, isc_h = np_(ic), np_(isc)
    for b, n in enumerate(lens):
        if n == 0:
            continue
        keys = O.entry_keys(ic_h[b, :n], isc_h[b, :n])
        ref = O.indexer_scores(np_(q_idx[b]).astype(np.float64), np_(w[b]), keys)
        tol = Hh.score_tolerance(np_(q_idx[b]), np_(w[b]), keys)
        err = np.abs(np_(scores[b, :n]).astype(np.float64) - ref)
        assert np.all(err <= tol), (b, float((err / tol).max()))


def test_indexer_scores_on_candidates():
    B, N, P = 2, 1500, 700
    cache, host = _small_cache(B, N)
    _, q_idx, w = WL.queries(2, "scan", B, 16, device="cuda")
    g = torch.Generator().manual_seed(3)
    cand = torch.stack([torch.sort(torch.randperm(N, generator=g)[:P - 5]).values for _ in range(B)])
    cand = torch.cat([cand, -torch.ones(B, 5, dtype=torch.long)], 1).to(torch.int32).cuda()
    scores = K.indexer_score(q_idx, w, cache.idx_codes, cache.idx_scales, cache.len, cand=cand)
    torch.cuda.synchronize()
    for b in range(B):
        c = np_(cand[b])
        keys = O.entry_keys(host.idx_codes[b, c[c >= 0]], host.idx_scales[b, c[c >= 0]])
        ref = O.indexer_scores(np_(q_idx[b]).astype(np.float64), np_(w[b]), keys)
        tol = Hh.score_tolerance(np_(q_idx[b]), np_(w[b]), keys)
        got = np_(scores[b])
        assert np.all(np.abs(got[:P - 5] - ref) <= tol)
        assert np.all(np.isneginf(got[P - 5:]))


# ============================================================== Top-k
@pytest.mark.parametrize("n,k,ties", [(1, 1, 0), (7, 512, 0), (511, 512, 0), (512, 512, 0), (513, 512, 0),
                                      (4096, 512, 0), (4096, 512, 7), (131072, 512, 0), (131072, 512, 3000),
                                      (40000, 16384, 0), (5000, 1, 0), (3000, 600, 1)])
def test_topk_bit_exact(n, k, ties):
    B = 3
    s = WL.scores(n * 7 + k, B, n, device="cpu", ties=ties)
    s[0, : min(n, 5)] = -0.0                       # negative zeros tie with +0
    nvec = torch.tensor([n, max(n - 3, 0), n // 2], dtype=torch.int32)
    out = K.topk_select(s.cuda(), k, n=nvec.cuda())
    torch.cuda.synchronize()
    for b in range(B):
        m = int(nvec[b])
        ref = O.topk_positions(s[b, :m].numpy().astype(np.float64), k)
        assert np.array_equal(np_(out[b]), ref), b


def test_topk_with_candidates():
    B, P, k = 2, 16384, 512
    s = WL.scores(9, B, P, device="cpu", ties=50)
    g = torch.Generator().manual_seed(4)
    cand = torch.stack([torch.sort(torch.randperm(100000, generator=g)[:P - 100]).values for _ in range(B)])
    cand = torch.cat([cand, -torch.ones(B, 100, dtype=torch.long)], 1).to(torch.int32)
    out = K.topk_select(s.cuda(), k, cand=cand.cuda())
    torch.cuda.synchronize()
    for b in range(B):
        c = cand[b].numpy()
        ok = c >= 0
        ref = O.topk_positions(s[b].numpy()[ok].astype(np.float64), k, positions=c[ok])
        assert np.array_equal(np_(out[b]), ref)


# ============================================================== attention
@pytest.mark.parametrize("H,k,W,dtype", [(16, 512, 0, torch.float32), (64, 512, 0, torch.bfloat16),
                                         (32, 300, 0, torch.bfloat16), (64, 512, 128, torch.bfloat16),
                                         (64, 1, 77, torch.bfloat16), (64, 0, 128, torch.bfloat16),
                                         (16, 129, 5, torch.float32), (64, 0, 0, torch.bfloat16),
                                         (64, 512, 0, torch.float32), (64, 700, 100, torch.bfloat16),
                                         (64, 1024, 0, torch.bfloat16), (64, 1000, 24, torch.float32)])
def test_attention_within_2e3(H, k, W, dtype):
    B, N = 2, 1200
    cache, host = _small_cache(B, N, seed=4)
    q, q_idx, w = WL.queries(4, "attn", B, H, dtype=dtype, device="cuda")
    idx = np.full((B, k), -1, np.int64)
    for b in range(B):
        keys = O.entry_keys(host.idx_codes[b, :N], host.idx_scales[b, :N])
        if k:
            idx[b] = O.topk_positions(O.indexer_scores(np_(q_idx[b]).astype(np.float64), np_(w[b]), keys), k)
    swa = WL.window(4, 0, B, W, device="cuda") if W else None
    out = K.sparse_latent_attn(q, cache, torch.from_numpy(idx).to(torch.int32).cuda() if k else None, swa=swa)
    torch.cuda.synchronize()
    assert K.sync_status() == 0
    for b in range(B):
        ref = O.attend(np_(q[b]).astype(np.float64), host.lat_codes[b], host.lat_scales[b], idx[b],
                       None if swa is None else np_(swa[b]).astype(np.float64))
        err = Hh.attn_rel_err(np_(out[b]), ref)
        assert err <= Hh.ATTN_TOL, (b, err)


@pytest.mark.parametrize("H,k,W", [(64, 512, 128), (64, 0, 77), (16, 300, 40), (64, 1000, 24)])
def test_attention_fp8_window_within_2e3(H, k, W):
    """Window rows given as FP8 (the csa2_swa_quant format): the attention equals the
    oracle's over the dequantised rows (key-split form at H = 64, chunked at 16)."""
    B, N = 2, 1500
    cache, host = _small_cache(B, N, seed=4)
    q, _, _ = WL.queries(5, 0, B, H, dtype=torch.bfloat16, device="cuda")
    rows = WL.window(5, 0, B, W, device="cuda")
    codes, scales = K.swa_quant(rows)
    rng = np.random.default_rng(H + k + W)
    idx = np.stack([np.sort(rng.choice(N, k, replace=False)) for _ in range(B)]).astype(np.int32) if k else None
    out = K.sparse_latent_attn(q, cache, torch.from_numpy(idx).cuda() if k else None, swa=(codes, scales))
    torch.cuda.synchronize()
    assert K.sync_status() == 0
    for b in range(B):
        rc, rs = O.quantize_swa(np_(rows[b]))
        ref = O.attend(np_(q[b]).astype(np.float64), host.lat_codes[b], host.lat_scales[b],
                       idx[b] if k else -np.ones(1, np.int64), O.dequantize_swa(rc, rs))
        assert Hh.attn_rel_err(np_(out[b]), ref) <= Hh.ATTN_TOL, b


def test_attention_index_past_len_is_flagged():
    B, N = 1, 300
    cache, host = _small_cache(B, N, seed=5)
    q, _, _ = WL.queries(5, "attn", B, 64, device="cuda")
    idx = torch.arange(512, dtype=torch.int32, device="cuda")[None]
    K.sparse_latent_attn(q, cache, idx)
    assert K.sync_status() == K.A.ERR_BOUNDS
    assert K.sync_status() == 0


@pytest.mark.parametrize("sampled_high", [True, False])
def test_topk_unrepresentative_sample_takes_the_exact_fallback(sampled_high):
    """Scores built so that the evenly spaced sample misleads the threshold: either
    too few (sampled slots high) or too many (sampled slots low) keys pass the
    filter. The result must still be the exact Top-k."""
    B, n, k = 2, 131072, 512
    S = 4096  # sample size used for k <= 1024
    s = WL.scores(11, B, n, device="cpu") * 0.5 + 0.25
    sampled = (torch.arange(S) * n) // S
    if sampled_high:
        s[:, sampled] += 1.0          # only ~r slots reach the sampled threshold
    else:
        s[:, sampled] -= 0.25         # nearly every slot beats the sampled threshold
    out = K.topk_select(s.cuda(), k)
    torch.cuda.synchronize()
    for b in range(B):
        ref = O.topk_positions(s[b].numpy().astype(np.float64), k)
        assert np.array_equal(np_(out[b]), ref)


# rows at every cluster shape's limit and just past it (four 512-thread blocks up to
# 73,728 slots, eight up to 147,456, sixteen 1,024-thread blocks up to 589,824, then
# sixteen 512-thread blocks re-reading their slices: coalesced unordered passes,
# ordered rounds for the list gather (k = 512) and the output (k = 16,384)), and one
# of the decode cache's appended lengths; heavy ties send the bounded select to the
# histogram levels
@pytest.mark.parametrize("n,k", [(524288, 16384), (65536 + 77, 512), (20000, 1500), (147456, 512),
                                 (147456 + 13, 512), (135200, 512), (300001, 2048), (73728, 512),
                                 (73728 + 4, 512), (589824, 512), (589824 + 8, 2048), (600000, 512),
                                 (600003, 16384)])
def test_topk_large_rows(n, k):
    B = 2
    s = WL.scores(n + k, B, n, device="cpu", ties=100000)
    out = K.topk_select(s.cuda(), k)
    torch.cuda.synchronize()
    for b in range(B):
        ref = O.topk_positions(s[b].numpy().astype(np.float64), k)
        assert np.array_equal(np_(out[b]), ref)


@pytest.mark.parametrize("k,scale", [(512, 2.0 ** -12), (0, 2.0 ** -12), (512, 2.0 ** 12), (0, 2.0 ** 12)])
def test_attention_window_magnitudes_within_2e3(k, scale):
    """bf16 window rows far from unit scale but inside the fp16 range the window goes
    through: 2^-12 N(0,1) (many values fp16 subnormals) and 2^12 N(0,1) (up to about
    2e4), with and without selected entries."""
    B, N, H, W = 2, 1200, 64, 128
    cache, host = _small_cache(B, N, seed=6)
    q, _, _ = WL.queries(6, "attn", B, H, dtype=torch.bfloat16, device="cuda")
    rows = (WL.window(6, 0, B, W, device="cuda").float() * scale).to(torch.bfloat16)
    rng = np.random.default_rng(k + 7)
    idx = np.stack([np.sort(rng.choice(N, k, replace=False)) for _ in range(B)]).astype(np.int32) if k else None
    out = K.sparse_latent_attn(q, cache, torch.from_numpy(idx).cuda() if k else None, swa=rows)
    torch.cuda.synchronize()
    assert K.sync_status() == 0
    for b in range(B):
        ref = O.attend(np_(q[b]).astype(np.float64), host.lat_codes[b], host.lat_scales[b],
                       idx[b] if k else -np.ones(1, np.int64), np_(rows[b]).astype(np.float64))
        assert Hh.attn_rel_err(np_(out[b]), ref) <= Hh.ATTN_TOL, b


@pytest.mark.parametrize("per_row,W,qscale,win,dtype", [
    (1, 128, 1.0, "bf16", torch.bfloat16), (1, 128, 64.0, "bf16", torch.bfloat16),
    (1, 128, 64.0, "fp8", torch.bfloat16), (1, 0, 64.0, None, torch.bfloat16),
    (2, 128, 64.0, "bf16", torch.bfloat16), (3, 0, 64.0, None, torch.bfloat16),
    (1, 128, 64.0, "bf16", torch.float32)])
def test_attention_rows_beyond_the_sms_within_2e3(per_row, W, qscale, win, dtype):
    """More (sequence, 64-head) rows than SMs / per_row: the key-split form gives each
    row per_row blocks that take several 128-key chunks each (one block a row, no
    merge, at per_row = 1), with a running softmax per head. Queries scaled by 2^6
    make the softmax peaked, so later chunks pass a head's reference by more than
    2^8 and the accumulated O and sum are rescaled. fp32 queries keep one chunk per
    block whatever the row count."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B = sms + 12 if per_row == 1 else sms // per_row
    N, H, k, seed = 640, 64, 512, 8
    cache = Hh.build_gpu_cache("lognormal", seed, B, N, 1, N)
    q, _, _ = WL.queries(seed, "attn", B, H, dtype=dtype, device="cuda")
    q = (q.float() * qscale).to(dtype)  # a power of two: exact in either type
    rng = np.random.default_rng(per_row * 1000 + W + int(qscale))
    idx = np.stack([np.sort(rng.choice(N, k, replace=False)) for _ in range(B)]).astype(np.int32)
    rows = WL.window(seed, 0, B, W, device="cuda") if W else None
    swa = rows if win == "bf16" else K.swa_quant(rows) if win == "fp8" else None
    out = K.sparse_latent_attn(q, cache, torch.from_numpy(idx).cuda(), swa=swa)
    torch.cuda.synchronize()
    assert K.sync_status() == 0
    for b in sorted({0, 1, B // 2, B - 2, B - 1} | set(rng.choice(B, 5, replace=False).tolist())):
        host = Hh.host_cache_from_rows([Hh.oracle_cache_rows("lognormal", seed, b, N, 1)], N)
        wref = None
        if win == "bf16":
            wref = np_(rows[b]).astype(np.float64)
        elif win == "fp8":
            wref = O.dequantize_swa(*O.quantize_swa(np_(rows[b])))
        ref = O.attend(np_(q[b]).astype(np.float64), host.lat_codes[0], host.lat_scales[0], idx[b], wref)
        assert Hh.attn_rel_err(np_(out[b]), ref) <= Hh.ATTN_TOL, b
