"""Oracle pins: the footprint arithmetic printed on the pages."""
import numpy as np

from oracle import csa2
from tests.oracle_pins import golden

G = golden("footprint.json")


def test_entry_bytes_288_and_68():
    assert csa2.entry_bytes(512, 16) == G["main_entry_bytes"]["value"]
    assert csa2.entry_bytes(512, None) == G["main_entry_bytes"]["data"]
    assert csa2.entry_bytes(128, 32) == G["indexer_entry_bytes"]["value"]
    assert csa2.entry_bytes(128, None) == G["indexer_entry_bytes"]["data"]
    # and the oracle's packed record sizes agree with them
    assert csa2.MAIN_CODE_BYTES + csa2.MAIN_SCALE_BYTES == 288
    assert csa2.IDX_CODE_BYTES + csa2.IDX_SCALE_BYTES == 68


def test_per_layer_table_and_890():
    main, idx = csa2.entry_bytes(512, 16), csa2.entry_bytes(128, 32)
    for layer, zone, ratio, m, i, tot in G["per_layer"]["rows"]:
        assert (main / ratio, idx / ratio, (main + idx) / ratio) == (m, i, tot), layer
    rows = G["per_layer"]["rows"]
    assert [sum(r[k] for r in rows) for k in (3, 4, 5)] == G["per_layer"]["total"]
    assert csa2.bytes_per_token() == G["bytes_per_token"]["value"]


def test_packed_append_writes_178_and_356_bytes_per_token():
    rng = np.random.default_rng(2)
    T = 64
    lat = rng.standard_normal((1, T, 512)).astype(np.float32)
    key = rng.standard_normal((1, T, 128)).astype(np.float32)
    w = [rng.uniform(0, 1, n).astype(np.float32) for n in (512, 512, 128, 128)]
    for ratio, per_token in ((2, 178.0), (1, 356.0)):
        c = csa2.Cache(1, T)
        csa2.append(c, lat, key, ratio, *w)
        n = int(c.len[0])
        written = n * (c.lat_codes.shape[2] + c.lat_scales.shape[2] + c.idx_codes.shape[2] + c.idx_scales.shape[2])
        assert written / T == per_token


def test_context_table():
    per_tok = csa2.bytes_per_token()
    for tokens, value, unit, places in G["context_table"]["rows"]:
        div = 2 ** 20 if unit == "MiB" else 2 ** 30
        assert round(tokens * per_tok / div, places) == value, tokens


def test_swa_and_ratios():
    swa = csa2.swa_bytes_per_sequence()
    assert round(swa / 2 ** 20, 2) == G["swa_per_sequence"]["value"]
    share = swa / (1048576 * csa2.bytes_per_token()) * 100
    assert round(share, 1) == G["swa_share_at_1M"]["value_percent"]
    # FP4 data against FP16: 4 bits instead of 16 per value
    fp16 = 512 * 2
    assert (1 - csa2.entry_bytes(512, None) / fp16) * 100 == G["fp4_vs_fp16_saving"]["value_percent"]
    s = G["session_1M_tokens"]
    assert round(1e6 * csa2.bytes_per_token() / 1e9, 1) == s["value_gb"]
    assert round(1e6 * s["previous_bytes_per_token"] / 1e9, 1) == s["previous_gb"]


def test_printed_880_and_832_do_not_follow_from_the_formula():
    with32 = csa2.bytes_per_token(main_block=32, idx_block=32)
    noscale = csa2.bytes_per_token(main_block=None, idx_block=None)
    assert (with32, noscale) == (850.0, 800.0)
    assert [with32, noscale] != G["not_reproducible"]["printed"]


def test_four_layer_store_writes_890_bytes_per_token():
    """Packing T tokens into the four source layers stores 890 bytes per token, with
    T/2 entries in each ratio-2 layer and T in the ratio-1 layer ('Le compte par
    couche', table and eq. 890)."""
    rng = np.random.default_rng(4)
    T = 96
    src = [(rng.standard_normal((T, 512)).astype(np.float32), rng.standard_normal((T, 128)).astype(np.float32))
           for _ in range(4)]
    w = [[rng.uniform(0, 1, n).astype(np.float32) for n in (512, 512, 128, 128)] if ratio == 2 else None
         for _, _, ratio in csa2.SOURCE_LAYERS]
    rows = csa2.store_entries(src, weights=w)
    stored = sum(sum(a.nbytes for a in r) for r in rows)
    assert stored / T == G["bytes_per_token"]["value"]
    assert [r[0].shape[0] for r in rows] == [T // 2, T // 2, T // 2, T]
    for (lat, key), (_, _, ratio), ww, r in zip(src, csa2.SOURCE_LAYERS, w, rows):
        ref = csa2.encode_entries(lat, key, ratio, *(ww or [None] * 4))
        assert all(np.array_equal(a, b) for a, b in zip(r, ref))
    # a 1,048,576-token session: 0.87 GiB
    per_tok = stored / T
    assert round(1048576 * per_tok / 2 ** 30, 2) == 0.87
