"""Oracle pins: scalar formats (E2M1, E4M3, E8M0) and the quantisers."""
import numpy as np

from oracle import csa2, formats as F
from tests import oracle_pins as P


def test_e2m1_decode_matches_format_definition():
    P.check_e2m1_decode(F.e2m1_decode)


def test_e2m1_encode_round_nearest_even_vs_exact_brute_force():
    P.check_e2m1_encode(F.e2m1_encode)


def test_e4m3_decode_matches_library_float8_e4m3fn():
    P.check_e4m3_decode(F.e4m3_decode)


def test_e4m3_encode_matches_library_cast_and_saturates():
    P.check_e4m3_encode(F.e4m3_encode)


def test_e8m0_and_exponent():
    P.check_e8m0(F.e8m0_decode, F.floor_log2)


def test_quantize_main_vs_exact_rational_brute_force():
    P.check_quantize_main_brute(csa2.quantize_main)


def test_quantize_main_invariants():
    P.check_quantize_main_invariants(csa2.quantize_main, csa2.dequantize_main)


def test_quantize_indexer_vs_brute_force_and_invariants():
    P.check_quantize_indexer(csa2.quantize_indexer, csa2.dequantize_indexer)


def test_nibble_packing_order():
    P.check_pack(csa2.pack_nibbles, csa2.unpack_nibbles)


def test_merge_ratio2_float32_rounding():
    P.check_merge(csa2.merge_ratio2)


def test_bf16_bits_exact():
    import torch
    x = torch.randn(1000).to(torch.bfloat16)
    got = F.bf16_bits_to_float(x.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(got, x.to(torch.float64).numpy())


def test_ratio2_with_unit_weights_equals_ratio1_of_even_tokens():
    rng = np.random.default_rng(1)
    lat = (rng.standard_normal((10, 512)) * 3).astype(np.float32)
    key = (rng.standard_normal((10, 128)) * 3).astype(np.float32)
    one = lambda n: np.ones(n, np.float32)  # noqa: E731
    zero = lambda n: np.zeros(n, np.float32)  # noqa: E731
    r2 = csa2.encode_entries(lat, key, 2, one(512), zero(512), one(128), zero(128))
    r1 = csa2.encode_entries(lat[0::2], key[0::2], 1)
    for a, b in zip(r2, r1):
        assert np.array_equal(a, b)


def test_fp8_window_rows_vs_exact_brute_force():
    from oracle import csa2
    P.check_quantize_swa(csa2.quantize_swa, csa2.dequantize_swa)
