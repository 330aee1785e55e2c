"""The multi-layer store ("Le cache KV en FP4", "Le compte par couche"): one
csa2_store_append writes every source layer -- 2, 8 and 14 at ratio 2, 20 at
ratio 1 -- bit-exact against the oracle, 890 bytes per token."""
import numpy as np
import pytest
import torch

import fp4_compressed_kv_append_b300 as K
from fp4_compressed_kv_append_b300 import configs as CF
from oracle import csa2 as O
from tests import harness as Hh
from tests import oracle_pool as OP
from tests.harness import np_

pytestmark = pytest.mark.gpu


def _layer_ref(st, li, t0, t1):
    """The oracle's rows of layer li for source tokens [t0, t1) of sequence 0."""
    (lat, ikey), (_, ratio), w = st.sources[li], st.c["layers"][li], st.weights[li]
    ww = None if w is None else [np_(x) for x in w]
    return OP.encode_rows(np_(lat[0, t0:t1]), np_(ikey[0, t0:t1]), ratio, ww)


def _check_rows(st, li, e0, rows):
    cache = st.caches[li]
    n = rows[0].shape[0]
    for name, ref in zip(("lat_codes", "lat_scales", "idx_codes", "idx_scales"), rows):
        got = np_(getattr(cache, name)[0, e0:e0 + n])
        assert np.array_equal(got, ref), (li, name, e0)


def test_store_four_layers_in_two_calls_bit_exact_890_bytes_per_token():
    c = CF.config(5)
    T = 6000
    st = CF.StoreWorkload(c, T=T)
    half = T // 2
    for t0 in (0, half):  # two appends of 3,000 tokens each
        K.store_append([(lat[:, t0:t0 + half].contiguous(), ikey[:, t0:t0 + half].contiguous(), ratio, cache, w)
                        for (lat, ikey, ratio, cache, w) in st.layers()])
    torch.cuda.synchronize()
    assert Hh.K.sync_status() == 0
    for li, (_, ratio) in enumerate(c["layers"]):
        assert int(st.caches[li].len[0]) == T // ratio
        _check_rows(st, li, 0, _layer_ref(st, li, 0, T))
    assert st.stored_bytes() / T == 890


@pytest.mark.slow
def test_store_one_million_tokens_is_0_87_GiB_and_sampled_rows_bit_exact():
    c = CF.config(5)
    st = CF.StoreWorkload(c)
    st()
    torch.cuda.synchronize()
    assert Hh.K.sync_status() == 0
    T = c["tokens"]
    assert st.stored_bytes() == 890 * T
    assert round(st.stored_bytes() / 2 ** 30, 2) == 0.87
    for li, (_, ratio) in enumerate(c["layers"]):
        n = T // ratio
        for e0 in (0, n // 2 - 1000, n - 2048):  # start, middle, end
            _check_rows(st, li, e0, _layer_ref(st, li, e0 * ratio, (e0 + 2048) * ratio))
