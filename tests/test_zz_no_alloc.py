"""csa2_decode_step_static: the decode step for callers that cannot allocate device
memory (its scratch lives in an array built into the library).

It must give what the regular csa2_decode_step gives on the same inputs, call
after call (the built-in scratch is reused and keeps the previous call's
contents), and refuse a step whose scratch would not fit the array. This file
is collected last so that a run stopping at the first failure has run every
other test before it.
"""
import ctypes as C

import pytest
import torch

import fp4_compressed_kv_append_b300 as K
from fp4_compressed_kv_append_b300 import _abi as A
from fp4_compressed_kv_append_b300 import configs as CF
from tests import harness as Hh
from tests.harness import np_

pytestmark = pytest.mark.gpu


def _descs_with_fresh_outputs(wl):
    """The workload's layer descriptors, each with new out / idx_out buffers."""
    layers = []
    for L in wl.layers:
        layers.append(K.Layer(L.mode, L.q, torch.full_like(L.out, float("nan")), cache=L.cache, q_idx=L.q_idx,
                              w_idx=L.w_idx, own_idx_codes=L.own_idx_codes, own_idx_scales=L.own_idx_scales,
                              pool=L.pool, q_idx2=L.q_idx2, w_idx2=L.w_idx2, swa=L.swa,
                              idx_out=torch.full_like(L.idx_out, -7)))
    return layers, (A.LayerDesc * len(layers))(*[L.desc() for L in layers])


def test_static_step_matches_the_regular_step_twice():
    c = CF.config(4, B=3, tokens=3000)  # Full, Reindex, Reuse, Reuse with a 128-row window
    wl = CF.DecodeWorkload(c)
    wl()  # the regular step, caller-provided workspace
    torch.cuda.synchronize()
    assert K.sync_status() == 0
    ref_out = [L.out.clone() for L in wl.layers]
    ref_idx = [L.idx_out.clone() for L in wl.layers]

    layers, descs = _descs_with_fresh_outputs(wl)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        for L in layers:
            L.out.fill_(float("nan"))
            L.idx_out.fill_(-7)
        st = A.lib().csa2_decode_step_static(descs, len(layers), c["B"], c["H"], CF.TOPK, A.BF16, stream)
        assert st == A.OK, A.status_str(st)
        torch.cuda.synchronize()
        assert K.sync_status() == 0
        for li, L in enumerate(layers):
            assert torch.equal(L.idx_out, ref_idx[li]), (call, li)
            err = Hh.attn_rel_err(np_(L.out), np_(ref_out[li]))
            assert err <= Hh.ATTN_TOL, (call, li, err)


def test_static_step_refuses_a_step_larger_than_its_scratch():
    # 64 sequences x 1,048,576 entries of scores alone need 256 MiB > 24 MiB; the
    # refusal comes from the host-side size check, before anything touches memory
    base = 0x10000000
    cv = A.CacheView(base, base + 0x1000, base + 0x2000, base + 0x3000, base + 0x4000, 1 << 20, 64)
    lay = (A.LayerDesc * 1)()
    lay[0].mode, lay[0].cache = A.FULL, C.pointer(cv)
    lay[0].q, lay[0].out, lay[0].q_idx, lay[0].w_idx = base + 0x5000, base + 0x6000, base + 0x7000, base + 0x8000
    assert A.lib().csa2_workspace_size(64, 1 << 20, 64, 512, 0, 0) > A.STATIC_WS_BYTES
    st = A.lib().csa2_decode_step_static(lay, 1, 64, 64, 512, A.BF16, torch.cuda.current_stream().cuda_stream)
    assert st == A.ERR_WORKSPACE
