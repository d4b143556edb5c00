"""Serving mix on the GPU: block pool, copy-on-write device copies, append and decode vs the oracle."""
import numpy as np
import pytest
import torch

from oracle import paging as opaging
import workloads
from parity import check_attention, check_cache_bits, owned_slots

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kw", [dict(B=20, group=4, prefix_len=64, ctx_lo=2, ctx_hi=140), dict()])
def test_serving_mix(kw):
    from paged_kv_cache_27_gb300 import harness, kvc_device_error_flags
    mix = workloads.shared_prefix_mix(**kw)
    got = harness.serving_mix(mix)
    ref = opaging.serving_mix(mix)
    assert kvc_device_error_flags(clear=True) == 0
    assert got["tables_before"] == ref["tables_before"]
    assert np.array_equal(got["block_table"], ref["block_table"])
    assert [tuple(map(int, c)) for c in got["copies"]] == [tuple(c) for c in ref["copies"]]
    assert len(ref["copies"]) > 0
    assert np.array_equal(got["slots"], ref["slots"])
    slots = owned_slots(ref["block_table"], mix.ctx, mix.bs)
    check_cache_bits(got["k_cache"], ref["k_cache"], slots, poison=False)
    check_cache_bits(got["v_cache"], ref["v_cache"], slots, poison=False)
    check_attention(got["out"], ref["out"], mix.name)


def test_block_cow_copies_every_layer():
    import paged_kv_cache_27_gb300 as kvc
    cfg = kvc.KvcConfig(num_layers=3, num_blocks=8, num_kv_heads=2, head_dim=64)
    k = torch.randn(cfg.pool_shape, device="cuda").half()
    v = torch.randn(cfg.pool_shape, device="cuda").half()
    h = kvc.kv_cache_create(cfg, k, v)
    try:
        a = kvc.kv_block_alloc(h)
        assert kvc.kv_block_cow(h, a) == a  # refcount 1: nothing to copy
        kvc.kv_block_share(h, a)
        k0, v0 = k.clone(), v.clone()
        nb = kvc.kv_block_cow(h, a)
        torch.cuda.synchronize()
        assert nb != a and kvc.kv_block_refcount(h, a) == 1 and kvc.kv_block_refcount(h, nb) == 1
        assert torch.equal(k[:, nb].view(torch.int16), k0[:, a].view(torch.int16))
        assert torch.equal(v[:, nb].view(torch.int16), v0[:, a].view(torch.int16))
        others = [i for i in range(8) if i != nb]
        assert torch.equal(k[:, others].view(torch.int16), k0[:, others].view(torch.int16))
        # a batch of copies
        k1, v1 = k.clone(), v.clone()
        kvc.kv_copy_blocks(h, [0, 1, 2], [5, 6, 7])
        torch.cuda.synchronize()
        assert torch.equal(k[:, 5:8].view(torch.int16), k1[:, 0:3].view(torch.int16))
        assert torch.equal(v[:, 5:8].view(torch.int16), v1[:, 0:3].view(torch.int16))
        assert torch.equal(k[:, 0:5].view(torch.int16), k1[:, 0:5].view(torch.int16))
    finally:
        kvc.kv_cache_destroy(h)
