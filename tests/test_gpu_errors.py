"""Error behaviour on the GPU: checked mode, device error flags, bad arguments (no fault, no hang).

Every bad index here is caught by a bounds check on the host or inside the
kernel before any memory access; nothing in this file faults the device.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture
def kvc():
    import paged_kv_cache_27_gb300 as m
    m.kvc_device_error_flags(clear=True)
    yield m
    m.kvc_set_checked_mode(False)
    m.kvc_device_error_flags(clear=True)


def session(wl):
    from paged_kv_cache_27_gb300.harness import DecodeSession
    return DecodeSession(wl).fill()


def test_checked_mode_rejects_bad_tables_and_contexts(kvc):
    wl = workloads.small_decode(1, B=2, Hq=4, Hkv=2, D=64, ctx=[20, 40])
    s = session(wl)
    kvc.kvc_set_checked_mode(True)
    s.step()  # valid inputs pass
    bad = s.block_table.clone()
    bad[1, 1] = wl.NB + 5
    with pytest.raises(kvc.KvcError) as e:
        kvc.paged_decode_attention(s.q[0], s.k_pool[0], s.v_pool[0], bad, s.context_lens, wl.scale, s.out[0],
                                   s.workspace, s.max_ctx)
    assert e.value.name == "KVC_ERR_INVALID"
    ctx0 = s.context_lens.clone()
    ctx0[0] = 0
    with pytest.raises(kvc.KvcError) as e:
        kvc.paged_decode_attention(s.q[0], s.k_pool[0], s.v_pool[0], s.block_table, ctx0, wl.scale, s.out[0],
                                   s.workspace, s.max_ctx)
    assert e.value.name == "KVC_ERR_CAPACITY"
    slots = torch.tensor([wl.NB * 16, 0], dtype=torch.int64, device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.kv_append(s.h, 0, s.k_new[0], s.v_new[0], slots)
    assert e.value.name == "KVC_ERR_CAPACITY"
    s.close()


def test_unchecked_bad_inputs_set_device_flags_without_faulting(kvc):
    wl = workloads.small_decode(2, B=3, Hq=4, Hkv=2, D=64, ctx=[20, 40, 60])
    s = session(wl)
    s.step()  # every position < ctx now holds real data (the pool is NaN-poisoned elsewhere)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    bad = s.block_table.clone()
    bad[1, 1] = -7  # in-kernel range check skips the block
    ctx = s.context_lens.clone()
    ctx[2] = 0  # in-kernel check writes zeros for this sequence
    out = torch.full_like(s.out[0], 5.0)
    kvc.paged_decode_attention(s.q[0], s.k_pool[0], s.v_pool[0], bad, ctx, wl.scale, out, s.workspace, s.max_ctx)
    torch.cuda.synchronize()
    f = kvc.kvc_device_error_flags(clear=True)
    assert f & kvc.DEVERR["BLOCK_ID"] and f & kvc.DEVERR["CONTEXT"]
    assert torch.isfinite(out).all()
    assert (out[2] == 0).all()
    # a slot past the pool is skipped by the append kernel and flagged
    before = s.k_pool.clone()
    slots = torch.tensor([wl.NB * 16 + 3, -1, -1], dtype=torch.int64, device="cuda")
    kvc.kv_append(s.h, 0, s.k_new[0], s.v_new[0], slots)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) & kvc.DEVERR["SLOT"]
    assert torch.equal(before.view(torch.int16), s.k_pool.view(torch.int16))
    s.close()


def test_bad_contexts_in_a_several_wave_batch(kvc):
    """400 ragged sequences (more CTAs than the GPU holds, dispatched longest first) with two bad context
    lengths: those two rows come out zero with the context flag set, every other row matches the oracle."""
    from oracle import paging as opaging
    from parity import check_attention
    ctx = np.random.default_rng(11).integers(1, 300, size=400)
    wl = workloads.small_decode(12, B=400, Hq=14, Hkv=2, D=64, ctx=ctx.tolist())
    s = session(wl)
    s.step()
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    ref, _, _ = opaging.decode_step(wl, 0)
    bad_ctx = s.context_lens.clone()
    bad_ctx[7] = 0
    bad_ctx[300] = s.max_ctx + 100
    out = torch.full_like(s.out[0], 5.0)
    kvc.paged_decode_attention(s.q[0], s.k_pool[0], s.v_pool[0], s.block_table, bad_ctx, wl.scale, out,
                               s.workspace, s.max_ctx)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) & kvc.DEVERR["CONTEXT"]
    assert (out[7] == 0).all() and (out[300] == 0).all()
    keep = np.ones(400, dtype=bool)
    keep[[7, 300]] = False
    check_attention(out[torch.from_numpy(keep).cuda()], ref[keep], "several-wave batch, good rows")
    s.close()


def test_argument_errors(kvc):
    wl = workloads.small_decode(3, B=2, Hq=4, Hkv=2, D=64, ctx=[20, 300])
    s = session(wl)
    small_ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    ns, bps, need = kvc.paged_decode_plan(2, 4, 2, 64, 300, blocks_per_split=1)
    assert ns == 19 and bps == 1 and need > 16  # 1 block per cluster of 1 CTA -> 19 partials in the workspace
    with pytest.raises(kvc.KvcError) as e:
        kvc.paged_decode_attention(s.q[0], s.k_pool[0], s.v_pool[0], s.block_table, s.context_lens, wl.scale,
                                   s.out[0], small_ws, s.max_ctx, blocks_per_split=1)
    assert e.value.name == "KVC_ERR_INVALID"
    q65 = torch.zeros((2, 130, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.paged_decode_attention(q65, s.k_pool[0], s.v_pool[0], s.block_table, s.context_lens, wl.scale,
                                   torch.empty_like(q65, dtype=torch.float32), s.workspace, s.max_ctx)
    assert e.value.name == "KVC_ERR_UNSUPPORTED"  # group of 65 query heads per KV head: beyond the 64 taken
    with pytest.raises(kvc.KvcError) as e:
        kvc.paged_decode_attention(s.q[0], s.k_pool[0], s.v_pool[0], s.block_table, s.context_lens, wl.scale,
                                   s.out[0], s.workspace, 10 ** 6)
    assert e.value.name == "KVC_ERR_CAPACITY"
    s.close()
