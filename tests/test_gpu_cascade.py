"""Cascade (shared-prefix) decode on the GPU vs the oracle's plain decode over the full tables."""
import numpy as np
import pytest
import torch

import oracle
from oracle import paging as opaging
import workloads
from parity import check_attention

pytestmark = pytest.mark.gpu

DEFAULT_MIN_SAVED = 36000  # the library's default routing threshold (saved block reads)


@pytest.fixture(autouse=True)
def always_cascade():
    """These tests exercise the cascade kernels themselves: route every call to them, whatever its prefix."""
    import paged_kv_cache_27_gb300 as kvc
    kvc.kvc_set_cascade_min_saved_blocks(0)
    yield
    kvc.kvc_set_cascade_min_saved_blocks(DEFAULT_MIN_SAVED)


def run_cascade(wl, out_dtype=torch.float32, checked=False, group_start=None, shared=None, max_shared=None):
    import paged_kv_cache_27_gb300 as kvc
    dev = "cuda"
    q = torch.from_numpy(wl.q).to(dev)
    kp, vp = torch.from_numpy(wl.k_pool).to(dev), torch.from_numpy(wl.v_pool).to(dev)
    table = torch.from_numpy(wl.block_table).to(dev)
    ctx = torch.from_numpy(wl.ctx).to(dev)
    gs_h = wl.group_start if group_start is None else group_start
    sh_h = wl.shared_blocks if shared is None else shared
    mx = int(sh_h.max()) if max_shared is None else max_shared
    gs, sh = torch.from_numpy(gs_h).to(dev), torch.from_numpy(sh_h).to(dev)
    B = wl.q.shape[0]
    max_ctx = int(wl.ctx.max())
    ws = kvc.paged_decode_cascade_plan(B, wl.Hq, wl.Hkv, wl.D, max_ctx, len(gs_h) - 1, mx)
    workspace = torch.full((max(ws, 16),), 0x7F, dtype=torch.uint8, device=dev)  # no reliance on zeroed scratch
    out = torch.empty((B, wl.Hq, wl.D), dtype=out_dtype, device=dev)
    kvc.kvc_set_checked_mode(checked)
    try:
        kvc.paged_decode_cascade_attention(q, kp, vp, table, ctx, gs, sh, mx, wl.scale, out, workspace, max_ctx)
        torch.cuda.synchronize()
    finally:
        kvc.kvc_set_checked_mode(False)
    # the plain decode on the same inputs, for a tight agreement check
    _, _, pws = kvc.paged_decode_plan(B, wl.Hq, wl.Hkv, wl.D, max_ctx)
    pout = torch.empty_like(out, dtype=torch.float32)
    kvc.paged_decode_attention(q, kp, vp, table, ctx, wl.scale, pout,
                               torch.empty(max(pws, 16), dtype=torch.uint8, device=dev), max_ctx)
    torch.cuda.synchronize()
    return out, pout


def oracle_out(wl):
    return oracle.decode(wl.q, wl.k_pool, wl.v_pool, wl.block_table, wl.ctx, wl.scale)


CASES = [
    # group sizes, shared blocks per group, private tokens per sequence, Hq, Hkv, D
    ([8, 8, 8], [32, 5, 0], None, 14, 2, 64),
    ([1, 2, 3, 8], [1, 7, 40, 3], [1, 16, 17, 2, 3, 200, 1, 1, 15, 16, 17, 31, 32, 33], 14, 2, 64),
    ([4, 4], [10, 2], None, 8, 8, 128),
    ([8], [300], [1, 2, 3, 50, 100, 16, 17, 8], 14, 2, 64),
    ([5, 1, 7], [64, 12, 1], None, 16, 2, 128),
    ([8, 3], [24, 9], None, 64, 4, 64),  # 16 query heads per KV head: 128 prefix rows, the mma.sync prefix
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_cascade_matches_oracle(case, out_dtype):
    import paged_kv_cache_27_gb300 as kvc
    sizes, shared, extra, Hq, Hkv, D = CASES[case]
    B = sum(sizes)
    if extra is None:
        extra = list(np.random.default_rng(case).integers(1, 400, size=B))
    wl = workloads.cascade_decode(1000 + case, sizes, shared, extra, Hq=Hq, Hkv=Hkv, D=D)
    out, pout = run_cascade(wl, out_dtype, checked=(case % 2 == 0))
    assert kvc.kvc_device_error_flags(clear=True) == 0
    check_attention(out, oracle_out(wl), f"cascade case {case}")
    if out_dtype == torch.float32:  # same math, different merge order: agrees with the plain decode closely
        assert (out - pout).abs().max().item() < 1e-5


def test_cascade_serving_mix():
    """The shared-prefix mix after its step: the groups the pool left sharing their prefix blocks, read once each."""
    import paged_kv_cache_27_gb300 as kvc
    from paged_kv_cache_27_gb300 import harness
    mix = workloads.shared_prefix_mix()
    got = harness.serving_mix(mix)
    ref = opaging.serving_mix(mix)
    table = got["block_table"]
    gs, sh, mx = kvc.kv_cascade_groups(table, mix.ctx)
    assert mx == mix.prefix_len // mix.bs
    dev = "cuda"
    max_ctx = int(mix.ctx.max())
    ws = kvc.paged_decode_cascade_plan(mix.B, mix.Hq, mix.Hkv, mix.D, max_ctx, len(gs) - 1, mx)
    out = torch.empty((mix.B, mix.Hq, mix.D), dtype=torch.float32, device=dev)
    kvc.paged_decode_cascade_attention(
        torch.from_numpy(mix.q).to(dev), got["k_cache"], got["v_cache"], torch.from_numpy(table).to(dev),
        torch.from_numpy(mix.ctx).to(dev), torch.from_numpy(gs).to(dev), torch.from_numpy(sh).to(dev), mx,
        mix.scale, out, torch.empty(ws, dtype=torch.uint8, device=dev), max_ctx)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    check_attention(out, ref["out"], "serving mix, cascade")


def test_cascade_checked_mode_rejects_bad_groups():
    import paged_kv_cache_27_gb300 as kvc
    wl = workloads.cascade_decode(7, [4, 4], [6, 3], [5] * 8)
    # a member whose row does not really begin with the group's blocks
    bad = wl.block_table.copy()
    bad[2, 4], bad[2, 6] = bad[2, 6], bad[2, 4]  # a shared entry swapped with the member's private block
    wl_bad = workloads.CascadeWorkload(**{**wl.__dict__, "block_table": bad})
    with pytest.raises(kvc.KvcError) as e:
        run_cascade(wl_bad, checked=True)
    assert "KVC_ERR_INVALID" in str(e.value)
    # more shared blocks than the members' contexts hold (16 * 7 > 6 * 16 + 5)
    sh = wl.shared_blocks.copy()
    sh[:4] = 7
    with pytest.raises(kvc.KvcError):
        run_cascade(wl, checked=True, shared=sh)
    # a group of nine
    wl9 = workloads.cascade_decode(8, [9], [2], [3] * 9)
    with pytest.raises(kvc.KvcError):
        run_cascade(wl9, checked=True)
    assert kvc.kvc_device_error_flags(clear=True) == 0


def test_cascade_unchecked_oversized_group_sets_flag():
    """Unchecked, a group of nine is reported through the device error word (its outputs are undefined)."""
    import paged_kv_cache_27_gb300 as kvc
    wl9 = workloads.cascade_decode(9, [9], [2], [3] * 9)
    run_cascade(wl9, checked=False)
    assert kvc.kvc_device_error_flags(clear=True) & kvc.DEVERR["CONTEXT"]


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 14, 2), (128, 8, 8)])
def test_cascade_unchecked_bad_shared_block_flagged(D, Hq, Hkv):
    """Unchecked, an out-of-range id among a group's shared blocks is skipped and flagged, every output stays finite,
    and the other group is still right (D = 64 runs the tensor-core prefix pass, D = 128 the mma.sync one)."""
    import paged_kv_cache_27_gb300 as kvc
    kvc.kvc_device_error_flags(clear=True)
    wl = workloads.cascade_decode(21, [4, 4], [6, 3], [5] * 8, Hq=Hq, Hkv=Hkv, D=D)
    bad = wl.block_table.copy()
    bad[:4, 2] = wl.NB + 7  # the first group's third shared block, in every member's row
    wl_bad = workloads.CascadeWorkload(**{**wl.__dict__, "block_table": bad})
    out, _ = run_cascade(wl_bad, checked=False)
    assert kvc.kvc_device_error_flags(clear=True) & kvc.DEVERR["BLOCK_ID"]
    assert torch.isfinite(out).all()
    ref = oracle_out(wl)
    check_attention(out[4:], ref[4:], f"cascade D={D}, the group without the bad block")


@pytest.mark.parametrize("scale_sign", [1.0, -1.0])
def test_cascade_full_group_rows_and_scale_sign(scale_sign):
    """Groups of 8 sequences with 8 query heads per KV head: 64 query rows, two full TMEM lane quarters of the
    tensor-core prefix pass; a negative scale as well (the running max then comes from the smallest score)."""
    import dataclasses
    extra = list(np.random.default_rng(31).integers(1, 300, size=19))
    wl = workloads.cascade_decode(31, [8, 8, 3], [40, 9, 17], extra, Hq=16, Hkv=2, D=64)
    wl = dataclasses.replace(wl, scale=scale_sign * wl.scale)
    out, pout = run_cascade(wl)
    ref = oracle_out(wl)
    check_attention(out, ref, f"cascade, 64 rows, scale sign {scale_sign}")
    assert (out - pout).abs().max().item() < 1e-4


def test_routing_by_saved_block_reads():
    """A cascade call saves at most (B - n_groups) * max_shared_blocks block reads per KV head.  Below the routing
    threshold it runs the plain decode kernel (output bit-identical to paged_decode_attention's); at the threshold
    it runs the cascade kernels (agreeing within the tolerance, in another summation order).  Both are checked
    against the oracle; the default threshold sends this small case to the plain decode."""
    import paged_kv_cache_27_gb300 as kvc
    wl = workloads.cascade_decode(71, [8, 8], [32, 20], list(np.random.default_rng(3).integers(1, 300, size=16)))
    saved = (16 - 2) * 32
    ref = oracle_out(wl)
    kvc.kvc_set_cascade_min_saved_blocks(DEFAULT_MIN_SAVED)
    out_default, pout = run_cascade(wl)
    assert torch.equal(out_default, pout)
    kvc.kvc_set_cascade_min_saved_blocks(saved + 1)
    out_plain, pout = run_cascade(wl)
    assert torch.equal(out_plain, pout)
    kvc.kvc_set_cascade_min_saved_blocks(saved)
    out_c, pout = run_cascade(wl)
    assert not torch.equal(out_c, pout)  # a different summation order: the cascade kernels ran
    check_attention(out_plain, ref, "routed to the plain decode")
    check_attention(out_c, ref, "cascade kernels")
    with pytest.raises(kvc.KvcError):
        kvc.kvc_set_cascade_min_saved_blocks(-1)
