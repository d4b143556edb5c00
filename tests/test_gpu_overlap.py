"""Launch overlap (programmatic dependent launch) on the multi-token, cascade and fp8 paths: calls chained in a CUDA
graph, each call's q being the previous call's output (filled with NaN before the replay), so a kernel that read
q before its dependency wait would see NaN or a partly written q.  Each call is checked against the oracle on the q
it actually received.  Also the decode step fed from pinned host memory with its copies overlapped with the calls."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_attention

pytestmark = pytest.mark.gpu


def _graph(fn):
    import paged_kv_cache_27_gb300 as kvc
    kvc.kvc_set_launch_overlap(True)
    try:
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                fn()
    finally:
        kvc.kvc_set_launch_overlap(False)
    return g


@pytest.mark.parametrize("T,ctx", [(2, [40, 2049, 300]), (5, [5, 16, 17, 20000])])
def test_multi_token_chain_in_graph(T, ctx):
    import paged_kv_cache_27_gb300 as kvc
    wl = workloads.multi_token_decode(41 + T, ctx, T)
    dev = "cuda"
    kp, vp = torch.from_numpy(wl.k_pool).to(dev), torch.from_numpy(wl.v_pool).to(dev)
    table, ctx_d = torch.from_numpy(wl.block_table).to(dev), torch.from_numpy(wl.ctx).to(dev)
    max_ctx = int(wl.ctx.max())
    ws = torch.zeros(max(kvc.paged_decode_multi_plan(len(ctx), wl.Hq, wl.Hkv, wl.D, max_ctx, T), 16),
                     dtype=torch.uint8, device=dev)
    q0 = torch.from_numpy(wl.q).to(dev)
    outs = [torch.empty_like(q0) for _ in range(3)]  # call i reads outs[i - 1] (q0 for the first)

    def chain():
        src = q0
        for o in outs:
            kvc.paged_decode_multi_attention(src, kp, vp, table, ctx_d, wl.scale, o, ws, max_ctx)
            src = o
    g = _graph(chain)
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    src = wl.q
    for i, o in enumerate(outs):
        ref = oracle.decode_multi(src, wl.k_pool, wl.v_pool, wl.block_table, wl.ctx, wl.scale)
        check_attention(o.reshape(-1, wl.Hq, wl.D), ref.reshape(-1, wl.Hq, wl.D), f"multi-token chain call {i}")
        src = o.cpu().numpy()  # the next call's q, as the GPU wrote it


@pytest.fixture
def always_cascade():
    import paged_kv_cache_27_gb300 as kvc
    kvc.kvc_set_cascade_min_saved_blocks(0)  # the cascade kernels, whatever the prefix length
    yield
    kvc.kvc_set_cascade_min_saved_blocks(36000)


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 14, 2), (128, 8, 8)])
def test_cascade_chain_in_graph(D, Hq, Hkv, always_cascade):
    import paged_kv_cache_27_gb300 as kvc
    extra = list(np.random.default_rng(5).integers(1, 200, size=16))
    wl = workloads.cascade_decode(43, [8, 5, 3], [40, 7, 0], extra, Hq=Hq, Hkv=Hkv, D=D)
    dev = "cuda"
    B = len(extra)
    kp, vp = torch.from_numpy(wl.k_pool).to(dev), torch.from_numpy(wl.v_pool).to(dev)
    table, ctx_d = torch.from_numpy(wl.block_table).to(dev), torch.from_numpy(wl.ctx).to(dev)
    gs, sh = torch.from_numpy(wl.group_start).to(dev), torch.from_numpy(wl.shared_blocks).to(dev)
    mx = int(wl.shared_blocks.max())
    max_ctx = int(wl.ctx.max())
    ws = torch.zeros(max(kvc.paged_decode_cascade_plan(B, Hq, Hkv, D, max_ctx, len(wl.group_start) - 1, mx), 16),
                     dtype=torch.uint8, device=dev)
    q0 = torch.from_numpy(wl.q).to(dev)
    outs = [torch.empty_like(q0) for _ in range(3)]

    def chain():
        src = q0
        for o in outs:
            kvc.paged_decode_cascade_attention(src, kp, vp, table, ctx_d, gs, sh, mx, wl.scale, o, ws, max_ctx)
            src = o
    g = _graph(chain)
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    src = wl.q
    for i, o in enumerate(outs):
        ref = oracle.decode(src, wl.k_pool, wl.v_pool, wl.block_table, wl.ctx, wl.scale)
        check_attention(o, ref, f"cascade chain call {i}, D={D}")
        src = o.cpu().numpy()


def test_fp8_decode_chain_in_graph():
    """The fp8-cache decode chained the same way (contexts over one cluster, so the combine kernel runs too)."""
    import paged_kv_cache_27_gb300 as kvc
    from test_gpu_fp8 import oracle_fp8, quantized_cache
    wl = workloads.multi_token_decode(47, [3000, 17, 40000, 2048], 1)
    rec, _ = quantized_cache(wl)
    dev = "cuda"
    B = len(wl.ctx)
    table, ctx_d = torch.from_numpy(wl.block_table).to(dev), torch.from_numpy(wl.ctx).to(dev)
    max_ctx = int(wl.ctx.max())
    _, _, w = kvc.paged_decode_plan(B, wl.Hq, wl.Hkv, wl.D, max_ctx)
    ws = torch.zeros(max(w, 16), dtype=torch.uint8, device=dev)
    q0 = torch.from_numpy(np.ascontiguousarray(wl.q[:, 0])).to(dev)
    outs = [torch.empty_like(q0) for _ in range(3)]

    def chain():
        src = q0
        for o in outs:
            kvc.paged_decode_attention_fp8(src, rec, table, ctx_d, wl.scale, o, ws, max_ctx)
            src = o
    g = _graph(chain)
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    src = wl.q[:, 0]
    for i, o in enumerate(outs):
        check_attention(o, oracle_fp8(src, rec, wl), f"fp8 chain call {i}")
        src = o.cpu().numpy()


def test_decode_chain_with_idle_combine_in_graph():
    """Decode calls planned for a context far longer than any actual one (forced short splits, so the plan has many
    parts and the combine kernel is launched) while every context fits one split: every combine CTA has nothing to
    merge.  The combine grid must still complete only after the decode kernel it follows, or the next call in the
    chain could read its q (the previous output) before it is written."""
    import paged_kv_cache_27_gb300 as kvc
    from oracle import paging as opaging
    from paged_kv_cache_27_gb300.harness import DecodeSession
    B, Hq, Hkv, D = 96, 14, 2, 64
    wl = workloads.small_decode(67, B=B, Hq=Hq, Hkv=Hkv, D=D, ctx=[16 + (7 * b) % 240 for b in range(B)])
    s = DecodeSession(wl).fill()
    s.append(0)
    _, kc, vc = opaging.decode_step(wl, 0)  # the pools after the step's append
    dev = "cuda"
    bps = 16  # blocks per split: 256 tokens, more than any context here
    max_ctx = 8192
    _, got_bps, wsb = kvc.paged_decode_plan(B, Hq, Hkv, D, max_ctx, bps)
    assert got_bps == bps and wsb > 0  # several parts: the combine kernel is part of every call
    wide = np.full((B, max_ctx // 16), -1, dtype=np.int32)
    wide[:, :wl.block_table.shape[1]] = wl.block_table
    table = torch.from_numpy(wide).to(dev)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    q0 = s.q[0]
    outs = [torch.empty_like(q0) for _ in range(4)]

    def chain():
        src = q0
        for o in outs:
            kvc.paged_decode_attention(src, s.k_pool[0], s.v_pool[0], table, s.context_lens, wl.scale, o, ws, max_ctx,
                                       bps)
            src = o
    g = _graph(chain)
    for rep in range(3):
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert kvc.kvc_device_error_flags(clear=True) == 0
        src = wl.q[0]
        for i, o in enumerate(outs):
            ref = oracle.decode(src, kc, vc, wl.block_table, wl.ctx, wl.scale)
            check_attention(o, ref, f"idle-combine chain call {i}, replay {rep}")
            src = o.cpu().numpy()
    s.close()


def test_cascade_chain_without_shared_blocks_in_graph(always_cascade):
    """A cascade call told to expect shared prefixes when no group shares a block: every CTA of the prefix pass
    leaves at once.  Chained calls in a graph still see the previous call's complete output."""
    import paged_kv_cache_27_gb300 as kvc
    extra = list(np.random.default_rng(9).integers(1, 300, size=12))
    wl = workloads.cascade_decode(45, [4, 4, 4], [0, 0, 0], extra)
    dev = "cuda"
    B = len(extra)
    kp, vp = torch.from_numpy(wl.k_pool).to(dev), torch.from_numpy(wl.v_pool).to(dev)
    table, ctx_d = torch.from_numpy(wl.block_table).to(dev), torch.from_numpy(wl.ctx).to(dev)
    gs, sh = torch.from_numpy(wl.group_start).to(dev), torch.from_numpy(wl.shared_blocks).to(dev)
    mx = 8  # an upper bound the groups do not reach
    max_ctx = int(wl.ctx.max())
    ws = torch.zeros(max(kvc.paged_decode_cascade_plan(B, wl.Hq, wl.Hkv, wl.D, max_ctx, len(wl.group_start) - 1, mx),
                         16), dtype=torch.uint8, device=dev)
    q0 = torch.from_numpy(wl.q).to(dev)
    outs = [torch.empty_like(q0) for _ in range(3)]

    def chain():
        src = q0
        for o in outs:
            kvc.paged_decode_cascade_attention(src, kp, vp, table, ctx_d, gs, sh, mx, wl.scale, o, ws, max_ctx)
            src = o
    g = _graph(chain)
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    src = wl.q
    for i, o in enumerate(outs):
        ref = oracle.decode(src, wl.k_pool, wl.v_pool, wl.block_table, wl.ctx, wl.scale)
        check_attention(o, ref, f"cascade chain without shared blocks, call {i}")
        src = o.cpu().numpy()


@pytest.mark.parametrize("fused", [True, False])
def test_host_step_copies_overlapped_with_calls(fused):
    """The step fed from pinned host memory with its copies overlapped with the calls (HostStep: staging-copy
    kernels in the calls' stream bring the inputs in, in pieces alongside earlier calls, and take the outputs back,
    eight layers at a time alongside a later call), replayed from a CUDA graph with launch overlap and then run
    eagerly.  Before each run the device inputs hold wrong but valid values
    (block 0, context 1, slot 0, NaN activations) and the device and host outputs NaN, so a call that ran ahead
    of its input copy, or a copy back that ran ahead of its call, shows up."""
    from oracle import paging as opaging
    from parity import check_cache_bits, owned_slots
    from paged_kv_cache_27_gb300.harness import DecodeSession, HostStep
    import paged_kv_cache_27_gb300 as kvc
    # 10 layers: inputs staged in all four pieces (layers 0-1, 2-3, 4-7, 8-9), outputs of layers 0-7 copied
    # back alongside layer 8's call with layer 9's still to come; the 40000-token context adds the combine kernel
    wl = workloads.small_decode(61, B=5, Hq=14, Hkv=2, D=64, ctx=[3000, 17, 40000, 2048, 1], L=10)
    s = DecodeSession(wl, out_dtype=torch.float16).fill()
    hs = HostStep(s)
    g = _graph(lambda: hs.run(fused))

    def poison():
        torch.cuda.synchronize()
        hs.block_table.zero_()
        hs.context_lens.fill_(1)
        hs.slots.zero_()
        for t in hs.q + hs.k_new + hs.v_new:
            t.fill_(float("nan"))
        s.out.fill_(float("nan"))
        hs.h_out.fill_(float("nan"))

    refs = [opaging.decode_step(wl, layer) for layer in range(wl.L)]
    slots = owned_slots(wl.block_table, wl.ctx, wl.bs)
    for how in ("graph", "eager"):
        poison()
        kvc.kvc_set_launch_overlap(True)
        try:
            g.replay() if how == "graph" else hs.run(fused)
        finally:
            kvc.kvc_set_launch_overlap(False)
        torch.cuda.synchronize()
        assert kvc.kvc_device_error_flags(clear=True) == 0
        for layer, (ref, kc, vc) in enumerate(refs):
            check_attention(hs.h_out[layer], ref, f"{how}, fused={fused}, layer {layer}")
            check_cache_bits(s.k_pool[layer], kc, slots)
            check_cache_bits(s.v_pool[layer], vc, slots)
    s.close()


@pytest.mark.parametrize("nbytes", [16, 4096 + 16, 3 * (1 << 20) + 48])
@pytest.mark.parametrize("ahead", [False, True])
def test_staging_copy_directions(nbytes, ahead):
    """kvc_copy_async between pinned host and device memory both ways and device to device, byte for byte, at
    sizes that leave a ragged last pass of the kernel's grid."""
    import paged_kv_cache_27_gb300 as kvc
    rng = np.random.default_rng(nbytes)
    host = torch.from_numpy(rng.integers(0, 256, size=nbytes, dtype=np.uint8)).pin_memory()
    dev_a = torch.full((nbytes,), 7, dtype=torch.uint8, device="cuda")
    dev_b = torch.zeros_like(dev_a)
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    kvc.kvc_set_launch_overlap(ahead)
    try:
        kvc.kvc_copy_async(dev_a, host, ahead=ahead)
        kvc.kvc_copy_async(dev_b, dev_a, ahead=False)
        kvc.kvc_copy_async(back, dev_b, ahead=False)
    finally:
        kvc.kvc_set_launch_overlap(False)
    torch.cuda.synchronize()
    assert torch.equal(dev_a.cpu(), host)
    assert torch.equal(back, host)


def test_staging_copy_refuses_pageable_memory():
    import paged_kv_cache_27_gb300 as kvc
    dev = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_copy_async(dev, torch.zeros(64, dtype=torch.uint8))
    assert "pinned" in str(e.value)
    with pytest.raises(ValueError):
        kvc.kvc_copy_async(dev, torch.zeros(48, dtype=torch.uint8, device="cuda"))


def test_prepared_call_matches_direct_call():
    """A decode call in its prepare=True form launches the same work as the direct call (bit for bit), on the
    current stream or a given one."""
    import paged_kv_cache_27_gb300 as kvc
    from paged_kv_cache_27_gb300.harness import DecodeSession
    wl = workloads.small_decode(63, B=3, Hq=14, Hkv=2, D=64, ctx=[100, 30000, 1])
    s = DecodeSession(wl).fill()
    s.append(0)  # the new token's K/V (without it the last slot of every context still holds the NaN poison)
    s.decode(0)
    torch.cuda.synchronize()
    ref = s.out[0].clone()
    assert torch.isfinite(ref).all()
    call = kvc.paged_decode_attention(s.q[0], s.k_pool[0], s.v_pool[0], s.block_table, s.context_lens, wl.scale,
                                      s.out[0], s.workspace, s.max_ctx, prepare=True)
    assert isinstance(call, kvc.PreparedCall)
    for stream in (None, torch.cuda.Stream()):
        s.out.fill_(float("nan"))
        torch.cuda.synchronize()
        call(stream)
        torch.cuda.synchronize()
        assert torch.equal(s.out[0], ref)
    assert kvc.kvc_device_error_flags(clear=True) == 0
    s.close()
