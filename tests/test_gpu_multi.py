"""Multi-token decode (several new tokens per sequence, causal among them) on the GPU vs the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_attention

pytestmark = pytest.mark.gpu


def poisoned_pools(wl, dev="cuda"):
    """The workload's pools on the device, every row past a sequence's context set to NaN."""
    k = torch.from_numpy(wl.k_pool).to(dev)
    v = torch.from_numpy(wl.v_pool).to(dev)
    for b, c in enumerate(wl.ctx):
        last, used = int(wl.block_table[b, (int(c) - 1) // wl.bs]), int(c) % wl.bs
        if used:
            k[last, :, used:] = float("nan")
            v[last, :, used:] = float("nan")
    return k, v


def run_multi(wl, out_dtype=torch.float32, checked=False, ctx=None):
    import paged_kv_cache_27_gb300 as kvc
    dev = "cuda"
    kp, vp = poisoned_pools(wl)
    ctx_h = wl.ctx if ctx is None else ctx
    q = torch.from_numpy(wl.q).to(dev)
    table, ctx_d = torch.from_numpy(wl.block_table).to(dev), torch.from_numpy(np.asarray(ctx_h, np.int32)).to(dev)
    B = wl.q.shape[0]
    max_ctx = int(np.max(wl.ctx))
    ws = kvc.paged_decode_multi_plan(B, wl.Hq, wl.Hkv, wl.D, max_ctx, wl.T)
    workspace = torch.full((max(ws, 16),), 0x7F, dtype=torch.uint8, device=dev)
    out = torch.empty(wl.q.shape, dtype=out_dtype, device=dev)
    kvc.kvc_set_checked_mode(checked)
    try:
        kvc.paged_decode_multi_attention(q, kp, vp, table, ctx_d, wl.scale, out, workspace, max_ctx)
        torch.cuda.synchronize()
    finally:
        kvc.kvc_set_checked_mode(False)
    return out, kp, vp, q, table, ctx_d, max_ctx


CASES = [
    # seed, contexts, T, Hq, Hkv, D
    (1, [1], 1, 1, 1, 64),
    (2, [2, 17, 300], 2, 14, 2, 64),
    (3, [4, 16, 33, 1000], 4, 8, 1, 64),
    (4, [8, 4096], 8, 8, 8, 128),
    (5, [3, 15, 16, 17, 20000], 3, 14, 2, 64),
    (6, [8, 9, 23, 24, 25, 31, 32, 33], 8, 14, 2, 64),
    (7, [130, 5000], 5, 16, 2, 128),
    # 64 query rows (two row groups of four n-tiles), 8 rows (one n-tile) at D=128, 18 rows over two row groups
    (8, [8, 100, 2049], 8, 16, 2, 64),
    (9, [2, 31, 32, 33, 9000], 2, 16, 4, 128),
    (10, [6, 64, 65, 3000], 6, 12, 4, 128),
    # wider query groups than 8 heads per KV head
    (11, [3, 40, 5000], 3, 32, 2, 64),
    (12, [1, 700], 1, 16, 1, 64),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_multi_token_matches_oracle(case, out_dtype):
    import paged_kv_cache_27_gb300 as kvc
    seed, ctx, T, Hq, Hkv, D = CASES[case]
    wl = workloads.multi_token_decode(seed, ctx, T, Hq=Hq, Hkv=Hkv, D=D)
    out = run_multi(wl, out_dtype, checked=(case % 2 == 1))[0]
    assert kvc.kvc_device_error_flags(clear=True) == 0
    ref = oracle.decode_multi(wl.q, wl.k_pool, wl.v_pool, wl.block_table, wl.ctx, wl.scale)
    check_attention(out.reshape(-1, Hq, D), ref.reshape(-1, Hq, D), f"multi-token case {case}")


def test_single_token_agrees_with_decode():
    import paged_kv_cache_27_gb300 as kvc
    wl = workloads.multi_token_decode(11, [1, 16, 17, 700, 3000], 1)
    out, kp, vp, q, table, ctx, max_ctx = run_multi(wl)
    _, _, ws = kvc.paged_decode_plan(len(wl.ctx), wl.Hq, wl.Hkv, wl.D, max_ctx)
    ref = torch.empty((len(wl.ctx), wl.Hq, wl.D), dtype=torch.float32, device="cuda")
    kvc.paged_decode_attention(q[:, 0].contiguous(), kp, vp, table, ctx, wl.scale, ref,
                               torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda"), max_ctx)
    torch.cuda.synchronize()
    assert (out[:, 0] - ref).abs().max().item() < 1e-5


def test_multi_token_argument_errors():
    import paged_kv_cache_27_gb300 as kvc
    with pytest.raises(kvc.KvcError) as e:
        kvc.paged_decode_multi_plan(2, 14, 2, 64, 100, 9)
    assert "KVC_ERR_UNSUPPORTED" in str(e.value)
    wl = workloads.multi_token_decode(12, [5, 40], 4)
    # checked mode: a context shorter than the new tokens
    with pytest.raises(kvc.KvcError) as e:
        run_multi(wl, checked=True, ctx=np.array([3, 40], np.int32))
    assert "KVC_ERR_CAPACITY" in str(e.value)
    # unchecked: the sequence is flagged and its rows are zero; the other is still right
    out = run_multi(wl, ctx=np.array([3, 40], np.int32))[0]
    assert kvc.kvc_device_error_flags(clear=True) & kvc.DEVERR["CONTEXT"]
    assert torch.all(out[0] == 0)
    ref = oracle.decode_multi(wl.q[1:], wl.k_pool, wl.v_pool, wl.block_table[1:], wl.ctx[1:], wl.scale)
    check_attention(out[1:].reshape(-1, wl.Hq, wl.D), ref.reshape(-1, wl.Hq, wl.D), "multi-token, other sequence")


def test_multi_token_bad_inputs_flagged_without_faulting():
    """Unchecked bad inputs with several clusters per context (partials + combine): a context shorter than the
    new tokens gives zero rows, an out-of-range block id is skipped; both are flagged, the rest is right."""
    import paged_kv_cache_27_gb300 as kvc
    kvc.kvc_device_error_flags(clear=True)
    wl = workloads.multi_token_decode(13, [20000, 5000, 700], 3)
    assert kvc.paged_decode_multi_plan(3, wl.Hq, wl.Hkv, wl.D, 20000, 3) > 0  # partial states: several clusters
    ctx = np.array(wl.ctx, np.int32)
    ctx[1] = 2
    out = run_multi(wl, ctx=ctx)[0]
    assert kvc.kvc_device_error_flags(clear=True) & kvc.DEVERR["CONTEXT"]
    assert torch.all(out[1] == 0)
    ref = oracle.decode_multi(wl.q, wl.k_pool, wl.v_pool, wl.block_table, wl.ctx, wl.scale)
    check_attention(out[0].reshape(-1, wl.Hq, wl.D), ref[0].reshape(-1, wl.Hq, wl.D), "multi-token, long context")
    check_attention(out[2].reshape(-1, wl.Hq, wl.D), ref[2].reshape(-1, wl.Hq, wl.D), "multi-token, third sequence")
    # an out-of-range block id in the first sequence's table: skipped and flagged, every output finite
    bad_table = wl.block_table.copy()
    bad_table[0, 3] = -5
    wl2 = dataclasses.replace(wl, block_table=bad_table)
    out2 = run_multi(wl2)[0]
    assert kvc.kvc_device_error_flags(clear=True) & kvc.DEVERR["BLOCK_ID"]
    assert torch.isfinite(out2).all()
    check_attention(out2[1:].reshape(-1, wl.Hq, wl.D), ref[1:].reshape(-1, wl.Hq, wl.D), "multi-token, other rows")


TC_CASES = [i for i, c in enumerate(CASES) if c[5] == 64 and c[2] >= 2 and c[2] * (c[3] // c[4]) <= 64]


@pytest.mark.parametrize("case", TC_CASES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_multi_token_tensor_core_kernel_matches_oracle(case, out_dtype):
    """The opt-in tensor-core multi-token kernel (keys as the products' M side, query rows as N) on the same cases:
    several row counts (14 to 64), contexts at block and tile edges, several clusters per context, poisoned pools."""
    import paged_kv_cache_27_gb300 as kvc
    seed, ctx, T, Hq, Hkv, D = CASES[case]
    wl = workloads.multi_token_decode(seed, ctx, T, Hq=Hq, Hkv=Hkv, D=D)
    kvc.kvc_set_multi_tc(True)
    try:
        out = run_multi(wl, out_dtype, checked=(case % 2 == 1))[0]
    finally:
        kvc.kvc_set_multi_tc(False)
    assert kvc.kvc_device_error_flags(clear=True) == 0
    ref = oracle.decode_multi(wl.q, wl.k_pool, wl.v_pool, wl.block_table, wl.ctx, wl.scale)
    check_attention(out.reshape(-1, Hq, D), ref.reshape(-1, Hq, D), f"multi-token (tensor cores) case {case}")


def test_multi_token_tensor_core_kernel_bad_inputs():
    """The tensor-core kernel with a short context (zero rows, flagged) and an out-of-range block id (skipped,
    flagged, outputs finite) over several clusters per context."""
    import paged_kv_cache_27_gb300 as kvc
    kvc.kvc_device_error_flags(clear=True)
    kvc.kvc_set_multi_tc(True)
    try:
        wl = workloads.multi_token_decode(13, [20000, 5000, 700], 3)
        ctx = np.array(wl.ctx, np.int32)
        ctx[1] = 2
        out = run_multi(wl, ctx=ctx)[0]
        assert kvc.kvc_device_error_flags(clear=True) & kvc.DEVERR["CONTEXT"]
        assert torch.all(out[1] == 0)
        ref = oracle.decode_multi(wl.q, wl.k_pool, wl.v_pool, wl.block_table, wl.ctx, wl.scale)
        check_attention(out[0].reshape(-1, wl.Hq, wl.D), ref[0].reshape(-1, wl.Hq, wl.D), "tensor cores, long context")
        check_attention(out[2].reshape(-1, wl.Hq, wl.D), ref[2].reshape(-1, wl.Hq, wl.D), "tensor cores, third")
        bad_table = wl.block_table.copy()
        bad_table[0, 3] = -5
        out2 = run_multi(dataclasses.replace(wl, block_table=bad_table))[0]
        assert kvc.kvc_device_error_flags(clear=True) & kvc.DEVERR["BLOCK_ID"]
        assert torch.isfinite(out2).all()
        check_attention(out2[1:].reshape(-1, wl.Hq, wl.D), ref[1:].reshape(-1, wl.Hq, wl.D), "tensor cores, others")
    finally:
        kvc.kvc_set_multi_tc(False)
