"""Varlen causal prefill into the paged cache, then a decode step, vs the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_attention, check_cache_bits, owned_slots

pytestmark = pytest.mark.gpu


def oracle_flow(wl, causal):
    out = oracle.prefill(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.scale, causal=causal)
    n = len(wl.seqlens)
    kc = np.zeros((wl.NB, wl.Hkv, wl.bs, wl.D), np.float16)
    vc = np.zeros_like(kc)
    slots = []
    for s in range(n):
        for p in range(wl.seqlens[s]):
            slots.append(int(wl.block_table[s][p // wl.bs]) * wl.bs + p % wl.bs)
    oracle.append(kc, vc, wl.k, wl.v, np.array(slots, np.int64))
    step = [int(wl.block_table[s][wl.seqlens[s] // wl.bs]) * wl.bs + wl.seqlens[s] % wl.bs for s in range(n)]
    oracle.append(kc, vc, wl.k_dec, wl.v_dec, np.array(step, np.int64))
    ctx = np.array(wl.seqlens, np.int32) + 1
    dec = oracle.decode(wl.q_dec, kc, vc, wl.block_table, ctx, wl.scale)
    return out, dec, kc, vc, ctx


@pytest.mark.parametrize("make", [workloads.varlen_prefill, workloads.gqa_prefill])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_small_prefills(make, causal, out_dtype):
    from paged_kv_cache_27_gb300 import harness, kvc_device_error_flags
    wl = make()
    got = harness.prefill_then_decode(wl, causal=causal, out_dtype=out_dtype)
    assert kvc_device_error_flags(clear=True) == 0
    out, dec, kc, vc, ctx = oracle_flow(wl, causal)
    check_attention(got["prefill_out"], out, f"{wl.name} prefill causal={causal}")
    check_attention(got["decode_out"], dec, f"{wl.name} decode")
    slots = owned_slots(wl.block_table, ctx, wl.bs)
    check_cache_bits(got["k_cache"], kc, slots)
    check_cache_bits(got["v_cache"], vc, slots)


@pytest.mark.parametrize("seqlens,Hq,Hkv,D", [
    ((1,), 2, 1, 64),
    ((63, 64, 65, 1, 130), 4, 2, 64),
    ((200, 3, 129), 8, 8, 128),
    ((333,), 14, 2, 64),
    ((255, 256, 257, 384, 129, 128, 1, 640), 4, 2, 64),  # around the 256-row blocks of two query tiles
    ((600, 250, 513, 64), 8, 2, 128),
    # head dim 64 with at least 65,536 (token, query head) pairs: the two-query-tile kernel
    ((255, 256, 257, 384, 129, 128, 1, 640), 32, 8, 64),
    ((1500, 700), 32, 4, 64),
])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("precise", [False, True])
def test_prefill_ragged(seqlens, Hq, Hkv, D, causal, precise):
    import paged_kv_cache_27_gb300 as kvc
    wl = workloads._prefill("ragged", [99, sum(seqlens), D], seqlens, Hq, Hkv, D)
    q, k, v = (torch.from_numpy(x).cuda() for x in (wl.q, wl.k, wl.v))
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    kvc.prefill_attention(q, k, v, cu, max(seqlens), wl.scale, causal, out, precise=precise)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    ref = oracle.prefill(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.scale, causal=causal)
    err = check_attention(out, ref, f"prefill {seqlens}")
    if precise:  # fp16 high part + residual: the weights keep ~22 bits
        assert err < 5e-5, err


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("precise", [False, True])
def test_prefill_long_peaked(D, causal, precise):
    """Long segments whose scores jump by far more than 2^8 between key tiles (keys scaled x6 every 97
    positions, growing along the segment): the running max moves and O is rescaled in place many times."""
    import paged_kv_cache_27_gb300 as kvc
    seqlens = (1500, 517)
    wl = workloads._prefill("peaked", [7, sum(seqlens), D], seqlens, 4, 2, D)
    k = wl.k.astype(np.float32)
    pos = np.arange(k.shape[0])
    boost = np.where(pos % 97 == 5, 2.0 + 4.0 * (pos / k.shape[0]), 1.0).astype(np.float32)
    wl.k = (k * boost[:, None, None]).astype(np.float16)
    q, kk, v = (torch.from_numpy(x).cuda() for x in (wl.q, wl.k, wl.v))
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    kvc.prefill_attention(q, kk, v, cu, max(seqlens), wl.scale, causal, out, precise=precise)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    ref = oracle.prefill(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.scale, causal=causal)
    err = check_attention(out, ref, f"prefill peaked D={D} causal={causal}")
    if precise:
        assert err < 5e-5, err


@pytest.mark.parametrize("scale", [-0.09, 0.0, 0.5])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_scale_sign(scale, causal):
    """Any real scale: a negative one makes the smallest raw score the largest scaled one; zero gives
    uniform weights over the visible keys."""
    import paged_kv_cache_27_gb300 as kvc
    seqlens = (300, 77, 520)
    wl = workloads._prefill("scale", [11, sum(seqlens), 64], seqlens, 4, 1, 64)
    q, k, v = (torch.from_numpy(x).cuda() for x in (wl.q, wl.k, wl.v))
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    kvc.prefill_attention(q, k, v, cu, max(seqlens), scale, causal, out)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    ref = oracle.prefill(wl.q, wl.k, wl.v, wl.cu_seqlens, scale, causal=causal)
    check_attention(out, ref, f"prefill scale={scale} causal={causal}")


def test_prefill_bad_precision_rejected():
    import paged_kv_cache_27_gb300 as kvc
    q = torch.zeros((4, 2, 64), dtype=torch.float16, device="cuda")
    k = torch.zeros((4, 1, 64), dtype=torch.float16, device="cuda")
    cu = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
    out = torch.empty((4, 2, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.prefill_attention_ex(q, k, k, cu, 4, 0.125, True, 7, out)
    assert "KVC_ERR_INVALID" in str(e.value)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("precise", [False, True])
def test_prefill_empty_segments(D, precise):
    """Zero-length segments anywhere in cu_seqlens (first, middle, last, repeated) are no-ops; the others are
    computed as usual and no output row is left unwritten."""
    import paged_kv_cache_27_gb300 as kvc
    seqlens = (0, 130, 0, 0, 1, 257, 0)
    wl = workloads._prefill("empty", [12, sum(seqlens), D], seqlens, 4, 2, D)
    q, k, v = (torch.from_numpy(x).cuda() for x in (wl.q, wl.k, wl.v))
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    assert list(wl.cu_seqlens) == [0, 0, 130, 130, 130, 131, 388, 388]
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    kvc.prefill_attention(q, k, v, cu, max(seqlens), wl.scale, True, out, precise=precise)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    ref = oracle.prefill(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.scale, causal=True)
    check_attention(out, ref, f"prefill with empty segments D={D}")
