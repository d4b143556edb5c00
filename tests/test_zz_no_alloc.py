"""The allocation-free decode entry point.

Some callers cannot allocate device memory while they run (allocator code that
would re-enter itself, plug-ins handed only their input and output buffers,
serving loops that forbid cudaMalloc after start-up).  For them,
paged_decode_attention_static_workspace keeps its split scratch in a fixed
16 MiB array inside the library.  These tests call it through the C ABI and
check it against paged_decode_attention with a caller workspace and against
the fp64 oracle.

They run after every other test: the conftest moves this module to the end of
the collected items (its file name also sorts last), so that if one of them
fails, a run that stops at the first failure has already run the rest.  They
pass the same way when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import paging
from parity import ATOL, check_attention

pytestmark = pytest.mark.gpu


def test_static_workspace_matches_caller_workspace_twice():
    import paged_kv_cache_27_gb300 as kvc
    from paged_kv_cache_27_gb300.harness import DecodeSession
    wl = workloads.small_decode(31, B=3, Hq=14, Hkv=2, D=64, ctx=[3000, 1500, 37], peak_frac=0.01)
    bps = 8  # 188 blocks -> 24 clusters of one CTA: the split partials go through the scratch
    s = DecodeSession(wl, blocks_per_split=bps).fill()
    s.step()
    torch.cuda.synchronize()
    nsplit, _, need = kvc.paged_decode_plan(wl.B, wl.Hq, wl.Hkv, wl.D, s.max_ctx, bps)
    assert need > 0
    ref = torch.empty_like(s.out[0])
    kvc.paged_decode_attention(s.q[0], s.k_pool[0], s.v_pool[0], s.block_table, s.context_lens, wl.scale, ref,
                               s.workspace, s.max_ctx, bps)
    oracle_out, _, _ = paging.decode_step(wl, 0)  # the fp64 oracle after the same append
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        kvc.paged_decode_attention_static_workspace(s.q[0], s.k_pool[0], s.v_pool[0], s.block_table,
                                                    s.context_lens, wl.scale, out, s.max_ctx, bps)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all(), call
        err = (out.double() - ref.double()).abs().max().item()
        assert err <= ATOL, (call, err)
        check_attention(out, oracle_out, f"static workspace, call {call}")
    assert kvc.kvc_device_error_flags(clear=True) == 0
    s.close()


def test_static_workspace_rejects_sizes_beyond_its_limit():
    import paged_kv_cache_27_gb300 as kvc
    B, Hq, Hkv, D, ctx = 64, 8, 8, 64, 4096
    _, _, need = kvc.paged_decode_plan(B, Hq, Hkv, D, ctx, blocks_per_split=1)
    assert need > 16 << 20
    dev = "cuda"
    q = torch.zeros((B, Hq, D), dtype=torch.float16, device=dev)
    kc = torch.zeros((4, Hkv, 16, D), dtype=torch.float16, device=dev)
    table = torch.zeros((B, ctx // 16), dtype=torch.int32, device=dev)
    lens = torch.full((B,), ctx, dtype=torch.int32, device=dev)
    out = torch.zeros((B, Hq, D), dtype=torch.float32, device=dev)
    with pytest.raises(kvc.KvcError) as e:
        kvc.paged_decode_attention_static_workspace(q, kc, kc, table, lens, 0.125, out, ctx, blocks_per_split=1)
    assert e.value.name == "KVC_ERR_CAPACITY"
    assert "16 MiB" in str(e.value)
