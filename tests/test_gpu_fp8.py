"""Quantized (fp8 e4m3) KV cache on the GPU: the quantizing append bit-exact against the oracle, the decode
over the fp8 cache against the oracle's decode of the same codes."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_attention

pytestmark = pytest.mark.gpu


def used_slots(wl):
    """Every cached position of every sequence: (slot int64 [n], pool row index (block, offset) pairs)."""
    slots = []
    for b, c in enumerate(wl.ctx):
        for j in range(int(c)):
            slots.append(int(wl.block_table[b, j // wl.bs]) * wl.bs + j % wl.bs)
    return np.array(slots, dtype=np.int64)


# the fp8 V pool's layout as the header states it: per (block, KV head), a row of 16 token codes per dim, token
# tau at byte 4 * ((tau & 7) >> 1) + 2 * (tau >> 3) + (tau & 1)
VT_POS = np.array([4 * ((t & 7) >> 1) + 2 * (t >> 3) + (t & 1) for t in range(16)])


def v_natural(vc):
    """Device V codes [NB][Hkv][D][16] -> [NB][Hkv][16][D] in token order (host numpy)."""
    v = vc.cpu().numpy()
    return np.ascontiguousarray(v[:, :, :, VT_POS].transpose(0, 1, 3, 2))


def test_v_positions_are_a_permutation():
    import paged_kv_cache_27_gb300 as kvc
    assert sorted(VT_POS) == list(range(16))
    assert [kvc.fp8_v_position(t) for t in range(16)] == list(VT_POS)
    for t in range(4):  # lane t's mma fragment (tokens 2t, 2t+1, 2t+8, 2t+9) is bytes 4t..4t+3
        assert [VT_POS[2 * t], VT_POS[2 * t + 1], VT_POS[2 * t + 8], VT_POS[2 * t + 9]] == [4 * t + i for i in range(4)]


def quantized_cache(wl, dev="cuda"):
    """The workload's used rows quantized on the GPU into NaN-poisoned fp8 pools; returns device codes/scales
    and the host rows that were appended."""
    import paged_kv_cache_27_gb300 as kvc
    slots = used_slots(wl)
    blk, off = slots // wl.bs, slots % wl.bs
    k_rows = wl.k_pool[blk, :, off]  # [n][Hkv][D]
    v_rows = wl.v_pool[blk, :, off]
    shape = wl.k_pool.shape
    kc = torch.full(shape, 0x7F, dtype=torch.uint8, device=dev)  # 0x7F is an e4m3 NaN
    vc = torch.full(shape[:2] + (shape[3], shape[2]), 0x7F, dtype=torch.uint8, device=dev)
    ks = torch.full(shape[:3], float("nan"), dtype=torch.float32, device=dev)
    vs = torch.full(shape[:3], float("nan"), dtype=torch.float32, device=dev)
    kvc.kv_append_fp8(torch.from_numpy(np.ascontiguousarray(k_rows)).to(dev),
                      torch.from_numpy(np.ascontiguousarray(v_rows)).to(dev), torch.from_numpy(slots).to(dev),
                      kc, vc, ks, vs)
    torch.cuda.synchronize()
    return kc, vc, ks, vs, slots


@pytest.mark.parametrize("D", [64, 128])
def test_append_fp8_bit_exact(D):
    import paged_kv_cache_27_gb300 as kvc
    wl = workloads.multi_token_decode(31 + D, [1, 17, 300, 1000], 1, Hq=8, Hkv=2, D=D)
    # rows of very different magnitudes, and all-zero rows
    scale = np.exp2(np.random.default_rng(D).integers(-10, 6, wl.k_pool.shape[:3]))[..., None]
    wl.k_pool = (wl.k_pool.astype(np.float32) * scale).astype(np.float16)
    wl.k_pool[0, 0, :4] = 0
    kc, vc, ks, vs, slots = quantized_cache(wl)
    assert kvc.kvc_device_error_flags(clear=True) == 0
    rk, rks = oracle.quantize_fp8(wl.k_pool)
    rv, rvs = oracle.quantize_fp8(wl.v_pool)
    blk, off = slots // wl.bs, slots % wl.bs
    used = np.zeros(wl.k_pool.shape[:3], bool)
    used[blk, :, off] = True
    for g, ref in ((kc.cpu().numpy(), rk), (v_natural(vc), rv)):
        assert np.array_equal(g[used], ref[used])
        assert np.all(g[~used] == 0x7F)  # untouched rows keep the poison
    for got, ref in ((ks, rks), (vs, rvs)):
        g = got.cpu().numpy()
        assert np.array_equal(g[used].view(np.uint32), ref[used].view(np.uint32))
        assert np.all(np.isnan(g[~used]))
    # a negative slot is skipped
    k1 = torch.from_numpy(np.ascontiguousarray(wl.k_pool[:1, :, 0])).cuda()
    before = kc.clone()
    kvc.kv_append_fp8(k1, k1, torch.tensor([-1], dtype=torch.int64, device="cuda"), kc, vc, ks, vs)
    torch.cuda.synchronize()
    assert torch.equal(kc, before)


CASES = [
    # seed, contexts, Hq, Hkv, D, blocks_per_split
    (1, [1], 1, 1, 64, 0),
    (2, [1, 17, 300, 2048], 14, 2, 64, 0),
    (3, [5, 64, 65, 700], 8, 1, 64, 0),
    (4, [2, 999, 4096], 8, 8, 128, 0),
    (5, [300, 1025, 2048], 14, 2, 64, 3),
    (6, [40000, 5000, 1], 14, 2, 64, 0),
    (7, [129, 2000], 16, 2, 128, 2),
    (8, [3, 900, 5000], 48, 2, 64, 0),  # 24 query heads per KV head: three chunks of 8
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_decode_fp8_matches_oracle(case, out_dtype):
    import paged_kv_cache_27_gb300 as kvc
    seed, ctx, Hq, Hkv, D, bps = CASES[case]
    wl = workloads.multi_token_decode(100 + seed, ctx, 1, Hq=Hq, Hkv=Hkv, D=D)
    kc, vc, ks, vs, _ = quantized_cache(wl)
    dev = "cuda"
    B = len(ctx)
    q = torch.from_numpy(np.ascontiguousarray(wl.q[:, 0])).to(dev)
    table, ctx_d = torch.from_numpy(wl.block_table).to(dev), torch.from_numpy(wl.ctx).to(dev)
    max_ctx = int(wl.ctx.max())
    _, _, ws = kvc.paged_decode_plan(B, Hq, Hkv, D, max_ctx, bps)
    out = torch.empty((B, Hq, D), dtype=out_dtype, device=dev)
    kvc.paged_decode_attention_fp8(q, kc, vc, ks, vs, table, ctx_d, wl.scale, out,
                                   torch.full((max(ws, 16),), 0x7F, dtype=torch.uint8, device=dev), max_ctx, bps)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    ref = oracle.decode_fp8(wl.q[:, 0], kc.cpu().numpy(), v_natural(vc), ks.cpu().numpy(), vs.cpu().numpy(),
                            wl.block_table, wl.ctx, wl.scale)
    check_attention(out, ref, f"fp8 decode case {case}")


def test_decode_fp8_model_step_shape():
    """One layer of the 24-layer benchmark shape (32 x 2048, 14 / 2 heads) on an fp8 cache."""
    import paged_kv_cache_27_gb300 as kvc
    wl = workloads.multi_token_decode(77, [2048] * 32, 1)
    kc, vc, ks, vs, _ = quantized_cache(wl)
    dev = "cuda"
    q = torch.from_numpy(np.ascontiguousarray(wl.q[:, 0])).to(dev)
    _, _, ws = kvc.paged_decode_plan(32, 14, 2, 64, 2048)
    out = torch.empty((32, 14, 64), dtype=torch.float32, device=dev)
    kvc.paged_decode_attention_fp8(q, kc, vc, ks, vs, torch.from_numpy(wl.block_table).to(dev),
                                   torch.from_numpy(wl.ctx).to(dev), wl.scale, out,
                                   torch.empty(max(ws, 16), dtype=torch.uint8, device=dev), 2048)
    torch.cuda.synchronize()
    ref = oracle.decode_fp8(wl.q[:, 0], kc.cpu().numpy(), v_natural(vc), ks.cpu().numpy(), vs.cpu().numpy(),
                            wl.block_table, wl.ctx, wl.scale)
    check_attention(out, ref, "fp8 decode, 32 x 2048")
