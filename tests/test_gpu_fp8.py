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


# the fp8 record layout as the header states it, per (block, KV head): K codes (16 token rows of D, the 16-byte
# chunks of row r permuted by p(r)), 16 K scales, V codes (D dim rows of 16 token codes, token tau at byte
# VT_POS[tau]), 16 V scales
VT_POS = np.array([4 * ((t & 7) >> 1) + 2 * (t >> 3) + (t & 1) for t in range(16)])


def k_chunk_perm(D, r):
    return ((r >> 1) & 3) if D == 64 else (r & 7)


def unpack_records(rec, D):
    """Device records uint8 [NB][Hkv][32 D + 128] -> host (K codes [NB][Hkv][16][D], K scales [NB][Hkv][16],
    V codes [NB][Hkv][16][D] in token order, V scales), by the layout above."""
    r = rec.cpu().numpy()
    NB, Hkv, nbytes = r.shape
    assert nbytes == 32 * D + 128
    kc = np.empty((NB, Hkv, 16, D), np.uint8)
    for row in range(16):
        for c in range(D // 16):
            src = row * D + ((c ^ k_chunk_perm(D, row)) << 4)
            kc[:, :, row, 16 * c:16 * c + 16] = r[:, :, src:src + 16]
    ks = np.ascontiguousarray(r[:, :, 16 * D:16 * D + 64]).view(np.float32)
    v0 = 16 * D + 64
    vt = r[:, :, v0:v0 + 16 * D].reshape(NB, Hkv, D, 16)
    vc = np.ascontiguousarray(vt[:, :, :, VT_POS].transpose(0, 1, 3, 2))
    vs = np.ascontiguousarray(r[:, :, v0 + 16 * D:v0 + 16 * D + 64]).view(np.float32)
    return kc, ks, vc, vs


def test_v_positions_are_a_permutation():
    import paged_kv_cache_27_gb300 as kvc
    assert sorted(VT_POS) == list(range(16))
    assert [kvc.fp8_v_position(t) for t in range(16)] == list(VT_POS)
    for t in range(4):  # lane t's mma fragment (tokens 2t, 2t+1, 2t+8, 2t+9) is bytes 4t..4t+3
        assert [VT_POS[2 * t], VT_POS[2 * t + 1], VT_POS[2 * t + 8], VT_POS[2 * t + 9]] == [4 * t + i for i in range(4)]
    assert kvc.kv_fp8_record_bytes(64) == 2176 and kvc.kv_fp8_record_bytes(128) == 4224


def quantized_cache(wl, dev="cuda"):
    """The workload's used rows quantized on the GPU into a poisoned fp8 record pool (0xFF bytes: NaN codes and
    NaN scales); returns the device records and the slots that were appended."""
    import paged_kv_cache_27_gb300 as kvc
    slots = used_slots(wl)
    blk, off = slots // wl.bs, slots % wl.bs
    k_rows = wl.k_pool[blk, :, off]  # [n][Hkv][D]
    v_rows = wl.v_pool[blk, :, off]
    NB, Hkv, _, D = wl.k_pool.shape
    rec = torch.full((NB, Hkv, kvc.kv_fp8_record_bytes(D)), 0xFF, dtype=torch.uint8, device=dev)
    kvc.kv_append_fp8(torch.from_numpy(np.ascontiguousarray(k_rows)).to(dev),
                      torch.from_numpy(np.ascontiguousarray(v_rows)).to(dev), torch.from_numpy(slots).to(dev), rec)
    torch.cuda.synchronize()
    return rec, slots


def oracle_fp8(q, rec, wl):
    kc, ks, vc, vs = unpack_records(rec, wl.D)
    return oracle.decode_fp8(q, kc, vc, ks, vs, wl.block_table, wl.ctx, wl.scale)


@pytest.mark.parametrize("D", [64, 128])
def test_append_fp8_bit_exact(D):
    import paged_kv_cache_27_gb300 as kvc
    wl = workloads.multi_token_decode(31 + D, [1, 17, 300, 1000], 1, Hq=8, Hkv=2, D=D)
    # rows of very different magnitudes, and all-zero rows
    scale = np.exp2(np.random.default_rng(D).integers(-10, 6, wl.k_pool.shape[:3]))[..., None]
    wl.k_pool = (wl.k_pool.astype(np.float32) * scale).astype(np.float16)
    wl.k_pool[0, 0, :4] = 0
    rec, slots = quantized_cache(wl)
    assert kvc.kvc_device_error_flags(clear=True) == 0
    kc, ks, vc, vs = unpack_records(rec, D)
    rk, rks = oracle.quantize_fp8(wl.k_pool)
    rv, rvs = oracle.quantize_fp8(wl.v_pool)
    blk, off = slots // wl.bs, slots % wl.bs
    used = np.zeros(wl.k_pool.shape[:3], bool)
    used[blk, :, off] = True
    for g, ref in ((kc, rk), (vc, rv)):
        assert np.array_equal(g[used], ref[used])
        assert np.all(g[~used] == 0xFF)  # untouched rows keep the poison
    for g, ref in ((ks, rks), (vs, rvs)):
        assert np.array_equal(g[used].view(np.uint32), ref[used].view(np.uint32))
        assert np.all(np.isnan(g[~used]))
    # a negative slot is skipped
    k1 = torch.from_numpy(np.ascontiguousarray(wl.k_pool[:1, :, 0])).cuda()
    before = rec.clone()
    kvc.kv_append_fp8(k1, k1, torch.tensor([-1], dtype=torch.int64, device="cuda"), rec)
    torch.cuda.synchronize()
    assert torch.equal(rec, before)


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
    # 400 ragged contexts: more CTAs than the GPU holds at once, dispatched longest context first
    (9, [int(c) for c in np.random.default_rng(9).integers(1, 600, size=400)], 14, 2, 64, 0),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_decode_fp8_matches_oracle(case, out_dtype):
    import paged_kv_cache_27_gb300 as kvc
    seed, ctx, Hq, Hkv, D, bps = CASES[case]
    wl = workloads.multi_token_decode(100 + seed, ctx, 1, Hq=Hq, Hkv=Hkv, D=D)
    rec, _ = quantized_cache(wl)
    dev = "cuda"
    B = len(ctx)
    q = torch.from_numpy(np.ascontiguousarray(wl.q[:, 0])).to(dev)
    table, ctx_d = torch.from_numpy(wl.block_table).to(dev), torch.from_numpy(wl.ctx).to(dev)
    max_ctx = int(wl.ctx.max())
    _, _, ws = kvc.paged_decode_plan(B, Hq, Hkv, D, max_ctx, bps)
    out = torch.empty((B, Hq, D), dtype=out_dtype, device=dev)
    kvc.paged_decode_attention_fp8(q, rec, table, ctx_d, wl.scale, out,
                                   torch.full((max(ws, 16),), 0x7F, dtype=torch.uint8, device=dev), max_ctx, bps)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    check_attention(out, oracle_fp8(wl.q[:, 0], rec, wl), f"fp8 decode case {case}")


@pytest.mark.parametrize("i", range(8))
def test_decode_fp8_random_shapes(i):
    """Seeded random shapes on the fp8 cache: batch up to 180 (several waves), GQA groups up to 16, both head dims,
    ragged contexts with single tokens, the planner's split or an explicit one."""
    import paged_kv_cache_27_gb300 as kvc
    rng = np.random.default_rng(900 + i)
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2]))
    G = int(rng.choice([1, 4, 7, 16] if D == 64 else [1, 4, 8]))
    B = int(rng.choice([2, 31, 180]))
    ctx = rng.integers(1, int(rng.choice([50, 900, 2500])) + 1, size=B)
    ctx[rng.random(B) < 0.1] = 1
    bps = int(rng.choice([0, 0, 5]))
    wl = workloads.multi_token_decode(300 + i, ctx.tolist(), 1, Hq=G * Hkv, Hkv=Hkv, D=D)
    rec, _ = quantized_cache(wl)
    dev = "cuda"
    q = torch.from_numpy(np.ascontiguousarray(wl.q[:, 0])).to(dev)
    table, ctx_d = torch.from_numpy(wl.block_table).to(dev), torch.from_numpy(wl.ctx).to(dev)
    max_ctx = int(wl.ctx.max())
    _, _, ws = kvc.paged_decode_plan(B, G * Hkv, Hkv, D, max_ctx, bps)
    out = torch.empty((B, G * Hkv, D), dtype=torch.float32, device=dev)
    kvc.paged_decode_attention_fp8(q, rec, table, ctx_d, wl.scale, out,
                                   torch.full((max(ws, 16),), 0x7F, dtype=torch.uint8, device=dev), max_ctx, bps)
    torch.cuda.synchronize()
    assert kvc.kvc_device_error_flags(clear=True) == 0
    check_attention(out, oracle_fp8(wl.q[:, 0], rec, wl), f"fp8 random case {i}")


def test_decode_fp8_model_step_shape():
    """One layer of the 24-layer benchmark shape (32 x 2048, 14 / 2 heads) on an fp8 cache."""
    import paged_kv_cache_27_gb300 as kvc
    wl = workloads.multi_token_decode(77, [2048] * 32, 1)
    rec, _ = quantized_cache(wl)
    dev = "cuda"
    q = torch.from_numpy(np.ascontiguousarray(wl.q[:, 0])).to(dev)
    _, _, ws = kvc.paged_decode_plan(32, 14, 2, 64, 2048)
    out = torch.empty((32, 14, 64), dtype=torch.float32, device=dev)
    kvc.paged_decode_attention_fp8(q, rec, torch.from_numpy(wl.block_table).to(dev),
                                   torch.from_numpy(wl.ctx).to(dev), wl.scale, out,
                                   torch.empty(max(ws, 16), dtype=torch.uint8, device=dev), 2048)
    torch.cuda.synchronize()
    check_attention(out, oracle_fp8(wl.q[:, 0], rec, wl), "fp8 decode, 32 x 2048")
