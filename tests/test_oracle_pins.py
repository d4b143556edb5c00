"""Pins for the fp64 oracle, against things other than itself (CPU only).

Each test ties an oracle function to the pages' printed numbers, a closed
form, a library routine (torch float64 scaled_dot_product_attention, numpy's
float16 widening) or a brute force, chosen so that a dropped term, a wrong
sign or index or a transposed operand fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import paging
import workloads

RNG = np.random.default_rng(7)


def f16(*shape, scale=1.0):
    return (RNG.standard_normal(shape).astype(np.float32) * scale).astype(np.float16)


def paged_single(K, V, bs=16, perm_seed=0, NB=None):
    """Place one contiguous sequence K, V ([n][Hkv][D] f16) on permuted pages (test-side placement)."""
    n, Hkv, D = K.shape
    nblk = -(-n // bs)
    NB = NB or nblk
    perm = np.random.default_rng(perm_seed).permutation(NB)[:nblk].astype(np.int32)
    kc = np.zeros((NB, Hkv, bs, D), np.float16)
    vc = np.zeros_like(kc)
    for j in range(n):
        kc[perm[j // bs], :, j % bs] = K[j]
        vc[perm[j // bs], :, j % bs] = V[j]
    return kc, vc, perm[None, :]


# ---------------------------------------------------------------- widening
def test_half_widening_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ------------------------------------------------------------ brute force
@pytest.mark.parametrize("n", [1, 2, 15, 16, 17, 33, 256])
def test_decode_equals_last_row_of_full_causal(n):
    """The cached row equals row n-1 of the n x n causal attention (gustavoai.dev page)."""
    D = 64
    Q, K, V = f16(n, 1, D), f16(n, 1, D), f16(n, 1, D)
    kc, vc, table = paged_single(K, V, perm_seed=n)
    out = oracle.decode(Q[n - 1:n], kc, vc, table, np.array([n], np.int32), 0.125)
    full = oracle.causal_attention(Q[:, 0].astype(np.float64), K[:, 0].astype(np.float64),
                                   V[:, 0].astype(np.float64), 0.125)
    assert np.max(np.abs(out[0, 0] - full[n - 1])) <= 1e-12
    if n == 256:
        # every row of the brute force is the decode of its own prefix
        for t in (0, 100, 200):
            o = oracle.decode(Q[t:t + 1], kc, vc, table, np.array([t + 1], np.int32), 0.125)
            assert np.max(np.abs(o[0, 0] - full[t])) <= 1e-12


@pytest.mark.parametrize("n,T", [(1, 1), (2, 2), (17, 2), (40, 4), (100, 8), (16, 8)])
def test_decode_multi_equals_last_rows_of_full_causal(n, T):
    """T new tokens verified at once: token t's output is row n - T + t of the n x n causal attention."""
    D = 64
    Q, K, V = f16(n, 1, D), f16(n, 1, D), f16(n, 1, D)
    kc, vc, table = paged_single(K, V, perm_seed=n + 100 * T)
    out = oracle.decode_multi(Q[None, n - T:n], kc, vc, table, np.array([n], np.int32), 0.125)
    full = oracle.causal_attention(Q[:, 0].astype(np.float64), K[:, 0].astype(np.float64),
                                   V[:, 0].astype(np.float64), 0.125)
    for t in range(T):
        assert np.max(np.abs(out[0, t, 0] - full[n - T + t])) <= 1e-12


def test_decode_multi_gqa_vs_torch_sdpa():
    """Several sequences, 8 query / 2 KV heads: torch float64 SDPA with the offset causal mask."""
    Hq, Hkv, D, T = 8, 2, 64, 3
    ctxs = [3, 20, 77]
    for b, n in enumerate(ctxs):
        Q, K, V = f16(T, Hq, D), f16(n, Hkv, D), f16(n, Hkv, D)
        kc, vc, table = paged_single(K, V, perm_seed=b)
        out = oracle.decode_multi(Q[None], kc, vc, table, np.array([n], np.int32), 1 / math.sqrt(D))
        q = torch.from_numpy(Q.astype(np.float64)).permute(1, 0, 2)                 # [Hq][T][D]
        k = torch.from_numpy(K.astype(np.float64)).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        v = torch.from_numpy(V.astype(np.float64)).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        mask = torch.arange(n)[None, :] <= (n - T + torch.arange(T))[:, None]     # [T][n]
        ref = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=1 / math.sqrt(D))
        assert np.max(np.abs(out[0] - ref.permute(1, 0, 2).numpy())) <= 1e-12


def test_full_causal_vs_torch_sdpa():
    n, D = 48, 64
    Q, K, V = (RNG.standard_normal((n, D)) for _ in range(3))
    ours = oracle.causal_attention(Q, K, V, 0.3)
    ref = F.scaled_dot_product_attention(torch.tensor(Q)[None], torch.tensor(K)[None],
                                         torch.tensor(V)[None], is_causal=True, scale=0.3)[0].numpy()
    assert np.max(np.abs(ours - ref)) <= 1e-12


@pytest.mark.parametrize("Hq,Hkv,D", [(14, 2, 64), (8, 8, 64), (4, 1, 128), (6, 3, 32)])
def test_decode_vs_torch_sdpa_gqa(Hq, Hkv, D):
    """Paged GQA decode equals torch's float64 SDPA with grouped heads (xformers BMGHK article)."""
    ctx = [1, 7, 16, 40, 100]
    wl = workloads.small_decode(3, B=len(ctx), Hq=Hq, Hkv=Hkv, D=D, ctx=ctx)
    out, kc, vc = paging.decode_step(wl, 0)
    G = Hq // Hkv
    for b, n in enumerate(ctx):
        h0, h1 = wl.hist_off[b], wl.hist_off[b + 1]
        K = np.concatenate([wl.k_hist[0, h0:h1], wl.k_new[0, b:b + 1]]).astype(np.float64)  # [n][Hkv][D]
        V = np.concatenate([wl.v_hist[0, h0:h1], wl.v_new[0, b:b + 1]]).astype(np.float64)
        q = torch.tensor(wl.q[0, b].astype(np.float64))[:, None, :]  # [Hq][1][D]
        Kt = torch.tensor(K).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq][n][D]
        Vt = torch.tensor(V).permute(1, 0, 2).repeat_interleave(G, dim=0)
        ref = F.scaled_dot_product_attention(q, Kt, Vt, scale=wl.scale)[:, 0].numpy()
        assert np.max(np.abs(out[b] - ref)) <= 1e-12, b


# ------------------------------------------------------------- closed forms
def test_one_token_context_returns_v0_exactly():
    K, V, q = f16(1, 1, 64), f16(1, 1, 64), f16(1, 1, 64, scale=10.0)
    kc, vc, table = paged_single(K, V)
    out = oracle.decode(q, kc, vc, table, np.array([1], np.int32), 0.125)
    assert np.array_equal(out[0, 0], V[0, 0].astype(np.float64))


def test_identical_keys_give_mean_of_values():
    n = 37
    K = np.repeat(f16(1, 1, 64), n, axis=0)
    V = f16(n, 1, 64)
    q = f16(1, 1, 64, scale=3.0)
    kc, vc, table = paged_single(K, V, perm_seed=5)
    out = oracle.decode(q, kc, vc, table, np.array([n], np.int32), 0.125)
    assert np.max(np.abs(out[0, 0] - V[:, 0].astype(np.float64).mean(0))) <= 1e-14


def test_two_tokens_logistic_form():
    """Two keys: o = v1 + (v2 - v1) * sigmoid(s2 - s1); scores set by construction."""
    D = 2
    for a in (-3.0, 0.0, 0.5, 2.0, 7.0):
        q = np.array([[[a, 0.0]]], np.float16)
        K = np.array([[[0.0, 1.0]], [[1.0, 0.0]]], np.float16)  # s1 = 0, s2 = a * scale
        V = np.array([[[1.5, -2.0]], [[-0.25, 4.0]]], np.float16)
        kc, vc, table = paged_single(K, V, bs=16)
        scale = 0.75
        out = oracle.decode(q, kc, vc, table, np.array([2], np.int32), scale)
        sig = 1.0 / (1.0 + math.exp(-a * scale))
        v1, v2 = V[0, 0].astype(np.float64), V[1, 0].astype(np.float64)
        assert np.max(np.abs(out[0, 0] - (v1 + (v2 - v1) * sig))) <= 1e-15


def test_dominant_key_selects_its_value():
    n, D = 50, 64
    q = np.zeros((1, 1, D), np.float16)
    q[0, 0, 0] = 1.0
    K = f16(n, 1, D, scale=0.01)
    K[17, 0, 0] = 600.0  # score gap >= 600*0.125 - small
    V = f16(n, 1, D)
    kc, vc, table = paged_single(K, V)
    out = oracle.decode(q, kc, vc, table, np.array([n], np.int32), 0.125)
    assert np.max(np.abs(out[0, 0] - V[17, 0].astype(np.float64))) <= 1e-30 + math.exp(-70) * 10


def test_scale_enters_the_scores():
    """Doubling the scale equals doubling q (a dropped or misplaced scale fails this)."""
    K, V = f16(30, 1, 64), f16(30, 1, 64)
    q = f16(1, 1, 64, scale=0.5)
    kc, vc, table = paged_single(K, V)
    a = oracle.decode(q, kc, vc, table, np.array([30], np.int32), 0.25)
    b = oracle.decode((q.astype(np.float32) * 2).astype(np.float16), kc, vc, table,
                      np.array([30], np.int32), 0.125)
    assert np.max(np.abs(a - b)) <= 1e-14
    c = oracle.decode(q, kc, vc, table, np.array([30], np.int32), 0.125)
    assert np.max(np.abs(a - c)) > 1e-6


# ----------------------------------------------------------------- paging
def test_block_permutation_invariance_bit_exact():
    n = 200
    K, V, q = f16(n, 2, 64), f16(n, 2, 64), f16(1, 6, 64)
    outs = []
    for seed in range(4):
        kc, vc, table = paged_single(K, V, perm_seed=seed, NB=40)
        outs.append(oracle.decode(q, kc, vc, table, np.array([n], np.int32), 0.125))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_prefix_sharing_equals_private_copies():
    """Two sequences pointing at the same prefix pages give the same result as private copies."""
    bs, D, Hkv = 16, 64, 2
    pre = 64
    K = f16(pre + 20, Hkv, D)
    V = f16(pre + 20, Hkv, D)
    K2 = np.concatenate([K[:pre], f16(30, Hkv, D)])
    V2 = np.concatenate([V[:pre], f16(30, Hkv, D)])
    q = f16(2, 4, D)
    NB = 20
    kc = np.zeros((NB, Hkv, bs, D), np.float16)
    vc = np.zeros_like(kc)
    shared = [3, 9, 0, 14]
    t1 = shared + [5, 11]
    t2 = shared + [1, 7]
    for tbl, KK, VV in ((t1, K, V), (t2, K2, V2)):
        for j in range(len(KK)):
            kc[tbl[j // bs], :, j % bs] = KK[j]
            vc[tbl[j // bs], :, j % bs] = VV[j]
    table = np.array([t1, t2], np.int32)
    ctx = np.array([len(K), len(K2)], np.int32)
    shared_out = oracle.decode(q, kc, vc, table, ctx, 0.125)
    priv = np.array([[2, 4, 6, 8, 5, 11], [10, 12, 13, 15, 1, 7]], np.int32)
    kc2, vc2 = kc.copy(), vc.copy()
    for s, (a, b) in enumerate(zip(shared, priv[0][:4])):
        kc2[b], vc2[b] = kc[a], vc[a]
    for s, (a, b) in enumerate(zip(shared, priv[1][:4])):
        kc2[b], vc2[b] = kc[a], vc[a]
    priv_out = oracle.decode(q, kc2, vc2, priv, ctx, 0.125)
    assert np.array_equal(shared_out, priv_out)


def test_gqa_equals_mha_with_replicated_kv_heads():
    """A KV head shared by G query heads equals MHA with that head copied G times (neuralialabs page)."""
    n, Hq, Hkv, D = 70, 14, 2, 64
    G = Hq // Hkv
    K, V, q = f16(n, Hkv, D), f16(n, Hkv, D), f16(1, Hq, D)
    kc, vc, table = paged_single(K, V, perm_seed=1)
    gqa = oracle.decode(q, kc, vc, table, np.array([n], np.int32), 0.125)
    Kr, Vr = np.repeat(K, G, axis=1), np.repeat(V, G, axis=1)
    kc2, vc2, table2 = paged_single(Kr, Vr, perm_seed=2)
    mha = oracle.decode(q, kc2, vc2, table2, np.array([n], np.int32), 0.125)
    assert np.array_equal(gqa, mha)


def test_append_then_gather_roundtrip_bit_exact():
    """Filling a cache by slot scatter and reading it back through the table returns the history."""
    wl = workloads.small_decode(11, B=3, Hq=4, Hkv=2, D=64, ctx=[5, 33, 64])
    kc, vc = paging.fill_layer(wl, 0)
    bs = wl.bs
    for b in range(wl.B):
        n = int(wl.ctx[b]) - 1
        # read back by reshaping the pool to per-head token rows (independent of the slot formula)
        rows_k = kc.transpose(1, 0, 2, 3).reshape(wl.Hkv, wl.NB * bs, wl.D)
        phys = np.repeat(wl.block_table[b], bs)[:n] * bs + np.tile(np.arange(bs), wl.max_blocks)[:n]
        got = rows_k[:, phys].transpose(1, 0, 2)
        assert np.array_equal(got.view(np.uint16),
                              wl.k_hist[0, wl.hist_off[b]:wl.hist_off[b + 1]].view(np.uint16))
    # pages not named by any table stay zero
    used = set(wl.block_table[wl.block_table >= 0].tolist())
    for p in range(wl.NB):
        if p not in used:
            assert not kc[p].any()


def test_append_skips_negative_slots_and_rejects_overflow():
    kc, vc = paging.empty_cache(4, 1, 16, 8)
    kn, vn = f16(3, 1, 8), f16(3, 1, 8)
    oracle.append(kc, vc, kn, vn, np.array([5, -1, 63], np.int64))
    assert np.array_equal(kc[0, 0, 5], kn[0, 0]) and np.array_equal(kc[3, 0, 15], kn[2, 0])
    assert np.count_nonzero(np.any(kc != 0, axis=-1)) == 2
    with pytest.raises(IndexError):
        oracle.append(kc, vc, kn, vn, np.array([64, 0, 0], np.int64))


# --------------------------------------------------------- split + merge
def test_partial_merge_partition_invariance():
    """Merging partial softmaxes over any partition equals the unsplit row (FlashAttention article)."""
    n, D = 300, 64
    q = RNG.standard_normal(D)
    K = RNG.standard_normal((n, D)) * 2
    V = RNG.standard_normal((n, D))
    m, l, acc = oracle.partial(q, K, V, 0, n, 0.125)
    whole = acc / l
    full = oracle.causal_attention(np.vstack([np.zeros((n - 1, D)), q]), K, V, 0.125)[n - 1]
    assert np.max(np.abs(whole - full)) <= 1e-13
    for trial in range(5):
        cuts = np.sort(RNG.choice(np.arange(1, n), size=trial + 2, replace=False))
        edges = [0, *cuts.tolist(), n]
        if trial == 3:
            edges = [0, 0, *cuts.tolist(), n, n]  # empty parts contribute nothing
        parts = [oracle.partial(q, K, V, a, b, 0.125) for a, b in zip(edges[:-1], edges[1:])]
        o = oracle.merge([p[0] for p in parts], [p[1] for p in parts], np.array([p[2] for p in parts]))
        assert np.max(np.abs(o - whole)) <= 1e-13


def test_merge_rescales_by_max_difference():
    """Two one-row parts merge to the two-token logistic form."""
    D = 3
    v1, v2 = np.array([1.0, 2.0, 3.0]), np.array([-1.0, 0.5, 8.0])
    m = np.array([0.3, 2.3])
    o = oracle.merge(m, np.array([1.0, 1.0]), np.array([v1, v2]))
    sig = 1 / (1 + math.exp(-2.0))
    assert np.max(np.abs(o - (v1 + (v2 - v1) * sig))) <= 1e-15


# ---------------------------------------------------------------- prefill
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_segments_vs_torch_sdpa(causal):
    """Every packed segment equals standalone attention on it (xformers article, part 4)."""
    wl = workloads.varlen_prefill()
    out = oracle.prefill(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.scale, causal=causal)
    for s in range(len(wl.seqlens)):
        a, b = wl.cu_seqlens[s], wl.cu_seqlens[s + 1]
        q = torch.tensor(wl.q[a:b].astype(np.float64)).permute(1, 0, 2)
        k = torch.tensor(wl.k[a:b].astype(np.float64)).permute(1, 0, 2)
        v = torch.tensor(wl.v[a:b].astype(np.float64)).permute(1, 0, 2)
        ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=wl.scale)
        assert np.max(np.abs(out[a:b] - ref.permute(1, 0, 2).numpy())) <= 1e-12


def test_prefill_gqa_vs_torch_sdpa():
    wl = workloads.gqa_prefill()
    G = wl.Hq // wl.Hkv
    for causal in (True, False):
        out = oracle.prefill(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.scale, causal=causal)
        for s in range(len(wl.seqlens)):
            a, b = wl.cu_seqlens[s], wl.cu_seqlens[s + 1]
            q = torch.tensor(wl.q[a:b].astype(np.float64)).permute(1, 0, 2)
            k = torch.tensor(wl.k[a:b].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
            v = torch.tensor(wl.v[a:b].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
            ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=wl.scale)
            assert np.max(np.abs(out[a:b] - ref.permute(1, 0, 2).numpy())) <= 1e-12


def test_prefill_last_row_equals_paged_decode():
    """The causal prefill's last row of a segment equals the decode over a cache holding that segment."""
    wl = workloads.gqa_prefill(B=1, M=100)
    out = oracle.prefill(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.scale, causal=True)
    kc, vc, table = paged_single(wl.k, wl.v, perm_seed=3)
    dec = oracle.decode(wl.q[-1:], kc, vc, table, np.array([100], np.int32), wl.scale)
    assert np.max(np.abs(dec[0] - out[-1])) <= 1e-12
