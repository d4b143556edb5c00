"""Seeded synthetic inputs for the paged KV-cache attention workloads.

This module is shared by the test suite, the benchmark and the oracle side.
It holds only random draws, shapes and placements: no attention arithmetic,
no slot arithmetic, no block-pool logic.  Both the CUDA path and the oracle
consume the arrays it returns and each derives everything else on its own.

Conventions:
  * values are drawn as float32 N(0, 1) from ``numpy.random.default_rng``
    and rounded to float16 (round-to-nearest-even, numpy's astype);
  * ``ctx[b]`` is the context length of sequence b AFTER this step's token is
    appended (the new token attends to itself);
  * the cached history of sequence b (positions ``0 .. ctx[b]-2``) is stored
    logically contiguous, packed over sequences: rows
    ``hist_off[b] .. hist_off[b+1]`` of ``k_hist``/``v_hist`` (``[L][rows][Hkv][D]``);
  * block tables are a seeded random placement of logical blocks on physical
    blocks (a permutation of the pool), ``-1`` past a sequence's last block.

Workload shapes follow the five configurations this library is measured on:
  1  one sequence, Hq = Hkv = 1, D = 64, context 256, 16 permuted blocks;
  2  24 layers, B = 32, Hq = 14, Hkv = 2, D = 64, context 2048, pool of
     32 x 2048 tokens;
  3  200 sequences, contexts U{16..4096}, groups of 8 sharing a 512-token
     prefix (copy-on-write blocks);
  4  B in {1, 4, 16} x context in {4096, 16384, 65536, 131072}, keys x3 on a
     seeded 1 % of positions;
  5  varlen prefill (37, 120, 8, 200) with 8 heads and GQA prefill B = 2,
     M = 256, 8 q / 2 KV heads, then one decode token per sequence.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BASE_SEED = 42


def normal_f16(rng: np.random.Generator, shape) -> np.ndarray:
    """float32 N(0,1) draws rounded to float16."""
    return rng.standard_normal(size=shape, dtype=np.float32).astype(np.float16)


def _ceil_div(a, b):
    return -(-a // b)


@dataclass
class DecodeWorkload:
    """One decode step over a paged cache, for every layer."""

    name: str
    L: int
    B: int
    Hq: int
    Hkv: int
    D: int
    bs: int
    NB: int
    max_blocks: int
    scale: float
    ctx: np.ndarray  # int32 [B], including the new token
    block_table: np.ndarray  # int32 [B][max_blocks], -1 past the end
    hist_off: np.ndarray  # int64 [B+1], packed history offsets (ctx-1 rows each)
    k_hist: np.ndarray  # f16 [L][sum(ctx-1)][Hkv][D]
    v_hist: np.ndarray  # f16 [L][sum(ctx-1)][Hkv][D]
    q: np.ndarray  # f16 [L][B][Hq][D]
    k_new: np.ndarray  # f16 [L][B][Hkv][D]
    v_new: np.ndarray  # f16 [L][B][Hkv][D]
    extra: dict = field(default_factory=dict)

    @property
    def kv_tokens(self) -> int:
        return int(self.ctx.astype(np.int64).sum())


def _placement(rng, ctx, bs, NB=None, max_blocks=None):
    """Seeded random placement of each sequence's logical blocks on the pool."""
    nblk = [_ceil_div(int(c), bs) for c in ctx]
    total = int(sum(nblk))
    NB = total if NB is None else NB
    assert NB >= total
    perm = rng.permutation(NB).astype(np.int32)
    mb = max(nblk) if max_blocks is None else max_blocks
    table = np.full((len(ctx), mb), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[off:off + n]
        off += n
    return NB, mb, table


def _decode(name, seed, L, B, Hq, Hkv, D, ctx, bs=16, NB=None, peak_frac=0.0, peak_factor=3.0):
    """Placement and peaked positions come from ``default_rng(seed)``; layer l's values from
    ``default_rng([*seed, 1000 + l])`` (drawn in parallel threads: numpy releases the GIL)."""
    seed = list(np.atleast_1d(seed).tolist())
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, dtype=np.int32)
    NB, mb, table = _placement(rng, ctx, bs, NB)
    hist = (ctx.astype(np.int64) - 1)
    hist_off = np.zeros(B + 1, dtype=np.int64)
    hist_off[1:] = np.cumsum(hist)
    rows = int(hist_off[-1])
    peaks = []
    if peak_frac > 0:
        # keys x3 on round(frac * ctx) seeded positions of each sequence (all KV heads, all dims)
        for b in range(B):
            n = int(round(peak_frac * int(ctx[b])))
            peaks.append(np.sort(rng.permutation(int(ctx[b]))[:n]))
    k_hist = np.empty((L, rows, Hkv, D), np.float16)
    v_hist = np.empty((L, rows, Hkv, D), np.float16)
    q = np.empty((L, B, Hq, D), np.float16)
    k_new = np.empty((L, B, Hkv, D), np.float16)
    v_new = np.empty((L, B, Hkv, D), np.float16)

    def layer(l):
        r = np.random.default_rng(seed + [1000 + l])
        k32 = r.standard_normal(size=(rows, Hkv, D), dtype=np.float32)
        v_hist[l] = normal_f16(r, (rows, Hkv, D))
        q[l] = normal_f16(r, (B, Hq, D))
        kn32 = r.standard_normal(size=(B, Hkv, D), dtype=np.float32)
        v_new[l] = normal_f16(r, (B, Hkv, D))
        for b, pos in enumerate(peaks):
            cached = pos[pos < ctx[b] - 1]
            k32[hist_off[b] + cached] *= peak_factor
            if (pos == ctx[b] - 1).any():
                kn32[b] *= peak_factor
        k_hist[l] = k32
        k_new[l] = kn32

    with ThreadPoolExecutor(max_workers=min(L, os.cpu_count() or 1)) as ex:
        list(ex.map(layer, range(L)))
    return DecodeWorkload(
        name=name, L=L, B=B, Hq=Hq, Hkv=Hkv, D=D, bs=bs, NB=NB, max_blocks=mb,
        scale=1.0 / float(np.sqrt(D)), ctx=ctx, block_table=table, hist_off=hist_off,
        k_hist=k_hist, v_hist=v_hist, q=q, k_new=k_new, v_new=v_new,
        extra={"peaks": peaks, "seed": seed})


def single_sequence_256() -> DecodeWorkload:
    """1 sequence, Hq = Hkv = 1, D = 64, context 256, 16 permuted blocks, 1 layer."""
    return _decode("single_seq_ctx256", BASE_SEED + 1, L=1, B=1, Hq=1, Hkv=1, D=64, ctx=[256])


def model_decode_step(L=24, B=32, ctx=2048, Hq=14, Hkv=2, D=64) -> DecodeWorkload:
    """24 layers, 32 sequences at context 2048, 14 q / 2 KV heads, D = 64.

    The pool holds exactly B * ctx tokens (32 x 2048 = 4096 blocks of 16)."""
    return _decode(f"model_step_L{L}_B{B}_ctx{ctx}_gqa{Hq}x{Hkv}", BASE_SEED + 2, L=L, B=B, Hq=Hq, Hkv=Hkv,
                   D=D, ctx=[ctx] * B)


def long_context(B: int, ctx: int, Hq=14, Hkv=2, D=64) -> DecodeWorkload:
    """Long context: B sequences at one context length, keys x3 on 1 % of positions."""
    cells = [(b, c) for b in (1, 4, 16) for c in (4096, 16384, 65536, 131072)]
    cell = cells.index((B, ctx)) if (B, ctx) in cells else 100 + B * 7 + ctx
    return _decode(f"long_ctx_B{B}_ctx{ctx}_peaked", [BASE_SEED + 4, cell], L=1, B=B, Hq=Hq, Hkv=Hkv,
                   D=D, ctx=[ctx] * B, peak_frac=0.01)


@dataclass
class ServingMix:
    """200 sequences whose groups of 8 share a 512-token prefix.

    No block tables here: they come from running the block pool (each side
    runs its own).  ``free_order`` is the seeded order in which a fresh pool
    of NB blocks is first drained and refilled, so that FIFO allocation
    places blocks in a random physical order.
    """

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    bs: int
    NB: int
    scale: float
    group: int
    prefix_len: int
    ctx: np.ndarray  # int32 [B], including the new token
    free_order: np.ndarray  # int32 [NB] permutation
    prefix_k: np.ndarray  # f16 [ngroups][prefix_len][Hkv][D]
    prefix_v: np.ndarray
    suffix_off: np.ndarray  # int64 [B+1]; member b owns max(0, ctx-1-prefix_len) rows
    suffix_k: np.ndarray  # f16 [rows][Hkv][D]
    suffix_v: np.ndarray
    q: np.ndarray  # f16 [B][Hq][D]
    k_new: np.ndarray  # f16 [B][Hkv][D]
    v_new: np.ndarray


def shared_prefix_mix(B=200, group=8, prefix_len=512, ctx_lo=16, ctx_hi=4096, Hq=14, Hkv=2, D=64,
            bs=16) -> ServingMix:
    rng = np.random.default_rng(BASE_SEED + 3)
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=B).astype(np.int32)
    ngroups = _ceil_div(B, group)
    suffix = np.maximum(ctx.astype(np.int64) - 1 - prefix_len, 0)
    suffix_off = np.zeros(B + 1, dtype=np.int64)
    suffix_off[1:] = np.cumsum(suffix)
    # capacity: every sequence's blocks privately, plus the prefixes and one spare per sequence
    NB = int(sum(_ceil_div(int(c), bs) for c in ctx)) + ngroups * _ceil_div(prefix_len, bs) + B
    free_order = rng.permutation(NB).astype(np.int32)
    prefix_k = normal_f16(rng, (ngroups, prefix_len, Hkv, D))
    prefix_v = normal_f16(rng, (ngroups, prefix_len, Hkv, D))
    rows = int(suffix_off[-1])
    suffix_k = normal_f16(rng, (rows, Hkv, D))
    suffix_v = normal_f16(rng, (rows, Hkv, D))
    q = normal_f16(rng, (B, Hq, D))
    k_new = normal_f16(rng, (B, Hkv, D))
    v_new = normal_f16(rng, (B, Hkv, D))
    return ServingMix(
        name=f"shared_prefix_B{B}_ctx{ctx_lo}-{ctx_hi}_prefix{prefix_len}x{group}", B=B, Hq=Hq,
        Hkv=Hkv, D=D, bs=bs, NB=NB, scale=1.0 / float(np.sqrt(D)), group=group,
        prefix_len=prefix_len, ctx=ctx, free_order=free_order, prefix_k=prefix_k,
        prefix_v=prefix_v, suffix_off=suffix_off, suffix_k=suffix_k, suffix_v=suffix_v, q=q,
        k_new=k_new, v_new=v_new)


@dataclass
class PrefillWorkload:
    """Packed varlen prefill, then one decode token per sequence over the paged cache."""

    name: str
    Hq: int
    Hkv: int
    D: int
    bs: int
    scale: float
    seqlens: tuple
    cu_seqlens: np.ndarray  # int32 [nseq+1]
    q: np.ndarray  # f16 [T][Hq][D]
    k: np.ndarray  # f16 [T][Hkv][D]
    v: np.ndarray
    NB: int
    max_blocks: int
    block_table: np.ndarray  # int32 [nseq][max_blocks], covers seqlen+1 tokens
    q_dec: np.ndarray  # f16 [nseq][Hq][D] for the decode token
    k_dec: np.ndarray  # f16 [nseq][Hkv][D]
    v_dec: np.ndarray


def _prefill(name, seed, seqlens, Hq, Hkv, D, bs=16) -> PrefillWorkload:
    rng = np.random.default_rng(seed)
    seqlens = tuple(int(s) for s in seqlens)
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens)
    T = int(cu[-1])
    q = normal_f16(rng, (T, Hq, D))
    k = normal_f16(rng, (T, Hkv, D))
    v = normal_f16(rng, (T, Hkv, D))
    NB, mb, table = _placement(rng, [s + 1 for s in seqlens], bs)
    n = len(seqlens)
    return PrefillWorkload(
        name=name, Hq=Hq, Hkv=Hkv, D=D, bs=bs, scale=1.0 / float(np.sqrt(D)), seqlens=seqlens,
        cu_seqlens=cu, q=q, k=k, v=v, NB=NB, max_blocks=mb, block_table=table,
        q_dec=normal_f16(rng, (n, Hq, D)), k_dec=normal_f16(rng, (n, Hkv, D)),
        v_dec=normal_f16(rng, (n, Hkv, D)))


def varlen_prefill(seqlens=(37, 120, 8, 200), H=8, D=64) -> PrefillWorkload:
    return _prefill("varlen_prefill_" + "-".join(map(str, seqlens)), [BASE_SEED + 5, 0], seqlens, H, H, D)


def gqa_prefill(B=2, M=256, Hq=8, Hkv=2, D=64) -> PrefillWorkload:
    return _prefill(f"gqa_prefill_B{B}_M{M}_{Hq}x{Hkv}", [BASE_SEED + 5, 1], (M,) * B, Hq, Hkv, D)


def small_decode(seed, B, Hq, Hkv, D, ctx, L=1, bs=16, peak_frac=0.0) -> DecodeWorkload:
    """A small decode case for parity sweeps (ragged contexts allowed)."""
    return _decode(f"small_B{B}_{Hq}x{Hkv}_D{D}", [BASE_SEED, 1000 + seed], L=L, B=B, Hq=Hq,
                   Hkv=Hkv, D=D, ctx=list(ctx), bs=bs, peak_frac=peak_frac)


@dataclass
class CascadeWorkload:
    """Groups of consecutive sequences whose block tables begin with the same blocks (one layer)."""

    name: str
    Hq: int
    Hkv: int
    D: int
    bs: int
    scale: float
    NB: int
    q: np.ndarray            # f16 [B][Hq][D]
    k_pool: np.ndarray       # f16 [NB][Hkv][bs][D]
    v_pool: np.ndarray
    block_table: np.ndarray  # int32 [B][max_blocks], -1 past each context
    ctx: np.ndarray          # int32 [B]
    group_start: np.ndarray  # int32 [n_groups + 1]
    shared_blocks: np.ndarray  # int32 [B]: the leading blocks of b's group


def cascade_decode(seed, group_sizes, shared, extra, Hq=14, Hkv=2, D=64, bs=16) -> CascadeWorkload:
    """Group g (group_sizes[g] consecutive sequences) shares shared[g] leading blocks; sequence b then owns
    extra[b] >= 1 more tokens in private blocks. Physical blocks are a seeded permutation; every K/V row of the
    pool, used or not, is N(0,1) fp16."""
    rng = np.random.default_rng(seed)
    B = int(sum(group_sizes))
    assert len(extra) == B and len(shared) == len(group_sizes) and min(extra) >= 1
    need = int(sum(shared)) + sum(_ceil_div(int(e), bs) for e in extra)
    NB = need + 3
    perm = iter(rng.permutation(NB).astype(np.int32).tolist())
    rows, ctx, sh = [], [], []
    b = 0
    for g, n in enumerate(group_sizes):
        common = [next(perm) for _ in range(int(shared[g]))]
        for _ in range(n):
            own = [next(perm) for _ in range(_ceil_div(int(extra[b]), bs))]
            rows.append(common + own)
            ctx.append(bs * int(shared[g]) + int(extra[b]))
            sh.append(int(shared[g]))
            b += 1
    mb = max(len(r) for r in rows)
    table = np.full((B, mb), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        table[i, :len(r)] = r
    gs = np.zeros(len(group_sizes) + 1, dtype=np.int32)
    gs[1:] = np.cumsum(group_sizes)
    return CascadeWorkload(
        name=f"cascade_{seed}", Hq=Hq, Hkv=Hkv, D=D, bs=bs, scale=1.0 / float(np.sqrt(D)), NB=NB,
        q=normal_f16(rng, (B, Hq, D)), k_pool=normal_f16(rng, (NB, Hkv, bs, D)),
        v_pool=normal_f16(rng, (NB, Hkv, bs, D)), block_table=table, ctx=np.array(ctx, dtype=np.int32),
        group_start=gs, shared_blocks=np.array(sh, dtype=np.int32))


@dataclass
class MultiTokenWorkload:
    """Each sequence's T newest tokens (already in the cache) to be verified at once (one layer)."""

    name: str
    T: int
    Hq: int
    Hkv: int
    D: int
    bs: int
    scale: float
    NB: int
    q: np.ndarray            # f16 [B][T][Hq][D]
    k_pool: np.ndarray       # f16 [NB][Hkv][bs][D]
    v_pool: np.ndarray
    block_table: np.ndarray  # int32 [B][max_blocks], -1 past each context
    ctx: np.ndarray          # int32 [B], including the T new tokens


def multi_token_decode(seed, ctx, T, Hq=14, Hkv=2, D=64, bs=16) -> MultiTokenWorkload:
    """Contexts ctx (each >= T) on seeded-permuted blocks; every K/V row of the pool N(0,1) fp16."""
    rng = np.random.default_rng(seed)
    ctx = np.array(ctx, dtype=np.int32)
    assert np.all(ctx >= T)
    nblk = [_ceil_div(int(c), bs) for c in ctx]
    NB = sum(nblk) + 2
    perm = rng.permutation(NB).astype(np.int32)
    table = np.full((len(ctx), max(nblk)), -1, dtype=np.int32)
    a = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[a:a + n]
        a += n
    return MultiTokenWorkload(
        name=f"multi_{seed}_T{T}", T=T, Hq=Hq, Hkv=Hkv, D=D, bs=bs, scale=1.0 / float(np.sqrt(D)), NB=NB,
        q=normal_f16(rng, (len(ctx), T, Hq, D)), k_pool=normal_f16(rng, (NB, Hkv, bs, D)),
        v_pool=normal_f16(rng, (NB, Hkv, bs, D)), block_table=table, ctx=ctx)
