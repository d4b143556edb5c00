"""Slot arithmetic, cache filling and the serving-mix protocol -- TEST INFRASTRUCTURE ONLY.

Sources:
  * "Aufmerksamkeit" feed (chatgpz.de), PagedAttention article, SECTION 2:
    token position p of a request lives on page ``block_table[p // PAGE_SIZE]``
    at offset ``p % PAGE_SIZE``; a new page is claimed when the token count
    reaches a page boundary.
  * same article, SECTION 3: requests sharing a system prompt point their
    tables at the same pages (refcount up); a request that writes a diverging
    token into a shared page first takes a private copy (copy-on-write).
  * "La caché de claves y valores" (gustavoai.dev), section "Las claves y los
    valores de una posición no cambian": per decode token, k_t and v_t are
    appended to the cache first, then the row attends over the whole cache.

The physical cache layout is this library's choice (the pages fix none):
one layer is ``[NB][Hkv][bs][D]``; slot = physical_block * bs + offset.
Attention results do not depend on it (pinned by the permutation tests).
"""
from __future__ import annotations

import numpy as np

from . import append as _append
from . import decode as _decode
from .page_pool import PagePool


def slot_of(table_row, pos: int, bs: int) -> int:
    return int(table_row[pos // bs]) * bs + pos % bs


def history_slots(block_table, hist_off, bs) -> np.ndarray:
    """Slot of every cached history token, packed like the workload's history rows."""
    B = len(hist_off) - 1
    out = np.empty(int(hist_off[-1]), dtype=np.int64)
    for b in range(B):
        n = int(hist_off[b + 1] - hist_off[b])
        pos = np.arange(n, dtype=np.int64)
        out[hist_off[b]:hist_off[b + 1]] = block_table[b][pos // bs].astype(np.int64) * bs + pos % bs
    return out


def step_slots(block_table, ctx, bs) -> np.ndarray:
    """Slot of the token appended in this step (position ctx - 1) of every sequence."""
    return np.array([slot_of(block_table[b], int(ctx[b]) - 1, bs) for b in range(len(ctx))],
                    dtype=np.int64)


def empty_cache(NB, Hkv, bs, D):
    return (np.zeros((NB, Hkv, bs, D), dtype=np.float16), np.zeros((NB, Hkv, bs, D), dtype=np.float16))


def fill_layer(wl, layer):
    """One layer's cache holding every sequence's history (positions 0 .. ctx-2)."""
    kc, vc = empty_cache(wl.NB, wl.Hkv, wl.bs, wl.D)
    slots = history_slots(wl.block_table, wl.hist_off, wl.bs)
    _append(kc, vc, wl.k_hist[layer], wl.v_hist[layer], slots)
    return kc, vc


def decode_step(wl, layer, kc=None, vc=None, nthreads=None):
    """Append this step's token, then decode; returns (out fp64 [B][Hq][D], kc, vc)."""
    if kc is None:
        kc, vc = fill_layer(wl, layer)
    _append(kc, vc, wl.k_new[layer], wl.v_new[layer], step_slots(wl.block_table, wl.ctx, wl.bs))
    out = _decode(wl.q[layer], kc, vc, wl.block_table, wl.ctx, wl.scale, nthreads=nthreads)
    return out, kc, vc


# ---------------------------------------------------------------------------
# Serving mix: groups sharing a prefix through refcounted pages.
# ---------------------------------------------------------------------------
def serving_mix(mix, nthreads=None):
    """Run the serving-mix protocol on the restated pool.

    Protocol (both this oracle and the library's harness follow it):
      1. allocate all NB pages, then release them in ``mix.free_order``, so
         FIFO allocation walks a seeded random physical order;
      2. per group in order: allocate the prefix pages; each member in order
         shares the first ceil(min(prefix_len, ctx-1) / bs) of them; the
         prefix tokens that at least one member holds are written into the
         shared pages; the prompt's own reference is then released (pages
         nobody needs return to the pool); members in order then allocate
         private pages until their table covers ctx-1 tokens and their
         suffix tokens are written there;
      3. the decode step, members in order: position p = ctx-1; if p falls on
         a new page, allocate it; else if its page has refcount > 1, take a
         copy-on-write private copy (the whole page is copied, then the old
         reference is released); the token's K/V are then appended at p and
         every sequence attends over its ctx tokens.
    Returns a dict with the block tables, copy pairs, slots, caches and output.
    """
    bs, B, G = mix.bs, mix.B, mix.group
    pool = PagePool(mix.NB)
    for _ in range(mix.NB):
        pool.allocate()
    for pid in mix.free_order:
        pool.release(int(pid))
    kc, vc = empty_cache(mix.NB, mix.Hkv, bs, mix.D)
    tables: list[list[int]] = [[] for _ in range(B)]
    npre = -(-mix.prefix_len // bs)
    for g in range(-(-B // G)):
        members = range(g * G, min(B, (g + 1) * G))
        prefix_pages = [pool.allocate() for _ in range(npre)]
        for b in members:
            need = -(-min(mix.prefix_len, int(mix.ctx[b]) - 1) // bs)
            for pid in prefix_pages[:need]:
                pool.share(pid)
            tables[b] = list(prefix_pages[:need])
        # prefix tokens some member holds go into the shared pages, then the prompt's reference is dropped
        n_pre = max(min(mix.prefix_len, int(mix.ctx[b]) - 1) for b in members)
        slots = np.array([prefix_pages[p // bs] * bs + p % bs for p in range(n_pre)], dtype=np.int64)
        _append(kc, vc, mix.prefix_k[g, :n_pre], mix.prefix_v[g, :n_pre], slots)
        for pid in prefix_pages:
            pool.release(pid)
        for b in members:
            while len(tables[b]) * bs < int(mix.ctx[b]) - 1:
                tables[b].append(pool.allocate())
            n_suf = int(mix.suffix_off[b + 1] - mix.suffix_off[b])
            if n_suf:
                pos = mix.prefix_len + np.arange(n_suf)
                slots = np.array([slot_of(tables[b], int(p), bs) for p in pos], dtype=np.int64)
                sl = slice(int(mix.suffix_off[b]), int(mix.suffix_off[b + 1]))
                _append(kc, vc, mix.suffix_k[sl], mix.suffix_v[sl], slots)
    tables_before = [list(t) for t in tables]
    # the decode step
    copies = []
    for b in range(B):
        p = int(mix.ctx[b]) - 1
        if p // bs == len(tables[b]):
            tables[b].append(pool.allocate())
        else:
            old = tables[b][p // bs]
            if pool.refcount(old) > 1:
                new = pool.cow_copy(old)
                copies.append((old, new))
                tables[b][p // bs] = new
    for old, new in copies:  # private copies are taken before any token of the step is written
        kc[new] = kc[old]
        vc[new] = vc[old]
    slots = np.array([slot_of(tables[b], int(mix.ctx[b]) - 1, bs) for b in range(B)], dtype=np.int64)
    _append(kc, vc, mix.k_new, mix.v_new, slots)
    mb = max(len(t) for t in tables)
    table = np.full((B, mb), -1, dtype=np.int32)
    for b in range(B):
        table[b, :len(tables[b])] = tables[b]
    out = _decode(mix.q, kc, vc, table, mix.ctx, mix.scale, nthreads=nthreads)
    return {"tables_before": tables_before, "block_table": table, "copies": copies, "slots": slots,
            "k_cache": kc, "v_cache": vc, "out": out, "pool": pool}
