"""Pins for the restated block pool, the byte-count formula and the serving-mix protocol (CPU)."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import geometry, paging
from oracle.page_pool import PagedRequest, PagePool, PoolOOM
import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_kv_bytes_golden():
    g = load("kv_bytes.json")
    for c in g["cases"]:
        per = geometry.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], c["elem_bytes"])
        if "bytes_per_token" in c:
            assert per == c["bytes_per_token"], c["what"]
        if "tokens" in c:
            assert geometry.kv_cache_bytes(c["tokens"], c["layers"], c["kv_heads"], c["head_dim"],
                                           c["elem_bytes"]) == c["bytes"], c["what"]
        if "tokens_b" in c:
            assert c["tokens_b"] * per == c["bytes_b"]
        if "mib" in c:
            assert c["bytes"] == c["mib"] * 2**20
    # the allocator measurement: a key and a value tensor of shape (1, 2, 295, 64) fp16 per layer, 24 layers
    assert 2 * (1 * 2 * 295 * 64) * 2 * 24 == 3624960
    # MHA/GQA ratio is exactly the group size 14 / 2
    assert geometry.kv_bytes_per_token(24, 14, 64, 2) == 7 * geometry.kv_bytes_per_token(24, 2, 64, 2)
    # the same 65,536 tokens split three ways cost the same
    assert len({geometry.kv_cache_bytes(u * t, 24, 2, 64, 2) for u, t in ((32, 2048), (64, 1024), (128, 512))}) == 1
    # a pool of 4096 pages of 16 tokens is exactly those 768 MiB
    assert geometry.paged_pool_bytes(4096, 16, 24, 2, 64, 2) == 805306368


def test_pool_section2_worked_example():
    g = load("page_pool.json")["section2"]
    pool = PagePool(g["total_pages"])
    reqs = [PagedRequest(f"req-{i}", pool, 16) for i in range(len(g["token_counts"]))]
    for r, n in zip(reqs, g["token_counts"]):
        for _ in range(n):
            r.generate_token()
    assert [len(r.block_table) for r in reqs] == g["pages"]
    waste = [(16 - r.tokens % 16) % 16 for r in reqs]
    assert waste == g["last_page_waste"]
    assert round(pool.utilisation, 1) == g["utilisation_pct_1dp"]
    before = len(pool.free)
    reqs[g["released_request"]].free()
    assert len(pool.free) - before == g["pages_returned"]
    # FIFO: request 0 holds pages 0..19, request 1 pages 20..22 (now at the tail of the free list)
    assert reqs[0].block_table == list(range(20))
    assert list(pool.free)[-3:] == [20, 21, 22]


def test_pool_section3_copy_on_write_example():
    g = load("page_pool.json")["section3"]
    pool = PagePool(g["total_pages"])
    n_pages = math.ceil(g["system_tokens"] / 16)
    assert n_pages == g["system_pages"]
    shared = [pool.allocate() for _ in range(n_pages)]
    assert shared == g["shared_pids"]
    tables = []
    for _ in range(g["users"]):
        for pid in shared:
            pool.share(pid)
        tables.append(list(shared))
    assert all(pool.refcount(p) == g["refcount_after_share"] for p in shared)
    mb_per_token = geometry.kv_bytes_per_token(32, 32, 128, 2) / 2**20
    saved = (n_pages * g["users"] - n_pages) * 16 * mb_per_token
    assert (n_pages * g["users"], n_pages) == (g["naive_pages"], g["cow_pages"])
    assert saved == g["saved_mb"]
    old = tables[g["diverging_user"]][-1]
    new = pool.cow_copy(old)
    assert (old, new) == (g["old_pid"], g["new_pid"])
    assert pool.refcount(old) == g["refcount_after_share"] - 1 and pool.refcount(new) == 1


def test_naive_allocation_section1_arithmetic():
    g = load("page_pool.json")["section1"]
    mb = geometry.kv_bytes_per_token(32, 32, 128, 2) / 2**20
    pre, used = g["max_seq_len"] * mb, g["avg_response"] * mb
    assert (pre, used) == (g["pre_allocated_mb"], g["used_mb"])
    assert round(used / pre * 100, 1) == g["utilisation_pct_1dp"]
    assert pre - used == g["wasted_mb"]
    assert int((pre - used) * g["users"] / 1024) == g["wasted_gb_approx"]


def test_pool_errors():
    pool = PagePool(2)
    a, b = pool.allocate(), pool.allocate()
    with pytest.raises(PoolOOM):
        pool.allocate()
    pool.release(a)
    with pytest.raises(ValueError):
        pool.release(a)  # already free
    with pytest.raises(ValueError):
        pool.share(a)
    with pytest.raises(ValueError):
        pool.release(7)
    assert pool.utilisation == 50.0


def test_paged_utilisation_near_98_percent():
    """Paged waste is at most one partial page per request (PagedAttention article, SECTION 4)."""
    rng = np.random.default_rng(42)
    for n in (10, 25, 50, 100, 200):
        toks = np.clip(rng.normal(500, 200, n).astype(int), 200, 2048)
        pool = PagePool(int(np.ceil(toks / 16).sum()))
        for t in toks:
            r = PagedRequest(0, pool)
            for _ in range(int(t)):
                r.generate_token()
        paged = toks.sum() / ((pool.total - len(pool.free)) * 16) * 100
        assert 97.0 < paged <= 100.0
        assert abs(toks.sum() / (2048 * n) * 100 - 24.4) < 4.0


def test_serving_mix_protocol_small():
    """The serving-mix protocol: refcounts, copy-on-write and the decode result vs private contiguous K/V."""
    mix = workloads.shared_prefix_mix(B=20, group=4, prefix_len=64, ctx_lo=2, ctx_hi=140, Hq=4, Hkv=2, D=32)
    r = paging.serving_mix(mix)
    tables = [list(t[t >= 0]) for t in r["block_table"]]
    # every live page's refcount equals the number of tables naming it
    count = {}
    for t in tables:
        for p in t:
            count[p] = count.get(p, 0) + 1
    for p, c in count.items():
        assert r["pool"].refcount(p) == c
    # the page written by each sequence in this step is private to it
    for b in range(mix.B):
        p = int(mix.ctx[b]) - 1
        assert count[tables[b][p // 16]] == 1
    assert len(r["copies"]) > 0
    # decode result equals attention over each sequence's logical history (no pages involved)
    for b in range(mix.B):
        g = b // mix.group
        n = int(mix.ctx[b]) - 1
        pre = min(n, mix.prefix_len)
        sl = slice(int(mix.suffix_off[b]), int(mix.suffix_off[b + 1]))
        K = np.concatenate([mix.prefix_k[g, :pre], mix.suffix_k[sl], mix.k_new[b:b + 1]])
        V = np.concatenate([mix.prefix_v[g, :pre], mix.suffix_v[sl], mix.v_new[b:b + 1]])
        G = mix.Hq // mix.Hkv
        for h in range(mix.Hq):
            Q = np.zeros((n + 1, mix.D))
            Q[-1] = mix.q[b, h].astype(np.float64)
            ref = oracle.causal_attention(Q, K[:, h // G].astype(np.float64), V[:, h // G].astype(np.float64),
                                          mix.scale)[-1]
            assert np.max(np.abs(r["out"][b, h] - ref)) <= 1e-12
