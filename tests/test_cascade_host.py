"""Host logic of the cascade decode: forming the groups and their shared block counts (no GPU).

A group is a run of consecutive sequences whose block-table rows begin with the same block (at most 8);
its shared count is the number of leading entries all members have in common, capped so that every member
keeps its newest token outside the shared blocks. Checked against a brute-force restatement on random
tables with planted sharing, and on the serving mix's tables from the oracle's own pool protocol.
"""
import numpy as np
import pytest

import workloads
from oracle import paging as opaging


def groups_brute(table, ctx, max_group=8, bs=16):
    B = len(ctx)
    gs, sh = [0], np.zeros(B, dtype=np.int32)
    b = 0
    while b < B:
        e = b + 1
        while e < B and e - b < max_group and table[e][0] == table[b][0]:
            e += 1
        s = 0
        if e - b > 1:
            cap = min((int(ctx[i]) - 1) // bs for i in range(b, e))
            while s < cap and all(table[i][s] == table[b][s] for i in range(b, e)):
                s += 1
        sh[b:e] = s
        gs.append(e)
        b = e
    return np.array(gs, dtype=np.int32), sh


def check_invariants(table, ctx, gs, sh, max_group=8, bs=16):
    assert gs[0] == 0 and gs[-1] == len(ctx) and np.all(np.diff(gs) >= 1) and np.all(np.diff(gs) <= max_group)
    for g in range(len(gs) - 1):
        m = range(gs[g], gs[g + 1])
        s = int(sh[gs[g]])
        assert all(int(sh[b]) == s for b in m)
        assert all(bs * s <= int(ctx[b]) - 1 for b in m)
        for j in range(s):
            assert len({int(table[b][j]) for b in m}) == 1


def planted(seed, B=60, mb=12):
    rng = np.random.default_rng(seed)
    table = rng.integers(0, 10_000, size=(B, mb)).astype(np.int32)
    ctx = rng.integers(1, mb * 16 + 1, size=B).astype(np.int32)
    b = 0
    while b < B:  # runs of 1..11 sequences copy a leading stretch of the first one's row
        n = int(rng.integers(1, 12))
        k = int(rng.integers(0, mb + 1))
        table[b:b + n, :k] = table[b, :k]
        b += n
    return table, ctx


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("max_group", [1, 3, 8])
def test_groups_match_brute_force(seed, max_group):
    import paged_kv_cache_27_gb300 as kvc
    table, ctx = planted(seed)
    gs, sh, mx = kvc.kv_cascade_groups(table, ctx, max_group=max_group)
    rgs, rsh = groups_brute(table, ctx, max_group)
    assert np.array_equal(gs, rgs) and np.array_equal(sh, rsh) and mx == int(rsh.max())
    check_invariants(table, ctx, gs, sh, max_group)


def test_groups_edge_cases():
    import paged_kv_cache_27_gb300 as kvc
    # nine sequences with identical rows: 8 + 1, the ninth alone shares nothing
    table = np.tile(np.arange(10, dtype=np.int32), (9, 1))
    ctx = np.full(9, 160, dtype=np.int32)
    gs, sh, mx = kvc.kv_cascade_groups(table, ctx)
    assert list(gs) == [0, 8, 9] and list(sh) == [9] * 8 + [0] and mx == 9
    # the cap: a member whose context ends inside the common stretch keeps its newest token private
    ctx = np.array([160, 33, 160], dtype=np.int32)
    gs, sh, _ = kvc.kv_cascade_groups(table[:3], ctx)
    assert list(sh) == [2, 2, 2]  # (33 - 1) // 16
    ctx = np.array([160, 32, 160], dtype=np.int32)
    _, sh, _ = kvc.kv_cascade_groups(table[:3], ctx)
    assert list(sh) == [1, 1, 1]
    # one sequence, and no sharing at all
    gs, sh, mx = kvc.kv_cascade_groups(table[:1], ctx[:1])
    assert list(gs) == [0, 1] and list(sh) == [0] and mx == 0
    gs, sh, mx = kvc.kv_cascade_groups(np.arange(12, dtype=np.int32).reshape(4, 3), np.full(4, 40, np.int32))
    assert list(gs) == [0, 1, 2, 3, 4] and mx == 0


def test_groups_of_generated_structures():
    import paged_kv_cache_27_gb300 as kvc
    wl = workloads.cascade_decode(5, [3, 1, 8, 2], [4, 2, 7, 0], [1, 16, 17, 5, 300, 1, 2, 3, 4, 5, 6, 7, 40, 41])
    gs, sh, mx = kvc.kv_cascade_groups(wl.block_table, wl.ctx)
    check_invariants(wl.block_table, wl.ctx, gs, sh)
    # the planted sharing is found exactly (private tails use fresh blocks); a lone sequence and the last
    # group, which shares nothing, become groups of one
    assert list(gs) == [0, 3, 4, 12, 13, 14]
    assert list(sh) == [4, 4, 4, 0] + [7] * 8 + [0, 0] and mx == 7


def test_groups_on_serving_mix_tables():
    """The shared-prefix mix after its step (the oracle's pool protocol): groups of at most 8 that share the prefix
    blocks the copy-on-write left shared."""
    import paged_kv_cache_27_gb300 as kvc
    mix = workloads.shared_prefix_mix()
    ref = opaging.serving_mix(mix)
    table = ref["block_table"]
    gs, sh, mx = kvc.kv_cascade_groups(table, mix.ctx)
    rgs, rsh = groups_brute(table, mix.ctx)
    assert np.array_equal(gs, rgs) and np.array_equal(sh, rsh)
    check_invariants(table, mix.ctx, gs, sh)
    assert mx == mix.prefix_len // mix.bs  # some group keeps the whole 512-token prefix shared
    assert np.count_nonzero(sh) >= mix.B // 2
