"""The C ABI without a GPU: exported symbols, the native block pool and host slot logic (CPU).

The native pool and slot code are compared with the oracle's restatement of
the PagedAttention article's PagePool / PagedRequest (page ids bit-exact).
"""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_kv_cache_27_gb300 as kvc
from oracle.page_pool import PagedRequest, PagePool
from oracle import paging as opaging
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:kvc_status|const char\s*\*|int)\s+(\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(kvc.lib_path())
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the binding wraps every one of them under the same name
    for n in names:
        if n != "kvc_last_error_string":
            assert hasattr(kvc, n), n


def test_pool_bytes_pins():
    # 24 layers x 2 KV heads x d 64 fp16 -> 12,288 B per token; 4096 blocks of 16 -> 768 MiB (K + V)
    cfg = kvc.KvcConfig(num_layers=24, num_blocks=4096, num_kv_heads=2, head_dim=64)
    assert 2 * kvc.kv_cache_pool_bytes(cfg) == 805306368
    assert 2 * kvc.kv_cache_pool_bytes(cfg) // (4096 * 16) == 12288
    with pytest.raises(kvc.KvcError) as e:
        kvc.kv_cache_pool_bytes(kvc.KvcConfig(1, 4, 2, 64, block_size=32))
    assert e.value.name == "KVC_ERR_UNSUPPORTED"


def host_cache(nb, layers=1):
    return kvc.kv_cache_create(kvc.KvcConfig(num_layers=layers, num_blocks=nb, num_kv_heads=2, head_dim=64))


def test_native_pool_matches_restated_pagepool_section2():
    h = host_cache(512)
    ref = PagePool(512)
    try:
        tables, rtabs = [], []
        for n in (320, 48, 160, 96, 272):
            req = PagedRequest(0, ref)
            tab = []
            for t in range(n):
                if t % 16 == 0:
                    tab.append(kvc.kv_block_alloc(h))
                req.generate_token()
            tables.append(tab)
            rtabs.append(req)
        assert [len(t) for t in tables] == [20, 3, 10, 6, 17]
        assert tables == [r.block_table for r in rtabs]
        assert round(kvc.kv_cache_utilisation(h), 1) == 10.9
        for b in tables[1]:
            kvc.kv_block_release(h, b)
        rtabs[1].free()
        assert kvc.kv_block_num_free(h) == len(ref.free) == 512 - 53
        # FIFO: the next allocations walk the untouched tail, then the released pages
        got = [kvc.kv_block_alloc(h) for _ in range(512 - 56 + 3)]
        want = [ref.allocate() for _ in range(512 - 56 + 3)]
        assert got == want and got[-3:] == [20, 21, 22]
        with pytest.raises(kvc.KvcError) as e:
            kvc.kv_block_alloc(h)
        assert e.value.name == "KVC_ERR_OOM"
    finally:
        kvc.kv_cache_destroy(h)


def test_native_pool_section3_sharing_and_errors():
    h = host_cache(512)
    try:
        shared = [kvc.kv_block_alloc(h) for _ in range(13)]
        assert shared == list(range(13))
        for _ in range(10):
            for b in shared:
                kvc.kv_block_share(h, b)
        assert all(kvc.kv_block_refcount(h, b) == 11 for b in shared)
        with pytest.raises(kvc.KvcError):
            kvc.kv_block_share(h, 100)  # not live
        with pytest.raises(kvc.KvcError):
            kvc.kv_block_release(h, 100)
        with pytest.raises(kvc.KvcError):
            kvc.kv_block_refcount(h, 512)
        # a host-only cache refuses device work
        with pytest.raises(kvc.KvcError) as e:
            kvc.kv_block_cow(h, 12)
        assert e.value.name == "KVC_ERR_INVALID"
        for _ in range(11):
            kvc.kv_block_release(h, 0)
        assert kvc.kv_block_refcount(h, 0) == 0
        with pytest.raises(kvc.KvcError):
            kvc.kv_block_release(h, 0)  # double free
    finally:
        kvc.kv_cache_destroy(h)


def test_slot_mapping_matches_oracle():
    wl = workloads.small_decode(5, B=6, Hq=2, Hkv=1, D=64, ctx=[1, 15, 16, 17, 100, 257])
    B = wl.B
    got = kvc.kv_slot_mapping(wl.block_table, np.zeros(B, np.int32), wl.ctx - 1)
    assert np.array_equal(got, opaging.history_slots(wl.block_table, wl.hist_off, 16))
    step = kvc.kv_slot_mapping(wl.block_table, wl.ctx - 1, np.ones(B, np.int32))
    assert np.array_equal(step, opaging.step_slots(wl.block_table, wl.ctx, 16))
    with pytest.raises(kvc.KvcError) as e:
        kvc.kv_slot_mapping(wl.block_table, wl.ctx, np.full(B, 17, np.int32))
    assert e.value.name == "KVC_ERR_CAPACITY"


def run_protocol_host(mix):
    """The serving-mix allocation protocol on the native pool, host side only (no data)."""
    h = kvc.kv_cache_create(kvc.KvcConfig(num_layers=1, num_blocks=mix.NB, num_kv_heads=mix.Hkv, head_dim=mix.D))
    try:
        for _ in range(mix.NB):
            kvc.kv_block_alloc(h)
        for pid in mix.free_order:
            kvc.kv_block_release(h, int(pid))
        bs, B, G = mix.bs, mix.B, mix.group
        npre = -(-mix.prefix_len // bs)
        tables = [[] for _ in range(B)]
        for g in range(-(-B // G)):
            members = range(g * G, min(B, (g + 1) * G))
            pre = [kvc.kv_block_alloc(h) for _ in range(npre)]
            for b in members:
                need = -(-min(mix.prefix_len, int(mix.ctx[b]) - 1) // bs)
                for pid in pre[:need]:
                    kvc.kv_block_share(h, pid)
                tables[b] = pre[:need]
            for pid in pre:
                kvc.kv_block_release(h, pid)
            for b in members:
                while len(tables[b]) * bs < int(mix.ctx[b]) - 1:
                    tables[b].append(kvc.kv_block_alloc(h))
        mb = max(-(-int(c) // bs) for c in mix.ctx)
        table = np.full((B, mb), -1, np.int32)
        nblk = np.array([len(t) for t in tables], np.int32)
        for b in range(B):
            table[b, :nblk[b]] = tables[b]
        slots, copies = kvc.kv_step_prepare(h, table, nblk, mix.ctx - 1)
        rc = {int(p): kvc.kv_block_refcount(h, int(p)) for p in np.unique(table[table >= 0])}
        return table, slots, copies, rc
    finally:
        kvc.kv_cache_destroy(h)


@pytest.mark.parametrize("kw", [dict(B=20, group=4, prefix_len=64, ctx_lo=2, ctx_hi=140),
                                dict(B=37, group=8, prefix_len=48, ctx_lo=1, ctx_hi=90),
                                dict()])
def test_step_prepare_matches_oracle_protocol(kw):
    mix = workloads.shared_prefix_mix(**kw)
    table, slots, copies, rc = run_protocol_host(mix)
    ref = opaging.serving_mix(mix) if mix.B <= 40 else None
    if ref is None:
        # full serving mix: compare the allocation only (the oracle's attention is run by the GPU tests)
        ref = _oracle_tables_only(mix)
    assert np.array_equal(table, ref["block_table"])
    assert np.array_equal(slots, ref["slots"])
    assert [tuple(map(int, c)) for c in copies] == [tuple(c) for c in ref["copies"]]
    for p, c in rc.items():
        assert ref["pool"].refcount(p) == c


def _oracle_tables_only(mix):
    """The oracle protocol with zero-sized head data, so only the pages matter."""
    import dataclasses
    small = dataclasses.replace(
        mix, Hkv=1, D=1, prefix_k=np.zeros(mix.prefix_k.shape[:2] + (1, 1), np.float16),
        prefix_v=np.zeros(mix.prefix_k.shape[:2] + (1, 1), np.float16),
        suffix_k=np.zeros((mix.suffix_k.shape[0], 1, 1), np.float16),
        suffix_v=np.zeros((mix.suffix_k.shape[0], 1, 1), np.float16),
        q=np.zeros((mix.B, 1, 1), np.float16), k_new=np.zeros((mix.B, 1, 1), np.float16),
        v_new=np.zeros((mix.B, 1, 1), np.float16), Hq=1)
    return opaging.serving_mix(small, nthreads=1)


def test_step_prepare_is_all_or_nothing_on_oom():
    h = host_cache(4)
    try:
        a = kvc.kv_block_alloc(h)
        kvc.kv_block_share(h, a)  # two sequences share block a, 3 blocks free
        b_, c_, d_ = (kvc.kv_block_alloc(h) for _ in range(3))
        table = np.array([[a, -1], [a, -1]], np.int32)
        nblk = np.array([1, 1], np.int32)
        before = table.copy()
        # sequence 0 writes position 3 of the shared block (needs a copy), sequence 1 needs a new block 1
        with pytest.raises(kvc.KvcError) as e:
            kvc.kv_step_prepare(h, table, nblk, [3, 16])
        assert e.value.name == "KVC_ERR_OOM"
        assert np.array_equal(table, before) and list(nblk) == [1, 1]
        kvc.kv_block_release(h, d_)
        kvc.kv_block_release(h, c_)
        slots, copies = kvc.kv_step_prepare(h, table, nblk, [3, 16])
        assert copies.tolist() == [[a, d_]]
        assert table.tolist() == [[d_, -1], [a, c_]] and nblk.tolist() == [1, 2]
        assert slots.tolist() == [d_ * 16 + 3, c_ * 16 + 0]
    finally:
        kvc.kv_cache_destroy(h)


def test_checked_mode_and_version():
    assert kvc.kvc_version() >= 100
    kvc.kvc_set_checked_mode(True)
    kvc.kvc_set_checked_mode(False)


def test_cache_layer_pointers_and_errors():
    """kv_cache_layer is pointer arithmetic over the caller's pools (never dereferenced here): layer l of a
    [L][NB][Hkv][bs][D] fp16 pool starts l * NB * Hkv * bs * D * 2 bytes in."""
    import ctypes
    import paged_kv_cache_27_gb300 as kvc
    L, NB, Hkv, D = 3, 10, 2, 64
    cfg = kvc._Config(L, NB, 16, Hkv, D, kvc.KVC_F16)
    kbase, vbase = 1 << 40, 1 << 41  # aligned addresses that are never touched
    h = ctypes.c_void_p()
    assert kvc._lib.kv_cache_create(ctypes.byref(cfg), ctypes.c_void_p(kbase), ctypes.c_void_p(vbase),
                                    ctypes.byref(h)) == 0
    try:
        per = NB * Hkv * 16 * D * 2
        for layer in range(L):
            assert kvc.kv_cache_layer(h.value, layer) == (kbase + per * layer, vbase + per * layer)
        for bad in (-1, L):
            with pytest.raises(kvc.KvcError) as e:
                kvc.kv_cache_layer(h.value, bad)
            assert "KVC_ERR_INVALID" in str(e.value)
    finally:
        kvc.kv_cache_destroy(h.value)
    # misaligned pools are refused; a host-only cache has no layers
    assert kvc._lib.kv_cache_create(ctypes.byref(cfg), ctypes.c_void_p(kbase + 8), ctypes.c_void_p(vbase),
                                    ctypes.byref(h)) != 0
    hh = kvc.kv_cache_create(kvc.KvcConfig(num_layers=L, num_blocks=NB, num_kv_heads=Hkv, head_dim=D))
    try:
        with pytest.raises(kvc.KvcError):
            kvc.kv_cache_layer(hh, 0)
    finally:
        kvc.kv_cache_destroy(hh)


def test_trace_read_needs_a_trace_build():
    import paged_kv_cache_27_gb300 as kvc
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_trace_read(16)
    assert "KVC_ERR_UNSUPPORTED" in str(e.value)


def test_copy_async_argument_errors():
    """kvc_copy_async refuses bad arguments synchronously, before any device work (no GPU needed)."""
    import paged_kv_cache_27_gb300 as kvc
    f = kvc._lib.kvc_copy_async
    buf = np.zeros(256, dtype=np.uint8)
    base = (buf.ctypes.data + 15) & ~15  # a 16-byte aligned pageable host address
    assert f(base, base + 64, 0, 0, None) == 0  # nothing to copy
    assert f(base, base + 64, 16, 2, None) == 1  # unknown flag
    assert f(None, base, 16, 0, None) == 1
    assert f(base, None, 16, 0, None) == 1
    assert f(base, base + 64, 24, 0, None) == 1  # not a multiple of 16
    assert f(base + 8, base + 64, 16, 0, None) == 1  # misaligned
    assert f(base, base + 16, 32, 0, None) == 1  # overlapping
    assert f(base, base + 64, 32, kvc.KVC_COPY_AHEAD, None) == 1  # pageable host memory
    assert "pinned" in kvc._lib.kvc_last_error_string().decode()
