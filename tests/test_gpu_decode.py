"""GPU parity of kv_append + paged_decode_attention against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import paging as opaging
import workloads
from parity import check_attention, check_cache_bits, owned_slots

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    import paged_kv_cache_27_gb300 as m
    return m


def run_session(kvc, wl, out_dtype=torch.float32, bps=0, fused=False, graph=False, overlap=False):
    """One decode step: eager, or replayed from a CUDA graph (with launch overlap) as the benchmark runs it."""
    from paged_kv_cache_27_gb300.harness import DecodeSession
    s = DecodeSession(wl, out_dtype=out_dtype, blocks_per_split=bps).fill()
    kvc.kvc_set_launch_overlap(overlap)
    try:
        if graph:
            g = s.capture(fused=fused)
            s.out.fill_(float("nan"))
            g.replay()
            g.replay()
        else:
            s.step(fused=fused)
        torch.cuda.synchronize()
    finally:
        kvc.kvc_set_launch_overlap(False)
    return s


def check_workload(kvc, wl, out_dtype=torch.float32, bps=0, layers=None, cache_bits=True, fused=False, graph=False,
                   overlap=False):
    s = run_session(kvc, wl, out_dtype, bps, fused, graph, overlap)
    assert kvc.kvc_device_error_flags(clear=True) == 0
    errs = []
    for layer in (range(wl.L) if layers is None else layers):
        ref, kc, vc = opaging.decode_step(wl, layer)
        errs.append(check_attention(s.out[layer], ref, f"{wl.name} layer {layer}"))
        if cache_bits:
            slots = owned_slots(wl.block_table, wl.ctx, wl.bs)
            check_cache_bits(s.k_pool[layer], kc, slots)
            check_cache_bits(s.v_pool[layer], vc, slots)
    s.close()
    return max(errs)


def test_single_sequence_256(kvc):
    wl = workloads.single_sequence_256()
    for dt in (torch.float32, torch.float16):
        check_workload(kvc, wl, dt)
    # the cached row equals the last row of the full 256 x 256 causal recompute
    s = run_session(kvc, wl)
    K = np.concatenate([wl.k_hist[0], wl.k_new[0]])[:, 0].astype(np.float64)
    V = np.concatenate([wl.v_hist[0], wl.v_new[0]])[:, 0].astype(np.float64)
    Q = np.zeros_like(K)
    Q[-1] = wl.q[0, 0, 0].astype(np.float64)
    full = oracle.causal_attention(Q, K, V, wl.scale)
    check_attention(s.out[0, 0], full[-1:], "single sequence vs 256x256 causal")


@pytest.mark.parametrize("B,Hq,Hkv,D,ctx", [
    (1, 1, 1, 64, [1]),
    (3, 4, 4, 64, [1, 2, 3]),
    (5, 14, 2, 64, [16, 17, 31, 32, 33]),
    (4, 8, 1, 64, [255, 256, 257, 1000]),
    (6, 7, 7, 128, [5, 64, 65, 200, 511, 700]),
    (2, 16, 2, 128, [300, 1500]),
    (9, 14, 2, 64, [4096, 1, 77, 2048, 3000, 16, 15, 999, 1024]),
])
@pytest.mark.parametrize("fused", [False, True])
def test_small_sweep(kvc, B, Hq, Hkv, D, ctx, fused):
    wl = workloads.small_decode(B * 100 + D, B=B, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx, L=2)
    for dt in (torch.float32, torch.float16):
        check_workload(kvc, wl, dt, fused=fused)


@pytest.mark.parametrize("B,Hq,Hkv,D,ctx", [
    (3, 64, 4, 64, [1, 500, 3000]),       # 16 query heads per KV head: two chunks of 8
    (2, 12, 1, 128, [17, 2049]),          # 12: a full chunk and a chunk of 4
    (2, 32, 1, 64, [300, 40000]),         # 32: four chunks, a context over several clusters
    (1, 64, 1, 64, [1024]),               # 64: the widest group the library takes
])
@pytest.mark.parametrize("fused", [False, True])
def test_wide_query_groups(kvc, B, Hq, Hkv, D, ctx, fused):
    """More than 8 query heads per KV head (the grouped-query paragraph of the neuralialabs.com page and the
    xformers article's part 5 fix no bound): the heads go in chunks of 8 to consecutive CTAs."""
    wl = workloads.small_decode(B * 1000 + Hq, B=B, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx, L=1)
    for dt in (torch.float32, torch.float16):
        check_workload(kvc, wl, dt, fused=fused)


def test_group_size_limit(kvc):
    with pytest.raises(kvc.KvcError) as e:
        kvc.paged_decode_plan(1, 65, 1, 64, 16)
    assert e.value.name == "KVC_ERR_UNSUPPORTED"


@pytest.mark.parametrize("bps", [1, 2, 3, 4, 7, 8, 64, 128])
@pytest.mark.parametrize("fused", [False, True])
def test_forced_split_sizes(kvc, bps, fused):
    """1 block per split (129 splits: combine kernel) up to 128 (a single split): both merge paths."""
    wl = workloads.small_decode(77, B=4, Hq=14, Hkv=2, D=64, ctx=[1, 300, 1025, 2048], peak_frac=0.01)
    check_workload(kvc, wl, torch.float32, bps=bps, fused=fused)


@pytest.mark.parametrize("bps", [0, 256, 512, 1024, 2048, 4096])
def test_long_context_cluster_slices(kvc, bps):
    """Clusters covering up to 4096 blocks each (the largest table slice a cluster stages): one part per
    sequence, or a few parts merged by the combine kernel."""
    wl = workloads.small_decode(91, B=3, Hq=14, Hkv=2, D=64, ctx=[70000, 5000, 1], peak_frac=0.01)
    check_workload(kvc, wl, torch.float32, bps=bps, fused=True)


def test_model_step_full_as_benchmarked(kvc):
    """24 layers x 32 sequences x context 2048, 14 q / 2 KV heads, in the benchmark's launch configuration
    (fused append + decode, CUDA graph, launch overlap): every layer and the whole cache against the oracle."""
    wl = workloads.model_decode_step()
    err = check_workload(kvc, wl, torch.float16, layers=range(wl.L), cache_bits=True, fused=True, graph=True,
                         overlap=True)
    assert err < 2e-3


def test_model_step_fp32_out_unfused_sampled_layers(kvc):
    wl = workloads.model_decode_step()
    check_workload(kvc, wl, torch.float32, layers=[0, 11, 23], cache_bits=False)


@pytest.mark.parametrize("B", [1, 4, 16])
@pytest.mark.parametrize("ctx", [4096, 16384, 65536, 131072])
def test_long_context(kvc, B, ctx):
    wl = workloads.long_context(B, ctx)
    check_workload(kvc, wl, torch.float32, cache_bits=(B * ctx <= 4 * 65536), fused=True, graph=True, overlap=True)


def test_workspace_reuse_across_context_lengths(kvc):
    """Growing contexts change the split count; one workspace serves every step (counters stay at zero)."""
    from paged_kv_cache_27_gb300.harness import DecodeSession
    base = workloads.small_decode(21, B=6, Hq=14, Hkv=2, D=64, ctx=[3000, 2000, 1000, 500, 4000, 64])
    s = DecodeSession(base).fill()
    ws = s.workspace
    for ctx_scale in (0.25, 0.5, 1.0, 0.1, 1.0):
        wl = workloads.small_decode(21, B=6, Hq=14, Hkv=2, D=64,
                                    ctx=[max(1, int(c * ctx_scale)) for c in base.ctx])
        s2 = DecodeSession(wl).fill()
        s2.workspace = ws  # shared workspace, same B and Hkv
        s2.step(fused=True)
        torch.cuda.synchronize()
        ref, _, _ = opaging.decode_step(wl, 0)
        check_attention(s2.out[0], ref, f"ctx scale {ctx_scale}")
        s2.close()
    s.close()


def _permuted(wl, perm):
    """The same sequences in the order perm (history repacked, physical blocks unchanged)."""
    import dataclasses
    off = wl.hist_off
    ctx = wl.ctx[perm]
    hist_off = np.zeros(wl.B + 1, dtype=np.int64)
    hist_off[1:] = np.cumsum(ctx.astype(np.int64) - 1)
    k = np.concatenate([wl.k_hist[:, off[i]:off[i + 1]] for i in perm], axis=1)
    v = np.concatenate([wl.v_hist[:, off[i]:off[i + 1]] for i in perm], axis=1)
    return dataclasses.replace(wl, ctx=ctx, block_table=wl.block_table[perm], hist_off=hist_off, k_hist=k, v_hist=v,
                               q=wl.q[:, perm], k_new=wl.k_new[:, perm], v_new=wl.v_new[:, perm])


@pytest.mark.parametrize("fused", [False, True])
def test_several_waves_longest_first(kvc, fused):
    """400 sequences x 2 KV heads: more CTAs than the GPU holds at once, so they take the sequences longest
    first.  Ragged lengths with ties, single tokens and the longest; every output and cache row against the
    oracle, and the same sequences in another order give the reordered outputs bit for bit."""
    rng = np.random.default_rng(5)
    ctx = rng.integers(1, 700, size=400)
    ctx[::9] = 1
    ctx[::7] = 350
    ctx[5] = ctx[123] = 700
    wl = workloads.small_decode(4040, B=400, Hq=14, Hkv=2, D=64, ctx=ctx.tolist())
    check_workload(kvc, wl, torch.float16, fused=fused, graph=True, overlap=True)
    s1 = run_session(kvc, wl, torch.float16, fused=fused)
    perm = np.random.default_rng(6).permutation(wl.B)
    s2 = run_session(kvc, _permuted(wl, perm), torch.float16, fused=fused)
    assert kvc.kvc_device_error_flags(clear=True) == 0
    assert torch.equal(s2.out[0], s1.out[0][torch.from_numpy(perm).to(s1.out.device)])
    s1.close()
    s2.close()


def test_several_waves_wide_groups(kvc):
    """160 sequences, 16 query heads per KV head (two head chunks per KV head): 640 CTAs, dispatched longest
    context first, against the oracle."""
    ctx = np.random.default_rng(8).integers(1, 500, size=160)
    ctx[::5] = 250
    wl = workloads.small_decode(4041, B=160, Hq=32, Hkv=2, D=64, ctx=ctx.tolist())
    check_workload(kvc, wl, torch.float32, fused=True)


def _random_case(i):
    """Seeded random decode shape: batch, heads (GQA groups 1..16), head dim, ragged contexts with ties and
    single tokens, an explicit split size or the planner's, the fused or separate append, eager or graph."""
    rng = np.random.default_rng(700 + i)
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 7, 8, 12, 16] if D == 64 else [1, 2, 4, 8]))
    B = int(rng.choice([1, 3, 17, 64, 180]))
    hi = int(rng.choice([40, 600, 3000]))
    ctx = rng.integers(1, hi + 1, size=B)
    ctx[rng.random(B) < 0.1] = 1
    ctx[rng.random(B) < 0.2] = hi
    bps = int(rng.choice([0, 0, 0, 1, 7, 64]))
    return dict(B=B, Hq=G * Hkv, Hkv=Hkv, D=D, ctx=ctx.tolist(), bps=bps, fused=bool(rng.random() < 0.5),
                graph=bool(rng.random() < 0.5))


@pytest.mark.parametrize("i", range(16))
def test_random_shapes_against_oracle(kvc, i):
    c = _random_case(i)
    wl = workloads.small_decode(5000 + i, B=c["B"], Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"], ctx=c["ctx"])
    check_workload(kvc, wl, torch.float32, bps=c["bps"], fused=c["fused"], graph=c["graph"], overlap=c["graph"])


def test_results_invariant_to_physical_placement(kvc):
    """Same logical data under two block permutations gives bit-identical outputs."""
    from paged_kv_cache_27_gb300.harness import DecodeSession
    wl = workloads.small_decode(9, B=3, Hq=14, Hkv=2, D=64, ctx=[100, 1000, 2000])
    outs = []
    for seed in (1, 2):
        perm = np.random.default_rng(seed).permutation(wl.NB).astype(np.int32)
        wl2 = type(wl)(**{**wl.__dict__, "block_table": np.where(wl.block_table >= 0, perm[wl.block_table], -1)})
        s = DecodeSession(wl2).fill()
        s.step()
        torch.cuda.synchronize()
        outs.append(s.out.clone())
        s.close()
    assert torch.equal(outs[0], outs[1])
