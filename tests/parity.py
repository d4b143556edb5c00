"""Shared checks for the GPU parity tests: tolerance and bit-exact cache comparison."""
import numpy as np

ATOL = 2e-3  # max-abs attention error allowed against the fp64 oracle (fp16 inputs, fp32 accumulation)
F16_NAN_BITS = 0x7E00


def f16_ulp(x):
    """Spacing of fp16 numbers at |x| (normal range), for fp16-output tolerances."""
    a = np.maximum(np.abs(x), 2.0 ** -14)
    return 2.0 ** (np.floor(np.log2(a)) - 10)


def check_attention(got, ref, what=""):
    """got: torch tensor (fp32 or fp16 output), ref: fp64 numpy.  Returns the max-abs error."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    if str(got.dtype) == "torch.float16":
        bound = np.maximum(ATOL, f16_ulp(ref))
        bad = err > bound
        assert not bad.any(), f"{what}: {bad.sum()} outputs beyond max(2e-3, 1 ulp fp16); max err {err.max():.3e}"
    else:
        assert err.max() <= ATOL, f"{what}: max err {err.max():.3e} > {ATOL}"
    return float(err.max())


def owned_slots(block_table, ctx, bs=16):
    """Slot of every token position < ctx[b] of every sequence (test-side arithmetic)."""
    out = []
    for b in range(len(ctx)):
        pos = np.arange(int(ctx[b]))
        out.append(block_table[b][pos // bs].astype(np.int64) * bs + pos % bs)
    return np.unique(np.concatenate(out)) if out else np.zeros(0, np.int64)


def check_cache_bits(gpu_pool, ref_pool, slots, poison=True):
    """Bit-exact comparison of the owned slots; every other slot must still hold the poison pattern."""
    g = gpu_pool.detach().cpu().numpy().view(np.uint16)  # [NB][Hkv][bs][D]
    r = ref_pool.view(np.uint16)
    NB, Hkv, bs, D = g.shape
    gt = g.transpose(0, 2, 1, 3).reshape(NB * bs, Hkv, D)
    rt = r.transpose(0, 2, 1, 3).reshape(NB * bs, Hkv, D)
    assert np.array_equal(gt[slots], rt[slots]), "owned cache slots differ from the oracle's"
    if poison:
        mask = np.ones(NB * bs, bool)
        mask[slots] = False
        assert (gt[mask] == F16_NAN_BITS).all(), "a slot outside every context was written"
