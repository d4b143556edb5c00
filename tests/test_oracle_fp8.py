"""Pins for the oracle's fp8 e4m3 cache extension (CPU only).

The e4m3 codec is tied to torch's float8_e4m3fn (a library routine): every code's value exactly, and the
nearest-even rounding of binary32 values inside the format's range (torch does not saturate past 448, so the
saturation rule is checked by its definition). The quantizer is tied to the same cast and to its closed-form
properties; the fp8 decode to the fp16 decode, which is pinned elsewhere, on caches whose dequantized values
are exactly fp16 values.
"""
import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(11)


def torch_e4m3_values(codes):
    t = torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_e4m3_codes(x32):
    return torch.from_numpy(np.asarray(x32, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_every_code_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = oracle.e4m3_to_float64(codes), torch_e4m3_values(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_encode_roundtrip_and_ties_vs_torch():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_to_float64(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_from_float32(vals), codes)
    # midpoints between consecutive positive values: ties go to the even fraction
    pos = np.sort(np.unique(oracle.e4m3_to_float64(np.arange(0, 0x7F, dtype=np.uint8))))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (pos[:-1] + pos[1:]) / 2)  # exact in binary32
    for x in (mids, -mids):
        ours = oracle.e4m3_from_float32(x)
        assert np.array_equal(ours, torch_e4m3_codes(x))
        assert np.all(ours & 1 == 0)  # the even neighbour


def test_encode_random_values_vs_torch():
    x = np.concatenate([
        RNG.uniform(-448, 448, 100_000),
        np.sign(RNG.standard_normal(100_000)) * np.exp2(RNG.uniform(-12, np.log2(448), 100_000)),
    ]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_from_float32(x), torch_e4m3_codes(x))


def test_encode_saturates_at_448():
    x = np.array([448.0, 455.0, 464.0, 480.0, 1e30, -500.0], np.float32)
    assert list(oracle.e4m3_from_float32(x)) == [0x7E] * 5 + [0xFE]
    assert oracle.e4m3_from_float32(np.array([np.nan], np.float32))[0] == 0x7F


def test_quantize_rows():
    x = (RNG.standard_normal((200, 64)) * np.exp2(RNG.uniform(-6, 6, (200, 1)))).astype(np.float16)
    x[3] = 0
    codes, scales = oracle.quantize_fp8(x)
    x32 = x.astype(np.float32)
    amax = np.abs(x32).max(axis=1)
    want = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    assert np.array_equal(scales, want)
    assert np.array_equal(codes, torch_e4m3_codes(x32 / scales[:, None]))
    assert np.all(codes[3] == 0) and scales[3] == 1.0
    # the largest magnitude of every non-zero row becomes +-448
    rows = np.arange(200) != 3
    top = codes[np.arange(200), np.abs(x32).argmax(axis=1)][rows]
    assert np.all((top & 0x7F) == 0x7E)
    # dequantized error: at most half a step of the row's e4m3 grid
    deq = oracle.e4m3_to_float64(codes) * scales[:, None]
    step = np.maximum(np.exp2(np.floor(np.log2(np.maximum(np.abs(x32) / scales[:, None], 2.0 ** -6))) - 3),
                      2.0 ** -9) * scales[:, None]
    assert np.all(np.abs(deq - x32) <= step / 2 + 1e-12)


@pytest.mark.parametrize("Hq,Hkv,D", [(14, 2, 64), (8, 8, 128)])
def test_decode_fp8_equals_fp16_decode_on_exact_values(Hq, Hkv, D):
    """Power-of-two scales keep every code value x scale an fp16 value: the two decodes see the same cache."""
    bs, NB, B = 16, 20, 3
    kq = RNG.integers(0, 256, (NB, Hkv, bs, D)).astype(np.uint8)
    vq = RNG.integers(0, 256, (NB, Hkv, bs, D)).astype(np.uint8)
    for c in (kq, vq):
        c[(c & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    ks = np.exp2(RNG.integers(-4, 3, (NB, Hkv, bs))).astype(np.float32)
    vs = np.exp2(RNG.integers(-4, 3, (NB, Hkv, bs))).astype(np.float32)
    kf = (oracle.e4m3_to_float64(kq) * ks[..., None]).astype(np.float16)
    vf = (oracle.e4m3_to_float64(vq) * vs[..., None]).astype(np.float16)
    assert np.array_equal(kf.astype(np.float64), oracle.e4m3_to_float64(kq) * ks[..., None])
    table = RNG.permutation(NB)[:18].astype(np.int32).reshape(B, 6)
    ctx = np.array([1, 50, 96], np.int32)
    q = (RNG.standard_normal((B, Hq, D)) * 0.05).astype(np.float16)
    a = oracle.decode_fp8(q, kq, vq, ks, vs, table, ctx, 1 / np.sqrt(D))
    b = oracle.decode(q, kf, vf, table, ctx, 1 / np.sqrt(D))
    assert np.array_equal(a, b)
