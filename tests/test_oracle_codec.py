"""Pins for the oracle's E4M3 decoder/encoder and 16-bit float decoders.

Each check compares the oracle against something other than itself: the
format facts the pages state (hand-derived golden table), exhaustive brute
force over every FP16/BF16 pattern, and PyTorch's float8_e4m3fn type as an
independent library implementation of the same format.
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden


def torch_grid():
    """Non-negative finite E4M3 values, index == code, decoded by PyTorch."""
    codes = torch.arange(0, 127, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def brute_nearest_e4m3(y32):
    """Independent E4M3 rounding: nearest grid value by search, ties to the
    even code, magnitudes above 448 clamp to 448, sign bit kept."""
    grid = torch_grid()
    y = np.asarray(y32, np.float32).astype(np.float64)
    sign = (np.signbit(y)).astype(np.uint8) << 7
    a = np.abs(y)
    idx = np.searchsorted(grid, a, side="left")
    hi = np.minimum(idx, 126)
    lo = np.maximum(idx - 1, 0)
    dlo = np.abs(a - grid[lo])
    dhi = np.abs(grid[hi] - a)
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= 448.0, 126, pick)
    return (pick.astype(np.uint8) | sign).astype(np.uint8)


# ------------------------------------------------------------------ decode
def test_decode_golden_table(oracle):
    for row in read_golden("e4m3_codes.txt"):
        code = int(row[0], 16)
        v = oracle.e4m3_decode(np.array([code], np.uint8))[0]
        if row[1] == "nan":
            assert math.isnan(v), hex(code)
        else:
            want = float(row[1])
            assert v == want, (hex(code), v, want)
            assert math.copysign(1.0, v) == math.copysign(1.0, want), hex(code)


def test_decode_all_codes_vs_torch(oracle):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_o, nan_r = np.isnan(ours), np.isnan(ref)
    assert np.array_equal(nan_o, nan_r)
    assert np.array_equal(ours[~nan_o], ref[~nan_r])
    assert np.array_equal(np.signbit(ours[~nan_o]), np.signbit(ref[~nan_r]))


def test_decode_structure(oracle):
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_decode(codes)
    finite = ~np.isnan(v)
    assert finite.sum() == 254
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    pos = v[1:0x7F]
    assert (pos > 0).all() and pos.size == 126
    assert np.all(np.diff(v[0:0x7F]) > 0), "codes 0x00..0x7E must increase"
    assert np.array_equal(v[0x80:0xFF], -v[0x00:0x7F])
    assert np.nanmax(v) == 448.0 and np.nanmin(v) == -448.0
    # every value is an integer number of 2^-9 units, matching the exact decoder
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_units(c) * 2.0 ** -9 == v[c]


# ------------------------------------------------------------------ encode
def test_roundtrip_all_finite_codes(oracle):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_encode_exhaustive_16bit(oracle, dtype):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    y = oracle.to_float(bits, dtype)
    keep = np.isfinite(y)
    y = y[keep]
    assert np.array_equal(oracle.e4m3_encode(y), brute_nearest_e4m3(y))


def test_encode_midpoints_and_edges(oracle):
    grid = torch_grid()
    mids = (grid[:-1] + grid[1:]) / 2.0          # exact in float32
    pts = []
    for m in mids.astype(np.float32):
        pts += [np.nextafter(m, np.float32(0)), m, np.nextafter(m, np.float32(1e9))]
    pts += [np.float32(x) for x in (448.0, 463.99997, 464.0, 464.00003, 480.0, 1e30, np.inf,
                                    2.0 ** -10, 2.0 ** -11, 1e-45, 0.0)]
    pts = np.array(pts, np.float32)
    pts = np.concatenate([pts, -pts])
    assert np.array_equal(oracle.e4m3_encode(pts), brute_nearest_e4m3(pts))
    enc = lambda x: int(oracle.e4m3_encode(np.array([x], np.float32))[0])
    assert enc(2.0 ** -10) == 0x00          # tie between 0 and 2^-9 -> even (0)
    assert enc(-(2.0 ** -10)) == 0x80       # sign kept on a zero result
    assert enc(1.5 * 2.0 ** -9) == 0x02     # tie between codes 1 and 2 -> even
    assert enc(248.0) == 0x78               # tie 240/256 across a binade edge -> 256
    assert enc(464.0) == 0x7E and enc(1e9) == 0x7E and enc(-np.inf) == 0xFE


def test_encode_random_fp32(oracle):
    rng = np.random.default_rng(12345)
    # random binary32 patterns over the exponent range that E4M3 rounding sees
    e = rng.integers(127 - 14, 127 + 10, size=1_000_000, dtype=np.uint32)
    m = rng.integers(0, 1 << 23, size=e.size, dtype=np.uint32)
    s = rng.integers(0, 2, size=e.size, dtype=np.uint32)
    y = ((s << 31) | (e << 23) | m).view(np.float32)
    assert np.array_equal(oracle.e4m3_encode(y), brute_nearest_e4m3(y))


def test_encode_vs_torch_cast(oracle):
    rng = np.random.default_rng(7)
    y = (rng.standard_normal(200_000) * rng.choice([1e-3, 1e-1, 1.0, 30.0, 200.0], 200_000)).astype(np.float32)
    y = y[np.abs(y) <= 448.0]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(y), ref)


# ------------------------------------------------------- 16-bit decoders
def test_half_decoder_exhaustive(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_float(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decoder_exhaustive(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_float(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
