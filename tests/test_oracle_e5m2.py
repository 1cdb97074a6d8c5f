"""Pins for the oracle's E5M2 codec (5 exponent + 2 mantissa bits, bias 15).

The pages give only the bit split: "What is FP8 inference on H100" s2 and
the zyxy.net FP8 article s2.  References, all independent of the oracle's
integer arithmetic:
  * PyTorch's float8_e5m2 for decoding, and for encoding wherever PyTorch
    does not overflow to infinity (|y| < 61440; the oracle saturates, as
    the E4M3 path does);
  * E5M2 is the top byte of an FP16 pattern, so every FP16 value's code is
    the round-to-nearest-even of its pattern shifted right by 8 bits;
  * a nearest-value search over the finite grid.
"""
import numpy as np
import torch


def torch_decode():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).to(torch.float64).numpy()


def test_decode_every_code(oracle):
    got = oracle.e5m2_decode(np.arange(256, dtype=np.uint8))
    want = torch_decode()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    assert got[0x7B] == 57344.0 and got[0x7C] == np.inf and got[0x01] == 2.0 ** -16 and got[0x04] == 2.0 ** -14


def fp16_pattern_rne(h):
    """Code of every FP16 value by rounding its 16-bit pattern to its top byte
    (ties to even), then saturating what reached infinity."""
    h = h.astype(np.uint32)
    sign = (h & 0x8000) >> 8
    mag = h & 0x7FFF
    base = mag >> 8
    r = mag & 0xFF
    up = (r > 0x80) | ((r == 0x80) & ((base & 1) == 1))
    code = base + up
    code = np.minimum(code, 0x7B)          # 0x7C and above: infinity after rounding -> 57344
    return (code | sign).astype(np.uint8)


def test_encode_every_fp16_value(oracle):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = h.view(np.float16).astype(np.float32)
    keep = ~np.isnan(x)
    got = oracle.e5m2_encode(x[keep])
    assert np.array_equal(got, fp16_pattern_rne(h[keep]))


def test_encode_random_fp32_vs_torch_and_search(oracle):
    rng = np.random.default_rng(31)
    y = (rng.standard_normal(1_000_000) * 2.0 ** rng.uniform(-20, 16, 1_000_000)).astype(np.float32)
    y = y[np.abs(y) < 61440]
    got = oracle.e5m2_encode(y)
    want = torch.from_numpy(y).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(got, want)
    # nearest finite grid value, ties to the even code, on a subsample
    grid = torch_decode()[:0x7C]                                   # codes 0..0x7B, increasing
    sub = y[:20000].astype(np.float64)
    a = np.abs(sub)
    idx = np.clip(np.searchsorted(grid, a), 1, 0x7B)
    lo, hi = idx - 1, idx
    dlo, dhi = a - grid[lo], grid[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= grid[0x7B], 0x7B, pick)
    assert np.array_equal(got[:20000], (pick | (np.signbit(sub) << 7)).astype(np.uint8))


def test_round_trip_and_saturation(oracle):
    codes = np.array([c for c in range(256) if (c & 0x7F) < 0x7C], np.uint8)   # finite codes
    vals = oracle.e5m2_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e5m2_encode(vals), codes)
    sat = oracle.e5m2_encode(np.float32([61440.0, 1e30, np.inf, -np.inf, -70000.0, 61439.996]))
    assert list(sat) == [0x7B, 0x7B, 0x7B, 0xFB, 0xFB, 0x7B]
