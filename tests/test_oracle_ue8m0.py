"""Pins for the oracle's UE8M0 (power-of-two) scales, the groundwork of the
hardware block-scaled MMA path.

The transformers "Fine-grained FP8" guide ("UE8M0 scale format") stores FP8
weight scales as float8_e8m0fnu.  A code c is the value 2^(c - 127) (255 is
NaN).  The dynamic quantizers' scale is fl32(amax / 448), rounded up to the
next power of two and clamped to 2^-127.  The pins use exact rationals,
numpy's own frexp and IEEE float32 divide, and the brute-force E4M3
rounding; none of them calls the oracle's arithmetic.
"""
from fractions import Fraction

import numpy as np
import pytest

import synth
from test_oracle_codec import brute_nearest_e4m3


def test_decode_every_code(oracle):
    v = oracle.ue8m0_decode(np.arange(256, dtype=np.uint8))
    assert np.isnan(v[255])
    for c in range(255):
        assert Fraction(float(v[c])) == Fraction(2) ** (c - 127), c


def restated_code(amax32):
    """Smallest k with 2^k >= fl32(amax/448) (1 for amax 0), clamped to -127,
    plus the bias 127: by numpy's frexp, independent of the C code."""
    a = np.asarray(amax32, np.float32)
    with np.errstate(under="ignore"):
        s = np.where(a == 0, np.float32(1), (a / np.float32(448)).astype(np.float32)).astype(np.float32)
    m, e = np.frexp(s.astype(np.float64))
    k = np.where(m == 0.5, e - 1, e)
    return (np.maximum(k, -127) + 127).astype(np.uint8), s


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_code_of_every_amax(oracle, dtype):
    bits = np.arange(0, 0x8000, dtype=np.uint32).astype(np.uint16)   # every non-negative pattern
    a = synth.bits_to_f32(bits, dtype)
    a = a[np.isfinite(a)]
    got = np.array([oracle.ue8m0_of_amax(v) for v in a], np.uint8)
    want, s = restated_code(a)
    assert np.array_equal(got, want)
    p = np.ldexp(1.0, got.astype(np.int64) - 127)
    assert np.all(p >= s.astype(np.float64))                         # never below the FP32 scale
    assert np.all((p / 2 < s.astype(np.float64)) | (got == 0))       # the smallest such power of two
    assert oracle.ue8m0_of_amax(0.0) == 127


def test_quantizers_match_a_restatement(oracle):
    for dtype in ("f16", "bf16"):
        M, K = 9, 512
        x = synth.bits_to_f32(synth.random_bits((M, K), dtype, seed=25, tensor_id=7, std=5.0), dtype)
        x = x * (2.0 ** (np.arange(M) - 4)).astype(np.float32)[:, None]
        x[3, 128:256] = 0.0
        bits = synth.f32_to_bits(x.astype(np.float32), dtype)
        x = synth.bits_to_f32(bits, dtype)
        q, codes = oracle.quantize_token_group_ue8m0(bits, dtype)
        g = np.abs(x.reshape(M, K // 128, 128)).max(axis=2)              # [M, G]
        want_codes, _ = restated_code(g)
        assert np.array_equal(codes, want_codes.T)
        p = np.ldexp(np.float32(1), want_codes.astype(np.int32) - 127).astype(np.float32)   # [M, G]
        want_q = brute_nearest_e4m3((x.reshape(M, K // 128, 128) / p[:, :, None]).astype(np.float32))
        assert np.array_equal(q, want_q.reshape(M, K))
        assert codes[1, 3] == 127 and not np.any(q[3, 128:256] & 0x7F)

        w = synth.random_bits((200, 256), dtype, seed=26, tensor_id=8, std=0.02)
        qw, cw = oracle.quantize_weight_block_ue8m0(w, dtype)
        wf = synth.bits_to_f32(w, dtype)
        for bi in range(2):
            for bj in range(2):
                blk = wf[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
                c, _ = restated_code(np.abs(blk).max())
                assert cw[bi, bj] == c
                pw = np.float32(np.ldexp(1.0, int(c) - 127))
                assert np.array_equal(qw[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128],
                                      brute_nearest_e4m3((blk / pw).astype(np.float32)))


def test_power_of_two_amax_over_448_gives_the_fp32_quantizer(oracle):
    """Where fl32(amax/448) is already a power of two, rounding it up changes
    nothing: bytes and scale value equal the (pinned) FP32-scale quantizer's."""
    rng = np.random.default_rng(27)
    rows = []
    for k in range(-6, 7):
        v = (rng.standard_normal(128) * 0.1).astype(np.float32)
        v[5] = np.float32(448.0 * 2.0 ** k)                # amax / 448 = 2^k exactly
        rows.append(v)
    bits = synth.f32_to_bits(np.stack(rows), "f16")
    q1, c = oracle.quantize_token_group_ue8m0(bits, "f16")
    q2, s = oracle.quantize_token_group(bits, "f16")
    assert np.array_equal(q1, q2)
    assert np.array_equal(oracle.ue8m0_decode(c), s)
