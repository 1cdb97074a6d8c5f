"""GPU parity of the E5M2 codec (5 exponent + 2 mantissa bits; "What is FP8
inference on H100 (Transformer Engine)?" s2 and "FP8 mixed-precision
inference ... H100 Transformer Engine" s2) against the oracle's bit-level
encoder and decoder: every FP16 and every BF16 input pattern (zeros of both
signs, subnormals, the saturation range, infinities and NaNs included) and
all 256 codes, bytes and values exact; ragged lengths; outputs inside canary
bands and pre-filled with two different poison bytes, so an unwritten
element or a store outside the output cannot pass."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TD, Guarded, no_device_error  # noqa: F401

pytestmark = pytest.mark.gpu

F = pytest.importorskip("fp8_scaled_gemm_02_b300")


def all_patterns():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def encode_gpu(bits, dt, poison):
    x = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TD[dt]).cuda()
    g = Guarded(bits.shape, torch.uint8, poison)
    F.fp8_e5m2_encode(x, q=g.t)
    torch.cuda.synchronize()
    return g.check(allow_poison=True).cpu().numpy()


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_encode_every_16bit_pattern(dt):
    bits = all_patterns()
    want = oracle.e5m2_encode(oracle.to_float(bits, dt))
    for poison in (0x00, 0xFF):
        got = encode_gpu(bits, dt, poison)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, f"{bad.size} codes differ, e.g. input 0x{bits[bad[0]]:04x}: " \
                              f"0x{got[bad[0]]:02x} vs 0x{want[bad[0]]:02x}"


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_decode_every_code(dt):
    codes = np.tile(np.arange(256, dtype=np.uint16).astype(np.uint8), 3)   # 768 bytes: 48 vectors
    want = oracle.e5m2_decode(codes)
    q = torch.from_numpy(codes).cuda()
    for poison in (0x00, 0xFF):
        g = Guarded(codes.shape, TD[dt], poison)
        F.fp8_e5m2_decode(q, out_dtype=TD[dt], y=g.t)
        torch.cuda.synchronize()
        got = g.check(allow_poison=True).float().cpu().numpy().astype(np.float64)
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], want[~nan])
        # the sign of zero is kept
        assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


@pytest.mark.parametrize("n", [1, 7, 8, 9, 15, 16, 17, 4095, 4097, 65541])
def test_ragged_lengths_round_trip(n):
    """Encode then decode: the tails (n % 8 for the encoder, n % 16 for the
    decoder) go through the scalar path."""
    rng = np.random.default_rng(n)
    v = (rng.standard_normal(n) * 2.0 ** rng.integers(-18, 17, n)).astype(np.float32)
    with np.errstate(over="ignore"):   # values past the FP16 range become infinities: inputs too
        bits = v.astype(np.float16).view(np.uint16)
    want_q = oracle.e5m2_encode(oracle.to_float(bits, "f16"))
    for poison in (0x00, 0xFF):
        got_q = encode_gpu(bits, "f16", poison)
        assert np.array_equal(got_q, want_q)
        g = Guarded((n,), torch.float16, poison)
        F.fp8_e5m2_decode(torch.from_numpy(got_q).cuda(), out_dtype=torch.float16, y=g.t)
        torch.cuda.synchronize()
        got = g.check(allow_poison=True).float().cpu().numpy().astype(np.float64)
        assert np.array_equal(got, oracle.e5m2_decode(want_q))


def test_large_stream():
    """A tensor far larger than one wave of CTAs (the grid-stride loop with
    four vectors in flight per thread), against the oracle."""
    n = (1 << 24) + 24
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    got = encode_gpu(bits, "bf16", 0xFF)
    assert np.array_equal(got, oracle.e5m2_encode(oracle.to_float(bits, "bf16")))
