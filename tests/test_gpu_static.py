"""GPU parity of static and delayed per-tensor scaling against the CPU oracle.

fp8_quantize_per_tensor_static quantizes with a scale the caller holds
(calibrated, or from an amax history as in the Transformer Engine recipe
DelayedScaling(margin, interval) of "Technical assignment: implement FP8
inference on H100", stage 3); fp8_scale_from_amax_history derives the next
scale.  Bytes, amaxes and scales must be bit-exact.

The kernel takes three routes by scale: a power of two (exact reciprocal),
a general scale in [2^-90, 2^90] (double-word reciprocal, with vectors whose
quotients sit on or next to an E4M3 rounding boundary redone by the IEEE
divide) and anything else (IEEE divide throughout).  The cases cover each,
with quotients that saturate, underflow and hit E4M3 midpoints.  Threads
cast 32-byte units (two 16-byte vectors): sizes cover an odd vector count
(the last vector done apart) and 1-7 trailing elements."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import host, no_device_error, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu

F = pytest.importorskip("fp8_scaled_gemm_02_b300")


def dev_scale(s):
    return torch.tensor([np.float32(s)], dtype=torch.float32, device="cuda")


def check_static(bits, dtype, s, with_amax=True):
    x = to_dev(bits, dtype)
    amax = torch.full((4,), -1.0, dtype=torch.float32, device="cuda")[:1] if with_amax else None
    q = F.fp8_quantize_per_tensor_static(x, dev_scale(s), amax=amax)
    want = oracle.quantize_with_scale(bits, dtype, np.float32(s))
    bad = np.argwhere(host(q) != want)
    assert bad.size == 0, f"scale {s!r}: {len(bad)} bytes differ, first {bad[:5].tolist()}"
    if with_amax:
        assert host(amax)[0].view(np.uint32) == oracle.amax(bits, dtype).view(np.uint32)


def scale_kinds(bits, dtype):
    _, s_dyn = oracle.quantize_per_tensor(bits, dtype)
    s_dyn = np.float32(s_dyn)
    return {
        "dynamic": s_dyn,                                      # guarded route, |x/s| <= 448
        "saturating": np.float32(s_dyn / np.float32(37.3)),    # most large |x| clamp to 448
        "underflowing": np.float32(s_dyn * np.float32(3000)),  # many quotients below 2^-10
        "pow2": np.float32(2.0 ** np.round(np.log2(s_dyn))),   # exact reciprocal route
        "fixed": np.float32(0.0123),
        "tiny": np.float32(2.0 ** -100),                        # IEEE-divide route, all saturate
        "huge": np.float32(2.0 ** 95),                          # IEEE-divide route, all underflow
    }


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("numel", [1, 7, 9, 24, 1000, 8014, 65536 + 3, 1000003, (1 << 24) + 5])
def test_static_parity(dtype, numel):
    bits = synth.random_bits((numel,), dtype, seed=41, tensor_id=numel, std=3.0)
    for kind, s in scale_kinds(bits, dtype).items():
        check_static(bits, dtype, s)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_static_every_input_at_adversarial_scales(dtype):
    """Every finite 16-bit input, at random scales and at scales built so
    that some quotient x/s lands on an E4M3 rounding midpoint or one FP32
    step from it (the cases the guard exists for)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = synth.bits_to_f32(bits, dtype)
    bits = np.ascontiguousarray(bits[np.isfinite(x)])
    x = synth.bits_to_f32(bits, dtype)
    rng = np.random.default_rng(77)
    lo, hi = (-30, 20) if dtype == "f16" else (-100, 100)
    scales = list((2.0 ** rng.uniform(lo, hi, 40)).astype(np.float32))
    # E4M3 midpoints: (2m+1)/16 * 2^e in the normal range, odd multiples of 2^-10 below it
    mids = [np.float32((2 * m + 1) / 16.0 * 2.0 ** e) for e in range(-6, 9) for m in range(8, 16)]
    mids += [np.float32(k * 2.0 ** -10) for k in (1, 3, 5, 7, 9, 11, 13, 15)]
    nz = x[(np.abs(x) > 1e-30) & (np.abs(x) < 1e30)]
    for _ in range(60):
        v = np.float32(rng.choice(nz))
        m = np.float32(rng.choice(mids))
        s = np.float32(np.abs(v) / m)
        for t in (s, np.nextafter(s, np.float32(0)), np.nextafter(s, np.float32(np.inf))):
            if 2.0 ** -126 <= t < 2.0 ** 127:
                scales.append(np.float32(t))
    want = oracle.quantize_scales_grid(bits, dtype, np.float32(scales))
    xd = to_dev(bits, dtype)
    for j, s in enumerate(scales):
        q = F.fp8_quantize_per_tensor_static(xd, dev_scale(s))
        bad = np.argwhere(host(q) != want[j])
        assert bad.size == 0, f"scale {s!r}: {len(bad)} bytes differ, first {bad[:5].tolist()}"


def test_static_zeros_and_negative_zero():
    for dtype in ("f16", "bf16"):
        bits = np.full(77, 0x8000, np.uint16)
        bits[::3] = 0
        for s in (0.5, 0.0123, 2.0 ** -100):
            check_static(bits, dtype, s)


def test_static_without_amax_and_into_a_ring_slot():
    bits = synth.random_bits((4096 + 5,), "bf16", seed=42, tensor_id=1, std=2.0)
    check_static(bits, "bf16", 0.01, with_amax=False)
    ring = torch.full((8,), 7.0, dtype=torch.float32, device="cuda")
    F.fp8_quantize_per_tensor_static(to_dev(bits, "bf16"), dev_scale(0.01), amax=ring[3:4])
    r = host(ring)
    assert r[3] == oracle.amax(bits, "bf16")
    assert np.all(np.delete(r, 3) == 7.0)


@pytest.mark.parametrize("H,margin", [(1, 0), (4, 0), (16, 2), (1000, -3), (70000, 1)])
def test_scale_from_history_parity(H, margin):
    rng = np.random.default_rng(H)
    h = (rng.random(H) * 10.0 ** rng.uniform(-3, 4, H)).astype(np.float32)
    s = F.fp8_scale_from_amax_history(torch.from_numpy(h).cuda(), margin)
    assert host(s)[0].view(np.uint32) == oracle.scale_from_history(h, margin).view(np.uint32)
    z = F.fp8_scale_from_amax_history(torch.zeros(H, dtype=torch.float32, device="cuda"), margin)
    assert host(z)[0] == np.float32(2.0 ** margin)


def test_delayed_scaling_loop():
    """Steps of delayed scaling: quantize with the current scale while
    recording this step's amax in a ring of H slots; every `interval` steps
    derive the next scale from the ring.  The CPU mirror runs the same
    recipe through the oracle."""
    H, interval, margin = 4, 2, 1
    ring = torch.zeros(H, dtype=torch.float32, device="cuda")
    scale = torch.ones(4, dtype=torch.float32, device="cuda")[:1]
    ring_c = np.zeros(H, np.float32)
    scale_c = np.float32(1.0)
    for t in range(9):
        std = [0.5, 3.0, 1.0, 40.0, 0.01, 2.0, 2.0, 900.0, 1.0][t]
        bits = synth.random_bits((3000 + 17 * t,), "f16", seed=43, tensor_id=t, std=std)
        q = F.fp8_quantize_per_tensor_static(to_dev(bits, "f16"), scale, amax=ring[t % H:t % H + 1])
        assert np.array_equal(host(q), oracle.quantize_with_scale(bits, "f16", scale_c)), f"step {t}"
        ring_c[t % H] = oracle.amax(bits, "f16")
        if (t + 1) % interval == 0:
            F.fp8_scale_from_amax_history(ring, margin, scale=scale)
            scale_c = oracle.scale_from_history(ring_c, margin)
        assert np.array_equal(host(ring).view(np.uint32), ring_c.view(np.uint32))
        assert host(scale)[0].view(np.uint32) == np.float32(scale_c).view(np.uint32)


def test_full_size_outlier_activation_static():
    """The 16384 x 8192 outlier activation at half its dynamic scale: the
    outlier channels saturate."""
    wl = synth.WORKLOADS["outlier_16384x8192x8192"]
    bits = synth.activation(wl, wl.linears[0])
    _, s_dyn = oracle.quantize_per_tensor(bits, "f16")
    check_static(bits, "f16", np.float32(s_dyn * np.float32(0.5)))
