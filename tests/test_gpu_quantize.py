"""GPU parity of the three quantizers against the CPU oracle: E4M3 bytes and
FP32 scales must be bit-exact.

Cases: several tiles with ragged edges, single-row / single-group minima,
all-zero and negative-zero units, exhaustive coverage of every FP16 and BF16
amax pattern, every FP16/BF16 input pattern at a set of scales, and the
full-size activation and weight tensors of the workloads.  Every output
sits inside canary bands and starts as poison (0xFF bytes, never a code or
scale a finite input produces): a store outside an output or an element
left unwritten fails the test."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import Guarded, host, no_device_error, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu

F = pytest.importorskip("fp8_scaled_gemm_02_b300")


def check_token_group(bits, dtype):
    M, K = bits.shape
    gq, gs = Guarded((M, K), torch.uint8), Guarded((K // 128, M), torch.float32)
    qa, sa = F.fp8_quantize_token_group(to_dev(bits, dtype), q=gq.t, sa=gs.t)
    torch.cuda.synchronize()
    gq.check()
    gs.check()
    oq, os_ = oracle.quantize_token_group(bits, dtype)
    q, s = host(qa), host(sa)
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32)), f"scales differ at {np.argwhere(s != os_)[:5]}"
    bad = np.argwhere(q != oq)
    assert bad.size == 0, f"{len(bad)} bytes differ, first {bad[:5].tolist()}"


def check_weight_block(bits, dtype):
    N, K = bits.shape
    gq, gs = Guarded((N, K), torch.uint8), Guarded(((N + 127) // 128, K // 128), torch.float32)
    qw, sw = F.fp8_quantize_weight_block(to_dev(bits, dtype), q=gq.t, sb=gs.t)
    torch.cuda.synchronize()
    gq.check()
    gs.check()
    oq, os_ = oracle.quantize_weight_block(bits, dtype)
    assert np.array_equal(host(sw).view(np.uint32), os_.view(np.uint32))
    bad = np.argwhere(host(qw) != oq)
    assert bad.size == 0, f"{len(bad)} bytes differ, first {bad[:5].tolist()}"


def check_per_tensor(bits, dtype):
    gq, gs = Guarded(bits.shape, torch.uint8), Guarded((1,), torch.float32)
    q, s = F.fp8_quantize_per_tensor(to_dev(bits, dtype), q=gq.t, scale=gs.t)
    torch.cuda.synchronize()
    gq.check()
    gs.check()
    oq, os_ = oracle.quantize_per_tensor(bits, dtype)
    assert host(s)[0].view(np.uint32) == np.float32(os_).view(np.uint32)
    assert np.array_equal(host(q), oq)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,K", [(1, 128), (5, 384), (17, 1024), (200, 2048), (1000, 640), (4100, 256)])
def test_token_group_parity(dtype, M, K):
    bits = synth.random_bits((M, K), dtype, seed=31, tensor_id=M * 7 + K, std=1.5)
    check_token_group(bits, dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N,K", [(1, 128), (128, 128), (300, 256), (129, 384), (1000, 640)])
def test_weight_block_parity(dtype, N, K):
    bits = synth.random_bits((N, K), dtype, seed=32, tensor_id=N * 7 + K, std=0.02)
    check_weight_block(bits, dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("numel", [1, 7, 8, 9, 1000, 65536 + 3, 1000003])
def test_per_tensor_parity(dtype, numel):
    bits = synth.random_bits((numel,), dtype, seed=33, tensor_id=numel, std=4.0)
    check_per_tensor(bits, dtype)


# The per-tensor quantizer switches paths by input size: one cluster of up
# to 16 CTAs (each slice <= 192 KB of shared memory) up to 16 * 192 KB of
# input, then a cooperative launch that keeps slices in shared memory up to
# 148 * 192 KB, and streams them beyond that.  These sizes sit on both sides
# of each switch, with and without a tail of numel % 8 elements.
SLICE_ELEMS = 192 * 1024 // 2


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("numel", [16 * SLICE_ELEMS, 16 * SLICE_ELEMS + 8, 16 * SLICE_ELEMS + 3,
                                   148 * SLICE_ELEMS - 8, 148 * SLICE_ELEMS + 8, 148 * SLICE_ELEMS + 5,
                                   3 * SLICE_ELEMS + 1])
def test_per_tensor_path_boundaries(dtype, numel):
    bits = synth.random_bits((numel,), dtype, seed=34, tensor_id=numel, std=3.0)
    check_per_tensor(bits, dtype)


def test_per_tensor_single_outlier_in_last_slice():
    """The maximum sits in the last CTA's slice (and in the tail): every
    other CTA must take it from the exchange."""
    for numel in (1000003, 16 * SLICE_ELEMS + 7, 148 * SLICE_ELEMS + 7):
        bits = synth.random_bits((numel,), "bf16", seed=35, tensor_id=numel, std=1.0)
        bits[-1] = 0x4700  # bf16 32768.0, far above the rest
        check_per_tensor(bits, "bf16")
        bits[-1] = 0x3F80
        bits[-9] = 0xC700  # -32768.0 in the last full vector
        check_per_tensor(bits, "bf16")


def test_zero_and_negative_zero_units():
    z = np.zeros((3, 384), np.uint16)
    z[1, 128:256] = 0x8000
    z[2, :] = synth.random_bits((384,), "f16", seed=1, tensor_id=1)
    z[2, 256:] = 0x8000
    for dt in ("f16", "bf16"):
        check_token_group(z, dt)
        check_weight_block(z, dt)
        check_per_tensor(np.zeros(77, np.uint16), dt)
        check_per_tensor(np.full(77, 0x8000, np.uint16), dt)


def _finite_patterns(dtype):
    p = np.arange(0x8000, dtype=np.uint32).astype(np.uint16)
    exp_mask = 0x7C00 if dtype == "f16" else 0x7F80
    return p[(p & exp_mask) != exp_mask]          # non-negative finite magnitudes, ascending


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_every_amax_pattern(dtype):
    """Every non-zero finite magnitude appears as a group amax (twice), with
    127 random companions of smaller magnitude and random signs."""
    mags = _finite_patterns(dtype)[1:]
    amax = np.repeat(mags, 2)
    n = amax.size
    rng = np.random.default_rng(41)
    frac = rng.random((n, 127))
    comp = np.floor(frac * (amax[:, None].astype(np.float64) + 1)).astype(np.uint16)
    comp |= (rng.integers(0, 2, (n, 127)) << 15).astype(np.uint16)
    groups = np.concatenate([(amax | (rng.integers(0, 2, n) << 15).astype(np.uint16))[:, None], comp], axis=1)
    pad = (-n) % 64
    groups = np.concatenate([groups, np.zeros((pad, 128), np.uint16)])
    bits = np.ascontiguousarray(groups.reshape(-1, 64 * 128))   # 64 groups per row
    check_token_group(bits, dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_every_input_pattern_at_many_scales(dtype):
    """Every finite input pattern is quantized under each of 24 amax values
    (each group carries its amax as element 0)."""
    mags = _finite_patterns(dtype)
    allp = np.concatenate([mags, mags | 0x8000])
    rng = np.random.default_rng(42)
    amaxes = np.concatenate([[mags[-1]], rng.choice(mags[1:], 23, replace=False)]).astype(np.uint16)
    rows = []
    for a in amaxes:
        xs = allp[(allp & 0x7FFF) <= a]
        pad = (-xs.size) % 127
        xs = np.concatenate([xs, np.zeros(pad, np.uint16)]).reshape(-1, 127)
        rows.append(np.concatenate([np.full((xs.shape[0], 1), a, np.uint16), xs], axis=1))
    groups = np.concatenate(rows)
    pad = (-groups.shape[0]) % 32
    groups = np.concatenate([groups, np.zeros((pad, 128), np.uint16)])
    check_token_group(np.ascontiguousarray(groups.reshape(-1, 32 * 128)), dtype)


def test_full_size_outlier_activation():
    wl = synth.WORKLOADS["outlier_16384x8192x8192"]
    bits = synth.activation(wl, wl.linears[0])
    check_token_group(bits, "f16")
    check_per_tensor(bits, "f16")


def test_full_size_llama_weights():
    wl = synth.WORKLOADS["llama2_7b_m4096"]
    for lin in wl.linears:
        check_weight_block(synth.weight(wl, lin), "bf16")
