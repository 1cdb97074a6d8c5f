"""GPU parity of the power-of-two (UE8M0) scale variants against the oracle
("UE8M0 scale format" of the transformers "Fine-grained FP8" guide): the
token-group and weight-block quantizers with scales rounded up to a power
of two and stored as 8-bit biased exponents.  E4M3 bytes and scale codes
must be bit-exact.  Outputs sit inside canary bands and start as poison
(0xFF bytes), so a store outside an output or an element never written
fails the test.

Cases: ragged shapes, zero units, every finite FP16/BF16 magnitude as a
group amax (every scale code a 16-bit input can produce, including the
subnormal FP32 scales of tiny BF16 groups and the clamp at 2^-127), and the
full-size outlier activation and Llama-2-7B weights."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TD, Guarded, no_device_error, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu

F = pytest.importorskip("fp8_scaled_gemm_02_b300")


def check_token_group(bits, dtype):
    M, K = bits.shape
    gq, gs = Guarded((M, K), torch.uint8), Guarded((K // 128, M), torch.uint8)
    F.fp8_quantize_token_group_ue8m0(to_dev(bits, dtype), q=gq.t, sa=gs.t)
    torch.cuda.synchronize()
    q, c = gq.check().cpu().numpy(), gs.check(allow_poison=True).cpu().numpy()
    oq, oc = oracle.quantize_token_group_ue8m0(bits, dtype)
    bad = np.argwhere(c != oc)
    assert bad.size == 0, f"{len(bad)} scale codes differ, first {bad[:5].tolist()}"
    bad = np.argwhere(q != oq)
    assert bad.size == 0, f"{len(bad)} bytes differ, first {bad[:5].tolist()}"


def check_weight_block(bits, dtype):
    N, K = bits.shape
    gq, gs = Guarded((N, K), torch.uint8), Guarded(((N + 127) // 128, K // 128), torch.uint8)
    F.fp8_quantize_weight_block_ue8m0(to_dev(bits, dtype), q=gq.t, sb=gs.t)
    torch.cuda.synchronize()
    q, c = gq.check().cpu().numpy(), gs.check(allow_poison=True).cpu().numpy()
    oq, oc = oracle.quantize_weight_block_ue8m0(bits, dtype)
    assert np.array_equal(c, oc), f"scale codes differ at {np.argwhere(c != oc)[:5].tolist()}"
    bad = np.argwhere(q != oq)
    assert bad.size == 0, f"{len(bad)} bytes differ, first {bad[:5].tolist()}"


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,K", [(1, 128), (5, 384), (17, 1024), (200, 2048), (1000, 640), (4100, 256)])
def test_token_group(dtype, M, K):
    check_token_group(synth.random_bits((M, K), dtype, seed=61, tensor_id=M * 7 + K, std=1.5), dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N,K", [(1, 128), (128, 128), (300, 256), (129, 384), (1000, 640)])
def test_weight_block(dtype, N, K):
    check_weight_block(synth.random_bits((N, K), dtype, seed=62, tensor_id=N * 7 + K, std=0.02), dtype)


def test_zero_units():
    z = np.zeros((3, 384), np.uint16)
    z[1, 128:256] = 0x8000
    z[2, :] = synth.random_bits((384,), "f16", seed=1, tensor_id=1)
    for dt in ("f16", "bf16"):
        check_token_group(z, dt)
        check_weight_block(z, dt)


def _finite_patterns(dtype):
    p = np.arange(0x8000, dtype=np.uint32).astype(np.uint16)
    exp_mask = 0x7C00 if dtype == "f16" else 0x7F80
    return p[(p & exp_mask) != exp_mask]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_every_amax_pattern(dtype):
    """Every non-zero finite magnitude as a group amax, with 127 random
    smaller companions of random sign: every code a 16-bit amax can give."""
    mags = _finite_patterns(dtype)[1:]
    n = mags.size
    rng = np.random.default_rng(63)
    comp = np.floor(rng.random((n, 127)) * (mags[:, None].astype(np.float64) + 1)).astype(np.uint16)
    comp |= (rng.integers(0, 2, (n, 127)) << 15).astype(np.uint16)
    groups = np.concatenate([(mags | (rng.integers(0, 2, n) << 15).astype(np.uint16))[:, None], comp], axis=1)
    pad = (-n) % 64
    groups = np.concatenate([groups, np.zeros((pad, 128), np.uint16)])
    check_token_group(np.ascontiguousarray(groups.reshape(-1, 64 * 128)), dtype)


def test_full_size_outlier_activation():
    wl = synth.WORKLOADS["outlier_16384x8192x8192"]
    check_token_group(synth.activation(wl, wl.linears[0]), "f16")


def test_full_size_llama_weights():
    wl = synth.WORKLOADS["llama2_7b_m4096"]
    for lin in wl.linears:
        check_weight_block(synth.weight(wl, lin), "bf16")


# ------------------------------------------------------------------- GEMM
def run_ue8_linear(a_bits, w_bits, in_dt, out_dt, rows=None):
    """UE8M0-quantize A and W on the GPU (checked bit-exact), run the GEMM
    in block_ue8m0 mode (scales applied by the tensor core), and compare the
    output with the oracle's block-scaled GEMM on the decoded power-of-two
    scales."""
    M, K = a_bits.shape
    N = w_bits.shape[0]
    qa, ca = F.fp8_quantize_token_group_ue8m0(to_dev(a_bits, in_dt))
    qw, cw = F.fp8_quantize_weight_block_ue8m0(to_dev(w_bits, in_dt))
    gc = Guarded((M, N), TD[out_dt])
    F.fp8_gemm_scaled(qa, ca, qw, cw, out_dtype=TD[out_dt], mode="block_ue8m0", c=gc.t)
    torch.cuda.synchronize()
    oqa, oca = oracle.quantize_token_group_ue8m0(a_bits, in_dt)
    oqw, ocw = oracle.quantize_weight_block_ue8m0(w_bits, in_dt)
    assert np.array_equal(qa.cpu().numpy(), oqa) and np.array_equal(ca.cpu().numpy(), oca)
    assert np.array_equal(qw.cpu().numpy(), oqw) and np.array_equal(cw.cpu().numpy(), ocw)
    R = oracle.gemm_block(oqa, oracle.ue8m0_decode(oca), oqw, oracle.ue8m0_decode(ocw), rows=rows)
    C = gc.check().float().cpu().numpy().astype(np.float64)
    if rows is not None:
        C = C[rows]
    ok, ratio = oracle.within_tolerance(C, R, out_dt)
    assert ok, f"worst |C-R|/bound = {ratio:.3f}"
    return ratio


SHAPES = [(1, 1, 128), (4, 128, 128), (200, 320, 512), (300, 520, 1024), (130, 4000, 640), (257, 37, 384),
          (128, 4096, 1024), (512, 2560, 2048), (1000, 2048, 1152)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("in_dt,out_dt", [("bf16", "bf16"), ("f16", "f16")])
def test_gemm(M, N, K, in_dt, out_dt):
    a = synth.random_bits((M, K), in_dt, seed=64, tensor_id=M, std=1.0)
    w = synth.random_bits((N, K), in_dt, seed=64, tensor_id=10000 + N, std=0.02)
    run_ue8_linear(a, w, in_dt, out_dt)


def _distinct(M, N, K, seed):
    """Every activation row and every (row, K block) group, and every weight
    block, at its own power-of-two magnitude: a scale factor read from the
    wrong row, column, K block or byte is far outside the tolerance."""
    rng = np.random.default_rng(seed)
    a = synth.bits_to_f32(synth.random_bits((M, K), "bf16", seed=seed, tensor_id=1), "bf16")
    a *= (2.0 ** rng.integers(-12, 12, (M, K // 128))).repeat(128, 1).astype(np.float32)
    w = synth.bits_to_f32(synth.random_bits((N, K), "bf16", seed=seed, tensor_id=2, std=0.02), "bf16")
    nb = (N + 127) // 128
    w *= (2.0 ** rng.integers(-12, 12, (nb, K // 128))).repeat(128, 0)[:N].repeat(128, 1).astype(np.float32)
    return synth.f32_to_bits(a, "bf16"), synth.f32_to_bits(w, "bf16")


@pytest.mark.parametrize("M,N,K", [(256, 384, 1024), (300, 700, 1408), (128, 2048, 2048)])
def test_gemm_distinct_scale_factors(M, N, K):
    a, w = _distinct(M, N, K, seed=65 + M)
    run_ue8_linear(a, w, "bf16", "bf16")


@pytest.mark.parametrize("bn,splits", [(32, 1), (64, 1), (128, 1), (192, 1), (256, 1), (64, 2), (128, 4), (192, 2),
                                       (32, 2)])
def test_gemm_every_tile(bn, splits):
    a, w = _distinct(300, 520, 1024, seed=66)
    F.fp8s_gemm_override(bn, splits)
    try:
        run_ue8_linear(a, w, "bf16", "bf16")
    finally:
        F.fp8s_gemm_override(0)


@pytest.mark.parametrize("M,N,K", [(300, 520, 1024), (600, 1000, 2048)])
def test_gemm_multicast_pairs(M, N, K):
    """Two CTAs of a cluster on a 256-row tile, each loading half of the
    256-wide weight tile by TMA multicast into both; the scale factors stay
    per CTA (an odd number of 128-row tiles leaves a pair's second CTA
    past M)."""
    a, w = _distinct(M, N, K, seed=67 + M)
    F.fp8s_gemm_override(256, 1, True)
    try:
        run_ue8_linear(a, w, "bf16", "bf16")
    finally:
        F.fp8s_gemm_override(0)


def _sample_rows(M, n=32, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, M - 1], rng.choice(M, size=min(n, M), replace=False)]))


@pytest.mark.parametrize("m", [1, 2, 4, 8, 16, 128])
def test_llama_decode_shapes(m):
    wl = synth.WORKLOADS[f"llama2_7b_m{m}"]
    for lin in wl.linears:
        run_ue8_linear(synth.activation(wl, lin), synth.weight(wl, lin), "bf16", "bf16")


def test_outlier_full_size():
    wl = synth.WORKLOADS["outlier_16384x8192x8192"]
    lin = wl.linears[0]
    run_ue8_linear(synth.activation(wl, lin), synth.weight(wl, lin), "f16", "f16", rows=_sample_rows(lin.M, n=24))
