"""GPU parity of the scaled FP8 GEMM against the CPU oracle.

The quantized operands are produced on the GPU and first checked bit-exact
against the oracle's; the GEMM output must then satisfy
|C - R| <= t*|R| + t*rms(R) with t = 1e-3 (FP16 out) or 2e-3 (BF16 out),
R being the oracle's unrounded FP64 result on the same bytes and scales.

Shapes span several tiles with ragged M / N / K edges, every tile width the
kernel instantiates, N not a multiple of 8 (scalar store path), single
rows/columns, and the workloads' full sizes on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TD, Guarded, host, no_device_error, out_bits_to_f64, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu

F = pytest.importorskip("fp8_scaled_gemm_02_b300")


def run_linear(a_bits, w_bits, in_dt, out_dt, mode, rows=None):
    """Quantize A and W on the GPU, run the GEMM; check bytes/scales against
    the oracle, then the output against the oracle GEMM on `rows`.  Every
    output sits inside canary bands and starts as poison (0xFF bytes), so a
    store past a ragged tile's edge or an element left unwritten fails."""
    a, w = to_dev(a_bits, in_dt), to_dev(w_bits, in_dt)
    (M, K), N = a_bits.shape, w_bits.shape[0]
    gqa, gqw = Guarded((M, K), torch.uint8), Guarded((N, K), torch.uint8)
    if mode == "block":
        gsa, gsw = Guarded((K // 128, M), torch.float32), Guarded(((N + 127) // 128, K // 128), torch.float32)
        qa, sa = F.fp8_quantize_token_group(a, q=gqa.t, sa=gsa.t)
        qw, sw = F.fp8_quantize_weight_block(w, q=gqw.t, sb=gsw.t)
        oqa, osa = oracle.quantize_token_group(a_bits, in_dt)
        oqw, osw = oracle.quantize_weight_block(w_bits, in_dt)
    else:
        gsa, gsw = Guarded((1,), torch.float32), Guarded((1,), torch.float32)
        qa, sa = F.fp8_quantize_per_tensor(a, q=gqa.t, scale=gsa.t)
        qw, sw = F.fp8_quantize_per_tensor(w, q=gqw.t, scale=gsw.t)
        oqa, osa = oracle.quantize_per_tensor(a_bits, in_dt)
        oqw, osw = oracle.quantize_per_tensor(w_bits, in_dt)
    gc = Guarded((M, N), TD[out_dt])
    c = F.fp8_gemm_scaled(qa, sa, qw, sw, out_dtype=TD[out_dt], mode=mode, c=gc.t)
    torch.cuda.synchronize()
    for g in (gqa, gqw, gsa, gsw, gc):
        g.check()
    assert np.array_equal(host(qa), oqa) and np.array_equal(host(qw), oqw), "operand bytes differ"
    if mode == "block":
        assert np.array_equal(host(sa), osa) and np.array_equal(host(sw), osw), "scales differ"
        R = oracle.gemm_block(oqa, osa, oqw, osw, rows=rows)
    else:
        assert host(sa)[0] == osa and host(sw)[0] == osw, "scales differ"
        R = oracle.gemm_per_tensor(oqa, osa, oqw, osw, rows=rows)
    C = out_bits_to_f64(c)
    if rows is not None:
        C = C[rows]
    ok, ratio = oracle.within_tolerance(C, R, out_dt)
    assert ok, f"worst |C-R|/bound = {ratio:.3f}"
    return ratio


SHAPES_PT = [
    (64, 64, 128),       # the 64x128 . 128x64 per-tensor case
    (1, 1, 16), (1, 8, 32), (3, 45, 144),      # K % 128 != 0; N % 8 != 0
    (300, 520, 640), (2048, 2048, 256), (512, 2560, 2048), (128, 4096, 1024),
    (130, 4000, 272), (257, 37, 1600),
]
SHAPES_BLK = [
    (1, 1, 128), (4, 128, 128), (200, 320, 512), (300, 520, 1024), (128, 4096, 1024),
    (512, 2560, 2048), (257, 37, 640), (1000, 2048, 384),
]


@pytest.mark.parametrize("M,N,K", SHAPES_PT)
@pytest.mark.parametrize("in_dt,out_dt", [("f16", "f16"), ("bf16", "bf16")])
def test_per_tensor(M, N, K, in_dt, out_dt):
    a = synth.random_bits((M, K), in_dt, seed=51, tensor_id=M, std=1.0)
    w = synth.random_bits((N, K), in_dt, seed=51, tensor_id=10000 + N, std=0.02)
    run_linear(a, w, in_dt, out_dt, "per_tensor")


@pytest.mark.parametrize("M,N,K", SHAPES_BLK)
@pytest.mark.parametrize("in_dt,out_dt", [("bf16", "bf16"), ("f16", "f16")])
def test_block(M, N, K, in_dt, out_dt):
    a = synth.random_bits((M, K), in_dt, seed=52, tensor_id=M, std=1.0)
    w = synth.random_bits((N, K), in_dt, seed=52, tensor_id=10000 + N, std=0.02)
    run_linear(a, w, in_dt, out_dt, "block")


def test_block_distinct_group_magnitudes():
    """Groups and blocks with very different magnitudes: a swapped scale index
    or a missed promotion would be far outside the tolerance."""
    M, N, K = 256, 384, 1024
    rng = np.random.default_rng(53)
    a = synth.bits_to_f32(synth.random_bits((M, K), "bf16", seed=53, tensor_id=1), "bf16")
    a *= (2.0 ** rng.integers(-8, 8, (M, K // 128))).repeat(128, 1).astype(np.float32)
    w = synth.bits_to_f32(synth.random_bits((N, K), "bf16", seed=53, tensor_id=2, std=0.02), "bf16")
    w *= (2.0 ** rng.integers(-8, 8, (3, K // 128))).repeat(128, 0).repeat(128, 1).astype(np.float32)
    run_linear(synth.f32_to_bits(a, "bf16"), synth.f32_to_bits(w, "bf16"), "bf16", "bf16", "block")


def test_repeat_calls_are_identical():
    a = synth.random_bits((300, 1024), "bf16", seed=54, tensor_id=1)
    w = synth.random_bits((520, 1024), "bf16", seed=54, tensor_id=2, std=0.02)
    qa, sa = F.fp8_quantize_token_group(to_dev(a, "bf16"))
    qw, sw = F.fp8_quantize_weight_block(to_dev(w, "bf16"))
    c1 = F.fp8_gemm_scaled(qa, sa, qw, sw)
    c2 = F.fp8_gemm_scaled(qa, sa, qw, sw)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


def _sample_rows(M, n=48, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, M - 1], rng.choice(M, size=min(n, M), replace=False)]))


@pytest.mark.parametrize("name", ["per_tensor_64x64x128", "block_128x4096x4096", "tinyllama_1.1b_m512",
                                  "llama2_7b_m128", "llama2_7b_m4096"])
def test_workload(name):
    wl = synth.WORKLOADS[name]
    for lin in wl.linears:
        a = synth.activation(wl, lin)
        w = synth.weight(wl, lin)
        rows = None if lin.M * lin.N * lin.K <= 2 ** 33 else _sample_rows(lin.M)
        for mode in wl.modes:
            run_linear(a, w, wl.in_dtype, wl.out_dtype, mode, rows=rows)


def test_workload_outlier_full_size():
    wl = synth.WORKLOADS["outlier_16384x8192x8192"]
    lin = wl.linears[0]
    run_linear(synth.activation(wl, lin), synth.weight(wl, lin), "f16", "f16", "block",
               rows=_sample_rows(lin.M, n=24))


def test_workload_outlier_per_tensor_full_size():
    """The full-size outlier shape with per-tensor scaling: the automatically
    chosen CTA-pair (cta_group::2) tiles, on sampled output rows."""
    wl = synth.WORKLOADS["outlier_16384x8192x8192"]
    lin = wl.linears[0]
    assert F.fp8s_gemm_plan(lin.M, lin.N, lin.K, "per_tensor")[2], "expected the CTA-pair configuration"
    run_linear(synth.activation(wl, lin), synth.weight(wl, lin), "f16", "f16", "per_tensor",
               rows=_sample_rows(lin.M, n=24, seed=1))
