"""GPU parity of the decode-batch GEMM (M <= 32 tokens, computed transposed
with the weight tile as the tensor core's 128-row operand) against the
oracle, through both entry points that use it: fp8_gemm_scaled in block
mode and the fused fp8_linear_token_group.  The block-scaled linear of the
transformers "Fine-grained FP8" guide at the decode batch sizes of the
Llama-2-7B / TinyLlama inference task (batch 1, 2, 4, 8 and up to 32).

Shapes cover both token widths of the kernel (16 and 32 columns), token
counts that leave most of those columns empty, a ragged last 128-row weight
tile, K ranges split over 1, 2, 4 and 8 CTAs (the split count follows from
the number of weight tiles), and the full Llama-2-7B decode linears.  Outputs
sit inside canary bands and start as poison (0xFF bytes)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TD, Guarded, no_device_error, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu

F = pytest.importorskip("fp8_scaled_gemm_02_b300")


def check(a_bits, w_bits, dt, fused):
    M, K = a_bits.shape
    N = w_bits.shape[0]
    qw, sw = F.fp8_quantize_weight_block(to_dev(w_bits, dt))
    oqa, osa = oracle.quantize_token_group(a_bits, dt)
    oqw, osw = oracle.quantize_weight_block(w_bits, dt)
    assert np.array_equal(qw.cpu().numpy(), oqw) and np.array_equal(sw.cpu().numpy(), osw)
    gc = Guarded((M, N), TD[dt])
    if fused:
        gqa, gsa = Guarded((M, K), torch.uint8), Guarded((K // 128, M), torch.float32)
        F.fp8_linear_token_group(to_dev(a_bits, dt), qw, sw, c=gc.t, qa=gqa.t, sa=gsa.t)
        torch.cuda.synchronize()
        assert np.array_equal(gqa.check().cpu().numpy(), oqa), "in-kernel activation bytes differ"
        assert np.array_equal(gsa.check().cpu().numpy().view(np.uint32), osa.view(np.uint32)), "scales differ"
    else:
        qa, sa = F.fp8_quantize_token_group(to_dev(a_bits, dt))
        F.fp8_gemm_scaled(qa, sa, qw, sw, out_dtype=TD[dt], mode="block", c=gc.t)
        torch.cuda.synchronize()
    R = oracle.gemm_block(oqa, osa, oqw, osw)
    C = gc.check().float().cpu().numpy().astype(np.float64)
    ok, ratio = oracle.within_tolerance(C, R, dt)
    assert ok, f"worst |C-R|/bound = {ratio:.3f}"


SHAPES = [(1, 1, 128), (1, 100, 1024), (2, 520, 384), (3, 4096, 1024), (8, 130, 2048), (16, 1000, 640),
          (17, 700, 1024), (24, 4096, 512), (31, 257, 1152), (32, 2048, 1024)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_decode(M, N, K, fused, dt):
    a = synth.random_bits((M, K), dt, seed=91, tensor_id=M, std=1.0)
    w = synth.random_bits((N, K), dt, seed=91, tensor_id=10000 + N, std=0.02)
    check(a, w, dt, fused)


@pytest.mark.parametrize("M,N", [(5, 128), (9, 640), (20, 3000), (32, 12288)])
@pytest.mark.parametrize("fused", [False, True])
def test_decode_distinct_magnitudes(M, N, fused):
    """Every (token, K block) group and every weight block at its own power
    of two: a token scale applied to the wrong column, a block scale to the
    wrong weight tile or K block, is far outside the tolerance."""
    K = 1536
    rng = np.random.default_rng(92 + M)
    a = synth.bits_to_f32(synth.random_bits((M, K), "bf16", seed=92, tensor_id=M), "bf16")
    a *= (2.0 ** rng.integers(-10, 10, (M, K // 128))).repeat(128, 1).astype(np.float32)
    w = synth.bits_to_f32(synth.random_bits((N, K), "bf16", seed=92, tensor_id=N, std=0.02), "bf16")
    nb = (N + 127) // 128
    w *= (2.0 ** rng.integers(-10, 10, (nb, K // 128))).repeat(128, 0)[:N].repeat(128, 1).astype(np.float32)
    check(synth.f32_to_bits(a, "bf16"), synth.f32_to_bits(w, "bf16"), "bf16", fused)


@pytest.mark.parametrize("m", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("fused", [False, True])
def test_llama_decode_linears(m, fused):
    wl = synth.WORKLOADS[f"llama2_7b_m{m}"]
    for lin in wl.linears:
        check(synth.activation(wl, lin), synth.weight(wl, lin), "bf16", fused)


def test_repeat_calls_are_identical():
    """Split-K sums the partials in a fixed order: bit-identical repeats."""
    a = synth.random_bits((7, 4096), "bf16", seed=93, tensor_id=1)
    w = synth.random_bits((4096, 4096), "bf16", seed=93, tensor_id=2, std=0.02)
    qa, sa = F.fp8_quantize_token_group(to_dev(a, "bf16"))
    qw, sw = F.fp8_quantize_weight_block(to_dev(w, "bf16"))
    c1 = F.fp8_gemm_scaled(qa, sa, qw, sw)
    c2 = F.fp8_gemm_scaled(qa, sa, qw, sw)
    f1 = F.fp8_linear_token_group(to_dev(a, "bf16"), qw, sw)
    f2 = F.fp8_linear_token_group(to_dev(a, "bf16"), qw, sw)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2) and torch.equal(f1, f2)
