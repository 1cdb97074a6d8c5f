"""GPU parity of the fused FP8 linear (fp8_linear_token_group): the
activation is quantized per 1x128 token group inside the block-scaled GEMM
kernel ("What is FP8 inference on H100 (Transformer Engine)?" s3 steps 2-6
with the 1x128 groups of the transformers "Fine-grained FP8" guide).

The optional copies of the in-kernel quantized activation and its scales
must be bit-exact against the oracle's token-group quantizer, and C within
the GEMM tolerance of the oracle's block-scaled GEMM on those bytes and
scales.  Shapes: the decode batches M = 1, 2, 4, 8, 16 (16-row activation
boxes) and M = 17 ... 300 (128-row boxes, ragged last M tile), ragged N,
every tile width and split-K factor the fused kernel has, groups of very
different magnitudes, and the Llama-2-7B decode linears.  Outputs sit inside
canary bands and start as poison."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TD, Guarded, no_device_error, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu

F = pytest.importorskip("fp8_scaled_gemm_02_b300")


def run_fused(a_bits, w_bits, dt, rows=None, copy_out=True):
    M, K = a_bits.shape
    N = w_bits.shape[0]
    qw, sw = F.fp8_quantize_weight_block(to_dev(w_bits, dt))
    gc = Guarded((M, N), TD[dt])
    gqa = Guarded((M, K), torch.uint8) if copy_out else None
    gsa = Guarded((K // 128, M), torch.float32) if copy_out else None
    F.fp8_linear_token_group(to_dev(a_bits, dt), qw, sw, c=gc.t, qa=gqa.t if copy_out else None,
                             sa=gsa.t if copy_out else None)
    torch.cuda.synchronize()
    oqa, osa = oracle.quantize_token_group(a_bits, dt)
    oqw, osw = oracle.quantize_weight_block(w_bits, dt)
    assert np.array_equal(qw.cpu().numpy(), oqw) and np.array_equal(sw.cpu().numpy(), osw)
    if copy_out:
        qa, sa = gqa.check().cpu().numpy(), gsa.check().cpu().numpy()
        bad = np.argwhere(qa != oqa)
        assert bad.size == 0, f"{len(bad)} activation bytes differ, first {bad[:5].tolist()}"
        assert np.array_equal(sa.view(np.uint32), osa.view(np.uint32)), "activation scales differ"
    R = oracle.gemm_block(oqa, osa, oqw, osw, rows=rows)
    C = gc.check().float().cpu().numpy().astype(np.float64)
    if rows is not None:
        C = C[rows]
    ok, ratio = oracle.within_tolerance(C, R, dt)
    assert ok, f"worst |C-R|/bound = {ratio:.3f}"
    return ratio


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (1, 4096, 1024), (2, 520, 384), (4, 300, 640), (8, 2048, 2048),
                                   (16, 1000, 1024), (17, 520, 512), (100, 37, 384), (128, 4096, 1024),
                                   (300, 520, 640)])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_fused(M, N, K, dt):
    a = synth.random_bits((M, K), dt, seed=81, tensor_id=M, std=1.0)
    w = synth.random_bits((N, K), dt, seed=81, tensor_id=10000 + N, std=0.02)
    run_fused(a, w, dt)


def test_fused_without_copies():
    a = synth.random_bits((8, 1024), "bf16", seed=82, tensor_id=1)
    w = synth.random_bits((700, 1024), "bf16", seed=82, tensor_id=2, std=0.02)
    run_fused(a, w, "bf16", copy_out=False)


def _distinct(M, N, K, seed):
    rng = np.random.default_rng(seed)
    a = synth.bits_to_f32(synth.random_bits((M, K), "bf16", seed=seed, tensor_id=1), "bf16")
    a *= (2.0 ** rng.integers(-10, 10, (M, K // 128))).repeat(128, 1).astype(np.float32)
    w = synth.bits_to_f32(synth.random_bits((N, K), "bf16", seed=seed, tensor_id=2, std=0.02), "bf16")
    nb = (N + 127) // 128
    w *= (2.0 ** rng.integers(-10, 10, (nb, K // 128))).repeat(128, 0)[:N].repeat(128, 1).astype(np.float32)
    return synth.f32_to_bits(a, "bf16"), synth.f32_to_bits(w, "bf16")


@pytest.mark.parametrize("M", [3, 16, 130])
def test_fused_distinct_group_magnitudes(M):
    a, w = _distinct(M, 384, 1536, seed=83 + M)
    run_fused(a, w, "bf16")


@pytest.mark.parametrize("bn,splits", [(64, 1), (128, 1), (192, 1), (64, 2), (128, 4), (128, 8), (64, 8)])
@pytest.mark.parametrize("M", [5, 128])
def test_fused_every_tile(bn, splits, M):
    a, w = _distinct(M, 520, 1024, seed=84)
    F.fp8s_gemm_override(bn, splits)
    try:
        run_fused(a, w, "bf16")
    finally:
        F.fp8s_gemm_override(0)


@pytest.mark.parametrize("m", [1, 2, 4, 8, 16, 128])
def test_fused_llama_decode(m):
    wl = synth.WORKLOADS[f"llama2_7b_m{m}"]
    for lin in wl.linears:
        run_fused(synth.activation(wl, lin), synth.weight(wl, lin), "bf16")


def test_fused_refuses_unbuilt_tiles():
    """192-wide tiles split K only for M <= 16; 256- and 32-wide tiles do not exist."""
    w = synth.random_bits((520, 1024), "bf16", seed=85, tensor_id=2, std=0.02)
    qw, sw = F.fp8_quantize_weight_block(to_dev(w, "bf16"))
    for M, bn, splits in [(20, 192, 2), (4, 256, 1), (4, 32, 1)]:
        a = synth.random_bits((M, 1024), "bf16", seed=85, tensor_id=1)
        F.fp8s_gemm_override(bn, splits)
        try:
            with pytest.raises(F.Fp8sError):
                F.fp8_linear_token_group(to_dev(a, "bf16"), qw, sw)
        finally:
            F.fp8s_gemm_override(0)


@pytest.mark.parametrize("splits", [2, 4, 8])
def test_fused_192_split_small_m(splits):
    """192-wide tiles with split-K (16-row activation boxes, M <= 16)."""
    a, w = _distinct(7, 700, 1024, seed=86)
    F.fp8s_gemm_override(192, splits)
    try:
        run_fused(a, w, "bf16")
    finally:
        F.fp8s_gemm_override(0)
