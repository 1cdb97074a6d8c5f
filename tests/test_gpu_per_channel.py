"""GPU parity of per-channel weight scaling against the CPU oracle.

"What is FP8 inference on H100" s5 names per-channel scaling for weights:
one scale per output channel (row of W).  fp8_quantize_per_channel must give
the oracle's E4M3 bytes and FP32 scales bit-exactly, and fp8_gemm_scaled in
mode "per_channel" (one activation scale, sb [N]) must stay within the
tolerance of the oracle's unrounded FP64 result, for every tile width,
split-K factor and CTA-pair tile, with ragged M, N and K."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TD, host, no_device_error, out_bits_to_f64, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu

F = pytest.importorskip("fp8_scaled_gemm_02_b300")


def weight_bits(N, K, dtype, seed):
    """Rows of very different magnitude (2^-8 .. 2^8 times N(0, 0.02)) and one
    all-zero row, so that per-row scales really differ."""
    w = synth.bits_to_f32(synth.random_bits((N, K), dtype, seed=seed, tensor_id=N + K, std=0.02), dtype)
    w = w * (2.0 ** (np.arange(N) % 17 - 8)).astype(np.float32)[:, None]
    if N > 2:
        w[N // 2] = 0.0
    return synth.f32_to_bits(w.astype(np.float32), dtype)


def check_quant(bits, dtype):
    q, sb = F.fp8_quantize_per_channel(to_dev(bits, dtype))
    oq, osb = oracle.quantize_per_channel(bits, dtype)
    assert np.array_equal(host(sb).view(np.uint32), osb.view(np.uint32)), "scales differ"
    bad = np.argwhere(host(q) != oq)
    assert bad.size == 0, f"{len(bad)} bytes differ, first {bad[:5].tolist()}"
    return q, sb, oq, osb


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N,K", [(1, 8), (3, 48), (128, 128), (300, 1040), (77, 4096), (1000, 11008),
                                 (5, 65536)])
def test_per_channel_quantize_parity(dtype, N, K):
    check_quant(weight_bits(N, K, dtype, seed=81), dtype)


def run(M, N, K, in_dt, out_dt, seed, rows=None):
    a = synth.random_bits((M, K), in_dt, seed=seed, tensor_id=1, std=1.0)
    qa, sa = F.fp8_quantize_per_tensor(to_dev(a, in_dt))
    qw, sb, oqw, osb = check_quant(weight_bits(N, K, in_dt, seed=seed), in_dt)
    oqa, osa = oracle.quantize_per_tensor(a, in_dt)
    c = F.fp8_gemm_scaled(qa, sa, qw, sb, out_dtype=TD[out_dt], mode="per_channel")
    torch.cuda.synchronize()
    R = oracle.gemm_per_channel(oqa, osa, oqw, osb, rows=rows)
    C = out_bits_to_f64(c)
    if rows is not None:
        C = C[rows]
    ok, ratio = oracle.within_tolerance(C, R, out_dt)
    assert ok, f"worst |C-R|/bound = {ratio:.3f}"
    return c


@pytest.mark.parametrize("M,N,K", [(64, 64, 128), (1, 8, 32), (3, 45, 144), (300, 520, 640), (128, 4096, 1024),
                                   (512, 2560, 2048), (257, 37, 1600)])
@pytest.mark.parametrize("in_dt,out_dt", [("f16", "f16"), ("bf16", "bf16")])
def test_per_channel_gemm(M, N, K, in_dt, out_dt):
    run(M, N, K, in_dt, out_dt, seed=82)


@pytest.fixture
def override():
    yield F.fp8s_gemm_override
    F.fp8s_gemm_override(0)


@pytest.mark.parametrize("bn,splits,pair", [(32, 1, 0), (64, 1, 0), (128, 1, 0), (192, 1, 0), (256, 1, 0),
                                            (32, 2, 0), (64, 4, 0), (128, 8, 0), (192, 2, 0), (64, 1, 1),
                                            (128, 1, 1), (256, 1, 1)])
def test_per_channel_forced_configs(override, bn, splits, pair):
    override(bn, splits, pair)
    c1 = run(200, 520, 1040, "bf16", "bf16", seed=83 + bn + splits)
    c2 = run(200, 520, 1040, "bf16", "bf16", seed=83 + bn + splits)
    assert torch.equal(c1, c2), "repeated calls differ"


def test_per_channel_llama_down_projection_sampled():
    """The 4096 x 4096 x 11008 down projection (CTA-pair tiles), sampled rows."""
    rng = np.random.default_rng(84)
    rows = np.unique(np.concatenate([[0, 4095], rng.choice(4096, 40, replace=False)]))
    run(4096, 4096, 11008, "bf16", "bf16", seed=84, rows=rows)


def test_uniform_per_channel_scales_equal_per_tensor():
    """sb[n] all equal to one per-tensor scale: the two modes give the same bits."""
    a = synth.random_bits((130, 640), "f16", seed=85, tensor_id=1, std=1.0)
    w = synth.random_bits((300, 640), "f16", seed=85, tensor_id=2, std=0.02)
    qa, sa = F.fp8_quantize_per_tensor(to_dev(a, "f16"))
    qw, sw = F.fp8_quantize_per_tensor(to_dev(w, "f16"))
    c_pt = F.fp8_gemm_scaled(qa, sa, qw, sw, out_dtype=torch.float16, mode="per_tensor")
    c_pc = F.fp8_gemm_scaled(qa, sa, qw, sw.expand(300).contiguous(), out_dtype=torch.float16, mode="per_channel")
    torch.cuda.synchronize()
    assert torch.equal(c_pt, c_pc)
