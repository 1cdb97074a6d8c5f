"""Seeded synthetic inputs for the FP8 quantize + scaled-GEMM workloads.

This module is the one piece shared by the CUDA path's tests/benchmark and
the CPU oracle: it draws random 16-bit inputs and holds none of the method's
arithmetic (no amax, scale, E4M3 rounding or GEMM).  Every tensor comes from
numpy's counter-based Philox generator keyed by (seed, tensor id), is drawn in
float64, rounded to float32 and then rounded to nearest-even into FP16 or
BF16.  Tensors are returned as raw ``np.uint16`` bit patterns plus a dtype tag.

Workloads (shapes and distributions of the pages' use cases: FP8 linear
layers of TinyLlama-1.1B and Llama-2-7B, per-tensor and fine-grained
block-scaled quantization) are described by ``WORKLOADS``; each linear is
A [M, K] activations times W [N, K] weights (nn.Linear layout).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

F16, BF16 = "f16", "bf16"


# ----------------------------------------------------------- random draws
def _gen(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[int(seed), int(tensor_id)]))


def f32_to_bits(x32: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to FP16 or BF16 (nearest-even); return uint16 bits."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == F16:
        with np.errstate(over="raise"):
            h = x32.astype(np.float16)
        if not np.all(np.isfinite(h)):
            raise OverflowError("input draw does not fit FP16")
        return h.view(np.uint16)
    if dtype == BF16:
        u = x32.view(np.uint32).astype(np.uint64)
        rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        out = rounded.astype(np.uint16)
        if np.any((out & 0x7F80) == 0x7F80):
            raise OverflowError("input draw does not fit BF16")
        return out
    raise ValueError(dtype)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Plain widening of FP16/BF16 bit patterns (for generators' own checks)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def normal(shape, std: float, dtype: str, seed: int, tensor_id: int,
           chunk: int = 1 << 24) -> np.ndarray:
    """N(0, std^2) draws rounded into ``dtype``; returns uint16 bits."""
    g = _gen(seed, tensor_id)
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for i in range(0, n, chunk):
        j = min(n, i + chunk)
        x = g.standard_normal(j - i, dtype=np.float64) * std
        out[i:j] = f32_to_bits(x.astype(np.float32), dtype)
    return out.reshape(shape)


def student_t_outliers(M: int, K: int, dtype: str, seed: int, tensor_id: int,
                       nu: int = 3, outlier_frac: float = 0.01, outlier_gain: float = 100.0,
                       chunk_rows: int = 1024) -> np.ndarray:
    """Activation stress tensor: Student-t(nu) entries, built as
    Z / sqrt(chi2_nu / nu) from nu+1 standard normals, with a seeded
    ``outlier_frac`` subset of the K channels multiplied by ``outlier_gain``."""
    g = _gen(seed, tensor_id)
    n_out = max(1, int(round(outlier_frac * K)))
    chan = np.sort(g.choice(K, size=n_out, replace=False))
    gain = np.ones(K, np.float64)
    gain[chan] = outlier_gain
    out = np.empty((M, K), np.uint16)
    for r0 in range(0, M, chunk_rows):
        r1 = min(M, r0 + chunk_rows)
        z = g.standard_normal((r1 - r0, K))
        chi2 = np.zeros((r1 - r0, K))
        for _ in range(nu):
            chi2 += g.standard_normal((r1 - r0, K)) ** 2
        t = z / np.sqrt(chi2 / nu)
        out[r0:r1] = f32_to_bits((t * gain).astype(np.float32), dtype)
    return out


# -------------------------------------------------------------- workloads
@dataclasses.dataclass(frozen=True)
class Linear:
    name: str
    M: int
    N: int
    K: int


@dataclasses.dataclass(frozen=True)
class Workload:
    """A set of FP8 linears with one input recipe."""
    name: str
    description: str
    in_dtype: str
    out_dtype: str
    modes: tuple            # ("per_tensor",), ("block",) or both
    linears: tuple          # of Linear
    act: str = "normal"     # "normal" or "student_t_outliers"
    act_std: float = 1.0
    w_std: float = 0.02
    seed: int = 1
    weight_kn: bool = False  # weights drawn as B [K, N] and transposed to [N, K]


def _llama2(M):
    return (Linear("qkv", M, 12288, 4096), Linear("o", M, 4096, 4096),
            Linear("gate_up", M, 22016, 4096), Linear("down", M, 4096, 11008))


WORKLOADS: Dict[str, Workload] = {
    w.name: w for w in [
        Workload("per_tensor_64x64x128",
                 "per-tensor FP8 GEMM, A 64x128 and B 128x64 FP16 (A~N(0,1), B~N(0,0.02), seed 0), FP16 out",
                 F16, F16, ("per_tensor",), (Linear("gemm", 64, 64, 128),), seed=0, weight_kn=True),
        Workload("block_128x4096x4096",
                 "fine-grained block-scaled GEMM, activations 128x4096 BF16 ~N(0,1) (1x128 groups), "
                 "weights 4096x4096 BF16 ~N(0,0.02) (128x128 blocks), BF16 out",
                 BF16, BF16, ("block",), (Linear("gemm", 128, 4096, 4096),), seed=2),
        Workload("tinyllama_1.1b_m512",
                 "TinyLlama-1.1B-shaped linears at M=512, FP16 ~N(0,1) activations, ~N(0,0.02) weights, "
                 "per-tensor and block-scaled, FP16 out",
                 F16, F16, ("per_tensor", "block"),
                 (Linear("qkv", 512, 2560, 2048), Linear("o", 512, 2048, 2048),
                  Linear("gate_up", 512, 11264, 2048), Linear("down", 512, 2048, 5632)), seed=3),
        Workload("llama2_7b_m128",
                 "Llama-2-7B-shaped linears at M=128 (decode batch), BF16, block-scaled, BF16 out",
                 BF16, BF16, ("block",), _llama2(128), seed=4),
        *[Workload(f"llama2_7b_m{m}",
                   f"Llama-2-7B-shaped linears at M={m} (decode, batch size {m}), BF16, block-scaled, BF16 out",
                   BF16, BF16, ("block",), _llama2(m), seed=4) for m in (1, 2, 4, 8, 16)],
        Workload("llama2_7b_m4096",
                 "Llama-2-7B-shaped linears at M=4096 (prefill), BF16, block-scaled, BF16 out",
                 BF16, BF16, ("block",), _llama2(4096), seed=4),
        Workload("outlier_16384x8192x8192",
                 "outlier stress: activations 16384x8192 Student-t(3) with 1% of channels x100, weights "
                 "8192x8192 ~N(0,0.02), FP16, token-group quantize + block-scaled GEMM, FP16 out",
                 F16, F16, ("block",), (Linear("gemm", 16384, 8192, 8192),),
                 act="student_t_outliers", seed=5),
    ]
}


def activation(wl: Workload, lin: Linear, M: Optional[int] = None) -> np.ndarray:
    """The activation tensor A [M, K] of one linear (uint16 bits).

    Linears of one workload that share K share the activation draw."""
    M = lin.M if M is None else M
    tid = 1000 + lin.K
    if wl.act == "student_t_outliers":
        return student_t_outliers(M, lin.K, wl.in_dtype, wl.seed, tid)
    return normal((M, lin.K), wl.act_std, wl.in_dtype, wl.seed, tid)


def weight(wl: Workload, lin: Linear) -> np.ndarray:
    """The weight tensor W [N, K] of one linear (uint16 bits)."""
    tid = 2000 + hash_name(lin.name)
    if wl.weight_kn:
        b = normal((lin.K, lin.N), wl.w_std, wl.in_dtype, wl.seed, tid)
        return np.ascontiguousarray(b.T)
    return normal((lin.N, lin.K), wl.w_std, wl.in_dtype, wl.seed, tid)


def hash_name(name: str) -> int:
    h = 0
    for ch in name.encode():
        h = (h * 131 + ch) % 1000003
    return h


def random_bits(shape, dtype: str, seed: int, tensor_id: int, std: float = 1.0) -> np.ndarray:
    """Generic N(0, std^2) tensor for edge-case tests."""
    return normal(shape, std, dtype, seed, tensor_id)


def all_workloads() -> List[str]:
    return list(WORKLOADS)
