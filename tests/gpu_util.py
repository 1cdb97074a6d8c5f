"""Helpers shared by the GPU parity tests (marshalling only)."""
import numpy as np
import pytest
import torch

TD = {"f16": torch.float16, "bf16": torch.bfloat16}


def to_dev(bits, dtype):
    """uint16 bit patterns -> CUDA tensor of the given 16-bit float type."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TD[dtype]).cuda()


def host(t):
    return t.cpu().numpy()


def out_bits_to_f64(c):
    return c.float().cpu().numpy().astype(np.float64)


@pytest.fixture(autouse=True)
def no_device_error():
    """Every GPU test also checks that no kernel's bounded wait expired."""
    import fp8_scaled_gemm_02_b300 as F
    yield
    assert F.fp8s_device_error() == 0, "a kernel's bounded wait expired"
