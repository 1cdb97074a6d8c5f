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


# ------------------------------------------------ guard bands and poison
# Stand-in for a memory checker: every output of a parity test can live
# inside a larger buffer whose bands before and after it hold a canary byte,
# with the output itself pre-filled with a poison pattern that no kernel
# writes for finite inputs (0xFF bytes: the NaN code of E4M3, a NaN as FP16,
# BF16 or FP32).  After the call the bands must be intact (no store outside
# the output) and the poison gone (no element left unwritten).
GUARD = 4096
CANARY = 0x5A
POISON = 0xFF


class Guarded:
    def __init__(self, shape, dtype, poison=POISON, device="cuda"):
        shape = tuple(shape)
        itemsize = torch.empty((), dtype=dtype).element_size()
        n = 1
        for d in shape:
            n *= d
        self.nbytes = n * itemsize
        padded = (self.nbytes + 15) // 16 * 16
        self.raw = torch.full((2 * GUARD + padded,), CANARY, dtype=torch.uint8, device=device)
        self.raw[GUARD:GUARD + self.nbytes] = poison
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)
        self.poison = poison

    def check(self, allow_poison=False):
        raw = self.raw.cpu().numpy()
        before, after = raw[:GUARD], raw[GUARD + self.nbytes:]
        assert (before == CANARY).all() and (after == CANARY).all(), "a kernel wrote outside its output"
        if not allow_poison:
            body = raw[GUARD:GUARD + self.nbytes]
            if self.t.element_size() == 1:
                left = int((body == self.poison).sum())
            else:
                words = body.view(np.uint16 if self.t.element_size() == 2 else np.uint32)
                full = np.iinfo(words.dtype).max if self.poison == 0xFF else None
                left = int((words == full).sum()) if full is not None else 0
            assert left == 0, f"{left} output elements were never written"
        return self.t


def guarded(shape, dtype, poison=POISON):
    return Guarded(shape, dtype, poison)
