"""The failure path of the kernels' bounded waits, made to run on purpose
without any fault: the per-tensor quantizer's grid-wide exchange spin (on a
tensor large enough that its CTAs stream their slices, so no asynchronous
copy is in flight while they wait) is given a limit of 1 ns.  A CTA that
gives up records its role (4 = quantizer) in the device error word and
carries on, so the call ends without a hang and the host reads
FP8S_ERR_DEVICE_TIMEOUT.  With the default limit restored, the next call
on the same context is bit-exact again."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import host, no_device_error, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu

F = pytest.importorskip("fp8_scaled_gemm_02_b300")


def test_exchange_spin_runs_out_and_reports():
    n = 20 * 1024 * 1024 + 8            # 40 MB of FP16: above the on-chip capacity, streamed slices
    bits = synth.random_bits((n,), "f16", seed=71, tensor_id=1, std=2.0)
    x = to_dev(bits, "f16")
    assert F.fp8s_device_error() == 0
    seen = []
    try:
        F.fp8s_set_exchange_timeout_ns(1)
        # every CTA but the last to arrive spins; with a 1 ns limit at least
        # one of them gives up (a few tries guard against a call whose CTAs
        # all arrived within one tick of the timer)
        for _ in range(5):
            F.fp8_quantize_per_tensor(x)
            seen.append(F.fp8s_device_error())
            if seen[-1]:
                break
    finally:
        F.fp8s_set_exchange_timeout_ns(0)
    assert 4 in seen, f"no exchange spin ran out: {seen}"
    assert set(seen) <= {0, 4}
    q, s = F.fp8_quantize_per_tensor(x)
    torch.cuda.synchronize()
    assert F.fp8s_device_error() == 0
    oq, os_ = oracle.quantize_per_tensor(bits, "f16")
    assert host(s)[0] == np.float32(os_)
    assert np.array_equal(host(q), oq)
