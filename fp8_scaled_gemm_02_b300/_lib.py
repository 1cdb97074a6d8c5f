"""ctypes binding of libfp8sgemm.so (the C ABI in include/fp8sgemm.h).

Argument marshalling only: every step of the quantize / GEMM path runs in the
library's CUDA kernels.  Loading fails loudly if the library is missing;
there is no fallback of any kind.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfp8sgemm.so")

FP8S_OK = 0
FP8S_ERR_CUDA = 5
STATUS_NAMES = {
    0: "FP8S_OK", 1: "FP8S_ERR_NULL", 2: "FP8S_ERR_SHAPE", 3: "FP8S_ERR_ALIGN", 4: "FP8S_ERR_DTYPE",
    5: "FP8S_ERR_CUDA", 6: "FP8S_ERR_DEVICE_TIMEOUT", 7: "FP8S_ERR_UNSUPPORTED_DEVICE",
}
FP8S_F16, FP8S_BF16 = 0, 1
FP8S_SCALE_PER_TENSOR, FP8S_SCALE_BLOCK, FP8S_SCALE_PER_CHANNEL, FP8S_SCALE_BLOCK_UE8M0 = 0, 1, 2, 3

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int

# name -> (restype, argtypes); mirrors include/fp8sgemm.h
SIGNATURES = {
    "fp8_quantize_per_tensor": (_I, [_P, _I, _I64, _P, _P, _P]),
    "fp8_quantize_per_tensor_static": (_I, [_P, _I, _I64, _P, _P, _P, _P]),
    "fp8_scale_from_amax_history": (_I, [_P, _I64, _I, _P, _P]),
    "fp8_quantize_token_group": (_I, [_P, _I, _I64, _I64, _P, _P, _P]),
    "fp8_quantize_weight_block": (_I, [_P, _I, _I64, _I64, _P, _P, _P]),
    "fp8_quantize_per_channel": (_I, [_P, _I, _I64, _I64, _P, _P, _P]),
    "fp8_gemm_scaled": (_I, [_P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _P]),
    "fp8_quantize_token_group_ue8m0": (_I, [_P, _I, _I64, _I64, _P, _P, _P]),
    "fp8_quantize_weight_block_ue8m0": (_I, [_P, _I, _I64, _I64, _P, _P, _P]),
    "fp8_linear_token_group": (_I, [_P, _I, _I64, _I64, _P, _P, _I64, _P, _P, _P, _P]),
    "fp8_e5m2_encode": (_I, [_P, _I, _I64, _P, _P]),
    "fp8_e5m2_decode": (_I, [_P, _I64, _P, _I, _P]),
    "fp8s_status_string": (ctypes.c_char_p, [_I]),
    "fp8s_last_cuda_error": (ctypes.c_char_p, []),
    "fp8s_device_error": (_I, [_P, ctypes.POINTER(_I)]),
    "fp8s_version": (_I, []),
    "fp8s_set_exchange_timeout_ns": (_I, [ctypes.c_ulonglong]),
    "fp8s_gemm_override": (_I, [_I, _I, _I]),
    "fp8s_gemm_plan": (_I, [_I64, _I64, _I64, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
}

_lib = None


class Fp8sError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = int(status)
        name = STATUS_NAMES.get(self.status, str(status))
        detail = status_string(self.status)
        if self.status == FP8S_ERR_CUDA:
            detail += f": {load().fp8s_last_cuda_error().decode()}"
        super().__init__(f"{where}: {name} ({detail})")


def load():
    """Load the library (once).  Raises ImportError when it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python fp8_scaled_gemm_02_b300/build.py`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().fp8s_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != FP8S_OK:
        raise Fp8sError(status, where)
