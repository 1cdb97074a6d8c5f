"""B300-native FP8 quantize + scaled-GEMM library (Python binding).

Functions carry the names of the C entry points in include/fp8sgemm.h and
only marshal torch tensors (device memory, current stream) into them:

  fp8_quantize_per_tensor(x)            -> (q, scale)        one FP32 scale
  fp8_quantize_per_tensor_static(x, scale [, amax])
                                        -> q                 given scale, one read of x
  fp8_scale_from_amax_history(history, margin)
                                        -> scale             delayed-scaling update
  fp8_quantize_token_group(x [M,K])     -> (q, sa [K/128,M]) 1x128 groups
  fp8_quantize_weight_block(w [N,K])    -> (q, sb [N/128,K/128]) 128x128 blocks
  fp8_quantize_per_channel(w [N,K])     -> (q, sb [N])       one scale per output channel
  fp8_gemm_scaled(qa, sa, qb, sb, ...)  -> C [M,N] FP16/BF16
  fp8_quantize_token_group_ue8m0(x)     -> (q, sa_code uint8 [K/128,M])   power-of-two scales
  fp8_quantize_weight_block_ue8m0(w)    -> (q, sb_code uint8 [N/128,K/128])
  fp8_linear_token_group(x, qw, sw)     -> C [M,N]         fused: x quantized inside the GEMM
  fp8_e5m2_encode(x) / fp8_e5m2_decode(q, dtype)
                                        E5M2 codec (5 exponent + 2 mantissa bits)

The path is the FP8 linear layer of "What is FP8 inference on H100
(Transformer Engine)?" s3 (amax -> scale = amax/448 -> x/scale rounded to
E4M3 -> FP32-accumulated GEMM -> rescale), with the fine-grained 1x128 /
128x128 scaling of the transformers "Fine-grained FP8" guide.
"""
import ctypes

import torch

from . import _lib
from ._lib import (FP8S_BF16, FP8S_F16, FP8S_SCALE_BLOCK, FP8S_SCALE_BLOCK_UE8M0, FP8S_SCALE_PER_CHANNEL,
                   FP8S_SCALE_PER_TENSOR, Fp8sError, check, load, status_string)

__all__ = [
    "fp8_quantize_per_tensor", "fp8_quantize_per_tensor_static", "fp8_scale_from_amax_history",
    "fp8_quantize_token_group", "fp8_quantize_per_channel", "fp8_quantize_weight_block", "fp8_gemm_scaled",
    "fp8_e5m2_encode", "fp8_e5m2_decode", "fp8_linear_token_group", "fp8_quantize_token_group_ue8m0", "fp8_quantize_weight_block_ue8m0",
    "fp8s_device_error", "fp8s_version", "fp8s_set_exchange_timeout_ns", "fp8s_gemm_override", "fp8s_gemm_plan", "Fp8sError", "status_string", "load", "LIB_PATH",
    "FP8S_F16", "FP8S_BF16", "FP8S_SCALE_PER_TENSOR", "FP8S_SCALE_BLOCK", "FP8S_SCALE_PER_CHANNEL",
    "FP8S_SCALE_BLOCK_UE8M0",
]

LIB_PATH = _lib.LIB_PATH
load()  # fail at import time if the CUDA library is missing

_DT = {torch.float16: FP8S_F16, torch.bfloat16: FP8S_BF16}
_MODE = {"per_tensor": FP8S_SCALE_PER_TENSOR, "block": FP8S_SCALE_BLOCK, "per_channel": FP8S_SCALE_PER_CHANNEL,
         "block_ue8m0": FP8S_SCALE_BLOCK_UE8M0}


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _in_dtype(t):
    if t.dtype not in _DT:
        raise TypeError(f"input must be float16 or bfloat16, got {t.dtype}")
    return _DT[t.dtype]


def _need_cuda(*ts):
    for t in ts:
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _need_f32(*ts):
    """Scales, amaxes and histories are read and written as raw FP32 words."""
    for t in ts:
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"scale / amax / history tensors must be float32, got {t.dtype}")


def _need_u8(*ts):
    """Byte outputs (E4M3 / E5M2 codes, UE8M0 scale codes)."""
    for t in ts:
        if t.dtype != torch.uint8 or not (t.is_cuda and t.is_contiguous()):
            raise TypeError(f"byte outputs must be contiguous uint8 CUDA tensors, got {t.dtype}")


def fp8_quantize_per_tensor(x, q=None, scale=None, stream=None):
    """x (any shape, FP16/BF16) -> (q uint8 same shape, scale float32 [1])."""
    _need_cuda(x)
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if q is None else q
    scale = torch.empty(4, dtype=torch.float32, device=x.device)[:1] if scale is None else scale
    st = load().fp8_quantize_per_tensor(_ptr(x), _in_dtype(x), x.numel(), _ptr(q), _ptr(scale), _stream(stream))
    check(st, "fp8_quantize_per_tensor")
    return q, scale


def fp8_quantize_per_tensor_static(x, scale, q=None, amax=None, stream=None):
    """x (any shape, FP16/BF16), scale float32 [1] on the device -> q uint8
    same shape, q = E4M3(fl32(x / scale)).  `amax` (a float32 CUDA tensor of
    which the first element is used, e.g. a slot of an amax-history ring)
    receives max|x|."""
    _need_cuda(x, scale)
    _need_f32(scale, amax)
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if q is None else q
    if amax is not None:
        _need_cuda(amax)
    st = load().fp8_quantize_per_tensor_static(_ptr(x), _in_dtype(x), x.numel(), _ptr(scale), _ptr(q),
                                               None if amax is None else _ptr(amax), _stream(stream))
    check(st, "fp8_quantize_per_tensor_static")
    return q


def fp8_scale_from_amax_history(history, margin=0, scale=None, stream=None):
    """history float32 [H] (recorded amaxes) -> scale float32 [1] =
    fl32(max(history) / 448) * 2**margin (1 * 2**margin when the max is 0)."""
    _need_cuda(history)
    _need_f32(history, scale)
    scale = torch.empty(4, dtype=torch.float32, device=history.device)[:1] if scale is None else scale
    st = load().fp8_scale_from_amax_history(_ptr(history), history.numel(), int(margin), _ptr(scale),
                                            _stream(stream))
    check(st, "fp8_scale_from_amax_history")
    return scale


def fp8_quantize_token_group(x, q=None, sa=None, stream=None):
    """x [M,K] FP16/BF16 -> (q uint8 [M,K], sa float32 [K/128, M])."""
    _need_cuda(x)
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device) if q is None else q
    sa = torch.empty((K // 128, M), dtype=torch.float32, device=x.device) if sa is None else sa
    st = load().fp8_quantize_token_group(_ptr(x), _in_dtype(x), M, K, _ptr(q), _ptr(sa), _stream(stream))
    check(st, "fp8_quantize_token_group")
    return q, sa


def fp8_quantize_weight_block(w, q=None, sb=None, stream=None):
    """w [N,K] FP16/BF16 -> (q uint8 [N,K], sb float32 [ceil(N/128), K/128])."""
    _need_cuda(w)
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device) if q is None else q
    sb = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=w.device) if sb is None else sb
    st = load().fp8_quantize_weight_block(_ptr(w), _in_dtype(w), N, K, _ptr(q), _ptr(sb), _stream(stream))
    check(st, "fp8_quantize_weight_block")
    return q, sb


def fp8_quantize_per_channel(w, q=None, sb=None, stream=None):
    """w [N,K] FP16/BF16 -> (q uint8 [N,K], sb float32 [N]): one scale per output channel."""
    _need_cuda(w)
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device) if q is None else q
    sb = torch.empty(N, dtype=torch.float32, device=w.device) if sb is None else sb
    _need_f32(sb)
    st = load().fp8_quantize_per_channel(_ptr(w), _in_dtype(w), N, K, _ptr(q), _ptr(sb), _stream(stream))
    check(st, "fp8_quantize_per_channel")
    return q, sb


def fp8_gemm_scaled(qa, sa, qb, sb, out_dtype=torch.bfloat16, mode="block", c=None, stream=None):
    """qa [M,K] uint8, qb [N,K] uint8 -> C [M,N] (FP16/BF16) = rescaled qa.qb^T.
    mode: "per_tensor" (sa, sb one float each), "block" (sa [K/128,M], sb
    [N/128,K/128]), "per_channel" (sa one float, sb [N]) or "block_ue8m0"
    (the block layout with uint8 UE8M0 codes, applied by the tensor core)."""
    _need_cuda(qa, sa, qb, sb)
    M, K = qa.shape
    N = qb.shape[0]
    if out_dtype not in _DT:
        raise TypeError("out_dtype must be float16 or bfloat16")
    c = torch.empty((M, N), dtype=out_dtype, device=qa.device) if c is None else c
    st = load().fp8_gemm_scaled(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), _ptr(c), _DT[c.dtype], M, N, K,
                                _MODE[mode], _stream(stream))
    check(st, "fp8_gemm_scaled")
    return c


def fp8_linear_token_group(x, qw, sw, c=None, qa=None, sa=None, stream=None):
    """Fused FP8 linear: x [M,K] FP16/BF16 (quantized per 1x128 token group
    inside the GEMM), qw [N,K] uint8 and sw [N/128,K/128] float32 from
    fp8_quantize_weight_block -> C [M,N] in x's dtype.  qa/sa (uint8 [M,K],
    float32 [K/128,M]) optionally receive the quantized activation."""
    _need_cuda(x, qw, sw)
    M, K = x.shape
    N = qw.shape[0]
    c = torch.empty((M, N), dtype=x.dtype, device=x.device) if c is None else c
    _need_cuda(c)
    if c.dtype != x.dtype:
        raise TypeError("the fused linear writes C in the activation's dtype")
    _need_f32(sw, sa)
    st = load().fp8_linear_token_group(_ptr(x), _in_dtype(x), M, K, _ptr(qw), _ptr(sw), N, _ptr(c),
                                       None if qa is None else _ptr(qa), None if sa is None else _ptr(sa),
                                       _stream(stream))
    check(st, "fp8_linear_token_group")
    return c


def fp8_quantize_token_group_ue8m0(x, q=None, sa=None, stream=None):
    """x [M,K] FP16/BF16 -> (q uint8 [M,K], sa uint8 [K/128, M] UE8M0 codes)."""
    _need_cuda(x)
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device) if q is None else q
    sa = torch.empty((K // 128, M), dtype=torch.uint8, device=x.device) if sa is None else sa
    _need_u8(q, sa)
    st = load().fp8_quantize_token_group_ue8m0(_ptr(x), _in_dtype(x), M, K, _ptr(q), _ptr(sa), _stream(stream))
    check(st, "fp8_quantize_token_group_ue8m0")
    return q, sa


def fp8_quantize_weight_block_ue8m0(w, q=None, sb=None, stream=None):
    """w [N,K] FP16/BF16 -> (q uint8 [N,K], sb uint8 [ceil(N/128), K/128] UE8M0 codes)."""
    _need_cuda(w)
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device) if q is None else q
    sb = torch.empty(((N + 127) // 128, K // 128), dtype=torch.uint8, device=w.device) if sb is None else sb
    _need_u8(q, sb)
    st = load().fp8_quantize_weight_block_ue8m0(_ptr(w), _in_dtype(w), N, K, _ptr(q), _ptr(sb), _stream(stream))
    check(st, "fp8_quantize_weight_block_ue8m0")
    return q, sb


def fp8_e5m2_encode(x, q=None, stream=None):
    """x (any shape, FP16/BF16) -> q uint8 same shape: E5M2 bytes, round to
    nearest even, saturating at +-57344."""
    _need_cuda(x)
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if q is None else q
    _need_cuda(q)
    st = load().fp8_e5m2_encode(_ptr(x), _in_dtype(x), x.numel(), _ptr(q), _stream(stream))
    check(st, "fp8_e5m2_encode")
    return q


def fp8_e5m2_decode(q, out_dtype=torch.float16, y=None, stream=None):
    """q uint8 E5M2 bytes (any shape) -> y FP16/BF16 same shape (exact)."""
    _need_cuda(q)
    if out_dtype not in _DT:
        raise TypeError("out_dtype must be float16 or bfloat16")
    y = torch.empty(q.shape, dtype=out_dtype, device=q.device) if y is None else y
    _need_cuda(y)
    st = load().fp8_e5m2_decode(_ptr(q), q.numel(), _ptr(y), _DT[y.dtype], _stream(stream))
    check(st, "fp8_e5m2_decode")
    return y


def fp8s_device_error(stream=None):
    """Synchronize and read/clear the device error word (0 = no wait expired)."""
    where = ctypes.c_int(0)
    st = load().fp8s_device_error(_stream(stream), ctypes.byref(where))
    if st not in (0, 6):
        check(st, "fp8s_device_error")
    return where.value


def fp8s_gemm_override(bn=0, splits=1, pair=False):
    """Force the GEMM tile width, split-K factor or CTA-pair tiles (bn=0: automatic choice)."""
    check(load().fp8s_gemm_override(int(bn), int(splits), int(bool(pair))), "fp8s_gemm_override")


def fp8s_gemm_plan(M, N, K, mode="block", sms=148):
    """(bn, splits, pair) that fp8_gemm_scaled picks for this shape (host only)."""
    bn, sp, pr = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    check(load().fp8s_gemm_plan(int(M), int(N), int(K), _MODE[mode], int(sms), ctypes.byref(bn), ctypes.byref(sp),
                                ctypes.byref(pr)), "fp8s_gemm_plan")
    return bn.value, sp.value, bool(pr.value)


def fp8s_set_exchange_timeout_ns(ns=0):
    """Test aid: the per-tensor quantizer's exchange-spin limit for inputs
    above ~29 MB (0 = the default 2 s)."""
    check(load().fp8s_set_exchange_timeout_ns(int(ns)), "fp8s_set_exchange_timeout_ns")


def fp8s_version():
    return load().fp8s_version()
