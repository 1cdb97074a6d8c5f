"""CPU oracle for the FP8 quantize + scaled-GEMM path (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package.  It shares no code with the CUDA path: the arithmetic lives in
``fp8_oracle.c`` (plain C, FP64 GEMM, integer-exact E4M3 rounding) and this
module only marshals numpy arrays into it.

Every function follows the steps of "What is FP8 inference on H100
(Transformer Engine)?" s3 (amax, scale = amax/448, x/scale rounded to E4M3,
FP32-or-better accumulation, rescale by scale_A*scale_B) and the block
geometry of the transformers "Fine-grained FP8" guide (1x128 token groups,
128x128 weight blocks).  See the C source for the readings taken where the
pages are silent.

Inputs are raw 16-bit patterns (``np.uint16``) with a dtype tag "f16"/"bf16".
"""
import ctypes
import os

import numpy as np

from . import build as _build

F16, BF16 = 0, 1
_DT = {"f16": F16, "fp16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16}

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        F = ctypes.c_float
        sig = {
            "oracle_set_threads": (None, [I]),
            "oracle_get_threads": (I, []),
            "oracle_half_to_float": (F, [ctypes.c_uint16]),
            "oracle_bf16_to_float": (F, [ctypes.c_uint16]),
            "oracle_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_e4m3_units": (I64, [ctypes.c_uint8]),
            "oracle_e4m3_encode": (ctypes.c_uint8, [F]),
            "oracle_quantize_per_tensor": (None, [P, I, I64, P, P]),
            "oracle_quantize_token_group": (None, [P, I, I64, I64, P, P]),
            "oracle_quantize_weight_block": (None, [P, I, I64, I64, P, P]),
            "oracle_gemm_per_tensor": (None, [P, F, P, F, I64, I64, P, I64, P]),
            "oracle_gemm_block": (None, [P, P, I64, P, P, I64, I64, P, I64, P]),
            "oracle_dot_units": (None, [P, P, I64, I64, I64, I64, I64, P]),
            "oracle_e4m3_decode_array": (None, [P, I64, P]),
            "oracle_e4m3_encode_array": (None, [P, I64, P]),
            "oracle_to_float_array": (None, [P, I, I64, P]),
            "oracle_quantize_with_scale": (None, [P, I, I64, F, P]),
            "oracle_quantize_scales_grid": (None, [P, I, I64, P, I64, P]),
            "oracle_scale_from_history": (F, [P, I64, I]),
            "oracle_quantize_per_channel": (None, [P, I, I64, I64, P, P]),
            "oracle_ue8m0_decode": (F, [ctypes.c_uint8]),
            "oracle_e5m2_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_e5m2_encode_array": (None, [P, I64, P]),
            "oracle_ue8m0_of_amax": (ctypes.c_uint8, [F]),
            "oracle_quantize_token_group_ue8m0": (None, [P, I, I64, I64, P, P]),
            "oracle_quantize_weight_block_ue8m0": (None, [P, I, I64, I64, P, P]),
            "oracle_gemm_per_channel": (None, [P, F, P, P, I64, I64, P, I64, P]),
            "oracle_amax": (F, [P, I, I64]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _dt(dtype) -> int:
    return _DT[str(dtype)]


def _u16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, "inputs are raw 16-bit patterns (np.uint16)"
    return x


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


# ------------------------------------------------------------------ codecs
def half_to_float(h) -> np.ndarray:
    h = _u16(h)
    out = np.empty(h.shape, np.float32)
    _load().oracle_to_float_array(_ptr(h), F16, h.size, _ptr(out))
    return out


def bf16_to_float(h) -> np.ndarray:
    h = _u16(h)
    out = np.empty(h.shape, np.float32)
    _load().oracle_to_float_array(_ptr(h), BF16, h.size, _ptr(out))
    return out


def to_float(h, dtype) -> np.ndarray:
    return bf16_to_float(h) if _dt(dtype) == BF16 else half_to_float(h)


def e4m3_decode(codes) -> np.ndarray:
    """O1: E4M3 byte -> exact value (float64)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_units(code: int) -> int:
    """Exact integer count of 2^-9 units of one E4M3 code."""
    return int(_load().oracle_e4m3_units(int(code)))


def e4m3_encode(y) -> np.ndarray:
    """O2: binary32 -> E4M3 byte (RNE, saturating, sign-preserving)."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(y), y.size, _ptr(out))
    return out


# -------------------------------------------------------------- quantizers
def quantize_per_tensor(x, dtype):
    """O3 per-tensor: returns (q uint8 same shape, scale float32 scalar)."""
    x = _u16(x)
    q = np.empty(x.shape, np.uint8)
    s = np.zeros(1, np.float32)
    _load().oracle_quantize_per_tensor(_ptr(x), _dt(dtype), x.size, _ptr(q), _ptr(s))
    return q, s[0]


def quantize_token_group(x, dtype):
    """O3 per token per 128-channel group: x [M,K] -> (q [M,K], sa [K/128, M])."""
    x = _u16(x)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), np.uint8)
    sa = np.empty((K // 128, M), np.float32)
    _load().oracle_quantize_token_group(_ptr(x), _dt(dtype), M, K, _ptr(q), _ptr(sa))
    return q, sa


def quantize_weight_block(w, dtype):
    """O3 per 128x128 block: w [N,K] -> (q [N,K], sb [ceil(N/128), K/128])."""
    w = _u16(w)
    N, K = w.shape
    assert K % 128 == 0
    q = np.empty((N, K), np.uint8)
    sb = np.empty(((N + 127) // 128, K // 128), np.float32)
    _load().oracle_quantize_weight_block(_ptr(w), _dt(dtype), N, K, _ptr(q), _ptr(sb))
    return q, sb


def quantize_per_channel(w, dtype):
    """O3 per output channel (one scale per row of W, "What is FP8 inference
    on H100" s5): w [N,K] -> (q [N,K], sb [N])."""
    w = _u16(w)
    N, K = w.shape
    q = np.empty((N, K), np.uint8)
    sb = np.empty(N, np.float32)
    _load().oracle_quantize_per_channel(_ptr(w), _dt(dtype), N, K, _ptr(q), _ptr(sb))
    return q, sb


def e5m2_decode(codes) -> np.ndarray:
    """E5M2 codes (5 exponent + 2 mantissa bits, bias 15) -> float64."""
    c = np.asarray(codes, np.uint8)
    lib = _load()
    return np.array([lib.oracle_e5m2_decode(int(v)) for v in c.ravel()], np.float64).reshape(c.shape)


def e5m2_encode(y) -> np.ndarray:
    """float32 -> E5M2 codes, round to nearest even, saturating at +-57344."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.shape, np.uint8)
    _load().oracle_e5m2_encode_array(_ptr(y), y.size, _ptr(out))
    return out


def ue8m0_decode(codes) -> np.ndarray:
    """UE8M0 scale codes -> float32 values 2^(c - 127) (255 -> NaN)."""
    c = np.asarray(codes, np.uint8)
    lib = _load()
    return np.array([lib.oracle_ue8m0_decode(int(v)) for v in c.ravel()], np.float32).reshape(c.shape)


def ue8m0_of_amax(amax) -> int:
    """The UE8M0 code of the power-of-two scale for an amax: fl32(amax/448)
    rounded up to a power of two (1 when amax == 0), clamped to 2^-127."""
    return int(_load().oracle_ue8m0_of_amax(float(np.float32(amax))))


def quantize_token_group_ue8m0(x, dtype):
    """Token-group quantizer with UE8M0 scales: x [M,K] -> (q [M,K], codes [K/128, M])."""
    x = _u16(x)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), np.uint8)
    c = np.empty((K // 128, M), np.uint8)
    _load().oracle_quantize_token_group_ue8m0(_ptr(x), _dt(dtype), M, K, _ptr(q), _ptr(c))
    return q, c


def quantize_weight_block_ue8m0(w, dtype):
    """Weight-block quantizer with UE8M0 scales: w [N,K] -> (q [N,K], codes [ceil(N/128), K/128])."""
    w = _u16(w)
    N, K = w.shape
    assert K % 128 == 0
    q = np.empty((N, K), np.uint8)
    c = np.empty(((N + 127) // 128, K // 128), np.uint8)
    _load().oracle_quantize_weight_block_ue8m0(_ptr(w), _dt(dtype), N, K, _ptr(q), _ptr(c))
    return q, c


def quantize_with_scale(x, dtype, s) -> np.ndarray:
    """The elementwise quantizer step E4M3(fl32(x / s)) for a given scale."""
    x = _u16(x)
    q = np.empty(x.shape, np.uint8)
    _load().oracle_quantize_with_scale(_ptr(x), _dt(dtype), x.size, float(np.float32(s)), _ptr(q))
    return q


def amax(x, dtype) -> np.float32:
    """max|x| over all elements, as FP32 (exact)."""
    x = _u16(x)
    return np.float32(_load().oracle_amax(_ptr(x), _dt(dtype), x.size))


def scale_from_history(history, margin=0) -> np.float32:
    """Delayed scaling: fl32(max(history) / 448) * 2**margin (1 * 2**margin
    when the max is 0), the recipe of "Technical assignment: implement FP8
    inference on H100" stage 3 step 1 (DelayedScaling(margin, interval))."""
    h = np.ascontiguousarray(history, dtype=np.float32).ravel()
    return np.float32(_load().oracle_scale_from_history(_ptr(h), h.size, int(margin)))


def quantize_scales_grid(x, dtype, scales) -> np.ndarray:
    """q[j, i] = E4M3(fl32(x[i] / scales[j])) for 1-D x."""
    x = _u16(x).ravel()
    s = np.ascontiguousarray(scales, dtype=np.float32).ravel()
    q = np.empty((s.size, x.size), np.uint8)
    _load().oracle_quantize_scales_grid(_ptr(x), _dt(dtype), x.size, _ptr(s), s.size, _ptr(q))
    return q


# -------------------------------------------------------------------- GEMM
def _rows(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(rows, dtype=np.int64)
    assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < M))
    return r, r.size


def gemm_per_tensor(qa, sa, qb, sb, rows=None) -> np.ndarray:
    """O4 per-tensor: R = (dec(qa) @ dec(qb)^T) * sa * sb in float64.

    qa [M,K] and qb [N,K] uint8; sa, sb scalars.  ``rows`` selects a subset
    of output rows (sampled parity at full sizes)."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    M, K = qa.shape
    N, K2 = qb.shape
    assert K == K2
    r, nr = _rows(rows, M)
    R = np.empty((nr, N), np.float64)
    _load().oracle_gemm_per_tensor(_ptr(qa), float(np.float32(sa)), _ptr(qb), float(np.float32(sb)),
                                   N, K, None if r is None else _ptr(r), nr, _ptr(R))
    return R


def gemm_per_channel(qa, sa, qb, sb, rows=None) -> np.ndarray:
    """O4 per-channel weights: R = (dec(qa) @ dec(qb)^T) * sa * sb[n] in float64
    (sa a scalar, sb [N])."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sb = np.ascontiguousarray(sb, dtype=np.float32).ravel()
    M, K = qa.shape
    N, K2 = qb.shape
    assert K == K2 and sb.size == N
    r, nr = _rows(rows, M)
    R = np.empty((nr, N), np.float64)
    _load().oracle_gemm_per_channel(_ptr(qa), float(np.float32(sa)), _ptr(qb), _ptr(sb), N, K,
                                    None if r is None else _ptr(r), nr, _ptr(R))
    return R


def gemm_block(qa, sa, qb, sb, rows=None) -> np.ndarray:
    """O4 block-scaled: R = sum_kb sa[kb,m] * sb[n//128,kb] * (partial over kb)."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    M, K = qa.shape
    N, K2 = qb.shape
    assert K == K2 and K % 128 == 0
    assert sa.shape == (K // 128, M) and sb.shape == ((N + 127) // 128, K // 128)
    r, nr = _rows(rows, M)
    R = np.empty((nr, N), np.float64)
    _load().oracle_gemm_block(_ptr(qa), _ptr(sa), M, _ptr(qb), _ptr(sb), N, K,
                              None if r is None else _ptr(r), nr, _ptr(R))
    return R


def dot_units(qa, qb, k0=0, k1=None) -> np.ndarray:
    """Exact int64 sums of units(qa)*units(qb) over k in [k0, k1), in 2^-18."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    M, K = qa.shape
    N, _ = qb.shape
    k1 = K if k1 is None else k1
    out = np.empty((M, N), np.int64)
    _load().oracle_dot_units(_ptr(qa), _ptr(qb), M, N, K, k0, k1, _ptr(out))
    return out


def within_tolerance(C, R, out_dtype):
    """The parity bar for GEMM outputs, against the unrounded FP64 result R:
        FP16 output:  |C - R| <= 1e-3*|R| + 1e-3*rms(R)
        BF16 output:  |C - R| <= 2e-3*|R| + 2e-3*rms(R) + ulp_bf16(R)/2
    The BF16 half-ulp term is the error of rounding R itself to BF16 to
    nearest (up to 2^-8*|R|, more than 2e-3*|R|), which no implementation can
    avoid; FP16's half-ulp (<= 2^-11*|R|) already fits inside its bound.
    Returns (ok, worst error / bound)."""
    bf16 = _dt(out_dtype) == BF16
    t = 2e-3 if bf16 else 1e-3
    C = np.asarray(C, np.float64)
    R = np.asarray(R, np.float64)
    if R.size == 0:
        return True, 0.0
    rms = float(np.sqrt(np.mean(R * R)))
    bound = t * np.abs(R) + t * rms
    if bf16:
        _, e = np.frexp(R)                       # |R| = f * 2^e, f in [0.5, 1)
        bound = bound + np.ldexp(1.0, np.maximum(e, -125) - 9)   # half of 2^(e-1-7)
    err = np.abs(C - R)
    ratio = float(np.max(err / np.maximum(bound, 1e-300)))
    return bool(np.all(err <= bound)), ratio
