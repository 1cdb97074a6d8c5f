"""The C-ABI library loads, exports every entry point its header declares,
and rejects bad arguments on the host before touching the GPU (these calls
return before any CUDA call, so they run on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from fp8_scaled_gemm_02_b300 import build
    build.build()
    from fp8_scaled_gemm_02_b300 import _lib
    return _lib.load()


def declared_symbols():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            names += re.findall(r"FP8S_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_header_declares_the_four_calls():
    names = declared_symbols()
    for n in ("fp8_quantize_per_tensor", "fp8_quantize_token_group", "fp8_quantize_weight_block",
              "fp8_gemm_scaled"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 7
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_binding_covers_header(lib):
    from fp8_scaled_gemm_02_b300 import _lib
    assert set(declared_symbols()) == set(_lib.SIGNATURES)


def test_last_cuda_error_is_text(lib):
    """The diagnostic text is static storage, never NULL."""
    from fp8_scaled_gemm_02_b300 import _lib
    assert isinstance(_lib.load().fp8s_last_cuda_error(), bytes)


def test_status_strings_and_version(lib):
    from fp8_scaled_gemm_02_b300 import _lib
    for code in range(8):
        s = _lib.status_string(code)
        assert s and s != "unknown status"
    assert _lib.status_string(99) == "unknown status"
    assert lib.fp8s_version() >= 100


P = ctypes.c_void_p
GOOD = P(1 << 20)      # a 16-byte aligned non-null address; never dereferenced
BAD_ALIGN = P((1 << 20) + 8)


def test_quantize_argument_checks(lib):
    # dtype is checked first, then pointers, then sizes, then alignment
    assert lib.fp8_quantize_token_group(GOOD, 7, 128, 128, GOOD, GOOD, None) == 4
    assert lib.fp8_quantize_token_group(None, 0, 128, 128, GOOD, GOOD, None) == 1
    assert lib.fp8_quantize_token_group(GOOD, 0, 128, 100, GOOD, GOOD, None) == 2
    assert lib.fp8_quantize_token_group(GOOD, 0, 0, 128, GOOD, GOOD, None) == 2
    assert lib.fp8_quantize_token_group(GOOD, 0, 128, 128, BAD_ALIGN, GOOD, None) == 3
    assert lib.fp8_quantize_weight_block(GOOD, 1, 0, 128, GOOD, GOOD, None) == 2
    assert lib.fp8_quantize_weight_block(GOOD, 1, 5, 129, GOOD, GOOD, None) == 2
    assert lib.fp8_quantize_weight_block(GOOD, 1, 5, 128, GOOD, None, None) == 1
    assert lib.fp8_quantize_weight_block(BAD_ALIGN, 1, 5, 128, GOOD, GOOD, None) == 3
    assert lib.fp8_quantize_per_tensor(GOOD, 0, 0, GOOD, GOOD, None) == 2
    assert lib.fp8_quantize_per_tensor(GOOD, 2, 10, GOOD, GOOD, None) == 4
    assert lib.fp8_quantize_per_tensor(GOOD, 0, 10, GOOD, BAD_ALIGN, None) == 3


def test_per_channel_argument_checks(lib):
    pc = lib.fp8_quantize_per_channel
    assert pc(GOOD, 3, 4, 128, GOOD, GOOD, None) == 4
    assert pc(GOOD, 0, 4, 128, None, GOOD, None) == 1
    assert pc(GOOD, 0, 0, 128, GOOD, GOOD, None) == 2
    assert pc(GOOD, 0, 4, 12, GOOD, GOOD, None) == 2          # K % 8
    assert pc(GOOD, 0, 4, 65544, GOOD, GOOD, None) == 2       # a row must fit in 128 KB of shared memory
    assert pc(GOOD, 1, 4, 128, GOOD, BAD_ALIGN, None) == 3
    # the GEMM's per-channel mode: same shape rules as per-tensor (K % 16, not K % 128)
    g = lib.fp8_gemm_scaled
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 0, 8, 8, 24, 2, None) == 2
    assert g(GOOD, GOOD, GOOD, BAD_ALIGN, GOOD, 0, 8, 8, 32, 2, None) == 3
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 0, 8, 8, 32, 4, None) == 4          # no mode 4


def test_per_channel_plan_is_the_per_tensor_plan(lib):
    from fp8_scaled_gemm_02_b300 import fp8s_gemm_plan
    for M, N, K in [(128, 4096, 4096), (512, 2560, 2048), (4096, 22016, 4096), (64, 64, 128)]:
        assert fp8s_gemm_plan(M, N, K, "per_channel") == fp8s_gemm_plan(M, N, K, "per_tensor")


def test_static_scaling_argument_checks(lib):
    ALIGN4 = P((1 << 20) + 4)   # 4-byte but not 16-byte aligned: enough for single floats
    q_static = lib.fp8_quantize_per_tensor_static
    assert q_static(GOOD, 2, 64, GOOD, GOOD, None, None) == 4
    assert q_static(GOOD, 0, 64, None, GOOD, None, None) == 1
    assert q_static(None, 0, 64, GOOD, GOOD, None, None) == 1
    assert q_static(GOOD, 0, 0, GOOD, GOOD, None, None) == 2
    assert q_static(BAD_ALIGN, 0, 64, GOOD, GOOD, None, None) == 3
    assert q_static(GOOD, 0, 64, GOOD, BAD_ALIGN, None, None) == 3
    assert q_static(GOOD, 0, 64, P((1 << 20) + 2), GOOD, None, None) == 3
    assert q_static(GOOD, 0, 64, GOOD, GOOD, P((1 << 20) + 1), None) == 3
    hist = lib.fp8_scale_from_amax_history
    assert hist(None, 4, 0, GOOD, None) == 1
    assert hist(GOOD, 4, 0, None, None) == 1
    assert hist(GOOD, 0, 0, GOOD, None) == 2
    assert hist(GOOD, (1 << 24) + 1, 0, GOOD, None) == 2
    assert hist(GOOD, 4, 65, GOOD, None) == 2
    assert hist(GOOD, 4, -65, GOOD, None) == 2
    assert hist(P((1 << 20) + 2), 4, 0, ALIGN4, None) == 3
    assert hist(GOOD, 4, 0, P((1 << 20) + 6), None) == 3


def test_gemm_argument_checks(lib):
    g = lib.fp8_gemm_scaled
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 3, 1, 1, 16, 0, None) == 4          # out dtype
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 0, 1, 1, 16, 5, None) == 4          # scale mode
    assert g(GOOD, None, GOOD, GOOD, GOOD, 0, 1, 1, 16, 0, None) == 1
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 0, 0, 1, 16, 0, None) == 2          # M < 1
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 0, 1, 1, 24, 0, None) == 2          # K % 16
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 0, 1, 1, 144, 1, None) == 2         # block: K % 128
    assert g(GOOD, GOOD, GOOD, GOOD, BAD_ALIGN, 0, 1, 1, 16, 0, None) == 3


def test_oracle_is_not_linked_into_the_library(lib):
    """The product library neither exports nor imports any oracle symbol."""
    import subprocess
    from fp8_scaled_gemm_02_b300 import _lib
    out = subprocess.run(["nm", "-D", _lib.LIB_PATH], capture_output=True, text=True).stdout
    assert "oracle_" not in out
    src = open(os.path.join(ROOT, "fp8_scaled_gemm_02_b300", "__init__.py")).read()
    assert "oracle" not in src.replace("no fallback", "")


def test_gemm_override_argument_checks(lib):
    assert lib.fp8s_gemm_override(3, 1, 0) == 2
    assert lib.fp8s_gemm_override(256, 16, 0) == 2
    assert lib.fp8s_gemm_override(256, 8, 0) == 2     # split-K only up to bn = 192
    assert lib.fp8s_gemm_override(192, 8, 0) == 0
    assert lib.fp8s_gemm_override(128, 3, 0) == 2
    assert lib.fp8s_gemm_override(128, 4, 0) == 0
    assert lib.fp8s_gemm_override(128, 2, 1) == 2     # a pair does not also split K
    assert lib.fp8s_gemm_override(32, 1, 1) == 2      # a pair needs bn >= 64
    assert lib.fp8s_gemm_override(256, 1, 1) == 0
    assert lib.fp8s_gemm_override(192, 4, 0) == 0
    assert lib.fp8s_gemm_override(96, 1, 0) == 2
    assert lib.fp8s_gemm_override(0, 0, 0) == 0


def plan(lib, M, N, K, mode):
    bn, sp, pr = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    st = lib.fp8s_gemm_plan(M, N, K, mode, 148, ctypes.byref(bn), ctypes.byref(sp), ctypes.byref(pr))
    assert st == 0
    return bn.value, sp.value, pr.value


def test_gemm_plan_matches_measured_choices(lib):
    """The tile choice for the workloads' shapes is the configuration that
    measured fastest on the B300 in sweeps of every configuration."""
    BLOCK, PT = 1, 0
    assert plan(lib, 128, 4096, 4096, BLOCK) == (128, 4, 0)      # decode: split K over clusters of 4
    assert plan(lib, 128, 4096, 11008, BLOCK) == (128, 4, 0)
    assert plan(lib, 128, 22016, 4096, BLOCK) == (192, 1, 0)     # 115 tiles already fill the GPU
    assert plan(lib, 512, 2560, 2048, BLOCK) == (128, 1, 0)
    assert plan(lib, 4096, 22016, 4096, BLOCK) == (256, 1, 0)    # large: widest single-CTA tile
    assert plan(lib, 16384, 8192, 8192, PT) == (256, 1, 1)       # large per-tensor: CTA pairs
    assert plan(lib, 512, 2048, 2048, PT)[2] == 0                # no pair when it cannot pay for its start-up
    assert plan(lib, 512, 11264, 2048, PT) == (192, 1, 0)      # M = 512: single-CTA 17.7 us vs paired 19.8 us
    assert plan(lib, 4096, 12288, 4096, PT)[2] == 1             # from M = 1024 up pairs pay off
    bn, sp, pr = plan(lib, 64, 64, 128, PT)
    assert sp == 1 and pr == 0


def test_gemm_plan_decode_batches(lib):
    """Block mode with M <= 32 runs the transposed decode kernel: 128 output
    columns a tile, K split over the largest power-of-two cluster (<= 8) with
    tiles * splits <= 2 * SMs and at least one K block a CTA."""
    BLOCK, UE8 = 1, 3
    assert plan(lib, 1, 12288, 4096, BLOCK) == (128, 2, 0)     # 96 tiles: 192 CTAs
    assert plan(lib, 16, 4096, 4096, BLOCK) == (128, 8, 0)     # 32 tiles: 256 CTAs
    assert plan(lib, 32, 4096, 11008, BLOCK) == (128, 8, 0)
    assert plan(lib, 8, 22016, 4096, BLOCK) == (128, 1, 0)     # 172 tiles: no split
    assert plan(lib, 1, 100, 256, BLOCK) == (128, 2, 0)        # two K blocks: at most two splits
    assert plan(lib, 1, 100, 128, BLOCK) == (128, 1, 0)
    # UE8M0 mode has no decode kernel: the general kernel's plan at any M
    bn, sp, pr = plan(lib, 1, 4096, 4096, UE8)
    assert pr == 0 and bn in (32, 64, 128, 192, 256)


def test_gemm_plan_argument_checks(lib):
    bn, sp, pr = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    args = (ctypes.byref(bn), ctypes.byref(sp), ctypes.byref(pr))
    assert lib.fp8s_gemm_plan(128, 128, 100, 1, 148, *args) == 2   # block mode needs K % 128 == 0
    assert lib.fp8s_gemm_plan(0, 128, 128, 1, 148, *args) == 2
    assert lib.fp8s_gemm_plan(128, 128, 128, 5, 148, *args) == 4
    assert lib.fp8s_gemm_plan(128, 128, 128, 1, 0, *args) == 2
    assert lib.fp8s_gemm_plan(128, 128, 128, 1, 148, None, *args[1:]) == 1


def test_e5m2_argument_checks(lib):
    enc, dec = lib.fp8_e5m2_encode, lib.fp8_e5m2_decode
    assert enc(GOOD, 2, 64, GOOD, None) == 4
    assert enc(None, 0, 64, GOOD, None) == 1
    assert enc(GOOD, 0, 0, GOOD, None) == 2
    assert enc(GOOD, 1, 64, BAD_ALIGN, None) == 3
    assert dec(GOOD, 64, GOOD, 5, None) == 4
    assert dec(GOOD, 64, None, 0, None) == 1
    assert dec(GOOD, -1, GOOD, 0, None) == 2
    assert dec(BAD_ALIGN, 64, GOOD, 1, None) == 3


def test_ue8m0_argument_checks(lib):
    tg, wb = lib.fp8_quantize_token_group_ue8m0, lib.fp8_quantize_weight_block_ue8m0
    assert tg(GOOD, 2, 4, 128, GOOD, GOOD, None) == 4
    assert tg(GOOD, 0, 4, 128, GOOD, None, None) == 1
    assert tg(GOOD, 0, 4, 200, GOOD, GOOD, None) == 2
    assert tg(GOOD, 0, 4, 128, GOOD, BAD_ALIGN, None) == 3
    assert wb(GOOD, 1, 0, 128, GOOD, GOOD, None) == 2
    assert wb(GOOD, 1, 5, 128, None, GOOD, None) == 1
    assert wb(GOOD, 1, 5, 256, GOOD, BAD_ALIGN, None) == 3
    g = lib.fp8_gemm_scaled
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 0, 8, 8, 144, 3, None) == 2      # UE8M0 block mode: K % 128
    assert g(GOOD, GOOD, GOOD, GOOD, BAD_ALIGN, 1, 8, 8, 128, 3, None) == 3
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 0, 8, 8, 128, 4, None) == 4


def test_ue8m0_plan_has_no_cta_pairs(lib):
    """The UE8M0 mode stages its scale factors per CTA: never a CTA pair,
    and split-K only up to 192-wide tiles."""
    for M, N, K in [(16384, 8192, 8192), (4096, 22016, 4096), (128, 4096, 4096), (1, 4096, 11008)]:
        bn, sp, pr = plan(lib, M, N, K, 3)
        assert pr == 0 and (sp == 1 or bn <= 192)


def test_exchange_timeout_setter(lib):
    assert lib.fp8s_set_exchange_timeout_ns(5) == 0
    assert lib.fp8s_set_exchange_timeout_ns(0) == 0
