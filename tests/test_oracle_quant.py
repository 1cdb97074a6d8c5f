"""Pins for the oracle's quantizers (per-tensor, 1x128 token group, 128x128
weight block).

Independent restatements use numpy's IEEE float32 divide and the brute-force
E4M3 rounding of test_oracle_codec; the invariants come straight from the
pages (the element equal to amax becomes +-448; nothing exceeds 448; groups
run along the input channels per token; blocks are 128x128).
"""
import numpy as np
import pytest

import synth
from test_oracle_codec import brute_nearest_e4m3


def f32(bits, dtype):
    return synth.bits_to_f32(bits, dtype)


def ref_scale(amax32):
    amax32 = np.asarray(amax32, np.float32)
    s = amax32 / np.float32(448.0)
    return np.where(amax32 == 0, np.float32(1.0), s).astype(np.float32)


def ref_quant(x32, s32):
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        return brute_nearest_e4m3((np.asarray(x32, np.float32) / np.asarray(s32, np.float32)).astype(np.float32))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_elementwise_step_all_inputs_many_scales(oracle, dtype):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = f32(bits, dtype)
    keep = np.isfinite(x)
    bits, x = bits[keep], x[keep]
    rng = np.random.default_rng(99)
    # scales as produced from amax values spread over the FP16/BF16 range
    lo, hi = (-24, 16) if dtype == "f16" else (-60, 60)
    amax = (2.0 ** rng.uniform(lo, hi, 150)).astype(np.float32)
    scales = ref_scale(amax)
    got = oracle.quantize_scales_grid(bits, dtype, scales)
    for j, s in enumerate(scales):
        assert np.array_equal(got[j], ref_quant(x, s)), f"scale {s!r}"


def test_amax_element_maps_to_448(oracle):
    rng = np.random.default_rng(5)
    for dtype in ("f16", "bf16"):
        # one 128-element group per trial; the largest |x| must encode to +-448
        for trial in range(300):
            mag = 2.0 ** (rng.uniform(-14, 13) if dtype == "f16" else rng.uniform(-100, 100))
            x32 = (rng.standard_normal(128) * mag).astype(np.float32)
            bits = synth.f32_to_bits(x32, dtype)
            xx = f32(bits, dtype)
            if not np.any(xx):
                continue
            q, sa = oracle.quantize_token_group(bits.reshape(1, 128), dtype)
            k = int(np.argmax(np.abs(xx)))
            assert q[0, k] in (0x7E, 0xFE)
            vals = oracle.e4m3_decode(q)
            assert np.all(np.abs(vals) <= 448.0)
            assert sa[0, 0] == ref_scale(np.abs(xx).max())


def test_per_tensor_matches_restatement(oracle):
    for dtype in ("f16", "bf16"):
        bits = synth.random_bits((37, 53), dtype, seed=11, tensor_id=1, std=3.0)
        q, s = oracle.quantize_per_tensor(bits, dtype)
        x = f32(bits, dtype)
        s_ref = ref_scale(np.abs(x).max())
        assert s == s_ref
        assert np.array_equal(q, ref_quant(x, s_ref))
        assert np.sum(np.isin(q, [0x7E, 0xFE])) >= 1


def test_token_group_layout_and_values(oracle):
    M, K = 5, 384
    for dtype in ("f16", "bf16"):
        bits = synth.random_bits((M, K), dtype, seed=12, tensor_id=2, std=2.0)
        # give each group a very different magnitude so a layout slip shows
        x = f32(bits, dtype) * (2.0 ** (np.arange(M * 3) - 7).reshape(M, 3, 1)).astype(np.float32).repeat(128, 2).reshape(M, K)
        bits = synth.f32_to_bits(x, dtype)
        x = f32(bits, dtype)
        q, sa = oracle.quantize_token_group(bits, dtype)
        assert sa.shape == (K // 128, M)
        for m in range(M):
            for g in range(K // 128):
                seg = x[m, g * 128:(g + 1) * 128]
                s = ref_scale(np.abs(seg).max())
                assert sa[g, m] == s
                assert np.array_equal(q[m, g * 128:(g + 1) * 128], ref_quant(seg, s))


def test_weight_block_layout_ragged_rows(oracle):
    N, K = 300, 256            # 3 row blocks, the last holds 44 rows
    for dtype in ("f16", "bf16"):
        bits = synth.random_bits((N, K), dtype, seed=13, tensor_id=3, std=0.02)
        x = f32(bits, dtype)
        # scale each block differently
        fac = (2.0 ** np.arange(6)).reshape(3, 1, 2, 1).astype(np.float32)
        xb = np.zeros((384, K), np.float32)
        xb[:N] = x
        xb = (xb.reshape(3, 128, 2, 128) * fac).reshape(384, K)[:N]
        bits = synth.f32_to_bits(xb, dtype)
        x = f32(bits, dtype)
        q, sb = oracle.quantize_weight_block(bits, dtype)
        assert sb.shape == (3, 2)
        for i in range(3):
            for j in range(2):
                blk = x[i * 128:min(N, i * 128 + 128), j * 128:(j + 1) * 128]
                s = ref_scale(np.abs(blk).max())
                assert sb[i, j] == s
                assert np.array_equal(q[i * 128:min(N, i * 128 + 128), j * 128:(j + 1) * 128], ref_quant(blk, s))


def test_all_zero_units_get_unit_scale(oracle):
    z = np.zeros((2, 256), np.uint16)
    z[1, :128] = 0x8000  # negative zeros in one group
    q, sa = oracle.quantize_token_group(z, "f16")
    assert np.all(sa == 1.0)
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0x80) and np.all(q[1, 128:] == 0)
    q, sb = oracle.quantize_weight_block(z, "bf16")
    assert np.all(sb == 1.0)
    q, s = oracle.quantize_per_tensor(np.zeros(10, np.uint16), "f16")
    assert s == 1.0 and np.all(q == 0)


def test_pseudocode_worked_example(oracle):
    """The per-tensor pseudocode on a 1x2 by 2x1 example worked by hand."""
    from conftest import read_golden
    rows = {r[0]: r[1:] for r in read_golden("pseudocode_worked_example.txt")}
    a = np.array([[float(v) for v in rows["a_f16"]]], np.float16).view(np.uint16)
    b_kxn = np.array([[float(v)] for v in rows["b_f16_kxn"]], np.float16)
    w = np.ascontiguousarray(b_kxn.T).view(np.uint16)      # weight layout [N, K]
    qa, sa = oracle.quantize_per_tensor(a, "f16")
    qw, sw = oracle.quantize_per_tensor(w, "f16")
    assert [int(c) for c in qa.ravel()] == [int(c, 16) for c in rows["a_codes"]]
    assert [int(c) for c in qw.ravel()] == [int(c, 16) for c in rows["b_codes"]]
    R = oracle.gemm_per_tensor(qa, sa, qw, sw)
    assert abs(R[0, 0] - float(rows["c"][0])) <= 3 * 2.0 ** -24 * 1.5
    assert np.float16(R[0, 0]) == np.float16(1.5)


# ------------------------------------------------- static / delayed scaling
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_elementwise_step_arbitrary_scales(oracle, dtype):
    """A static scale is any FP32 value, not fl32(amax/448): quotients then
    saturate (|x/s| > 448, including an FP32 overflow to inf), underflow to
    zero and land anywhere on the E4M3 grid."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = f32(bits, dtype)
    keep = np.isfinite(x)
    bits, x = bits[keep], x[keep]
    rng = np.random.default_rng(123)
    lo, hi = (-30, 20) if dtype == "f16" else (-120, 120)
    scales = (2.0 ** rng.uniform(lo, hi, 120)).astype(np.float32)
    scales = np.concatenate([scales, np.float32([2.0 ** -100, 2.0 ** 95, 0.125, 1.0, 3.0])])
    got = oracle.quantize_scales_grid(bits, dtype, scales)
    for j, s in enumerate(scales):
        assert np.array_equal(got[j], ref_quant(x, s)), f"scale {s!r}"
    # both saturation and underflow occur for the extreme scales
    assert np.all(np.isin(got[-5][np.abs(x) > 1e-20], [0x7E, 0xFE]))
    assert np.all(np.isin(got[-4][np.abs(x) < 2.0 ** 80], [0x00, 0x80]))


def _fl32_of_fraction(fr):
    """The FP32 value nearest to a positive Fraction, ties to even (found by
    bracketing with numpy's neighbours, independent of any float divide)."""
    from fractions import Fraction
    a = np.float32(float(fr))
    for _ in range(3):
        lo = np.nextafter(a, np.float32(0))
        hi = np.nextafter(a, np.float32(np.inf))
        cands = [lo, a, hi]
        d = [abs(Fraction(float(c)) - fr) for c in cands]
        best = min(d)
        picks = [c for c, dd in zip(cands, d) if dd == best]
        if len(picks) == 2:
            picks = [c for c in picks if (int(np.float32(c).view(np.uint32)) & 1) == 0]
        if picks[0] == a:
            return a
        a = picks[0]
    return a


def test_scale_from_history_closed_form(oracle):
    from fractions import Fraction
    cases = [([0.5, 3.0, 1.25], 0), ([0.5, 3.0, 1.25], 2), ([0.5, 3.0, 1.25], -3), ([7.0], 0),
             ([65504.0, 1.0], 1), ([1e-30, 0.0], 0), ([1e30, 2.5], -64), ([0.3, 0.7, 0.1, 0.7], 64)]
    for hist, margin in cases:
        h32 = np.float32(hist)
        m = max(Fraction(float(v)) for v in h32)
        s0 = _fl32_of_fraction(m / 448)
        want = Fraction(float(s0)) * Fraction(2) ** margin
        got = oracle.scale_from_history(h32, margin)
        assert Fraction(float(got)) == want, (hist, margin, got)


def test_scale_from_history_zero_window_and_order(oracle):
    assert oracle.scale_from_history(np.zeros(5, np.float32), 0) == np.float32(1.0)
    assert oracle.scale_from_history(np.zeros(5, np.float32), 3) == np.float32(8.0)
    rng = np.random.default_rng(4)
    h = (rng.random(64) * 100).astype(np.float32)
    a = oracle.scale_from_history(h, 1)
    assert a == oracle.scale_from_history(h[::-1].copy(), 1) == oracle.scale_from_history(np.sort(h), 1)
    # a window of one equals the dynamic scale of that amax
    bits = synth.random_bits((31, 17), "f16", seed=21, tensor_id=3, std=4.0)
    _, s_dyn = oracle.quantize_per_tensor(bits, "f16")
    assert oracle.scale_from_history(np.float32([oracle.amax(bits, "f16")]), 0) == s_dyn


def test_amax_matches_numpy(oracle):
    for dtype in ("f16", "bf16"):
        bits = synth.random_bits((3, 1001), dtype, seed=22, tensor_id=4, std=9.0)
        assert oracle.amax(bits, dtype) == np.abs(f32(bits, dtype)).max()


# ------------------------------------------------- per-channel weights
def test_per_channel_is_one_unit_per_row(oracle):
    for dtype in ("f16", "bf16"):
        N, K = 37, 640
        bits = synth.random_bits((N, K), dtype, seed=23, tensor_id=5, std=0.02)
        # rows of very different magnitude, one all-zero row
        scale_rows = (2.0 ** (np.arange(N) % 17 - 8)).astype(np.float32)   # 2^-8 .. 2^8
        x = f32(bits, dtype) * scale_rows[:, None]
        x[5] = 0.0
        bits = synth.f32_to_bits(x, dtype)
        xx = f32(bits, dtype)
        q, sb = oracle.quantize_per_channel(bits, dtype)
        want_s = ref_scale(np.abs(xx).max(axis=1))
        assert np.array_equal(sb, want_s)
        assert np.array_equal(q, ref_quant(xx, want_s[:, None]))
        assert sb[5] == 1.0 and not np.any(q[5] & 0x7F)


def test_per_channel_with_k128_is_the_token_group_quantizer(oracle):
    """With K = 128 a row is one 1x128 group: the per-channel quantizer must
    give the (pinned) token-group quantizer's bytes and scales."""
    bits = synth.random_bits((50, 128), "bf16", seed=24, tensor_id=6, std=3.0)
    q1, s1 = oracle.quantize_per_channel(bits, "bf16")
    q2, s2 = oracle.quantize_token_group(bits, "bf16")
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2[0])
