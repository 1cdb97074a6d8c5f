"""Exhaustive check of the quantizers' division: every pair of FP16 (and of
BF16) magnitudes |x| <= amax is quantized once, inside a 1x128 group whose
amax is that amax, through the token-group entry point, and the E4M3 bytes
and FP32 scales must equal the oracle's bit for bit.

Why these pairs are all the inputs there are: a quantization unit's scale
depends only on its amax, s = fl32(amax / 448), and every element of the
unit has |x| <= amax, so the byte of an element is a function of the pair
(|x|, amax) and the sign of x.  The quantizers derive the byte from a
reciprocal multiply with one refinement step rather than a per-element
divide ("What is FP8 inference on H100 (Transformer Engine)?", s3 step 3
fixes the quotient fl32(x / s) and its E4M3 rounding); this test is what
shows that shortcut never changes a byte.  The weight-block and per-tensor
quantizers share the same per-element code with the token-group kernel.

Group layout: slot 0 holds the amax pattern, slots 1..127 list the next 127
magnitudes x = 0, 1, 2, ... (patterns), padded with the amax itself after x
reaches it; signs alternate over slots and groups, so both signs and -0
occur."""
import numpy as np
import pytest

import oracle

F = pytest.importorskip("fp8_scaled_gemm_02_b300")

TOP = {"f16": 0x7BFF, "bf16": 0x7F7F}  # largest finite magnitude pattern
PER = 127                               # x values per group (slot 0 is the amax)


def pair_groups(a_lo, a_hi):
    """Groups covering every pair (a, x), a in [a_lo, a_hi], 0 <= x <= a
    (patterns), as a uint16 array [groups, 128]."""
    a = np.arange(a_lo, a_hi + 1, dtype=np.int64)
    n_g = (a + 1 + PER - 1) // PER
    ga = np.repeat(a, n_g)
    first = np.repeat(np.cumsum(n_g) - n_g, n_g)
    k = np.arange(len(ga), dtype=np.int64) - first  # group index within its amax
    xs = np.minimum(k[:, None] * PER + np.arange(PER, dtype=np.int64)[None, :], ga[:, None])
    g = np.empty((len(ga), 128), np.uint16)
    g[:, 0] = ga
    g[:, 1:] = xs
    sign = ((np.arange(128)[None, :] + np.arange(len(ga))[:, None]) & 1).astype(np.uint16) << np.uint16(15)
    return g | sign


def amax_chunks(top, max_groups):
    """Splits [1, top] into consecutive amax ranges of at most max_groups groups."""
    out, lo, acc = [], 1, 0
    for a in range(1, top + 1):
        n = (a + 1 + PER - 1) // PER
        if acc + n > max_groups and a > lo:
            out.append((lo, a - 1))
            lo, acc = a, 0
        acc += n
    out.append((lo, top))
    return out


def test_pair_groups_cover_every_pair():
    """Host-side pin of the layout: each (a, x) with 0 <= x <= a appears,
    and nothing exceeds its group's amax."""
    g = pair_groups(1, 700) & np.uint16(0x7FFF)
    a = g[:, 0].astype(np.int64)
    assert np.all(g[:, 1:] <= g[:, :1])
    seen = set()
    for row, am in zip(g, a):
        for x in row[1:]:
            seen.add((int(am), int(x)))
    assert seen == {(am, x) for am in range(1, 701) for x in range(am + 1)}
    chunks = amax_chunks(700, 300)
    assert chunks[0][0] == 1 and chunks[-1][1] == 700
    assert all(b + 1 == c for (_, b), (c, _) in zip(chunks, chunks[1:]))


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_every_amax_x_pair(dtype):
    from gpu_util import host, to_dev

    total = 0
    for lo, hi in amax_chunks(TOP[dtype], 1 << 20):
        bits = pair_groups(lo, hi)
        # pad the group count to a multiple of 4 with copies of the first group
        pad = (-len(bits)) % 4
        if pad:
            bits = np.concatenate([bits, np.repeat(bits[:1], pad, axis=0)])
        qa, sa = F.fp8_quantize_token_group(to_dev(bits, dtype))
        oq, osa = oracle.quantize_token_group(bits, dtype)
        q, s = host(qa), host(sa)
        assert np.array_equal(s.view(np.uint32), osa.view(np.uint32)), f"scales differ for amax {lo:#x}..{hi:#x}"
        bad = np.argwhere(q != oq)
        assert bad.size == 0, (f"{len(bad)} bytes differ for amax {lo:#x}..{hi:#x}; first (group, slot) "
                               f"{bad[:3].tolist()}, patterns {[hex(int(bits[i, j])) for i, j in bad[:3]]}")
        total += len(bits) * PER
    assert total >= (TOP[dtype] * (TOP[dtype] + 1)) // 2
