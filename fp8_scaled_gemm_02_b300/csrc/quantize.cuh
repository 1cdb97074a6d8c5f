// quantize.cuh -- E4M3 quantization kernels: dynamic per tensor, per 1x128
// token group, per 128x128 weight block and per output channel; per tensor
// with a given (static or delayed) scale.
//
// Method ("What is FP8 inference on H100 (Transformer Engine)?", s3 steps
// 2-4): amax = max|x| over the unit, s = fl32(amax / 448) (1 when amax == 0),
// q = E4M3_rne_satfinite(fl32(x / s)).  Units are the whole tensor, a group
// of 128 input channels of one token, a 128x128 weight block (the
// transformers "Fine-grained FP8" guide, opening bullets) or one output
// channel of a weight ("What is FP8 inference on H100", s5: per-channel
// scaling for weights).
//
// All kernels stream 16-byte vectors (8 FP16/BF16 elements) and keep the
// arithmetic bit-exact with IEEE single precision:
//  * amax is taken on the 16-bit patterns: with the sign bit cleared,
//    finite FP16/BF16 magnitudes order exactly like unsigned integers, so a
//    packed 16-bit unsigned max (__vmaxu2) is an exact max.
//  * the E4M3 byte of fl32(x / s) is obtained without a per-element divide.
//    Once per unit: y = RN(1/s), and ylo = RN(r*y) with the residual
//    r = 1 - s*y (exact through an FMA), so that y + ylo is 1/s to about
//    2^-47 (a double-word reciprocal: the FMA residual correction of
//    P. Markstein, "Computation of elementary functions on the IBM RISC
//    System/6000 processor", IBM J. Res. Dev. 34(1), 1990; see also Muller
//    et al., "Handbook of Floating-Point Arithmetic", division with an FMA).  Per element: q = RN(x*y + RN(x*ylo))
//    (a multiply and an FMA, two elements at a time with the packed .f32x2
//    instructions).  q can differ from fl32(x/s) in the last place, but
//    never across an E4M3 rounding boundary: for every pair of FP16 or BF16
//    magnitudes |x| <= amax (about 5 * 10^8 of each) the byte cvt(q) equals
//    cvt(fl32(x/s)), which an exhaustive test checks through the
//    token-group entry point against the oracle.  (RN(x*y) alone is not
//    enough: it differs at about 5 in 10^5 pairs, where x/s lies on or next
//    to an E4M3 midpoint.)  Elements never exceed their unit's amax, so
//    these pairs are every input the quantizers can see.
//    The sign of a zero quotient can come out wrong (x = -0 with ylo > 0
//    gives -0 + +0 = +0), and the E4M3 code of -0/s is 0x80: so the input's
//    sign bit is OR-ed into every code, which changes nothing else (a
//    negative non-zero quotient already has its sign bit, including one
//    that rounds to zero).  Units whose scale is tiny (s < 2^-90, possible
//    only for BF16 inputs below about 2^-81) use the IEEE divide __fdiv_rn.
//  * the E4M3 rounding is the hardware cvt.rn.satfinite.e4m3x2.f32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace fp8s {

enum : int { kInF16 = 0, kInBF16 = 1 };

// Device error word shared by every kernel of the library (first writer wins).
__device__ unsigned int g_fp8s_error;
enum : unsigned { kErrProducer = 1, kErrMma = 2, kErrEpilogue = 3, kErrQuant = 4 };
__device__ __forceinline__ void record_error(unsigned code) { atomicCAS(&g_fp8s_error, 0u, code); }
__device__ __forceinline__ void record_quant_error() { record_error(kErrQuant); }

// Two packed 16-bit values (low half first) -> two floats.  Exact.
template <int DT>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (DT == kInF16) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
  } else {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
}

// One 16-bit magnitude pattern -> float.  Exact.
template <int DT>
__device__ __forceinline__ float mag_to_float(uint32_t h) {
  if constexpr (DT == kInF16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
  } else {
    return __uint_as_float(h << 16);
  }
}

// Largest magnitude pattern among the 8 elements of a 16-byte vector.
__device__ __forceinline__ uint32_t amax_bits8(const uint4& v) {
  const uint32_t k = 0x7FFF7FFFu;
  uint32_t m = __vmaxu2(__vmaxu2(v.x & k, v.y & k), __vmaxu2(v.z & k, v.w & k));
  return max(m & 0xFFFFu, m >> 16);
}

// The quotient x / s of one quantization unit, to E4M3 precision (see the
// file comment).
struct UnitScale {
  float s;     // dequant factor written to memory
  float y;     // RN(1/s)
  float ylo;   // RN((1 - s*y) * y): 1/s ~ y + ylo to about 2^-47
  bool exact_div;

  __device__ __forceinline__ UnitScale() : s(1.0f), y(1.0f), ylo(0.0f), exact_div(false) {}
  __device__ __forceinline__ UnitScale(float s_, float y_, bool e_) : s(s_), y(y_), exact_div(e_) {
    ylo = __fmul_rn(__fmaf_rn(-s, y, 1.0f), y);
  }
  __device__ __forceinline__ explicit UnitScale(float amax) {
    s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
    y = __frcp_rn(s);
    ylo = __fmul_rn(__fmaf_rn(-s, y, 1.0f), y);  // the residual 1 - s*y is exact (FMA)
    exact_div = !(s >= 0x1p-90f);
  }

  // q = RN(x*y + RN(x*ylo)): x times the double-word reciprocal y + ylo,
  // valid when !exact_div.  For every FP16 and BF16 pair |x| <= amax this q
  // rounds to the same E4M3 byte as the IEEE quotient fl32(x/s) (checked
  // exhaustively over all such pairs; with RN(x*y) alone about 5 in 10^5
  // pairs differ, at quotients on or next to an E4M3 rounding midpoint).
  __device__ __forceinline__ float div_fast(float x) const { return __fmaf_rn(x, y, __fmul_rn(x, ylo)); }

  __device__ __forceinline__ float div_exact(float x) const { return __fdiv_rn(x, s); }
};

// Two packed 16-bit inputs -> {x_lo, x_hi} as an FP32 pair.  Exact.
template <int DT>
__device__ __forceinline__ uint64_t unpack2_f2(uint32_t w) {
  if constexpr (DT == kInF16) {
    const float2 f = unpack2<DT>(w);
    return ptx::f2_pack(f.x, f.y);
  } else {
    return ptx::f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
}

// The unit's reciprocal words as FP32 pairs: {y, y} and {ylo, ylo}.
struct UnitPair {
  uint64_t yy, ll;
  __device__ __forceinline__ explicit UnitPair(const UnitScale& us)
      : yy(ptx::f2_pack(us.y, us.y)), ll(ptx::f2_pack(us.ylo, us.ylo)) {}
};

// Power-of-two (UE8M0) scales (the "UE8M0 scale format" section of the
// transformers "Fine-grained FP8" guide: such checkpoints store each scale
// as an 8-bit biased exponent).  The unit's FP32 scale fl32(amax / 448) (1
// when amax == 0) is rounded up to the nearest power of two 2^k (the smallest
// with 2^k >= it; k >= -127, the smallest UE8M0 value), stored as the byte
// k + 127.  Then 1/s = 2^-k is exact, so x * 2^-k is the correctly rounded
// quotient fl32(x / s) itself, and the double-word reciprocal's low word is
// zero: the same element path computes RN(x * 2^-k).
__device__ __forceinline__ UnitScale ue8m0_unit(float amax, uint32_t* code) {
  const float s32 = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
  const uint32_t b = __float_as_uint(s32);
  const int e = static_cast<int>(b >> 23);
  const uint32_t m = b & 0x7FFFFFu;
  // a subnormal s32 lies in (0, 2^-126): 2^-126 covers it if it exceeds
  // 2^-127 (mantissa above 2^22), else the clamp at 2^-127 applies
  const int k = e == 0 ? (m > (1u << 22) ? -126 : -127) : e - 127 + (m != 0u ? 1 : 0);
  *code = static_cast<uint32_t>(k + 127);
  // 2^k (k = -127 is the subnormal 2^-127) and 2^-k (k <= 120: s32 < 2^121)
  const float s = k >= -126 ? __uint_as_float(static_cast<uint32_t>(k + 127) << 23) : __uint_as_float(1u << 22);
  const float y = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
  return UnitScale(s, y, false);   // ylo = RN((1 - s*y) * y) = 0
}

// Two packed 16-bit inputs -> two E4M3 bytes (low input in the low byte),
// without the sign of a -0 input (see quant4).
template <int DT>
__device__ __forceinline__ uint32_t quant2_fast(uint32_t w, const UnitPair& k) {
  const uint64_t x = unpack2_f2<DT>(w);
  const uint64_t q = ptx::f2_fma(x, k.yy, ptx::f2_mul(x, k.ll));  // as UnitScale::div_fast
  float lo, hi;
  ptx::f2_unpack(q, lo, hi);
  return ptx::cvt_e4m3x2(hi, lo);
}

template <int DT>
__device__ __forceinline__ uint32_t quant2_exact(uint32_t w, const UnitScale& us) {
  const float2 f = unpack2<DT>(w);
  return ptx::cvt_e4m3x2(us.div_exact(f.y), us.div_exact(f.x));
}

// Input sign bits of two packed 16-bit words, at the sign positions of the
// four E4M3 bytes they quantize to.
__device__ __forceinline__ uint32_t sign_bytes(uint32_t w0, uint32_t w1) {
  return __byte_perm(w0, w1, 0x7531) & 0x80808080u;
}

// 4 inputs (two words) -> 4 E4M3 bytes.
template <int DT, bool kExact>
__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1, const UnitScale& us, const UnitPair& k) {
  uint32_t c0, c1;
  if constexpr (kExact) {
    c0 = quant2_exact<DT>(w0, us);
    c1 = quant2_exact<DT>(w1, us);
  } else {
    c0 = quant2_fast<DT>(w0, k);
    c1 = quant2_fast<DT>(w1, k);
  }
  return __byte_perm(c0, c1, 0x5410) | sign_bytes(w0, w1);
}

// 8 input elements (one 16-byte vector) -> 8 E4M3 bytes.
template <int DT, bool kExact>
__device__ __forceinline__ uint2 quant8_impl(const uint4& v, const UnitScale& us, const UnitPair& k) {
  return make_uint2(quant4<DT, kExact>(v.x, v.y, us, k), quant4<DT, kExact>(v.z, v.w, us, k));
}

template <int DT, bool kExact>
__device__ __forceinline__ uint2 quant8_impl(const uint4& v, const UnitScale& us) {
  return quant8_impl<DT, kExact>(v, us, UnitPair(us));
}

// The per-unit choice of division path is made once, outside the element loop.
template <int DT>
__device__ __forceinline__ uint2 quant8(const uint4& v, const UnitScale& us) {
  if (__builtin_expect(us.exact_div, 0)) return quant8_impl<DT, true>(v, us);
  return quant8_impl<DT, false>(v, us);
}

template <int DT>
__device__ __forceinline__ uint8_t quant1(uint16_t h, const UnitScale& us) {
  float x = unpack2<DT>(static_cast<uint32_t>(h)).x;
  const float t = us.exact_div ? us.div_exact(x) : us.div_fast(x);
  return static_cast<uint8_t>(ptx::cvt_e4m3x2(0.0f, t) & 0xFFu);
}

// 16-byte load from this CTA's shared memory.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// The fused linear's activation quantizer for one warp: rows [r0, r0 + 16)
// of an FP16/BF16 box in shared memory (256-byte rows at xs, at least
// r0 + 16 of them; rows at or past `rows` count as zero and are not stored)
// become 1x128 token groups.  Half a warp holds a row (16-byte loads, eight
// rows a half), the amax is reduced by shuffles on pairs of rows packed into
// one word, lane l (< 16) computes the scale and reciprocal of row r0 + l
// (one divide and one reciprocal for all sixteen rows), and the half-warps
// take their rows' s and y back by shuffle; the elements then follow the
// quantizers' division path (bit-identical), the IEEE-divide fallback taken
// for all sixteen rows if any of them needs it.  No branch depends on a row,
// so the eight rows' work interleaves.  The E4M3 bytes go to the MMA's
// 128-byte swizzled tile at as (16-byte unit u of row r at u ^ (r % 8)), s
// to sa_rows[r] (shared memory); if qo is set, also the bytes to
// qo + r * qld and s to so[r].
template <int DT>
__device__ __forceinline__ void quant_box16_rows(uint32_t xs, uint32_t as, int r0, int rows, int lane,
                                                 float* sa_rows, uint8_t* qo, int64_t qld, float* so) {
  const int half = lane >> 4, hl = lane & 15;
  uint4 v[8];
  uint32_t a[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) v[q] = lds128(xs + static_cast<uint32_t>((r0 + 2 * q + half) * 256 + hl * 16));
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const bool live = r0 + 2 * q + half < rows;
    v[q].x = live ? v[q].x : 0u;
    v[q].y = live ? v[q].y : 0u;
    v[q].z = live ? v[q].z : 0u;
    v[q].w = live ? v[q].w : 0u;
    a[q] = amax_bits8(v[q]);
  }
#pragma unroll
  for (int q = 0; q < 8; q += 2) {
    uint32_t pk = a[q] | (a[q + 1] << 16);   // magnitudes are 15-bit: two per word
#pragma unroll
    for (int d = 8; d >= 1; d >>= 1) pk = __vmaxu2(pk, __shfl_xor_sync(0xFFFFFFFFu, pk, d));
    a[q] = pk & 0xFFFFu;
    a[q + 1] = pk >> 16;
  }
  uint32_t mine = 0;   // lane l < 16: the amax of row r0 + l (row 2q + h sits in half h)
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t t = __shfl_sync(0xFFFFFFFFu, a[q], (lane & 1) << 4);
    mine = (lane >> 1) == q ? t : mine;
  }
  const UnitScale own(mag_to_float<DT>(mine));   // lanes 16-31: amax 0, s = 1
  float sq[8], yq[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    sq[q] = __shfl_sync(0xFFFFFFFFu, own.s, 2 * q + half);
    yq[q] = __shfl_sync(0xFFFFFFFFu, own.y, 2 * q + half);
  }
  // UnitScale(s, y, ...) recomputes ylo exactly as UnitScale(amax) does
  uint2 q8[8];
  if (__any_sync(0xFFFFFFFFu, own.exact_div)) {
#pragma unroll
    for (int q = 0; q < 8; ++q) q8[q] = quant8<DT>(v[q], UnitScale(sq[q], yq[q], !(sq[q] >= 0x1p-90f)));
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) q8[q] = quant8_impl<DT, false>(v[q], UnitScale(sq[q], yq[q], false));
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int r = r0 + 2 * q + half;
    const uint32_t unit = static_cast<uint32_t>(hl >> 1) ^ static_cast<uint32_t>(r & 7);
    const uint32_t dst = as + static_cast<uint32_t>(r * 128) + (unit << 4) + static_cast<uint32_t>((hl & 1) * 8);
    const uint32_t sdst = ptx::smem_u32(sa_rows + r);
    asm volatile(
        "{\n\t.reg .pred p, h, ps;\n\t"
        "setp.lt.s32 p, %3, %4;\n\t"
        "setp.eq.s32 h, %7, 0;\n\t"
        "@p st.shared.v2.u32 [%0], {%1, %2};\n\t"
        "and.pred ps, p, h;\n\t"
        "@ps st.shared.f32 [%5], %6;\n\t}" ::"r"(dst),
        "r"(q8[q].x), "r"(q8[q].y), "r"(r), "r"(rows), "r"(sdst), "f"(sq[q]), "r"(hl)
        : "memory");
  }
  if (qo != nullptr) {   // warp-uniform
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int r = r0 + 2 * q + half;
      if (r < rows) {
        reinterpret_cast<uint2*>(qo + static_cast<int64_t>(r) * qld)[hl] = q8[q];
        if (hl == 0) so[r] = sq[q];
      }
    }
  }
}

// 16-byte load that does not allocate in L1 and asks L2 to keep the line
// (evict-last policy `pol`, from createpolicy): for data read again soon.
__device__ __forceinline__ uint4 ld_keep_l2(const uint4* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------------------------
// K3: per-token 1x128 groups.  Rows of A are contiguous, so the M*K/128
// groups form one contiguous sequence (group f = row f / G, column block
// f % G, starting at element 128 f).  Persistent CTAs of 8 consumer warps +
// 1 producer warp: the producer streams chunks of 8*GPW consecutive groups
// (GPW = 16: 32 KB of FP16/BF16, one 1-D bulk copy each) into a
// kTgStages-deep shared-memory ring.  Consumer warp w owns groups
// GPW*w .. GPW*w + GPW-1 of a chunk:
//   1. GPW/2 16-byte loads per lane (load j: group 2j on lanes 0-15, group
//      2j+1 on lanes 16-31) into registers, then the stage is released;
//      each half-warp reduces its group's amax with 4 shuffles;
//   2. lane i < GPW turns the amax of group i into its scale and correctly
//      rounded reciprocal (one divide per group, not per lane) and stores
//      the scale;
//   3. every lane fetches its group's scale by shuffle and casts its 8
//      elements per load.
// Small tensors use a small GPW so that the chunks still cover every SM.
constexpr int kTgStages = 3;
// Shared memory of one CTA: sized by GPW, so that the small-GPW launches of
// small tensors leave room for the next kernel's CTAs on the same SM
// (programmatic dependent launch can then start them early).
constexpr int tg_smem_bytes(int gpw) { return 1024 + kTgStages * 8 * gpw * 256 + 64; }

template <int DT, int GPW, bool UE8 = false>
__global__ void __launch_bounds__(288, 2)
    quant_token_group_kernel(const uint8_t* __restrict__ x, uint2* __restrict__ q, void* __restrict__ sa_out,
                             uint32_t M, uint32_t G, uint32_t num_groups, unsigned long long timeout_ns) {
  static_assert(GPW == 2 || GPW == 4 || GPW == 8 || GPW == 16, "groups per warp");
  constexpr int kTgChunkGroups = 8 * GPW;
  constexpr int kTgChunkBytes = kTgChunkGroups * 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kTgStages * kTgChunkBytes);
  uint64_t* empty_bar = full_bar + kTgStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t num_chunks = (num_groups + kTgChunkGroups - 1) / kTgChunkGroups;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTgStages; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 8);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::griddep_wait();  // the previous kernel's writes are visible from here on
  ptx::griddep_launch();

  if (warp == 8) {
    if (lane == 0) {
      uint32_t it = 0;
      for (uint32_t c = blockIdx.x; c < num_chunks; c += gridDim.x, ++it) {
        const int s = it % kTgStages;
        if (!ptx::mbar_wait_bounded(&empty_bar[s], ((it / kTgStages) & 1) ^ 1, timeout_ns)) {
          record_quant_error();
          break;
        }
        const uint32_t ng = min(num_groups - c * kTgChunkGroups, static_cast<uint32_t>(kTgChunkGroups));
        ptx::mbar_arrive_expect_tx(&full_bar[s], ng * 256);
        ptx::bulk_load(smem + s * kTgChunkBytes, x + static_cast<uint64_t>(c) * kTgChunkBytes, ng * 256,
                       &full_bar[s]);
      }
      // every issued copy lands before the CTA may exit
      const uint32_t first = it > kTgStages ? it - kTgStages : 0;
      for (uint32_t j = first; j < it; ++j)
        if (!ptx::mbar_wait_bounded(&full_bar[j % kTgStages], (j / kTgStages) & 1, timeout_ns)) record_quant_error();
    }
  } else {
    const int half = lane >> 4, hl = lane & 15;
    uint32_t it = 0;
    for (uint32_t c = blockIdx.x; c < num_chunks; c += gridDim.x, ++it) {
      const int s = it % kTgStages;
      if (!ptx::mbar_wait_bounded(&full_bar[s], (it / kTgStages) & 1, timeout_ns)) {
        record_quant_error();
        break;
      }
      const uint32_t gw = c * kTgChunkGroups + warp * GPW;  // first group of this warp
      const uint32_t tile = ptx::smem_u32(smem + s * kTgChunkBytes) + static_cast<uint32_t>(warp * GPW * 256);
      uint4 v[GPW / 2];
      uint32_t mine = 0;  // lanes 0..GPW-1: amax bits of group gw + lane
#pragma unroll
      for (int j = 0; j < GPW / 2; ++j) {
        // groups past the end hold stale data; never stored
        v[j] = lds128(tile + static_cast<uint32_t>(((2 * j + half) * 16 + hl) * 16));
        uint32_t a = amax_bits8(v[j]);
        a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 8));
        a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
        a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
        a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, a, 16);
        if (lane == 2 * j) mine = a;
        if (lane == 2 * j + 1) mine = other;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty_bar[s]);

      uint32_t code = 0;
      const UnitScale own = UE8 ? ue8m0_unit(mag_to_float<DT>(mine), &code) : UnitScale(mag_to_float<DT>(mine));
      const uint32_t my_group = gw + hl;
      if (lane < GPW && my_group < num_groups) {
        const uint32_t m = my_group / G;
        const uint64_t at = static_cast<uint64_t>(my_group - m * G) * M + m;
        if constexpr (UE8) static_cast<uint8_t*>(sa_out)[at] = static_cast<uint8_t>(code);
        else static_cast<float*>(sa_out)[at] = own.s;
      }
      // Warp-uniform choices, made once per chunk: every group present, and
      // no group needing the IEEE divide (then no per-group branches).
      const bool whole = gw + GPW <= num_groups;
      const bool any_exact = __any_sync(0xFFFFFFFFu, lane < GPW && own.exact_div);
      uint2* qw = q + static_cast<uint64_t>(gw) * 16 + hl;
      if (whole && !any_exact) {
#pragma unroll
        for (int j = 0; j < GPW / 2; ++j) {
          const int src = 2 * j + half;
          const UnitScale us(__shfl_sync(0xFFFFFFFFu, own.s, src), __shfl_sync(0xFFFFFFFFu, own.y, src), false);
          qw[src * 16] = quant8_impl<DT, false>(v[j], us);
        }
      } else {
#pragma unroll
        for (int j = 0; j < GPW / 2; ++j) {
          const int src = 2 * j + half;
          const UnitScale us(__shfl_sync(0xFFFFFFFFu, own.s, src), __shfl_sync(0xFFFFFFFFu, own.y, src),
                             __shfl_sync(0xFFFFFFFFu, own.exact_div ? 1 : 0, src) != 0);
          if (gw + src < num_groups) qw[src * 16] = quant8<DT>(v[j], us);
        }
      }
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------------
// K4: one persistent CTA per SM: a TMA producer warp and two consumer groups
// of 8 warps.  The producer streams whole 128x128 weight blocks (32 KB of
// FP16/BF16, one 2-D TMA box each) into a kWbStages-deep shared-memory ring;
// the CTA's i-th block goes to consumer group i % 2, so the two groups work
// on alternate blocks at once.  A group copies its block into registers
// (thread t: row t/16 + 16i, 16-byte column t%16, i = 0..7), frees the stage
// at once, reduces the block amax and casts from registers, so loads of the
// next blocks overlap the cast of this one.  One CTA per SM keeps the block
// count of the busiest SM at ceil(blocks / SMs).
// Waits are bounded.  The group's named barrier also ORs its threads' failed
// waits, so every warp of a group takes the same decision to leave; the
// producer gives up on its own.
constexpr int kWbStages = 6;
// Loads a CTA issues before waiting for its first block to land: the rest of
// the first ring pass follows one load per landed block, so the first
// blocks arrive sooner than when every SM asks for six at once (measured:
// 2% faster for a 4096 x 4096 weight, the same for larger ones).
constexpr int kWbRamp = 4;
constexpr int kWbGroups = 2;
constexpr int kWbThreads = 32 * (8 * kWbGroups + 1);
constexpr int kWbBlockBytes = 128 * 128 * 2;
constexpr int kWbSmemBytes = 1024 + kWbStages * kWbBlockBytes + 256;

template <int DT, bool UE8 = false>
__global__ void __launch_bounds__(kWbThreads, 1)
    quant_weight_block_tma_kernel(const __grid_constant__ CUtensorMap tmap_w, uint2* __restrict__ q,
                                  void* __restrict__ sb_out, int N, int KB, int num_blocks,
                                  unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kWbStages * kWbBlockBytes);
  uint64_t* empty_bar = full_bar + kWbStages;
  uint32_t* warp_max = reinterpret_cast<uint32_t*>(empty_bar + kWbStages);  // [group][2][8]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kWbStages; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 8);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::griddep_wait();  // the previous kernel's writes are visible from here on
  ptx::griddep_launch();

  if (warp == 8 * kWbGroups) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_w);
      uint32_t it = 0;
      for (int b = blockIdx.x; b < num_blocks; b += gridDim.x, ++it) {
        const int s = it % kWbStages;
        if (!ptx::mbar_wait_bounded(&empty_bar[s], ((it / kWbStages) & 1) ^ 1, timeout_ns)) {
          record_quant_error();
          break;
        }
        if (it >= static_cast<uint32_t>(kWbRamp) && it < static_cast<uint32_t>(kWbStages) &&
            !ptx::mbar_wait_bounded(&full_bar[it - kWbRamp], 0, timeout_ns)) {
          record_quant_error();
          break;
        }
        const int bi = b / KB, bj = b - (b / KB) * KB;
        ptx::mbar_arrive_expect_tx(&full_bar[s], kWbBlockBytes);
        ptx::tma_load_2d(smem + s * kWbBlockBytes, &tmap_w, &full_bar[s], bj * 128, bi * 128);
      }
      // every issued load lands before the CTA may exit
      const uint32_t first = it > kWbStages ? it - kWbStages : 0;
      for (uint32_t j = first; j < it; ++j)
        if (!ptx::mbar_wait_bounded(&full_bar[j % kWbStages], (j / kWbStages) & 1, timeout_ns)) record_quant_error();
    }
  } else {
    const int grp = warp >> 3;                 // consumer group
    const int gw = warp & 7;                   // warp within the group
    const int t = threadIdx.x & 255;           // thread within the group
    uint32_t* gmax = warp_max + grp * 16;
    const int64_t row_vec = static_cast<int64_t>(KB) * 16;
    uint32_t k = 0;                            // blocks this group has done
    for (uint32_t it = grp; blockIdx.x + static_cast<int64_t>(it) * gridDim.x < num_blocks; it += kWbGroups, ++k) {
      const int b = static_cast<int>(blockIdx.x + static_cast<int64_t>(it) * gridDim.x);
      const int s = it % kWbStages;
      const int bi = b / KB, bj = b - (b / KB) * KB;
      const bool ok = ptx::mbar_wait_bounded(&full_bar[s], (it / kWbStages) & 1, timeout_ns);
      uint4 v[8];
      uint32_t a = 0;
      const uint32_t tile = ptx::smem_u32(smem + s * kWbBlockBytes) + static_cast<uint32_t>(t * 16);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[i] = lds128(tile + static_cast<uint32_t>(i * 256 * 16));
        a = max(a, amax_bits8(v[i]));
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty_bar[s]);
      if (!ok) record_quant_error();
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
      if (lane == 0) gmax[(k & 1) * 8 + gw] = a;
      // the barrier ORs the group's failed waits: the whole group leaves together
      if (ptx::named_bar_sync_or(1 + grp, 256, !ok)) break;
      a = gmax[(k & 1) * 8];
#pragma unroll
      for (int i = 1; i < 8; ++i) a = max(a, gmax[(k & 1) * 8 + i]);
      uint32_t code = 0;
      const UnitScale us = UE8 ? ue8m0_unit(mag_to_float<DT>(a), &code) : UnitScale(mag_to_float<DT>(a));
      const UnitPair k(us);
      const int r0 = bi * 128 + (t >> 4);
      uint2* qrow = q + static_cast<int64_t>(r0) * row_vec + bj * 16 + (t & 15);
      const int64_t step = 16 * row_vec;  // 16 rows down
      if (__builtin_expect(!us.exact_div && bi * 128 + 128 <= N, 1)) {  // whole block, fast divide
#pragma unroll
        for (int i = 0; i < 8; ++i) qrow[i * step] = quant8_impl<DT, false>(v[i], us, k);
      } else if (!us.exact_div) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (r0 + 16 * i < N) qrow[i * step] = quant8_impl<DT, false>(v[i], us, k);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (r0 + 16 * i < N) qrow[i * step] = quant8_impl<DT, true>(v[i], us, k);
      }
      if (t == 0) {
        const int64_t at = static_cast<int64_t>(bi) * KB + bj;
        if constexpr (UE8) static_cast<uint8_t*>(sb_out)[at] = static_cast<uint8_t>(code);
        else static_cast<float*>(sb_out)[at] = us.s;
      }
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------------
// K1': per-tensor quantization in one cooperative launch (all CTAs resident).
// CTA b owns the contiguous vectors [b*nvec/G, (b+1)*nvec/G).
//  A. Amax of the slice.  When the host chose `resident` (every slice fits in
//     kPtSliceBytes) the slice is brought into shared memory with one 1-D bulk
//     copy and stays there, so x is read from HBM once; otherwise the slice is
//     streamed from global memory (and streamed again in C).
//  B. Grid exchange through the caller's own buffers, no scratch memory:
//     CTA b stores its slice amax in the b-th 32-bit word of q, then bumps the
//     arrival count held in *word (the caller's scale, zeroed before the
//     launch).  When the count reaches G every CTA reads the G slot words,
//     takes the maximum, and bumps the count again.
//  C. Cast of the slice.  The first ceil(G/2) output vectors (they overlap
//     the slot words) are written by CTA 0 only after the count reaches 2G,
//     i.e. after every CTA has read the slots; CTA 0 then stores the scale
//     over the count.
// With G = 1 there is no exchange.  Every wait is bounded (a timeout records
// the error and the CTA carries on, so no other CTA waits forever).
constexpr int kPtThreads = 512;
constexpr int kPtSliceBytes = 192 * 1024;  // input a CTA keeps in shared memory
constexpr int kPtSmemBytes = 1024 + kPtSliceBytes + 64;

// Brings a slice (bytes a multiple of 16) into shared memory as 16 KB bulk
// copies issued by the lanes of warp 0, all completing on `bar`: many copies
// in flight keep an SM's ingest rate up where one large copy would not.
__device__ __forceinline__ void pt_load_slice(uint8_t* dst, const uint4* src, uint32_t bytes, uint64_t* bar) {
  constexpr uint32_t kChunk = 16 * 1024;
  if (threadIdx.x == 0) ptx::mbar_arrive_expect_tx(bar, bytes);
  __syncwarp();
  if (threadIdx.x < 32) {
    for (uint32_t off = threadIdx.x * kChunk; off < bytes; off += 32 * kChunk) {
      const uint32_t n = bytes - off < kChunk ? bytes - off : kChunk;
      ptx::bulk_load(dst + off, reinterpret_cast<const uint8_t*>(src) + off, n, bar);
    }
  }
}

template <int DT, bool kExact>
__device__ __forceinline__ void pt_cast_range(const uint4* __restrict__ x, uint32_t slice_smem, bool resident,
                                              int64_t v0, int64_t a, int64_t b, uint2* __restrict__ q,
                                              const UnitScale& us) {
  const UnitPair k(us);
  int64_t i = a + threadIdx.x;
  if (!resident) {
    // from global memory: four loads in flight per thread before any cast
    for (; i + 3 * kPtThreads < b; i += 4 * kPtThreads) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = ld_stream(x + i + u * kPtThreads);
#pragma unroll
      for (int u = 0; u < 4; ++u) q[i + u * kPtThreads] = quant8_impl<DT, kExact>(v[u], us, k);
    }
  }
  for (; i < b; i += kPtThreads) {
    const uint4 v = resident ? lds128(slice_smem + static_cast<uint32_t>((i - v0) * 16)) : ld_stream(x + i);
    q[i] = quant8_impl<DT, kExact>(v, us, k);
  }
}

template <int DT>
__global__ void __launch_bounds__(kPtThreads, 1)
    quant_per_tensor_kernel(const uint4* __restrict__ x, int64_t nvec, const uint16_t* __restrict__ tail, int ntail,
                            uint2* __restrict__ q, uint8_t* __restrict__ q_tail, unsigned int* word, int resident_i,
                            unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* slice = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(slice + kPtSliceBytes);
  __shared__ uint32_t warp_max[kPtThreads / 32];
  __shared__ uint32_t amax_all;
  const bool resident = resident_i != 0;
  const unsigned G = gridDim.x;
  const int64_t v0 = static_cast<int64_t>(blockIdx.x) * nvec / G;
  const int64_t v1 = static_cast<int64_t>(blockIdx.x + 1) * nvec / G;
  const uint32_t slice_smem = ptx::smem_u32(slice);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::griddep_wait();

  // A. slice amax
  uint32_t a = 0;
  if (resident) {
    pt_load_slice(slice, x + v0, static_cast<uint32_t>((v1 - v0) * 16), bar);
    if (!ptx::mbar_wait_bounded(bar, 0, timeout_ns)) record_quant_error();
    for (int64_t i = threadIdx.x; i < v1 - v0; i += kPtThreads)
      a = max(a, amax_bits8(lds128(slice_smem + static_cast<uint32_t>(i * 16))));
  } else {
    // first of two passes over x: ask L2 to keep the lines for the cast pass
    const uint64_t pol = l2_evict_last_policy();
    int64_t i = v0 + threadIdx.x;
    for (; i + 7 * kPtThreads < v1; i += 8 * kPtThreads) {  // eight loads in flight per thread
      uint4 w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w[u] = ld_keep_l2(x + i + u * kPtThreads, pol);
#pragma unroll
      for (int u = 0; u < 8; ++u) a = max(a, amax_bits8(w[u]));
    }
    for (; i < v1; i += kPtThreads) a = max(a, amax_bits8(ld_keep_l2(x + i, pol)));
  }
  if (blockIdx.x == 0 && threadIdx.x < static_cast<unsigned>(ntail))
    a = max(a, static_cast<uint32_t>(tail[threadIdx.x] & 0x7FFFu));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
  __syncthreads();

  // B. grid exchange of the slice maxima (magnitude patterns)
  if (threadIdx.x == 0) {
    for (int w = 1; w < kPtThreads / 32; ++w) a = max(a, warp_max[w]);
    amax_all = a;
    if (G > 1) {
      reinterpret_cast<unsigned int*>(q)[blockIdx.x] = a;
      __threadfence();
      atomicAdd(word, 1u);
      volatile unsigned int* vword = word;
      const uint64_t t0 = ptx::globaltimer_ns();
      while (*vword < G) {
        if (ptx::globaltimer_ns() - t0 > timeout_ns) {
          record_quant_error();
          break;
        }
      }
      __threadfence();
    }
  }
  __syncthreads();
  if (G > 1) {
    // every thread reads a share of the G slot words (one L2 round trip)
    const unsigned int* slots = reinterpret_cast<const unsigned int*>(q);
    uint32_t m = 0;
    for (unsigned c = threadIdx.x; c < G; c += kPtThreads) m = max(m, __ldcg(slots + c));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    __syncthreads();  // warp_max is reused
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kPtThreads / 32; ++w) m = max(m, warp_max[w]);
      amax_all = max(m, warp_max[0]);
      __threadfence();
      atomicAdd(word, 1u);  // this CTA is done with the slots
    }
    __syncthreads();
  }
  const UnitScale us(mag_to_float<DT>(amax_all));

  // C. cast (CTA 0 leaves the slot-covering vectors for last)
  const int64_t nscr = (G > 1 && blockIdx.x == 0) ? (static_cast<int64_t>(G) + 1) / 2 : 0;
  if (us.exact_div) pt_cast_range<DT, true>(x, slice_smem, resident, v0, v0 + nscr, v1, q, us);
  else pt_cast_range<DT, false>(x, slice_smem, resident, v0, v0 + nscr, v1, q, us);
  if (blockIdx.x == 0) {
    if (threadIdx.x < static_cast<unsigned>(ntail)) q_tail[threadIdx.x] = quant1<DT>(tail[threadIdx.x], us);
    if (nscr > 0) {
      if (threadIdx.x == 0) {
        volatile unsigned int* vword = word;
        const uint64_t t0 = ptx::globaltimer_ns();
        while (*vword < 2 * G) {
          if (ptx::globaltimer_ns() - t0 > timeout_ns) {
            record_quant_error();
            break;
          }
        }
      }
      __syncthreads();
      if (us.exact_div) pt_cast_range<DT, true>(x, slice_smem, resident, v0, v0, v0 + nscr, q, us);
      else pt_cast_range<DT, false>(x, slice_smem, resident, v0, v0, v0 + nscr, q, us);
    }
    __syncthreads();
    if (threadIdx.x == 0) *reinterpret_cast<float*>(word) = us.s;
  }
}

// K1'': per-tensor quantization of a small tensor by one thread-block
// cluster of G <= 16 CTAs (grid = one cluster; G = 1 is a plain launch).
// The cluster is scheduled as a unit, so its CTAs may wait on each other
// without a cooperative launch, and the exchange of the slice maxima stays
// on chip: each CTA keeps its maximum in its own shared memory, and after a
// cluster barrier every CTA reads all G of them through distributed shared
// memory.  The slices (at most kPtSliceBytes each) are fetched with one bulk
// copy and cast from shared memory.  A second cluster barrier before exit
// keeps every CTA's shared memory alive until all peers have read it.
template <int DT>
__global__ void __launch_bounds__(kPtThreads, 1)
    quant_per_tensor_cluster_kernel(const uint4* __restrict__ x, int64_t nvec, const uint16_t* __restrict__ tail,
                                    int ntail, uint2* __restrict__ q, uint8_t* __restrict__ q_tail,
                                    float* __restrict__ scale, unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* slice = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(slice + kPtSliceBytes);
  __shared__ uint32_t warp_max[kPtThreads / 32];
  __shared__ uint32_t amax_cta;  // this CTA's slice maximum, read by the peers
  __shared__ uint32_t amax_all;
  const unsigned G = gridDim.x;
  const unsigned rank = blockIdx.x;
  const int64_t v0 = static_cast<int64_t>(rank) * nvec / G;
  const int64_t v1 = static_cast<int64_t>(rank + 1) * nvec / G;
  const uint32_t slice_smem = ptx::smem_u32(slice);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::griddep_wait();
  pt_load_slice(slice, x + v0, static_cast<uint32_t>((v1 - v0) * 16), bar);
  if (!ptx::mbar_wait_bounded(bar, 0, timeout_ns)) record_quant_error();
  uint32_t a = 0;
  for (int64_t i = threadIdx.x; i < v1 - v0; i += kPtThreads)
    a = max(a, amax_bits8(lds128(slice_smem + static_cast<uint32_t>(i * 16))));
  if (rank == 0 && threadIdx.x < static_cast<unsigned>(ntail))
    a = max(a, static_cast<uint32_t>(tail[threadIdx.x] & 0x7FFFu));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kPtThreads / 32; ++w) a = max(a, warp_max[w]);
    amax_cta = a;
  }
  if (G > 1) {
    ptx::cluster_arrive_release();
    ptx::cluster_wait();
    if (threadIdx.x == 0) {
      uint32_t m = 0;
      for (unsigned r = 0; r < G; ++r) m = max(m, ptx::ld_dsmem_u32(ptx::mapa(ptx::smem_u32(&amax_cta), r)));
      amax_all = m;
    }
    ptx::cluster_arrive_relaxed();  // this CTA's reads of its peers are done (waited for before exit)
  } else if (threadIdx.x == 0) {
    amax_all = a;
  }
  __syncthreads();
  const UnitScale us(mag_to_float<DT>(amax_all));
  if (us.exact_div) pt_cast_range<DT, true>(x, slice_smem, true, v0, v0, v1, q, us);
  else pt_cast_range<DT, false>(x, slice_smem, true, v0, v0, v1, q, us);
  if (rank == 0) {
    if (threadIdx.x < static_cast<unsigned>(ntail)) q_tail[threadIdx.x] = quant1<DT>(tail[threadIdx.x], us);
    if (threadIdx.x == 0) *scale = us.s;
  }
  if (G > 1) ptx::cluster_wait();
}

// ------------------------------------------------------------------------
// K1s: per-tensor quantization with a scale the caller supplies (static or
// delayed scaling, the Transformer Engine recipe with an amax history):
// q = E4M3(fl32(x / s)) with s = *scale, one read of x, and optionally the
// tensor's amax folded into *amax_out (zeroed before the launch; one
// atomicMax per CTA on the FP32 pattern, which orders like an unsigned
// integer for non-negative values).
//
// The exhaustive check behind the dynamic kernels covers |x| <= 448 s with
// s = fl32(amax/448) only; here s is arbitrary and |x / s| may saturate, so
// the double-word quotient q~ = RN(x*y + RN(x*ylo)) is used only with a
// guard that holds for every s in [2^-90, 2^90]:
//  * q~ is fl32(x/s) or one of its two FP32 neighbours: y + ylo is 1/s to
//    about 2^-47 and RN(x*ylo) adds at most 2^-48 relative, far below the
//    half ulp that separates two roundings;
//  * two adjacent FP32 values can fall on different E4M3 codes only if one
//    of them is an E4M3 rounding boundary (a midpoint of the E4M3 grid,
//    normal or subnormal), and every such boundary has its low 19 mantissa
//    bits zero (its significand has at most four bits after the leading 1);
//  * so where some q~ of four elements has low 19 bits 0x7FFFF, 0 or 1, the
//    four are recomputed with the IEEE divide.  An overflowed q~ (+-inf,
//    low bits 0) is caught the same way.
// A power-of-two s has an exact reciprocal (ylo = 0): q~ = x*y is then
// exactly fl32(x/s) and needs no guard.  Scales outside [2^-90, 2^90]
// divide every element.
enum : int { kPsPow2 = 0, kPsGuarded = 1, kPsDivide = 2 };
constexpr int kPsThreads = 256;
constexpr int kPsUnroll = 4;  // 32-byte units in flight per thread (eight 16-byte loads)

// (low 19 bits of f's pattern + 1) mod 2^19, moved to the top 19 bits (one
// IMAD): below 3 << 13 exactly when the low 19 bits are 0x7FFFF, 0 or 1,
// i.e. when f is on or next to a value whose significand has at most four
// bits after the leading 1, as every E4M3 rounding boundary has.  (Zeros also land here and take the
// exact route, as do E4M3-representable quotients: correct, just slower.)
__device__ __forceinline__ uint32_t boundary_key(float f) { return __float_as_uint(f) * 8192u + 8192u; }

template <int DT>
__device__ __forceinline__ uint32_t quant4_guarded(uint32_t w0, uint32_t w1, const UnitScale& us,
                                                   const UnitPair& k) {
  float q0, q1, q2, q3;
  ptx::f2_unpack(ptx::f2_fma(unpack2_f2<DT>(w0), k.yy, ptx::f2_mul(unpack2_f2<DT>(w0), k.ll)), q0, q1);
  ptx::f2_unpack(ptx::f2_fma(unpack2_f2<DT>(w1), k.yy, ptx::f2_mul(unpack2_f2<DT>(w1), k.ll)), q2, q3);
  const uint32_t key = min(min(boundary_key(q0), boundary_key(q1)), min(boundary_key(q2), boundary_key(q3)));
  if (__builtin_expect(key < (3u << 13), 0)) {
    return quant4<DT, true>(w0, w1, us, k);
  }
  return __byte_perm(ptx::cvt_e4m3x2(q1, q0), ptx::cvt_e4m3x2(q3, q2), 0x5410) | sign_bytes(w0, w1);
}

template <int DT, int kPath>
__device__ __forceinline__ uint2 quant8_static(const uint4& v, const UnitScale& us, const UnitPair& k) {
  if constexpr (kPath == kPsGuarded) {
    return make_uint2(quant4_guarded<DT>(v.x, v.y, us, k), quant4_guarded<DT>(v.z, v.w, us, k));
  } else {
    return quant8_impl<DT, kPath == kPsDivide>(v, us, k);
  }
}

// 16-byte store that does not allocate in L1.
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// The cast of every 32-byte unit (two input vectors -> one 16-byte output
// vector), grid-stride; returns this thread's amax pattern.
template <int DT, int kPath>
__device__ __forceinline__ uint32_t ps_cast_all(const uint4* __restrict__ x, int64_t nunit, uint4* __restrict__ q,
                                                const UnitScale& us) {
  const UnitPair k(us);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kPsThreads;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kPsThreads + threadIdx.x;
  uint32_t a = 0;
  for (; i + (kPsUnroll - 1) * stride < nunit; i += kPsUnroll * stride) {
    uint4 v[2 * kPsUnroll];
#pragma unroll
    for (int u = 0; u < kPsUnroll; ++u) {
      v[2 * u] = ld_stream(x + 2 * (i + u * stride));
      v[2 * u + 1] = ld_stream(x + 2 * (i + u * stride) + 1);
    }
#pragma unroll
    for (int u = 0; u < kPsUnroll; ++u) {
      a = max(a, max(amax_bits8(v[2 * u]), amax_bits8(v[2 * u + 1])));
      const uint2 lo = quant8_static<DT, kPath>(v[2 * u], us, k);
      const uint2 hi = quant8_static<DT, kPath>(v[2 * u + 1], us, k);
      st_stream(q + i + u * stride, make_uint4(lo.x, lo.y, hi.x, hi.y));
    }
  }
  for (; i < nunit; i += stride) {
    const uint4 v0 = ld_stream(x + 2 * i), v1 = ld_stream(x + 2 * i + 1);
    a = max(a, max(amax_bits8(v0), amax_bits8(v1)));
    const uint2 lo = quant8_static<DT, kPath>(v0, us, k);
    const uint2 hi = quant8_static<DT, kPath>(v1, us, k);
    st_stream(q + i, make_uint4(lo.x, lo.y, hi.x, hi.y));
  }
  return a;
}

// x: nvec 16-byte vectors (8 elements each) + ntail (< 8) trailing elements;
// the last vector of an odd nvec and the tail are done by CTA 0.
template <int DT>
__global__ void __launch_bounds__(kPsThreads)
    quant_static_kernel(const uint4* __restrict__ x, int64_t nvec, const uint16_t* __restrict__ tail, int ntail,
                        const float* __restrict__ scale, uint2* __restrict__ q, uint8_t* __restrict__ q_tail,
                        unsigned int* __restrict__ amax_out) {
  __shared__ uint32_t warp_max[kPsThreads / 32];
  ptx::griddep_wait();
  const float s = __ldg(scale);
  const int path = (s >= 0x1p-90f && s <= 0x1p90f) ? ((__float_as_uint(s) & 0x7FFFFFu) == 0 ? kPsPow2 : kPsGuarded)
                                                   : kPsDivide;
  const UnitScale us(s, __frcp_rn(s), path == kPsDivide);
  const int64_t nunit = nvec / 2;
  uint4* q16 = reinterpret_cast<uint4*>(q);
  uint32_t a;
  if (path == kPsPow2) a = ps_cast_all<DT, kPsPow2>(x, nunit, q16, us);
  else if (path == kPsGuarded) a = ps_cast_all<DT, kPsGuarded>(x, nunit, q16, us);
  else a = ps_cast_all<DT, kPsDivide>(x, nunit, q16, us);
  if (blockIdx.x == 0) {
    if ((nvec & 1) && threadIdx.x == 32) {
      const uint4 v = ld_stream(x + nvec - 1);
      a = max(a, amax_bits8(v));
      q[nvec - 1] = quant8_impl<DT, true>(v, us);
    }
    if (threadIdx.x < static_cast<unsigned>(ntail)) {
      const uint16_t h = tail[threadIdx.x];
      a = max(a, static_cast<uint32_t>(h & 0x7FFFu));
      const float t = us.div_exact(unpack2<DT>(static_cast<uint32_t>(h)).x);
      q_tail[threadIdx.x] =
          static_cast<uint8_t>(ptx::cvt_e4m3x2(0.0f, t) & 0xFFu) | static_cast<uint8_t>((h >> 8) & 0x80u);
    }
  }
  if (amax_out == nullptr) return;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kPsThreads / 32; ++w) a = max(a, warp_max[w]);
    atomicMax(amax_out, __float_as_uint(mag_to_float<DT>(a)));
  }
}

// Zeroes the amax slot before the static kernel folds its maxima into it.
// A kernel rather than a memset so that both launches keep programmatic
// dependent launch (a memset node between them would serialize the stream).
__global__ void zero_word_kernel(unsigned int* p) {
  ptx::griddep_wait();
  *p = 0u;
}

// ------------------------------------------------------------------------
// Per output channel (per-channel weight scaling, "What is FP8 inference on
// H100" s5): one quantization unit per row of W[N][K].  Persistent CTAs take
// rows in turn; a row (K/8 16-byte vectors) is loaded once into shared
// memory while its amax is reduced, then cast from there with the row's
// UnitScale -- the same exact quotient path as the other dynamic
// quantizers, since every element of a row is within its amax.
constexpr int kPcThreads = 256;

template <int DT>
__global__ void __launch_bounds__(kPcThreads)
    quant_per_channel_kernel(const uint4* __restrict__ w, int64_t N, int64_t kvec, uint2* __restrict__ q,
                             float* __restrict__ sb) {
  extern __shared__ uint4 row_s[];
  __shared__ uint32_t warp_max[kPcThreads / 32];
  __shared__ uint32_t amax_row;
  ptx::griddep_wait();
  for (int64_t n = blockIdx.x; n < N; n += gridDim.x) {
    const uint4* src = w + n * kvec;
    uint32_t a = 0;
    for (int64_t i = threadIdx.x; i < kvec; i += kPcThreads) {
      const uint4 v = ld_stream(src + i);
      row_s[i] = v;
      a = max(a, amax_bits8(v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int v = 1; v < kPcThreads / 32; ++v) a = max(a, warp_max[v]);
      amax_row = a;
    }
    __syncthreads();
    const UnitScale us(mag_to_float<DT>(amax_row));
    uint2* dst = q + n * kvec;
    for (int64_t i = threadIdx.x; i < kvec; i += kPcThreads) dst[i] = quant8<DT>(row_s[i], us);
    if (threadIdx.x == 0) sb[n] = us.s;
    __syncthreads();  // row_s, warp_max and amax_row are reused by the next row
  }
}

// Delayed scaling: the next scale from a window of recorded amaxes,
// s = fl32(max(history) / 448) * 2^margin (1 * 2^margin when the window's
// maximum is 0).  One CTA.
constexpr int kHsThreads = 256;
__global__ void __launch_bounds__(kHsThreads)
    scale_from_history_kernel(const float* __restrict__ history, int64_t H, int margin, float* __restrict__ scale) {
  __shared__ float warp_max[kHsThreads / 32];
  ptx::griddep_wait();
  float m = 0.0f;
  for (int64_t i = threadIdx.x; i < H; i += kHsThreads) m = fmaxf(m, history[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kHsThreads / 32; ++w) m = fmaxf(m, warp_max[w]);
    const float s0 = m == 0.0f ? 1.0f : __fdiv_rn(m, 448.0f);
    *scale = __fmul_rn(s0, __uint_as_float(static_cast<uint32_t>(127 + margin) << 23));
  }
}

}  // namespace fp8s
