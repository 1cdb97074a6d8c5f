// quantize.cuh -- dynamic E4M3 quantization kernels (per tensor, per 1x128
// token group, per 128x128 weight block).
//
// Method ("What is FP8 inference on H100 (Transformer Engine)?", s3 steps
// 2-4): amax = max|x| over the unit, s = fl32(amax / 448) (1 when amax == 0),
// q = E4M3_rne_satfinite(fl32(x / s)).  Units are the whole tensor, a group
// of 128 input channels of one token, or a 128x128 weight block (the
// transformers "Fine-grained FP8" guide, opening bullets).
//
// All kernels stream 16-byte vectors (8 FP16/BF16 elements) and keep the
// arithmetic bit-exact with IEEE single precision:
//  * amax is taken on the 16-bit patterns: with the sign bit cleared,
//    finite FP16/BF16 magnitudes order exactly like unsigned integers, so a
//    packed 16-bit unsigned max (__vmaxu2) is an exact max.
//  * fl32(x / s) is computed without a per-element divide.  With y the
//    correctly rounded reciprocal of s (computed once per unit), q0 = x*y is
//    refined twice by the remainder r = x - s*q (exact via FMA) and
//    q' = q + r*y.  The first refinement leaves q within one ulp of x/s; the
//    second then returns the correctly rounded quotient (Markstein, "IA-64
//    and Elementary Functions", theorem on division by reciprocal
//    refinement).  Zeros keep the sign of x (x/s with s > 0, so -0 stays
//    -0).  Units whose scale is tiny (s < 2^-90, possible only for BF16
//    inputs below about 2^-81) use the IEEE divide __fdiv_rn.
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

// Exact fl32(x / s) for one quantization unit (see the file comment).
struct UnitScale {
  float s;     // dequant factor written to memory
  float y;     // RN(1/s)
  bool exact_div;

  __device__ __forceinline__ explicit UnitScale(float amax) {
    s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
    y = __frcp_rn(s);
    exact_div = !(s >= 0x1p-90f);
  }

  // Reciprocal refinement (two Markstein steps); valid when !exact_div.
  // The remainder is formed negated, r' = s*q - x (exact), and the step is
  // q - r'*y: for x != 0 this is the same rounding of the same exact value as
  // q + r*y, and for x = -0 (or a quotient that underflows to zero) the sum
  // of two like-signed zeros keeps the sign of x, so no copysign is needed.
  __device__ __forceinline__ float div_fast(float x) const {
    float q = __fmul_rn(x, y);
    float r = __fmaf_rn(s, q, -x);
    q = __fmaf_rn(-r, y, q);
    r = __fmaf_rn(s, q, -x);
    q = __fmaf_rn(-r, y, q);
    return q;
  }

  __device__ __forceinline__ float div_exact(float x) const { return __fdiv_rn(x, s); }

  template <bool kExact>
  __device__ __forceinline__ float div(float x) const {
    if constexpr (kExact) return div_exact(x);
    else return div_fast(x);
  }
};

// 8 input elements (one 16-byte vector) -> 8 E4M3 bytes.
template <int DT, bool kExact>
__device__ __forceinline__ uint2 quant8_impl(const uint4& v, const UnitScale& us) {
  const float2 a = unpack2<DT>(v.x), b = unpack2<DT>(v.y), c = unpack2<DT>(v.z), d = unpack2<DT>(v.w);
  const uint32_t p0 = ptx::cvt_e4m3x2(us.div<kExact>(a.y), us.div<kExact>(a.x));
  const uint32_t p1 = ptx::cvt_e4m3x2(us.div<kExact>(b.y), us.div<kExact>(b.x));
  const uint32_t p2 = ptx::cvt_e4m3x2(us.div<kExact>(c.y), us.div<kExact>(c.x));
  const uint32_t p3 = ptx::cvt_e4m3x2(us.div<kExact>(d.y), us.div<kExact>(d.x));
  return make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
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

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------------------------
// K3: one 1x128 token group per half-warp (16 lanes x 8 elements).
// grid = (ceil(M/16/ROWS_PER_CTA_ITEMS) , K/128); the CTA (256 threads =
// 16 half-warps) handles UNROLL blocks of 16 consecutive rows of one group
// column, so each warp's 16 scale writes of a group column are contiguous.
template <int DT, int UNROLL>
__global__ void __launch_bounds__(256) quant_token_group_kernel(const uint4* __restrict__ x,
                                                                uint2* __restrict__ q,
                                                                float* __restrict__ sa, int M, int G) {
  const int hw = threadIdx.x >> 4;  // half-warp 0..15
  const int hl = threadIdx.x & 15;  // lane within the half-warp
  const int g = blockIdx.y;
  const int64_t row_vec = static_cast<int64_t>(G) * 16;  // 16-byte vectors per row
  int rows[UNROLL];
  uint4 v[UNROLL];
#pragma unroll
  for (int u = 0; u < UNROLL; ++u) {
    rows[u] = (blockIdx.x * UNROLL + u) * 16 + hw;
    v[u] = make_uint4(0, 0, 0, 0);
    if (rows[u] < M) v[u] = ld_stream(x + rows[u] * row_vec + g * 16 + hl);
  }
#pragma unroll
  for (int u = 0; u < UNROLL; ++u) {
    uint32_t a = amax_bits8(v[u]);
    a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 8));
    a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
    a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    const UnitScale us(mag_to_float<DT>(a));
    if (rows[u] < M) {
      q[rows[u] * row_vec + g * 16 + hl] = quant8<DT>(v[u], us);
      if (hl == 0) sa[static_cast<int64_t>(g) * M + rows[u]] = us.s;
    }
  }
}

// ------------------------------------------------------------------------
// K4: persistent CTAs of 8 consumer warps + 1 TMA producer warp.  The
// producer streams whole 128x128 weight blocks (32 KB of FP16/BF16, one 2-D
// TMA box each) into a kWbStages-deep shared-memory ring; consumers copy a
// block into registers (thread t: row t/16 + 16i, 16-byte column t%16,
// i = 0..7), free the stage at once, reduce the block amax and cast from
// registers, so loads of the next blocks overlap the cast of this one.
// Waits are bounded; a consumer that gives up raises a shared abort flag that
// every consumer reads after the same named barrier, so they leave together.
constexpr int kWbStages = 3;
constexpr int kWbBlockBytes = 128 * 128 * 2;
constexpr int kWbSmemBytes = 1024 + kWbStages * kWbBlockBytes + 256;

template <int DT>
__global__ void __launch_bounds__(288, 2)
    quant_weight_block_tma_kernel(const __grid_constant__ CUtensorMap tmap_w, uint2* __restrict__ q,
                                  float* __restrict__ sb, int N, int KB, int num_blocks,
                                  unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kWbStages * kWbBlockBytes);
  uint64_t* empty_bar = full_bar + kWbStages;
  uint32_t* warp_max = reinterpret_cast<uint32_t*>(empty_bar + kWbStages);  // [2][8]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(warp_max + 16);

  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  if (t == 0) {
    for (int s = 0; s < kWbStages; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 8);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();

  if (warp == 8) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_w);
      uint32_t it = 0;
      for (int b = blockIdx.x; b < num_blocks; b += gridDim.x, ++it) {
        const int s = it % kWbStages;
        if (!ptx::mbar_wait_bounded(&empty_bar[s], ((it / kWbStages) & 1) ^ 1, timeout_ns)) {
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
    const int64_t row_vec = static_cast<int64_t>(KB) * 16;
    uint32_t it = 0;
    for (int b = blockIdx.x; b < num_blocks; b += gridDim.x, ++it) {
      const int s = it % kWbStages;
      const int bi = b / KB, bj = b - (b / KB) * KB;
      const bool ok = ptx::mbar_wait_bounded(&full_bar[s], (it / kWbStages) & 1, timeout_ns);
      uint4 v[8];
      uint32_t a = 0;
      const uint4* tile = reinterpret_cast<const uint4*>(smem + s * kWbBlockBytes);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[i] = tile[t + 256 * i];
        a = max(a, amax_bits8(v[i]));
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty_bar[s]);
      if (!ok) {
        record_quant_error();
        *abort_flag = 1;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
      if (lane == 0) warp_max[(it & 1) * 8 + warp] = a;
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (*abort_flag) break;
      a = warp_max[(it & 1) * 8];
#pragma unroll
      for (int i = 1; i < 8; ++i) a = max(a, warp_max[(it & 1) * 8 + i]);
      const UnitScale us(mag_to_float<DT>(a));
      const int col = bj * 16 + (t & 15);
      if (__builtin_expect(!us.exact_div, 1)) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = bi * 128 + (t >> 4) + 16 * i;
          if (r < N) q[r * row_vec + col] = quant8_impl<DT, false>(v[i], us);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = bi * 128 + (t >> 4) + 16 * i;
          if (r < N) q[r * row_vec + col] = quant8_impl<DT, true>(v[i], us);
        }
      }
      if (t == 0) sb[static_cast<int64_t>(bi) * KB + bj] = us.s;
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------------
// K1: per-tensor amax.  Grid-stride over 16-byte vectors; the block maximum
// is folded into *amax_word (the float's bit pattern; non-negative floats
// order like unsigned integers) with one atomicMax per CTA.  *amax_word must
// be zero beforehand.  The tail (numel % 8 elements) is read by block 0.
template <int DT>
__global__ void __launch_bounds__(256) amax_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                   const uint16_t* __restrict__ tail, int ntail,
                                                   unsigned int* __restrict__ amax_word) {
  __shared__ uint32_t warp_max[8];
  uint32_t a = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    const uint4 v0 = ld_stream(x + i), v1 = ld_stream(x + i + stride);
    const uint4 v2 = ld_stream(x + i + 2 * stride), v3 = ld_stream(x + i + 3 * stride);
    a = max(a, max(max(amax_bits8(v0), amax_bits8(v1)), max(amax_bits8(v2), amax_bits8(v3))));
  }
  for (; i < nvec; i += stride) a = max(a, amax_bits8(ld_stream(x + i)));
  if (blockIdx.x == 0 && threadIdx.x < ntail) a = max(a, static_cast<uint32_t>(tail[threadIdx.x] & 0x7FFFu));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < (blockDim.x >> 5); ++k) a = max(a, warp_max[k]);
    atomicMax(amax_word, __float_as_uint(mag_to_float<DT>(a)));
  }
}

// K2: per-tensor cast with the scale derived from the finished amax.
template <int DT>
__global__ void __launch_bounds__(256) cast_per_tensor_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                              const uint16_t* __restrict__ tail, int ntail,
                                                              uint2* __restrict__ q, uint8_t* __restrict__ q_tail,
                                                              const unsigned int* __restrict__ amax_word) {
  const UnitScale us(__uint_as_float(*amax_word));
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + stride < nvec; i += 2 * stride) {
    const uint4 v0 = ld_stream(x + i), v1 = ld_stream(x + i + stride);
    q[i] = quant8<DT>(v0, us);
    q[i + stride] = quant8<DT>(v1, us);
  }
  for (; i < nvec; i += stride) q[i] = quant8<DT>(ld_stream(x + i), us);
  if (blockIdx.x == 0 && threadIdx.x < ntail) q_tail[threadIdx.x] = quant1<DT>(tail[threadIdx.x], us);
}

// Turns the finished amax (bits in *word) into the stored scale, in place.
__global__ void finalize_scale_kernel(unsigned int* word) {
  const float amax = __uint_as_float(*word);
  const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
  *reinterpret_cast<float*>(word) = s;
}

}  // namespace fp8s
