// codec.cuh -- the E5M2 encoding (5 exponent + 2 mantissa bits), the other
// FP8 format of "What is FP8 inference on H100 (Transformer Engine)?" s2 and
// of "FP8 mixed-precision inference ... H100 Transformer Engine" s2.  The
// pages give only the bit split; the reading taken is the IEEE-style one:
// bias 15, S.11111.00 = +-infinity, S.11111.xx (xx != 0) = NaN, largest
// finite value 57344.  Encoding rounds to nearest even; finite values past
// 57344 and +-infinity saturate to +-57344 (as the E4M3 quantizers
// saturate); a NaN input gives S.11111.11 with the input's sign.
//
// Both kernels are elementwise streams (HBM-bound: 3 bytes per element):
// 16-byte loads and stores, several in flight per thread, a grid-stride loop
// over one wave of CTAs.  Every E5M2 value is an FP16 value (same exponent
// range and bias, two of FP16's ten mantissa bits), so decoding to FP16 is
// the byte shifted into the high half, and decoding to BF16 goes through the
// exact FP16 -> FP32 -> BF16 widening (BF16 has the wider exponent range).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"
#include "quantize.cuh"

namespace fp8s {

constexpr int kCodecThreads = 256;
constexpr int kCodecUnroll = 4;   // 16-byte units in flight per thread

// Two FP32 values -> two E5M2 bytes (round to nearest even, saturate to
// +-57344); `hi` lands in the upper byte.
__device__ __forceinline__ uint16_t cvt_e5m2x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One 16-bit FP16/BF16 pattern: is it a NaN?
template <int DT>
__device__ __forceinline__ bool is_nan16(uint32_t h) {
  return DT == kInF16 ? (h & 0x7FFFu) > 0x7C00u : (h & 0x7FFFu) > 0x7F80u;
}

// Two packed 16-bit inputs -> two E5M2 bytes (low input in the low byte).
template <int DT>
__device__ __forceinline__ uint32_t e5m2_encode2(uint32_t w) {
  const float2 f = unpack2<DT>(w);
  uint32_t c = cvt_e5m2x2(f.y, f.x);
  // a NaN keeps its sign and becomes S.11111.11
  const uint32_t lo = w & 0xFFFFu, hi = w >> 16;
  if (__builtin_expect(is_nan16<DT>(lo) | is_nan16<DT>(hi), 0)) {
    if (is_nan16<DT>(lo)) c = (c & 0xFF00u) | ((lo >> 8) & 0x80u) | 0x7Fu;
    if (is_nan16<DT>(hi)) c = (c & 0x00FFu) | ((hi & 0x8000u) | 0x7F00u);
  }
  return c;
}

// 8 inputs (one 16-byte vector) -> 8 E5M2 bytes.
template <int DT>
__device__ __forceinline__ uint2 e5m2_encode8(const uint4& v) {
  return make_uint2(e5m2_encode2<DT>(v.x) | (e5m2_encode2<DT>(v.y) << 16),
                    e5m2_encode2<DT>(v.z) | (e5m2_encode2<DT>(v.w) << 16));
}

// Two E5M2 bytes (low byte first) -> two 16-bit outputs packed in a word.
template <int DT>
__device__ __forceinline__ uint32_t e5m2_decode2(uint32_t b2) {
  // the bytes, each moved into the high half of a 16-bit FP16 pattern
  const uint32_t h2 = __byte_perm(b2, 0, 0x1404);   // {0, b0, 0, b1} as bytes: lo half = b0 << 8, hi half = b1 << 8
  if constexpr (DT == kInF16) {
    return h2;
  } else {
    const __half2 h = *reinterpret_cast<const __half2*>(&h2);
    const float2 f = __half22float2(h);
    __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);   // exact: every E5M2 value is a BF16 value
    return *reinterpret_cast<uint32_t*>(&b);
  }
}

// x [nvec * 8 + ntail] FP16/BF16 -> q E5M2 bytes.
template <int DT>
__global__ void __launch_bounds__(kCodecThreads)
    e5m2_encode_kernel(const uint4* __restrict__ x, int64_t nvec, const uint16_t* __restrict__ tail, int ntail,
                       uint2* __restrict__ q, uint8_t* __restrict__ qtail) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + (kCodecUnroll - 1) * stride < nvec; i += kCodecUnroll * stride) {
    uint4 v[kCodecUnroll];
#pragma unroll
    for (int u = 0; u < kCodecUnroll; ++u) v[u] = ld_stream(x + i + u * stride);
#pragma unroll
    for (int u = 0; u < kCodecUnroll; ++u) q[i + u * stride] = e5m2_encode8<DT>(v[u]);
  }
  for (; i < nvec; i += stride) q[i] = e5m2_encode8<DT>(ld_stream(x + i));
  if (blockIdx.x == 0 && threadIdx.x < ntail) {
    const uint32_t h = tail[threadIdx.x];
    qtail[threadIdx.x] = static_cast<uint8_t>(e5m2_encode2<DT>(h) & 0xFFu);
  }
}

// q [nvec * 16 + ntail] E5M2 bytes -> y FP16/BF16.
template <int DT>
__global__ void __launch_bounds__(kCodecThreads)
    e5m2_decode_kernel(const uint4* __restrict__ q, int64_t nvec, const uint8_t* __restrict__ qtail, int ntail,
                       uint4* __restrict__ y, uint16_t* __restrict__ ytail) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  auto decode16 = [](const uint4& b, uint4* out) {
    const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 o;
      o.x = e5m2_decode2<DT>(w[2 * h] & 0xFFFFu);
      o.y = e5m2_decode2<DT>(w[2 * h] >> 16);
      o.z = e5m2_decode2<DT>(w[2 * h + 1] & 0xFFFFu);
      o.w = e5m2_decode2<DT>(w[2 * h + 1] >> 16);
      out[h] = o;
    }
  };
  for (; i + (kCodecUnroll - 1) * stride < nvec; i += kCodecUnroll * stride) {
    uint4 v[kCodecUnroll];
#pragma unroll
    for (int u = 0; u < kCodecUnroll; ++u) v[u] = ld_stream(q + i + u * stride);
#pragma unroll
    for (int u = 0; u < kCodecUnroll; ++u) decode16(v[u], y + 2 * (i + u * stride));
  }
  for (; i < nvec; i += stride) decode16(ld_stream(q + i), y + 2 * i);
  if (blockIdx.x == 0 && threadIdx.x < ntail) ytail[threadIdx.x] = static_cast<uint16_t>(e5m2_decode2<DT>(qtail[threadIdx.x]));
}

}  // namespace fp8s
