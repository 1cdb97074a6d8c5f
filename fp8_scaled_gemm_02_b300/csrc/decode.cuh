// decode.cuh -- the block-scaled FP8 GEMM for decode batches (M <= 32 tokens),
// computed transposed: C^T = W . A^T.
//
// Method: the block-scaled linear of the transformers "Fine-grained FP8"
// guide (1x128 token groups, 128x128 weight blocks) with FP32 promotion per
// 128-wide K block, as in gemm.cuh; only the operand roles change.  A decode
// batch has few tokens and a weight of megabytes, so the weight tile is the
// MMA's 128-row operand (A of tcgen05.mma) and the tokens are its N = MT
// columns (MT = 16 or 32, rows past M zero).  Per K block a stage holds 16 KB
// of weight and MT x 128 bytes of activation (instead of 16 + 16 KB with the
// tokens as rows), the TMEM partial is 128 x MT, and the promotion of a K
// block is MT columns per thread: the weight stream sets the pace.
//
//   warp 0      TMA producer: 128x128-byte weight tiles (and, unfused, the
//               MT x 128-byte E4M3 activation tiles), 128-byte swizzle, a
//               STAGES-deep ring.
//   warp 1      MMA issuer: tcgen05.mma kind::f8f6f4, M = 128, N = MT, four
//               per K block, a fresh TMEM buffer per K block.
//   warp 2      TMEM allocation.
//   warps 4-7   epilogue: thread = one weight row n of the tile (its lane
//               quarter of TMEM), MT token columns; per K block it adds
//               partial[n][m] * sa[kb][m] * sb[n/128][kb] into FP32 pairs.
// Fused (the activation arrives in FP16/BF16 and is quantized per 1x128
// token group inside the kernel), two forms:
//   resident    warps 2-7 first quantize the CTA's whole K range of the
//               activation from global memory into a shared-memory buffer
//               of E4M3 tiles (and its token scales); the MMA loop then
//               runs as unfused, with the activation tiles resident.
//   ring        the activation has a ring of its own: quantizer warps (2-3,
//               and 8-9 for MT = 32) load its M x 128 boxes by TMA ahead of
//               the MMA and quantize them into the ring's E4M3 tiles, the
//               token scales into a second ring the epilogue reads.
// Split-K: the S CTAs of a cluster share the tile, each a K range; the FP32
// partials are exchanged through distributed shared memory (rank r owns
// weight rows [r*128/S, (r+1)*128/S)) and summed in rank order, so results
// are deterministic; no global scratch memory.  Output C[m][n] is written
// transposed: for a fixed token the 32 lanes of a warp write 32 consecutive
// columns.
//
// The CUDA occupancy query reports one CTA per SM for any kernel that
// allocates tensor memory, but the hardware places two when shared memory
// and registers allow: the unfused kernel, the resident form and the ring
// form with MT = 16 keep ~100 KB and <= 128 registers so that two CTAs share
// an SM.  Every wait is bounded as in gemm.cuh.
#pragma once

#include "gemm.cuh"

namespace fp8s {

// FUSED: 0 = the E4M3 activation comes quantized; 1 = fused, the activation
// streamed through a ring of its own and quantized K block by K block; 2 =
// fused, the CTA's whole K range of the activation quantized once into a
// resident shared-memory buffer before the MMAs start.
template <int MT, bool SPLIT, int FUSED>
struct DecCfg {
  static constexpr bool kRing = FUSED == 1;
  static constexpr bool kRes = FUSED == 2;
  static_assert(MT == 16 || MT == 32, "token columns per MMA");
  static constexpr int kEpiWarps = 4;
  // Two CTAs per SM (~100 KB of shared memory, <= 128 registers) for the
  // unfused kernel and the fused MT = 16 one; the fused MT = 32 kernel takes
  // an SM alone.  Fused: kQWarps quantizer warps, 2-3 and 8.. (the epilogue
  // keeps warps 4-7, whose warp index modulo 4 is their TMEM lane quarter).
  static constexpr int kCtasPerSm = (kRing && MT == 32) ? 1 : 2;
  static constexpr int kQWarps = kRing ? (MT == 16 ? 2 : 4) : 0;
  static constexpr int kThreads = 128 + 32 * kEpiWarps + (kRing ? 32 * (kQWarps - 2) : 0);
  static constexpr int kWBytes = kBM * kBK;                 // 128 weight rows x one K block
  static constexpr int kXBytes = MT * kBK;                  // E4M3 activation rows
  // Unfused: a stage holds the weight tile and the E4M3 activation tile.
  // Fused: the stage holds the weight tile only; the activation has a ring of
  // its own, kXSlots slots of [FP16/BF16 box (MT x 256 B) | E4M3 tile
  // (MT x 128 B)], slot j owned by quantizer j % kQWarps.
  static constexpr int kStageBytes = FUSED ? kWBytes : kWBytes + kXBytes;
  // resident (FUSED == 2): up to kActKb K blocks of E4M3 activation tiles
  // and their token scales, for the CTA's whole K range
  static constexpr int kActKb = kRes ? (MT == 16 ? 16 : 8) : 0;
  static constexpr int kActBytes = kActKb * MT * kBK;
  static constexpr int kSaBufBytes = kActKb * MT * 4;
  static constexpr int kXSlots = 2 * kQWarps;
  static constexpr int kX16Bytes = MT * kBK * 2;
  static constexpr int kXSlotBytes = kRing ? kX16Bytes + kXBytes : 0;
  static constexpr int kXRingBytes = kXSlots * kXSlotBytes;
  static constexpr int kPitch = MT + 4;                     // staging row pitch (floats): 16-byte rows
  static constexpr int kStagingBytes = kBM * kPitch * 4;
  static constexpr int kRecvBytes = SPLIT ? 112 * kPitch * 4 : 0;
  static constexpr int kSaSlots = kRing ? 12 : 0;            // ring: token scales per K block
  static constexpr int kSaBytes = kSaSlots * MT * 4;
  static constexpr int kBudget = kCtasPerSm == 2 ? 104 * 1024 : 220 * 1024;
  static constexpr int kStagesRaw =
      (kBudget - kXRingBytes - kActBytes - kSaBufBytes - kRecvBytes - kSaBytes - 1024) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(!SPLIT || kStages * kStageBytes >= kStagingBytes, "staging fits in the ring");
  static constexpr int kNBuf = 8;
  static constexpr int kTmemCols = kNBuf * MT;               // 128 or 256: a power of two
  static constexpr int kBarBytes = 8 * (2 * kStages + 2 * kNBuf + 4 + (kRing ? 3 * kXSlots + 2 * kSaSlots : 0)) + 16;
  static constexpr int kSmemBytes =
      1024 + kStages * kStageBytes + kXRingBytes + kActBytes + kSaBufBytes + kRecvBytes + kSaBytes + kBarBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  // A quantizer runs at most kXSlots K blocks ahead of the MMA, which runs at
  // most kNBuf ahead of the epilogue; with 2 * kSaSlots above that lead no
  // wait on a scale slot is two phases behind.  Slot j of either ring is
  // always used by quantizer j % kQWarps.
  static_assert(kSaSlots == 0 || 2 * kSaSlots > kXSlots + kNBuf, "scale slots");
  static_assert(kSaSlots % (kQWarps > 0 ? kQWarps : 1) == 0, "scale slots per quantizer");
};

// Sums this CTA's R weight rows over the S partials in rank order and stores
// them transposed, C[m][tn*128 + row] for m < M (consecutive threads take
// consecutive rows, so each store of a warp covers 32 consecutive columns).
template <int MT, int OUT, int S>
__device__ __forceinline__ void dec_reduce(const float* send, const float* recv, uint32_t rank, int tid, int tn,
                                           const GemmParams& p) {
  constexpr int kPitch = MT + 4;
  constexpr int R = kBM / S;
  uint16_t* C = reinterpret_cast<uint16_t*>(p.c);
  const float* src[S];
#pragma unroll
  for (int q = 0; q < S; ++q)
    src[q] = q == static_cast<int>(rank) ? send + static_cast<int>(rank) * R * kPitch
                                         : recv + (q < static_cast<int>(rank) ? q : q - 1) * R * kPitch;
  const int mmax = p.M < MT ? p.M : MT;
  for (int idx = tid; idx < R * mmax; idx += 32 * DecCfg<MT, true, 0>::kEpiWarps) {
    const int m = idx / R, rr = idx - (idx / R) * R;
    float v[S];
#pragma unroll
    for (int q = 0; q < S; ++q) v[q] = src[q][rr * kPitch + m];
    float acc = v[0];
#pragma unroll
    for (int q = 1; q < S; ++q) acc += v[q];
    const int n = tn * kBM + static_cast<int>(rank) * R + rr;
    if (n < p.N) C[static_cast<int64_t>(m) * p.N + n] = one_out<OUT>(acc);
  }
}

template <int MT, int OUT, bool SPLIT, int FUSED>
__global__ void __launch_bounds__(DecCfg<MT, SPLIT, FUSED>::kThreads, DecCfg<MT, SPLIT, FUSED>::kCtasPerSm)
    fp8_decode_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                      const GemmParams p) {
  using Cfg = DecCfg<MT, SPLIT, FUSED>;
  constexpr int S_ = Cfg::kStages;
  constexpr int NBUF = Cfg::kNBuf;
  constexpr int DT = OUT;  // fused: the activation has the output's type

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int XS = Cfg::kXSlots > 0 ? Cfg::kXSlots : 1;   // (unfused: no activation slots)
  uint8_t* w_ring = smem;
  uint8_t* x_ring = w_ring + S_ * Cfg::kWBytes;             // unfused: E4M3 tiles, one per stage
  uint8_t* xq_ring = smem + S_ * Cfg::kStageBytes;          // ring: activation slots
  uint8_t* act_buf = xq_ring + Cfg::kXRingBytes;            // resident: E4M3 tiles, K block i at i * MT * 128
  float* sa_buf = reinterpret_cast<float*>(act_buf + Cfg::kActBytes);   // resident: [i][MT] token scales
  float* staging = reinterpret_cast<float*>(smem);  // split-K: after the ring has drained
  const float* recv = reinterpret_cast<const float*>(act_buf + Cfg::kActBytes + Cfg::kSaBufBytes);
  float* sa_ring = reinterpret_cast<float*>(act_buf + Cfg::kActBytes + Cfg::kSaBufBytes + Cfg::kRecvBytes);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sa_ring) + Cfg::kSaBytes);
  uint64_t* empty_bar = full_bar + S_;
  uint64_t* tfull_bar = empty_bar + S_;
  uint64_t* tempty_bar = tfull_bar + NBUF;
  uint64_t* mma_done_bar = tempty_bar + NBUF;
  uint64_t* staged_bar = mma_done_bar + 1;
  uint64_t* recv_bar = staged_bar + 1;
  uint64_t* act_ready_bar = recv_bar + 1;                        // resident: the activation is quantized
  uint64_t* x8_ready_bar = act_ready_bar + 1;                     // ring: slot's E4M3 rows written
  uint64_t* xfull_bar = x8_ready_bar + (Cfg::kRing ? XS : 0);     // ring: slot's activation box landed
  uint64_t* xempty_bar = xfull_bar + (Cfg::kRing ? XS : 0);       // ring: slot's MMAs done
  uint64_t* sa_full_bar = xempty_bar + (Cfg::kRing ? XS : 0);     // ring: a scale slot written
  uint64_t* sa_free_bar = sa_full_bar + Cfg::kSaSlots;            // fused: a scale slot read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sa_free_bar + Cfg::kSaSlots);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint32_t rank = 0, S = 1;
  if constexpr (SPLIT) {
    rank = ptx::cluster_ctarank();
    S = ptx::cluster_nctarank();
  }
  const int tn = static_cast<int>(blockIdx.x / S);   // one weight tile per cluster
  const int kb_begin = static_cast<int>((static_cast<int64_t>(rank) * p.num_kb) / S);
  const int kb_end = static_cast<int>((static_cast<int64_t>(rank + 1) * p.num_kb) / S);
  const int nkb = kb_end - kb_begin;  // >= 1: the host keeps S <= num_kb
  const int rot = tn % nkb;           // spread the shared activation's L2 requests over K blocks
  auto kb_at = [&](int i) { return kb_begin + (i + rot < nkb ? i + rot : i + rot - nkb); };

  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmap_w);
    ptx::tma_prefetch_desc(&tmap_x);
    for (int s = 0; s < S_; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      ptx::mbar_init(&tfull_bar[b], 1);
      ptx::mbar_init(&tempty_bar[b], Cfg::kEpiWarps);
    }
    ptx::mbar_init(mma_done_bar, 1);
    ptx::mbar_init(staged_bar, Cfg::kEpiWarps);
    ptx::mbar_init(recv_bar, 1);
    ptx::mbar_init(act_ready_bar, 6);   // resident: quantizer warps 2-7
    if constexpr (Cfg::kRing) {
      for (int j = 0; j < XS; ++j) {
        ptx::mbar_init(&x8_ready_bar[j], 1);   // the slot's quantizer warp
        ptx::mbar_init(&xfull_bar[j], 1);
        ptx::mbar_init(&xempty_bar[j], 1);     // the MMA issuer's commit
      }
      for (int j = 0; j < Cfg::kSaSlots; ++j) {
        ptx::mbar_init(&sa_full_bar[j], 1);
        ptx::mbar_init(&sa_free_bar[j], Cfg::kEpiWarps);
      }
    }
    ptx::fence_mbar_init();
  }
  if (warp == 2) {
    ptx::tmem_alloc<Cfg::kTmemCols>(tmem_slot);
    ptx::tmem_relinquish();
  }
  if constexpr (Cfg::kRes) {
    // rows past M are never written by the quantizers: zero bytes, scale 0
    for (int i = threadIdx.x; i < Cfg::kActBytes / 16; i += Cfg::kThreads)
      ptx::sts128(ptx::smem_u32(act_buf) + 16u * static_cast<uint32_t>(i), 0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < Cfg::kActKb * MT; i += Cfg::kThreads) sa_buf[i] = 0.0f;
    ptx::fence_proxy_async_shared();
  }
  if constexpr (Cfg::kRing) {
    // activation rows past M are never written by the quantizer: they stay
    // zero, and their token scales 0 (the products they meet are zero)
    for (int i = threadIdx.x; i < XS * Cfg::kXBytes / 16; i += Cfg::kThreads) {
      const int j = i / (Cfg::kXBytes / 16), u = i - j * (Cfg::kXBytes / 16);
      ptx::sts128(ptx::smem_u32(xq_ring + j * Cfg::kXSlotBytes + Cfg::kX16Bytes) + 16u * static_cast<uint32_t>(u), 0u,
                  0u, 0u, 0u);
    }
    for (int i = threadIdx.x; i < Cfg::kSaSlots * MT; i += Cfg::kThreads) sa_ring[i] = 0.0f;
    ptx::fence_proxy_async_shared();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (SPLIT) ptx::cluster_arrive_relaxed();  // peers' barriers: waited for before the exchange
  bool cluster_waited = !SPLIT;
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  ptx::griddep_wait();  // the previous kernel's writes (our operands) are visible from here on
  ptx::griddep_launch();

  // fused: the box holds the M token rows (M <= MT), 256 bytes each
  const uint32_t x16_box_bytes = static_cast<uint32_t>(p.M < MT ? p.M : MT) * kBK * 2u;

  // Resident: warps 2-7 quantize the CTA's whole K range of the activation
  // once, straight from global memory, while the producer already streams
  // the weight.  A lane takes half a 1x128 token group (64 elements: eight
  // 16-byte loads); its partner lane (the other half) completes the amax by
  // one shuffle; both compute s = fl32(amax / 448) and its reciprocal pair,
  // and the lane casts its 64 elements with the token-group quantizer's
  // arithmetic ([P5] groups, [P2] s3 steps 2-4; bit-identical) into four
  // 16-byte units of the K block's swizzled E4M3 tile (unit u of row m at
  // u ^ (m % 8)); the first half's lane stores s.  K block i of the CTA's
  // issue order sits at act_buf + i * MT * 128, its scales at sa_buf[i][m].
  auto res_quantize = [&]() {
    if constexpr (Cfg::kRes) {
      const int qw = warp - 2;   // 0..5
      // the host launches this form only when nkb <= kActKb; beyond that
      // nothing is written outside the buffer and the error word says so
      const int nkb_q = nkb <= Cfg::kActKb ? nkb : Cfg::kActKb;
      if (nkb > Cfg::kActKb && qw == 0 && lane == 0) record_error(kErrProducer);
      const int units = 2 * p.M * nkb_q;
      const uint16_t* X = reinterpret_cast<const uint16_t*>(p.x);
      const bool copy_out = p.qa_out != nullptr && tn == 0;
      for (int base = 32 * qw; base < units; base += 6 * 32) {   // warp-uniform
        const int u = base + lane;
        const bool live = u < units;   // units is even: partners are live together
        const int i = live ? u / (2 * p.M) : 0;
        const int rem = u - i * 2 * p.M;
        const int m = live ? rem >> 1 : 0, h = rem & 1;
        const int kb = kb_at(i);
        uint4 v[8];
        uint32_t a = 0;
        if (live) {
          const uint4* src = reinterpret_cast<const uint4*>(X + static_cast<int64_t>(m) * p.K + kb * kBK + h * 64);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            v[j] = __ldg(src + j);
            a = max(a, amax_bits8(v[j]));
          }
        }
        a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        if (live) {
          const UnitScale us(mag_to_float<DT>(a));
          uint2 q[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) q[j] = quant8<DT>(v[j], us);
          const uint32_t row = ptx::smem_u32(act_buf) + static_cast<uint32_t>(i * MT * kBK + m * kBK);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t unit = static_cast<uint32_t>(h * 4 + c) ^ static_cast<uint32_t>(m & 7);
            ptx::sts128(row + (unit << 4), q[2 * c].x, q[2 * c].y, q[2 * c + 1].x, q[2 * c + 1].y);
          }
          if (h == 0) sa_buf[i * MT + m] = us.s;
          if (copy_out) {
            uint4* dst = reinterpret_cast<uint4*>(p.qa_out + static_cast<int64_t>(m) * p.K + kb * kBK + h * 64);
#pragma unroll
            for (int c = 0; c < 4; ++c) dst[c] = make_uint4(q[2 * c].x, q[2 * c].y, q[2 * c + 1].x, q[2 * c + 1].y);
            if (h == 0) p.sa_out[static_cast<int64_t>(kb) * p.M + m] = us.s;
          }
        }
      }
      ptx::fence_proxy_async_shared();   // the E4M3 tiles, before the MMA reads them
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(act_ready_bar);
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int kb = kb_at(i);
        const int s = i % S_;
        if (!ptx::mbar_wait_bounded(&empty_bar[s], ((i / S_) & 1) ^ 1, p.timeout_ns)) {
          record_error(kErrProducer);
          break;
        }
        if constexpr (FUSED) {
          ptx::mbar_arrive_expect_tx(&full_bar[s], Cfg::kWBytes);   // the activation: the quantizers' loads
        } else {
          ptx::mbar_arrive_expect_tx(&full_bar[s], Cfg::kWBytes + Cfg::kXBytes);
          ptx::tma_load_2d(x_ring + s * Cfg::kXBytes, &tmap_x, &full_bar[s], kb * kBK, 0);
        }
        ptx::tma_load_2d(w_ring + s * Cfg::kWBytes, &tmap_w, &full_bar[s], kb * kBK, tn * kBM);
        ++issued;
      }
      // every issued load lands before the CTA may exit
      for (int j = issued > S_ ? issued - S_ : 0; j < issued; ++j)
        if (!ptx::mbar_wait_bounded(&full_bar[j % S_], (j / S_) & 1, p.timeout_ns)) record_error(kErrProducer);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_e4m3_f32(kBM, MT);
      const uint32_t w0 = ptx::smem_u32(w_ring), x0 = ptx::smem_u32(x_ring), xq0 = ptx::smem_u32(xq_ring);
      const uint32_t act0 = ptx::smem_u32(act_buf);
      bool act_ok = true;
      if constexpr (Cfg::kRes) act_ok = ptx::mbar_wait_bounded(act_ready_bar, 0, p.timeout_ns);
      for (int i = 0; i < nkb && act_ok; ++i) {
        const int buf = i % NBUF, s = i % S_;
        const int xj = Cfg::kRing ? i % XS : 0;
        if (!ptx::mbar_wait_bounded(&tempty_bar[buf], ((i / NBUF) & 1) ^ 1, p.timeout_ns) ||
            !ptx::mbar_wait_bounded(&full_bar[s], (i / S_) & 1, p.timeout_ns) ||
            (Cfg::kRing && !ptx::mbar_wait_bounded(&x8_ready_bar[xj], (i / XS) & 1, p.timeout_ns))) {
          record_error(kErrMma);
          break;
        }
        ptx::tc_fence_after();
        const uint64_t adesc = ptx::smem_desc_sw128_kmajor(w0 + s * Cfg::kWBytes);
        const uint64_t bdesc = ptx::smem_desc_sw128_kmajor(
            Cfg::kRes    ? act0 + static_cast<uint32_t>(i * MT * kBK)
            : Cfg::kRing ? xq0 + static_cast<uint32_t>(xj * Cfg::kXSlotBytes + Cfg::kX16Bytes)
                         : x0 + s * Cfg::kXBytes);
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * MT);
#pragma unroll
        for (int k = 0; k < kBK / kMmaK; ++k) ptx::mma_f8f6f4(d, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
        ptx::mma_commit(&empty_bar[s]);
        if constexpr (Cfg::kRing) ptx::mma_commit(&xempty_bar[xj]);
        ptx::mma_commit(&tfull_bar[buf]);
      }
      if (!act_ok) record_error(kErrMma);
      ptx::mma_commit(mma_done_bar);
      if (!ptx::mbar_wait_bounded(mma_done_bar, 0, p.timeout_ns)) record_error(kErrMma);
    }
  } else if (Cfg::kRes && (warp == 2 || warp == 3)) {
    res_quantize();
  } else if (Cfg::kRing && (warp == 2 || warp == 3 || warp >= 8)) {
    // ------------------------------- fused activation quantizer (ring)
    // K block i (in the CTA's issue order) goes to quantizer i % kQWarps and
    // activation slot j = i % kXSlots (two slots per quantizer).  A slot's
    // FP16/BF16 box is free again once its quantizer has read it, so the
    // quantizer reloads it (TMA) for K block i + kXSlots right after
    // quantizing K block i: the boxes run two K blocks of this quantizer
    // ahead.  The slot's E4M3 tile is free once the MMA of K block
    // i - kXSlots has committed.  Each row of a box is one 1x128 token group
    // ([P5] groups, [P2] s3 steps 2-4), quantized by quant_box16_rows sixteen
    // rows at a time into the slot's swizzled E4M3 tile, its scale into the
    // scale-ring slot of this K block.  Every barrier of a slot is waited
    // for and arrived on by its one quantizer, in order.
    if constexpr (Cfg::kRing) {
      const int qwarp = warp < 4 ? warp - 2 : warp - 6;   // 0 .. kQWarps - 1
      constexpr int NQ = Cfg::kQWarps;
      const bool copy_out = p.qa_out != nullptr && tn == 0;
      auto load_box = [&](int k) {   // lane 0: the box of K block k into its slot (the slot's box is free)
        const int j = k % XS;
        ptx::mbar_arrive_expect_tx(&xfull_bar[j], x16_box_bytes);
        ptx::tma_load_2d(xq_ring + j * Cfg::kXSlotBytes, &tmap_x, &xfull_bar[j], kb_at(k) * kBK, 0);
      };
      int next_issue = qwarp, next_wait = qwarp;   // lane 0's bookkeeping of this quantizer's loads
      if (lane == 0)
        for (; next_issue < nkb && next_issue < qwarp + XS; next_issue += NQ) load_box(next_issue);
      bool ok = true;
      for (int i = qwarp; i < nkb; i += NQ) {
        const int j = i % XS;
        const int slot = i % Cfg::kSaSlots;
        bool got = true;
        if (lane == 0) {
          got = ptx::mbar_wait_bounded(&xfull_bar[j], (i / XS) & 1, p.timeout_ns);
          if (got) next_wait = i + NQ;
          got = got && ptx::mbar_wait_bounded(&xempty_bar[j], ((i / XS) & 1) ^ 1, p.timeout_ns) &&
                ptx::mbar_wait_bounded(&sa_free_bar[slot], ((i / Cfg::kSaSlots) & 1) ^ 1, p.timeout_ns);
        }
        if (!__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0)) {
          if (lane == 0) record_error(kErrProducer);
          ok = false;
          break;
        }
        const int kb = kb_at(i);
        const uint32_t xs = ptx::smem_u32(xq_ring + j * Cfg::kXSlotBytes);
        const uint32_t as = xs + static_cast<uint32_t>(Cfg::kX16Bytes);
        uint8_t* qo = copy_out ? p.qa_out + static_cast<int64_t>(kb) * kBK : nullptr;
        float* so = copy_out ? p.sa_out + static_cast<int64_t>(kb) * p.M : nullptr;
        for (int r0 = 0; r0 < MT && r0 < p.M; r0 += 16)
          quant_box16_rows<DT>(xs, as, r0, p.M, lane, sa_ring + slot * MT, qo, p.K, so);
        // the E4M3 bytes before the MMA reads them, and this warp's reads of
        // the box before the next TMA write into it
        ptx::fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&x8_ready_bar[j]);
          ptx::mbar_arrive(&sa_full_bar[slot]);
          if (next_issue < nkb) {
            load_box(next_issue);
            next_issue += NQ;
          }
        }
      }
      // after an error: every load issued and not yet waited for lands
      // before the CTA may exit
      if (lane == 0 && !ok)
        for (int k = next_wait; k < next_issue; k += NQ)
          (void)ptx::mbar_wait_bounded(&xfull_bar[k % XS], (k / XS) & 1, p.timeout_ns);
    }
  } else if (warp >= 4 && warp < 8) {
    // ----------------------------------------------------------- epilogue
    const int epi_tid = threadIdx.x - 128;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;               // weight row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float* sb_row = p.sb + static_cast<int64_t>(tn) * p.num_kb;   // the tile is one weight block row
    float2 acc2[MT / 2];
#pragma unroll
    for (int j = 0; j < MT / 2; ++j) acc2[j] = make_float2(0.0f, 0.0f);
    bool ok = true;
    if constexpr (Cfg::kRes) {
      // these warps quantize their share of the activation first; every
      // warp's token scales are in sa_buf once all six have arrived
      res_quantize();
      bool got = true;
      if (lane == 0) got = ptx::mbar_wait_bounded(act_ready_bar, 0, p.timeout_ns);
      if (!__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0)) {
        if (lane == 0) record_error(kErrEpilogue);
        ok = false;
      }
      __syncwarp();  // lane 0's acquire orders the other lanes' reads too
    }
    // token scales of the next K block (unfused: from global memory, one K
    // block ahead; the tokens past M get 0)
    float sa_n[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) sa_n[m] = 0.0f;
    float sb_n = __ldg(sb_row + kb_at(0));
    if constexpr (!FUSED) {
#pragma unroll
      for (int m = 0; m < MT; ++m) sa_n[m] = m < p.M ? __ldg(p.sa + static_cast<int64_t>(kb_at(0)) * p.M + m) : 0.0f;
    }
    for (int i = 0; i < nkb && ok; ++i) {
      float sa_c[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) sa_c[m] = sa_n[m];
      const float sb_c = sb_n;
      if (i + 1 < nkb) {
        const int kn = kb_at(i + 1);
        sb_n = __ldg(sb_row + kn);
        if constexpr (!FUSED) {
#pragma unroll
          for (int m = 0; m < MT; ++m) sa_n[m] = m < p.M ? __ldg(p.sa + static_cast<int64_t>(kn) * p.M + m) : 0.0f;
        }
      }
      const int buf = i % NBUF;
      if (!ptx::mbar_wait_bounded(&tfull_bar[buf], (i / NBUF) & 1, p.timeout_ns)) {
        record_error(kErrEpilogue);
        ok = false;
        break;
      }
      if constexpr (Cfg::kRes) {
#pragma unroll
        for (int m = 0; m < MT; m += 4) {
          const float4 f = *reinterpret_cast<const float4*>(sa_buf + i * MT + m);
          sa_c[m] = f.x;
          sa_c[m + 1] = f.y;
          sa_c[m + 2] = f.z;
          sa_c[m + 3] = f.w;
        }
      }
      if constexpr (Cfg::kRing) {
        const int slot = i % Cfg::kSaSlots;
        bool got = true;
        if (lane == 0) got = ptx::mbar_wait_bounded(&sa_full_bar[slot], (i / Cfg::kSaSlots) & 1, p.timeout_ns);
        if (!__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0)) {
          if (lane == 0) record_error(kErrEpilogue);
          ok = false;
          break;
        }
        __syncwarp();  // lane 0's acquire orders the other lanes' reads too
#pragma unroll
        for (int m = 0; m < MT; ++m) sa_c[m] = sa_ring[slot * MT + m];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sa_free_bar[slot]);
      }
      ptx::tc_fence_after();
      uint32_t part[MT];
#pragma unroll
      for (int c = 0; c < MT; c += 16) tmem_load_nowait<16>(tmem_base + lane_off + static_cast<uint32_t>(buf * MT + c), &part[c]);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty_bar[buf]);
#pragma unroll
      for (int m = 0; m < MT; m += 2) promote2(acc2[m / 2], part[m], part[m + 1], make_float2(sa_c[m] * sb_c, sa_c[m + 1] * sb_c));
    }
    if (ok) {
      if constexpr (SPLIT) {
        float* srow = staging + row * Cfg::kPitch;
#pragma unroll
        for (int j = 0; j < MT / 2; j += 2)
          *reinterpret_cast<float4*>(srow + 2 * j) = make_float4(acc2[j].x, acc2[j].y, acc2[j + 1].x, acc2[j + 1].y);
        if (!cluster_waited) {
          ptx::cluster_wait();
          cluster_waited = true;
        }
        // push each peer's rows into its receive buffer (as gemm.cuh's split-K)
        constexpr int kPitch = Cfg::kPitch;
        const int R = kBM / static_cast<int>(S);
        const uint32_t slice_bytes = static_cast<uint32_t>(R * kPitch * 4);
        ptx::fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(staged_bar);
        if (epi_tid == 0) {
          if (!ptx::mbar_wait_bounded(staged_bar, 0, p.timeout_ns)) {
            record_error(kErrEpilogue);
            ok = false;
          } else {
            ptx::mbar_arrive_expect_tx(recv_bar, (S - 1) * slice_bytes);
            const uint32_t send0 = ptx::smem_u32(staging), recv0 = ptx::smem_u32(recv), rbar = ptx::smem_u32(recv_bar);
            for (uint32_t k = 1; k < S; ++k) {
              const uint32_t q = (rank + k) % S;
              const uint32_t slot = rank < q ? rank : rank - 1;
              ptx::bulk_copy_to_peer(ptx::mapa(recv0 + slot * slice_bytes, q), send0 + q * slice_bytes, slice_bytes,
                                     ptx::mapa(rbar, q));
            }
          }
        }
        if (ptx::mbar_wait_bounded(recv_bar, 0, p.timeout_ns)) {
          switch (S) {
            case 2: dec_reduce<MT, OUT, 2>(staging, recv, rank, epi_tid, tn, p); break;
            case 4: dec_reduce<MT, OUT, 4>(staging, recv, rank, epi_tid, tn, p); break;
            default: dec_reduce<MT, OUT, 8>(staging, recv, rank, epi_tid, tn, p); break;
          }
        } else {
          record_error(kErrEpilogue);
        }
      } else {
        const int n = tn * kBM + row;
        if (n < p.N) {
          uint16_t* C = reinterpret_cast<uint16_t*>(p.c);
#pragma unroll
          for (int m = 0; m < MT; m += 2) {
            if (m < p.M) C[static_cast<int64_t>(m) * p.N + n] = one_out<OUT>(acc2[m / 2].x);
            if (m + 1 < p.M) C[static_cast<int64_t>(m + 1) * p.N + n] = one_out<OUT>(acc2[m / 2].y);
          }
        }
      }
    }
  }

  if (!cluster_waited) ptx::cluster_wait();  // every thread waits out its split-K arrival before the last barrier
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<Cfg::kTmemCols>(tmem_base);
  }
  if constexpr (SPLIT) ptx::cluster_sync_all();  // no CTA leaves while a peer may touch its shared memory
}

}  // namespace fp8s
