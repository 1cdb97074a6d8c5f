// gemm.cuh -- scaled FP8 GEMM on the 5th-generation tensor cores (sm_103a).
//
// Method ("What is FP8 inference on H100 (Transformer Engine)?", s3 steps
// 5-6 and its pseudocode): acc = qA . qB^T with FP32 accumulation, then the
// output is rescaled by scale_A * scale_B and rounded to FP16/BF16.  The
// block-scaled variant follows the block geometry of the transformers
// "Fine-grained FP8" guide (1x128 activation groups, 128x128 weight blocks):
// the FP32 partial sum of each 128-wide K block is multiplied by its
// activation-group scale and weight-block scale and added into an FP32
// accumulator.
//
// Design (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0      TMA producer: streams 128x128-byte A tiles and BNx128-byte B
//               tiles into a STAGES-deep shared-memory ring (128-byte
//               swizzle), signalling `full` mbarriers by transaction bytes.
//   warp 1      MMA issuer (one thread): tcgen05.mma kind::f8f6f4, M=128,
//               N=BN, K=32, four per 128-byte K block, accumulating in TMEM.
//               tcgen05.commit frees the smem stage and publishes a TMEM
//               accumulator buffer.
//   warp 2      allocates / frees TMEM (NBUF buffers of BN FP32 columns).
//   warps 4-11  two epilogue warpgroups; warp w reads TMEM lanes
//               32*(w%4)..+31 (rows of the tile), warpgroup e reads columns
//               e*BN/2 .. (e+1)*BN/2.
//     per-tensor: the accumulator of a whole tile stays in TMEM; the
//               epilogue loads it once, multiplies by sA*sB, rounds and stores.
//     block:    every K block lands in its own TMEM buffer (the MMA starts a
//               fresh sum per K block); the epilogue loads it, releases the
//               buffer, and adds partial * sa[kb][m] * sb[n/128][kb] into
//               FP32 registers; after the last K block it rounds and stores.
// NBUF TMEM buffers let the MMA run ahead of the epilogue (by whole tiles in
// per-tensor mode, by K blocks in block mode).
//
// Every mbarrier wait is bounded in wall time; on expiry the waiting role
// records where it gave up in g_fp8s_error (quantize.cuh) and leaves its loop; in-flight
// TMA loads and MMAs are drained (also bounded) before TMEM is freed.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"
#include "quantize.cuh"

namespace fp8s {

constexpr int kBM = 128;   // tile rows = MMA M
constexpr int kBK = 128;   // K block: 128 E4M3 bytes = one swizzled smem row
constexpr int kMmaK = 32;  // K of one tcgen05.mma kind::f8f6f4

enum : int { kModePerTensor = 0, kModeBlock = 1 };
enum : int { kOutF16 = 0, kOutBF16 = 1 };

struct GemmParams {
  int M, N, K;
  int num_kb;     // ceil(K / 128)
  int tiles_m, tiles_n, num_tiles;
  int group_m;    // raster: tiles of this many M rows are swept across N together
  const float* sa;
  const float* sb;
  void* c;
  unsigned long long timeout_ns;
};

template <int BN, int MODE>
struct GemmCfg {
  static_assert(BN == 32 || BN == 64 || BN == 128 || BN == 256, "BN");
  static_assert(MODE == kModePerTensor || BN <= 128, "block mode keeps BN/2 accumulators per thread");
  static constexpr int kEpiWarps = 8;
  static constexpr int kThreads = 128 + 32 * kEpiWarps;
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = BN * kBK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStagesRaw = (200 * 1024) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
  // TMEM accumulator buffers: whole tiles (per-tensor) or single K blocks
  // (block mode; narrow tiles get up to 16 so the MMA can run far ahead).
  static constexpr int kNBufMax = MODE == kModeBlock ? 16 : 4;
  static constexpr int kNBuf = (512 / BN) > kNBufMax ? kNBufMax : (512 / BN);
  static constexpr int kTmemCols = kNBuf * BN;
  static constexpr int kColsPerThread = BN / 2;  // per epilogue warpgroup
  static constexpr int kChunk = kColsPerThread < 32 ? kColsPerThread : 32;
  // Block mode: K blocks the epilogue takes per TMEM hand-off (one
  // tcgen05.wait::ld per batch), capped by registers and by half the buffers.
  static constexpr int kBatchRaw = 64 / kColsPerThread;
  static constexpr int kBatch = MODE == kModeBlock ? (kBatchRaw > kNBuf / 2 ? kNBuf / 2 : kBatchRaw) : 1;
  static_assert(kBatch >= 1, "batch");
  static constexpr int kBarBytes = 8 * (2 * kStages + 2 * kNBuf + 1) + 16;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM columns");
};

// First K block of a tile.  Tiles start their K loop at different K blocks
// so that concurrently running CTAs that share an operand (all CTAs of a
// decode-sized GEMM share the whole activation) do not all request the same
// L2 lines at the same time.  Summation order changes per tile, nothing else.
__device__ __forceinline__ int kb_rotation(int tm, int tn, int num_kb) { return (tm + tn) % num_kb; }

__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& tm, int& tn) {
  const int per_group = p.group_m * p.tiles_n;
  const int gid = t / per_group;
  const int first_m = gid * p.group_m;
  const int rows = min(p.tiles_m - first_m, p.group_m);
  const int r = t - gid * per_group;
  tm = first_m + r % rows;
  tn = r / rows;
}

template <int OUT>
__device__ __forceinline__ uint32_t pack_out(float lo, float hi) {
  if constexpr (OUT == kOutF16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <int OUT>
__device__ __forceinline__ uint16_t one_out(float v) {
  if constexpr (OUT == kOutF16) {
    return __half_as_ushort(__float2half_rn(v));
  } else {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

// Rounds and stores W consecutive outputs of one row, starting at column n0.
template <int OUT, int W>
__device__ __forceinline__ void store_row(uint16_t* __restrict__ crow, int n0, int N, bool vec_ok, const float* v) {
  if (vec_ok && n0 + W <= N) {
#pragma unroll
    for (int j = 0; j < W; j += 8) {
      uint4 pk;
      pk.x = pack_out<OUT>(v[j + 0], v[j + 1]);
      pk.y = pack_out<OUT>(v[j + 2], v[j + 3]);
      pk.z = pack_out<OUT>(v[j + 4], v[j + 5]);
      pk.w = pack_out<OUT>(v[j + 6], v[j + 7]);
      *reinterpret_cast<uint4*>(crow + n0 + j) = pk;
    }
  } else {
#pragma unroll
    for (int j = 0; j < W; ++j)
      if (n0 + j < N) crow[n0 + j] = one_out<OUT>(v[j]);
  }
}

// Issues the TMEM load of W columns into r (no wait).
template <int W>
__device__ __forceinline__ void tmem_load_nowait(uint32_t taddr, uint32_t* r) {
  if constexpr (W == 32) {
    ptx::tmem_ld_32x32b_x32(taddr, *reinterpret_cast<uint32_t(*)[32]>(r));
  } else {
    static_assert(W == 16, "chunk width");
    ptx::tmem_ld_32x32b_x16(taddr, *reinterpret_cast<uint32_t(*)[16]>(r));
  }
}

template <int W>
__device__ __forceinline__ void tmem_load_chunk(uint32_t taddr, float* out) {
  if constexpr (W == 32) {
    uint32_t r[32];
    ptx::tmem_ld_32x32b_x32(taddr, r);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) out[j] = __uint_as_float(r[j]);
  } else {
    static_assert(W == 16, "chunk width");
    uint32_t r[16];
    ptx::tmem_ld_32x32b_x16(taddr, r);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) out[j] = __uint_as_float(r[j]);
  }
}

template <int BN, int MODE, int OUT>
__global__ void __launch_bounds__(GemmCfg<BN, MODE>::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const GemmParams p) {
  using Cfg = GemmCfg<BN, MODE>;
  constexpr int S = Cfg::kStages;
  constexpr int NBUF = Cfg::kNBuf;
  constexpr int CPT = Cfg::kColsPerThread;
  constexpr int CW = Cfg::kChunk;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + S * Cfg::kABytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem_b + S * Cfg::kBBytes);
  uint64_t* empty_bar = full_bar + S;
  uint64_t* tfull_bar = empty_bar + S;
  uint64_t* tempty_bar = tfull_bar + NBUF;
  uint64_t* mma_done_bar = tempty_bar + NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done_bar + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmap_a);
    ptx::tma_prefetch_desc(&tmap_b);
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      ptx::mbar_init(&tfull_bar[b], 1);
      ptx::mbar_init(&tempty_bar[b], Cfg::kEpiWarps);
    }
    ptx::mbar_init(mma_done_bar, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 2) {
    ptx::tmem_alloc<Cfg::kTmemCols>(tmem_slot);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int tm, tn;
        tile_coords(t, p, tm, tn);
        const int rot = kb_rotation(tm, tn, p.num_kb);
        for (int i = 0; i < p.num_kb; ++i) {
          const int kb = (i + rot) % p.num_kb;
          const int s = issued % S;
          const uint32_t ph = (issued / S) & 1;
          if (!ptx::mbar_wait_bounded(&empty_bar[s], ph ^ 1, p.timeout_ns)) {
            record_error(kErrProducer);
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full_bar[s], Cfg::kStageBytes);
          ptx::tma_load_2d(smem_a + s * Cfg::kABytes, &tmap_a, &full_bar[s], kb * kBK, tm * kBM);
          ptx::tma_load_2d(smem_b + s * Cfg::kBBytes, &tmap_b, &full_bar[s], kb * kBK, tn * BN);
          ++issued;
        }
      }
      // Drain: every issued load has landed before the CTA may exit.
      const uint32_t first = issued > S ? issued - S : 0;
      for (uint32_t j = first; j < issued; ++j)
        if (!ptx::mbar_wait_bounded(&full_bar[j % S], (j / S) & 1, p.timeout_ns)) record_error(kErrProducer);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_e4m3_f32(kBM, BN);
      const uint32_t a0 = ptx::smem_u32(smem_a);
      const uint32_t b0 = ptx::smem_u32(smem_b);
      uint32_t consumed = 0, unit = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        for (int kb = 0; kb < p.num_kb && ok; ++kb) {  // kb counts K blocks of the tile in issue order
          const bool new_unit = (MODE == kModeBlock) || kb == 0;
          const uint32_t buf = unit % NBUF;
          if (new_unit) {
            if (!ptx::mbar_wait_bounded(&tempty_bar[buf], ((unit / NBUF) & 1) ^ 1, p.timeout_ns)) {
              record_error(kErrMma);
              ok = false;
              break;
            }
            ptx::tc_fence_after();
          }
          const int s = consumed % S;
          if (!ptx::mbar_wait_bounded(&full_bar[s], (consumed / S) & 1, p.timeout_ns)) {
            record_error(kErrMma);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t adesc = ptx::smem_desc_sw128_kmajor(a0 + s * Cfg::kABytes);
          const uint64_t bdesc = ptx::smem_desc_sw128_kmajor(b0 + s * Cfg::kBBytes);
          const uint32_t d = tmem_base + buf * BN;
#pragma unroll
          for (int k = 0; k < kBK / kMmaK; ++k) {
            // advance 32 bytes (2 x 16-byte units) along K inside the swizzled row
            const uint32_t acc = (MODE == kModeBlock) ? (k > 0) : (kb > 0 || k > 0);
            ptx::mma_f8f6f4(d, adesc + 2 * k, bdesc + 2 * k, idesc, acc);
          }
          ptx::mma_commit(&empty_bar[s]);
          ++consumed;
          const bool unit_done = (MODE == kModeBlock) || kb == p.num_kb - 1;
          if (unit_done) {
            ptx::mma_commit(&tfull_bar[buf]);
            ++unit;
          }
        }
      }
      // Drain: all issued MMAs complete before TMEM can be released.
      ptx::mma_commit(mma_done_bar);
      if (!ptx::mbar_wait_bounded(mma_done_bar, 0, p.timeout_ns)) record_error(kErrMma);
    }
  } else if (warp >= 4) {
    // ----------------------------------------------------------- epilogue
    const int epi_warp = warp - 4;
    const int quarter = warp & 3;   // TMEM lane quarter this warp may access
    const int wg = epi_warp >> 2;   // column half of the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const bool vec_ok = (p.N % 8) == 0;
    uint16_t* C = reinterpret_cast<uint16_t*>(p.c);
    const int KB = p.num_kb;
    uint32_t unit = 0;
    bool ok = true;

    float pt_scale = 0.0f;
    if constexpr (MODE == kModePerTensor) pt_scale = __ldg(p.sa) * __ldg(p.sb);

    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      int tm, tn;
      tile_coords(t, p, tm, tn);
      const int row = tm * kBM + quarter * 32 + lane;
      const int n_base = tn * BN + wg * CPT;
      uint16_t* crow = C + static_cast<int64_t>(row) * p.N;

      if constexpr (MODE == kModePerTensor) {
        const uint32_t buf = unit % NBUF;
        if (!ptx::mbar_wait_bounded(&tfull_bar[buf], (unit / NBUF) & 1, p.timeout_ns)) {
          record_error(kErrEpilogue);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int c = 0; c < CPT / CW; ++c) {
          float v[CW];
          tmem_load_chunk<CW>(tmem_base + lane_off + buf * BN + wg * CPT + c * CW, v);
#pragma unroll
          for (int j = 0; j < CW; ++j) v[j] *= pt_scale;
          if (row < p.M) store_row<OUT, CW>(crow, n_base + c * CW, p.N, vec_ok, v);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&tempty_bar[buf]);
        ++unit;
      } else {
        constexpr int KBT = Cfg::kBatch;
        float acc[CPT];
#pragma unroll
        for (int j = 0; j < CPT; ++j) acc[j] = 0.0f;
        const int nb = n_base / 128;  // weight block row of this warpgroup's columns
        const float* sa_col = p.sa + (row < p.M ? row : 0);
        const float* sb_row = p.sb + static_cast<int64_t>(nb) * KB;
        const int rot = kb_rotation(tm, tn, KB);
        auto kb_at = [&](int i) { return i + rot < KB ? i + rot : i + rot - KB; };  // i-th K block issued
        float sa_n[KBT], sb_n[KBT];
#pragma unroll
        for (int j = 0; j < KBT; ++j) {
          sa_n[j] = j < KB ? __ldg(sa_col + static_cast<int64_t>(kb_at(j)) * p.M) : 0.0f;
          sb_n[j] = j < KB ? __ldg(sb_row + kb_at(j)) : 0.0f;
        }
        for (int kb0 = 0; kb0 < KB; kb0 += KBT) {
          const int nkb = min(KBT, KB - kb0);
          float sc[KBT];
#pragma unroll
          for (int j = 0; j < KBT; ++j) {
            sc[j] = sa_n[j] * sb_n[j];
            const int kn = kb0 + KBT + j;  // prefetch the next batch's scales
            sa_n[j] = kn < KB ? __ldg(sa_col + static_cast<int64_t>(kb_at(kn)) * p.M) : 0.0f;
            sb_n[j] = kn < KB ? __ldg(sb_row + kb_at(kn)) : 0.0f;
          }
          for (int j = 0; j < nkb && ok; ++j) {
            const uint32_t u = unit + j;
            if (!ptx::mbar_wait_bounded(&tfull_bar[u % NBUF], (u / NBUF) & 1, p.timeout_ns)) {
              record_error(kErrEpilogue);
              ok = false;
            }
          }
          if (!ok) break;
          ptx::tc_fence_after();
          uint32_t part[KBT][CPT];
#pragma unroll
          for (int j = 0; j < KBT; ++j) {
            if (j < nkb) {
              const uint32_t col0 = ((unit + j) % NBUF) * BN + wg * CPT;
#pragma unroll
              for (int c = 0; c < CPT / CW; ++c)
                tmem_load_nowait<CW>(tmem_base + lane_off + col0 + c * CW, &part[j][c * CW]);
            }
          }
          ptx::tmem_ld_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0)
            for (int j = 0; j < nkb; ++j) ptx::mbar_arrive(&tempty_bar[(unit + j) % NBUF]);
          unit += nkb;
#pragma unroll
          for (int j = 0; j < KBT; ++j)
            if (j < nkb) {
#pragma unroll
              for (int c = 0; c < CPT; ++c) acc[c] = fmaf(__uint_as_float(part[j][c]), sc[j], acc[c]);
            }
        }
        if (!ok) break;
        if (row < p.M) {
#pragma unroll
          for (int c = 0; c < CPT / CW; ++c) store_row<OUT, CW>(crow, n_base + c * CW, p.N, vec_ok, acc + c * CW);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<Cfg::kTmemCols>(tmem_base);
  }
}

}  // namespace fp8s
