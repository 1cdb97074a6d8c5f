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
// Design (persistent over output tiles of 128 x BN):
//   warp 0      TMA producer: streams 128x128-byte A tiles and BNx128-byte B
//               tiles into a STAGES-deep shared-memory ring (128-byte
//               swizzle), signalling `full` mbarriers by transaction bytes.
//   warp 1      MMA issuer (one thread): tcgen05.mma kind::f8f6f4, M=128,
//               N=BN, K=32, four per 128-byte K block, accumulating in TMEM.
//               tcgen05.commit frees the smem stage and publishes a TMEM
//               accumulator buffer.
//   warp 2      allocates / frees TMEM (NBUF buffers of BN FP32 columns).
//   warps 4..   epilogue warpgroups; warp w reads TMEM lanes 32*(w%4)..+31
//               (rows of the tile), warpgroup e reads columns
//               e*CPT .. (e+1)*CPT (CPT = BN / number of epilogue warpgroups).
//     per-tensor: the accumulator of a whole tile stays in TMEM; the
//               epilogue loads it once, multiplies by sA*sB, rounds and stores.
//     block:    every K block lands in its own TMEM buffer (the MMA starts a
//               fresh sum per K block); the epilogue loads it, releases the
//               buffer, and adds partial * sa[kb][m] * sb[n/128][kb] into
//               FP32 registers; after the last K block it rounds and stores.
// NBUF TMEM buffers let the MMA run ahead of the epilogue (by whole tiles in
// per-tensor mode, by K blocks in block mode).
//
// Split-K over a thread-block cluster (SPLIT = true, for shapes with too few
// output tiles to occupy the GPU): the S CTAs of a cluster share one output
// tile and CTA rank r takes K blocks [r*KB/S, (r+1)*KB/S).  Every cluster
// owns exactly one tile, so once its last MMA has retired the operand ring is
// idle and doubles as the staging buffer: each CTA leaves its FP32 partial
// tile (already rescaled) there, 128 columns per pass; after a cluster-wide
// mbarrier hand-off, rank r sums rows [r*128/S, (r+1)*128/S) of all S
// partials in rank order (distributed shared memory loads), rounds and
// stores them.  The summation order is fixed, so results are deterministic,
// and no global scratch memory is used.
//
// CTA pairs (PAIR = true, large shapes): the two CTAs of a cluster share an
// output tile of 256 x BN.  Each loads its own 128 rows of A and half (BN/2
// rows) of B per K block; the leader (even rank) issues tcgen05.mma
// .cta_group::2 with M = 256, which reads both CTAs' shared memory and writes
// each CTA's 128 rows into its own TMEM, and multicasts its commits to both
// CTAs.  Per CTA this halves the B operand traffic of a 128 x BN tile, so a
// 256 x 128 pair tile feeds the tensor core like a 128 x 256 single-CTA tile
// while each epilogue keeps a 128 x 128 accumulator.
//
// Every mbarrier wait is bounded in wall time; on expiry the waiting role
// records where it gave up in g_fp8s_error (quantize.cuh) and leaves its
// loop; in-flight TMA loads and MMAs are drained (also bounded) before TMEM is
// freed, and CTAs of a cluster leave together through one cluster barrier.
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

// Per-channel weights (one sB per output column) run the per-tensor kernel
// with a per-column epilogue scale.  kModeUE8 is the block geometry with
// power-of-two (UE8M0) scales, applied by the tensor core itself
// (kind::mxf8f6f4.block_scale): the accumulator then spans the whole K range
// like per-tensor mode, and the epilogue only rounds.
enum : int { kModePerTensor = 0, kModeBlock = 1, kModePerChannel = 2, kModeUE8 = 3 };
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
  // fused activation quantization: optional copies of the E4M3 activation
  // [M][K] and its token-group scales [K/128][M] (written by the CTAs of
  // tile column 0)
  uint8_t* qa_out;
  float* sa_out;
  // fused decode with a resident activation: the FP16/BF16 activation [M][K]
  const void* x;
};

// FR > 0: the fused linear.  A arrives as FP16/BF16 (the output's type) in
// boxes of FR rows x 128 columns and is quantized per 1x128 token group
// inside the kernel (block mode only).
template <int BN, int MODE, bool SPLIT, bool PAIR = false, int FR = 0>
struct GemmCfg {
  static_assert(BN == 32 || BN == 64 || BN == 128 || BN == 192 || BN == 256, "BN");
  static_assert(!(SPLIT && PAIR), "a CTA pair does not also split K");
  static_assert(!PAIR || BN >= 64, "a CTA pair holds at least 32 rows of B each");
  // (UE8M0 pairs share B by multicast: the scale factors stay per CTA)
  // Block mode keeps 64 FP32 accumulators per epilogue thread: BN = 192 and
  // 256 need three and four epilogue warpgroups.
  // UE8M0 mode with BN = 256 keeps a single TMEM accumulator, which the
  // epilogue must hand back quickly: four warpgroups of 64 columns load the
  // whole tile before any store.
  static constexpr int kEpiWarps = MODE == kModeUE8 ? (BN == 256 ? 16 : 8)
                                 : MODE != kModeBlock ? 8 : BN == 256 ? 16 : BN == 192 ? 12 : 8;
  static constexpr int kEpiWG = kEpiWarps / 4;
  static constexpr int kEpiThreads = 32 * kEpiWarps;
  static constexpr int kThreads = 128 + kEpiThreads;
  static constexpr bool kLowReg = kEpiWarps == 16;  // 640 threads: at most 96 registers each
  // Block mode with 12 or 16 epilogue warps (at most 128 or 96 registers a
  // thread) reads a K block's partial 32 or 16 columns per wait, so only one
  // chunk is staged next to the 64 accumulators.
  static constexpr bool kSeqChunks = MODE == kModeBlock && kEpiWarps >= 12;
  // Columns of a K block's partial loaded per wait.
  static constexpr int kSeqLoadCols = kLowReg ? 16 : 32;
  // PAIR: two CTAs of a cluster share a 256-row tile.  Per-tensor modes
  // issue cta_group::2 MMAs over both CTAs (kPairMma); the two block modes
  // keep single-CTA MMAs (the FP32 path's per-K-block TMEM hand-off and the
  // UE8M0 scale factors stay inside one CTA) and share the B tile instead:
  // each CTA loads half of it with a TMA multicast into both CTAs' shared
  // memory (kMcB).
  static constexpr bool kMcB = PAIR && (MODE == kModeBlock || MODE == kModeUE8);
  static constexpr bool kPairMma = PAIR && !kMcB;
  static_assert(!kMcB || BN == 256, "B multicast pairs: 256-wide tiles");
  static constexpr int kTileM = PAIR ? 2 * kBM : kBM;   // output rows per (pair) tile
  static constexpr int kBRows = kPairMma ? BN / 2 : BN;  // rows of B this CTA's shared memory holds
  static constexpr bool kFused = FR > 0;
  static_assert(!kFused || (MODE == kModeBlock && !PAIR && (BN <= 128 || (BN == 192 && (!SPLIT || FR == 16))) &&
                             (FR == 16 || FR == 128)),
                "fused activation quantization: block mode, single CTAs, 16- or 128-row boxes");
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = kBRows * kBK;
  static constexpr int kXBytes = FR * kBK * 2;            // fused: FP16/BF16 activation box
  static constexpr int kStageBytes = kABytes + kBBytes + kXBytes;
  static constexpr int kSaSlots = kFused ? 8 : 0;         // fused: ring of per-K-block token scales
  static constexpr int kSaBytes = kSaSlots * kBM * 4;
  // Split-K partial: 128 rows x BN FP32, rows padded by 4 words so that
  // 16-byte writes of 8 consecutive rows cover all 32 banks.  The outgoing
  // partial aliases the drained operand ring; the incoming slices of up to 7
  // peers (at most 112 rows in all) have a buffer of their own.
  static_assert(!SPLIT || BN <= 192, "split-K exchanges a 128 x BN partial in one pass");
  // A fused kernel with 16-row activation boxes serves M <= 16: its partial
  // has at most 16 valid rows, which is all it stages and exchanges.
  static constexpr int kPartRows = (FR > 0 && FR < kBM) ? FR : kBM;
  static constexpr int kStagePitch = BN + 4;
  static constexpr int kStagingBytes = kPartRows * kStagePitch * 4;
  static constexpr int kRecvBytes = SPLIT ? (kPartRows - kPartRows / 8) * kStagePitch * 4 : 0;
  // UE8M0 scale factors: per group of four K blocks, one 32-bit word (a
  // byte per K block) per row of A and per row of B.  Warp 3 stages them in
  // shared memory as tiles of 32 rows x 16 bytes, one per 128 rows of the
  // operand: row r of a tile holds the words of rows r, 32 + r, 64 + r and
  // 96 + r of those 128.  The MMA issuer copies each tile into four TMEM
  // columns (tcgen05.cp ... warpx4).  A ring of kSfSlots groups, each slot
  // with shared memory and TMEM columns of its own.
  static constexpr bool kUE8 = MODE == kModeUE8;
  static constexpr int kSfbTiles = kUE8 ? (BN + 127) / 128 : 0;   // scale tiles of B (one per 128 rows)
  static constexpr int kSfSlots = kUE8 ? (SPLIT ? 4 : 8) : 0;   // split-K: the ring also stages the partial
  static constexpr int kSfSlotBytes = 512 * (1 + kSfbTiles);
  static constexpr int kSfBytes = kSfSlots * kSfSlotBytes;
  static constexpr int kSfCols = 4 * (1 + kSfbTiles);               // TMEM columns per slot
  static constexpr int kStagesRaw = (214 * 1024 - kRecvBytes - kSfBytes - kSaBytes) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(!SPLIT || kStages * kStageBytes >= kStagingBytes, "staging fits in the ring");
  // TMEM accumulator buffers: whole tiles (per-tensor) or single K blocks
  // (block mode; narrow tiles get up to 16 so the MMA can run far ahead).
  static constexpr int kNBufMax = MODE == kModeBlock ? 16 : 4;
  static constexpr int kTmemMax = 512 - kSfSlots * kSfCols;
  static constexpr int kNBuf = (kTmemMax / BN) > kNBufMax ? kNBufMax : (kTmemMax / BN);
  static constexpr int kTmemAccCols = kNBuf * BN;
  static constexpr int kTmemCols = kTmemAccCols + kSfSlots * kSfCols;
  static constexpr int kTmemAlloc = kTmemCols <= 32 ? 32 : kTmemCols <= 64 ? 64 : kTmemCols <= 128 ? 128
                                  : kTmemCols <= 256 ? 256 : 512;  // allocations are powers of two
  static constexpr int kColsPerThread = BN / kEpiWG;
  static constexpr int kChunk = kLowReg ? 16 : (kColsPerThread < 32 ? kColsPerThread : 32);
  static_assert(kColsPerThread % kChunk == 0, "chunks tile a thread's columns");
  // Block mode: K blocks the epilogue takes per TMEM hand-off (one
  // tcgen05.wait::ld per batch), capped by registers and by half the buffers.
  static constexpr int kBatchRaw = 64 / kColsPerThread;
  static constexpr int kBatch =
      (MODE == kModeBlock && !kSeqChunks) ? (kBatchRaw > kNBuf / 2 ? kNBuf / 2 : kBatchRaw) : 1;
  static_assert(kBatch >= 1, "batch");
  static constexpr int kBarBytes =
      8 * (2 * kStages + 2 * kNBuf + 1 + 2 + 2 * kSfSlots + (kFused ? 2 * kStages + 2 * kSaSlots : 0)) + 16;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kRecvBytes + kSfBytes + kSaBytes + kBarBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kTmemCols <= 512, "TMEM columns");
};

// First K block (within the CTA's K range) of a tile.  Tiles start their K
// loop at different K blocks so that concurrently running CTAs that share an
// operand (all CTAs of a decode-sized GEMM share the whole activation) do not
// all request the same L2 lines at the same time.  Summation order changes
// per tile, nothing else.
__device__ __forceinline__ int kb_rotation(int tm, int tn, int nkb) { return (tm + tn) % nkb; }

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
  uint32_t r[W];
  tmem_load_nowait<W>(taddr, r);
  ptx::tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < W; ++j) out[j] = __uint_as_float(r[j]);
}

// acc += {p0, p1} * sc: one packed FMA for two accumulators (each half rounds
// exactly like fmaf).  The accumulators are kept as FP32 pairs (float2), so
// the packed FMA needs no moves to form its operands.
__device__ __forceinline__ void promote2(float2& acc, uint32_t p0, uint32_t p1, float2 sc) {
  acc = __ffma2_rn(make_float2(__uint_as_float(p0), __uint_as_float(p1)), sc, acc);
}

// As store_row, for W values held as W/2 FP32 pairs.
template <int OUT, int W>
__device__ __forceinline__ void store_row2(uint16_t* __restrict__ crow, int n0, int N, bool vec_ok, const float2* v) {
  if (vec_ok && n0 + W <= N) {
#pragma unroll
    for (int j = 0; j < W / 2; j += 4) {
      uint4 pk;
      pk.x = pack_out<OUT>(v[j + 0].x, v[j + 0].y);
      pk.y = pack_out<OUT>(v[j + 1].x, v[j + 1].y);
      pk.z = pack_out<OUT>(v[j + 2].x, v[j + 2].y);
      pk.w = pack_out<OUT>(v[j + 3].x, v[j + 3].y);
      *reinterpret_cast<uint4*>(crow + n0 + 2 * j) = pk;
    }
  } else {
#pragma unroll
    for (int j = 0; j < W / 2; ++j) {
      if (n0 + 2 * j < N) crow[n0 + 2 * j] = one_out<OUT>(v[j].x);
      if (n0 + 2 * j + 1 < N) crow[n0 + 2 * j + 1] = one_out<OUT>(v[j].y);
    }
  }
}

// Writes W consecutive FP32 values, held as W/2 pairs, of one staging row.
template <int W>
__device__ __forceinline__ void stage_row2(float* srow, const float2* v) {
#pragma unroll
  for (int j = 0; j < W / 2; j += 2)
    *reinterpret_cast<float4*>(srow + 2 * j) = make_float4(v[j].x, v[j].y, v[j + 1].x, v[j + 1].y);
}

// Writes W consecutive FP32 values of one staging row (16-byte stores).
template <int W>
__device__ __forceinline__ void stage_row(float* srow, const float* v) {
#pragma unroll
  for (int j = 0; j < W; j += 4) *reinterpret_cast<float4*>(srow + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
}

// Tells the MMA issuer a TMEM accumulator buffer has been read.  In a CTA
// pair the issuer (and the barrier) lives in the leader CTA.
template <bool PAIR>
__device__ __forceinline__ void release_tmem(uint64_t* bar) {
  // The TMEM reads are ordered by tcgen05.wait::ld and the before-sync fence
  // the caller issued; no memory operation needs releasing.
  if constexpr (PAIR) ptx::mbar_arrive_cluster_relaxed(ptx::mapa(ptx::smem_u32(bar), 0));
  else ptx::mbar_arrive(bar);
}

// Rows of a split-K tile each rank reduces: the tile's valid rows (all 128
// unless the tile holds the last rows of M) split evenly over the S ranks;
// S * R <= 128 always.  A decode batch of a few tokens exchanges a few rows.
__device__ __forceinline__ int split_rows(const GemmParams& p, int tm, int S) {
  const int mt = min(kBM, p.M - tm * kBM);
  return (mt + S - 1) / S;
}

// Sums this CTA's R rows over the S partials in rank order (its own in
// `send`, peer q's in receive slot q < rank ? q : q - 1), rounds and stores
// them.  S is a template parameter so that the S loads of an output vector
// are issued together; each thread takes two 4-column vectors per
// iteration.
template <int BN, int OUT, int S>
__device__ __forceinline__ void reduce_rows(const float* send, const float* recv, uint32_t rank, int tid, int nthreads,
                                            int tm, int tn, int R, const GemmParams& p) {
  constexpr int kPitch = BN + 4;
  constexpr int kVecPerRow = BN / 4;
  const int kTotal = R * kVecPerRow;
  uint16_t* C = reinterpret_cast<uint16_t*>(p.c);
  const bool vec_ok = (p.N % 4) == 0;
  const float* src[S];
#pragma unroll
  for (int q = 0; q < S; ++q)
    src[q] = q == static_cast<int>(rank) ? send + static_cast<int>(rank) * R * kPitch
                                         : recv + (q < static_cast<int>(rank) ? q : q - 1) * R * kPitch;
  for (int v0 = tid; v0 < kTotal; v0 += 2 * nthreads) {
    float4 t[2][S];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int v = v0 + u * nthreads;
      const int off = (v / kVecPerRow) * kPitch + (v % kVecPerRow) * 4;
#pragma unroll
      for (int q = 0; q < S; ++q)
        t[u][q] = v < kTotal ? *reinterpret_cast<const float4*>(src[q] + off) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int v = v0 + u * nthreads;
      if (v >= kTotal) continue;
      float4 acc = t[u][0];
#pragma unroll
      for (int q = 1; q < S; ++q) {
        acc.x += t[u][q].x;
        acc.y += t[u][q].y;
        acc.z += t[u][q].z;
        acc.w += t[u][q].w;
      }
      const int row = tm * kBM + static_cast<int>(rank) * R + v / kVecPerRow;
      const int n = tn * BN + (v % kVecPerRow) * 4;
      if (row >= p.M) continue;
      uint16_t* crow = C + static_cast<int64_t>(row) * p.N;
      if (vec_ok && n + 4 <= p.N) {
        uint2 pk;
        pk.x = pack_out<OUT>(acc.x, acc.y);
        pk.y = pack_out<OUT>(acc.z, acc.w);
        *reinterpret_cast<uint2*>(crow + n) = pk;
      } else {
        const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (n + j < p.N) crow[n + j] = one_out<OUT>(a4[j]);
      }
    }
  }
}

// Split-K exchange, pushed through the cluster's shared memory.  Rank r of
// S owns output rows [r*R, (r+1)*R), R = 128/S.  Once every epilogue warp of
// this CTA has written its part of the partial into `send` (signalled on the
// CTA-local `staged` barrier), one thread copies the R-row slice owned by
// each peer q straight into q's receive buffer with a bulk copy
// (cp.async.bulk shared::cta -> shared::cluster) that completes on q's
// `recv` barrier; the data arriving is the signal.  Each CTA then waits for
// its S-1 incoming slices, sums its rows over all S partials in rank order
// (local shared memory only), rounds and stores.  Slot j of the receive
// buffer holds the slice of peer q, j = q < r ? q : q - 1.  Every wait is
// bounded; returns false (after recording the error) if one gave up.
template <int BN, int OUT>
__device__ __forceinline__ bool exchange_and_reduce(uint64_t* staged_bar, uint64_t* recv_bar, const float* send,
                                                    const float* recv, uint32_t rank, uint32_t S, int tid,
                                                    int nthreads, int tm, int tn, const GemmParams& p) {
  constexpr int kPitch = BN + 4;
  const int R = split_rows(p, tm, static_cast<int>(S));
  const uint32_t slice_bytes = static_cast<uint32_t>(R * kPitch * 4);   // a multiple of 16 for every BN
  const int lane = tid & 31;
  ptx::fence_proxy_async_shared();  // this thread's ordinary stores, before the bulk copies read them
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(staged_bar);
  if (tid == 0) {
    if (!ptx::mbar_wait_bounded(staged_bar, 0, p.timeout_ns)) {
      record_error(kErrEpilogue);
      return false;
    }
    // After the staged wait, so that threads which see `recv` complete also
    // see every warp's part of this CTA's own slice.  Incoming bytes may land
    // before this; the phase cannot complete until this arrival.
    ptx::mbar_arrive_expect_tx(recv_bar, (S - 1) * slice_bytes);
    const uint32_t send0 = ptx::smem_u32(send), recv0 = ptx::smem_u32(recv), rbar = ptx::smem_u32(recv_bar);
    // peers in the order rank+1, rank+2, ...: the S CTAs start on S
    // different destinations instead of all sending to rank 0 first
    for (uint32_t i = 1; i < S; ++i) {
      const uint32_t q = (rank + i) % S;
      const uint32_t slot = rank < q ? rank : rank - 1;  // this CTA's slot in q's receive buffer
      // two copies per slice (both 16-byte multiples): more requests in flight
      const uint32_t h = (slice_bytes / 2) & ~15u;
      ptx::bulk_copy_to_peer(ptx::mapa(recv0 + slot * slice_bytes, q), send0 + q * slice_bytes, h,
                             ptx::mapa(rbar, q));
      ptx::bulk_copy_to_peer(ptx::mapa(recv0 + slot * slice_bytes + h, q), send0 + q * slice_bytes + h,
                             slice_bytes - h, ptx::mapa(rbar, q));
    }
  }
  if (!ptx::mbar_wait_bounded(recv_bar, 0, p.timeout_ns)) {
    record_error(kErrEpilogue);
    return false;
  }
  switch (S) {
    case 2: reduce_rows<BN, OUT, 2>(send, recv, rank, tid, nthreads, tm, tn, R, p); break;
    case 4: reduce_rows<BN, OUT, 4>(send, recv, rank, tid, nthreads, tm, tn, R, p); break;
    default: reduce_rows<BN, OUT, 8>(send, recv, rank, tid, nthreads, tm, tn, R, p); break;
  }
  return true;
}

// Per-tensor epilogue scaling of CW consecutive columns from n0: by the
// product sA*sB, or with per-channel weights by sA*sB[n] (the clamped column
// keeps a ragged tile's loads inside sB; those columns are never stored).
template <int MODE, int CW>
__device__ __forceinline__ void scale_chunk(float* v, float pt_scale, float sa, const GemmParams& p, int n0) {
  if constexpr (MODE == kModeUE8) {
    // the tensor core has applied the scales already
  } else if constexpr (MODE == kModePerChannel) {
#pragma unroll
    for (int j = 0; j < CW; ++j) v[j] *= sa * __ldg(p.sb + (n0 + j < p.N ? n0 + j : p.N - 1));
  } else {
#pragma unroll
    for (int j = 0; j < CW; ++j) v[j] *= pt_scale;
  }
}

template <int BN, int MODE, int OUT, bool SPLIT, bool PAIR, int FR = 0>
__global__ void __launch_bounds__(GemmCfg<BN, MODE, SPLIT, PAIR, FR>::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const GemmParams p) {
  using Cfg = GemmCfg<BN, MODE, SPLIT, PAIR, FR>;
  constexpr int DT = OUT;  // fused: the activation has the output's type (kInF16 == kOutF16, kInBF16 == kOutBF16)
  constexpr int TM = Cfg::kTileM;
  constexpr int S_ = Cfg::kStages;
  constexpr int NBUF = Cfg::kNBuf;
  constexpr int CPT = Cfg::kColsPerThread;
  constexpr int CW = Cfg::kChunk;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + S_ * Cfg::kABytes;
  uint8_t* smem_x = smem_b + S_ * Cfg::kBBytes;  // fused: FP16/BF16 activation boxes
  float* staging = reinterpret_cast<float*>(smem);  // split-K only: used after the ring has drained
  const float* recv = reinterpret_cast<const float*>(smem + S_ * Cfg::kStageBytes);  // split-K incoming slices
  uint8_t* sf_smem = smem + S_ * Cfg::kStageBytes + Cfg::kRecvBytes;  // UE8M0: scale-factor tiles
  float* sa_ring = reinterpret_cast<float*>(sf_smem + Cfg::kSfBytes);   // fused: [kSaSlots][128] token scales
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sa_ring) + Cfg::kSaBytes);
  uint64_t* empty_bar = full_bar + S_;
  uint64_t* tfull_bar = empty_bar + S_;
  uint64_t* tempty_bar = tfull_bar + NBUF;
  uint64_t* mma_done_bar = tempty_bar + NBUF;
  uint64_t* staged_bar = mma_done_bar + 1;  // split-K: every epilogue warp of this CTA staged its part
  uint64_t* recv_bar = staged_bar + 1;      // split-K: all S-1 incoming slices have landed
  uint64_t* sf_full_bar = recv_bar + 1;     // UE8M0: a scale-factor slot has been staged
  uint64_t* sf_empty_bar = sf_full_bar + Cfg::kSfSlots;  // UE8M0: its MMAs are done with it
  uint64_t* a8_ready_bar = sf_empty_bar + Cfg::kSfSlots;  // fused: stage's E4M3 activation written
  uint64_t* xfull_bar = a8_ready_bar + (Cfg::kFused ? S_ : 0);    // fused: stage's FP16/BF16 box landed
  uint64_t* sa_full_bar = xfull_bar + (Cfg::kFused ? S_ : 0);     // fused: a scale slot written
  uint64_t* sa_free_bar = sa_full_bar + Cfg::kSaSlots;            // fused: a scale slot read by the epilogue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sa_free_bar + Cfg::kSaSlots);
  volatile uint32_t* pair_bad = tmem_slot + 1;  // CTA pair: the two TMEM allocations disagree

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work split: without split-K every CTA is its own "cluster" of one; a CTA
  // pair is a cluster of two sharing one tile and the whole K range.
  uint32_t rank = 0, S = 1, prank = 0;
  if constexpr (SPLIT) {
    rank = ptx::cluster_ctarank();
    S = ptx::cluster_nctarank();
  }
  if constexpr (PAIR) prank = ptx::cluster_ctarank();
  const bool leader = !Cfg::kPairMma || prank == 0;   // issues the MMAs
  const int csize = PAIR ? 2 : static_cast<int>(S);
  const int cluster_id = static_cast<int>(blockIdx.x / csize);
  const int num_clusters = static_cast<int>(gridDim.x / csize);
  const int kb_begin = static_cast<int>((static_cast<int64_t>(rank) * p.num_kb) / S);
  const int kb_end = static_cast<int>((static_cast<int64_t>(rank + 1) * p.num_kb) / S);
  const int nkb = kb_end - kb_begin;  // >= 1: the host keeps S <= num_kb
  // Split-K reuses the operand ring as staging, which is only safe when every
  // cluster owns a single tile; the host guarantees it, this is a backstop.
  if (SPLIT && num_clusters < p.num_tiles) {
    if (threadIdx.x == 0 && rank == 0) record_error(kErrProducer);
    return;
  }

  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmap_a);
    ptx::tma_prefetch_desc(&tmap_b);
    for (int s = 0; s < S_; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      // B multicast: a stage is free once both CTAs' MMAs have read it
      ptx::mbar_init(&empty_bar[s], Cfg::kMcB ? 2 : 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      ptx::mbar_init(&tfull_bar[b], 1);
      ptx::mbar_init(&tempty_bar[b], (Cfg::kPairMma ? 2 : 1) * Cfg::kEpiWarps);
    }
    ptx::mbar_init(mma_done_bar, 1);
    ptx::mbar_init(staged_bar, Cfg::kEpiWarps);
    ptx::mbar_init(recv_bar, 1);
    for (int j = 0; j < Cfg::kSfSlots; ++j) {
      ptx::mbar_init(&sf_full_bar[j], 1);
      ptx::mbar_init(&sf_empty_bar[j], 1);
    }
    if constexpr (Cfg::kFused) {
      for (int j = 0; j < S_; ++j) {
        ptx::mbar_init(&a8_ready_bar[j], 2);   // the two quantizer warps
        ptx::mbar_init(&xfull_bar[j], 1);
      }
      for (int j = 0; j < Cfg::kSaSlots; ++j) {
        ptx::mbar_init(&sa_full_bar[j], 2);
        ptx::mbar_init(&sa_free_bar[j], Cfg::kEpiWarps);
      }
    }
    ptx::fence_mbar_init();
  }
  if (warp == 2) {
    if constexpr (Cfg::kPairMma) {
      ptx::tmem_alloc_pair<Cfg::kTmemAlloc>(tmem_slot);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc<Cfg::kTmemAlloc>(tmem_slot);
      ptx::tmem_relinquish();
    }
  }
  if constexpr (Cfg::kFused) {
    // Rows of the E4M3 activation stages that the quantizer never writes
    // (past M, or past the FR-row box) stay zero, and the scales of rows past
    // M stay 1, so the MMA and the promotion see plain zeros there.
    for (int i = threadIdx.x; i < S_ * Cfg::kABytes / 16; i += Cfg::kThreads)
      ptx::sts128(ptx::smem_u32(smem_a) + 16u * static_cast<uint32_t>(i), 0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < Cfg::kSaSlots * kBM; i += Cfg::kThreads) sa_ring[i] = 1.0f;
    ptx::fence_proxy_async_shared();  // the zeros, before the tensor core reads the stages
  }
  ptx::tc_fence_before();
  __syncthreads();
  // Peers' barriers must be initialised before any remote arrive.  A pair
  // signals its peer from the first K block on; split-K only in the
  // epilogue, so there the wait is deferred until the first exchange.
  if constexpr (PAIR) ptx::cluster_sync_all();
  if constexpr (SPLIT) ptx::cluster_arrive_relaxed();
  bool cluster_waited = !SPLIT;
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if constexpr (Cfg::kPairMma) {
    // The pair's MMAs write the leader's TMEM address in both CTAs; make sure
    // both allocations returned it (both CTAs see the same answer).
    if (threadIdx.x == 0) {
      const uint32_t other = ptx::ld_dsmem_u32(ptx::mapa(ptx::smem_u32(tmem_slot), prank ^ 1));
      *pair_bad = other != tmem_base ? 1u : 0u;
      if (other != tmem_base) record_error(kErrMma);
    }
    __syncthreads();
  }
  const bool run_roles = !(Cfg::kPairMma && *pair_bad);
  ptx::griddep_wait();  // the previous kernel's writes (our operands) are visible from here on
  ptx::griddep_launch();


  if (!run_roles) {
    // nothing: the CTA pair could not share its accumulators
  } else if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t full0 = PAIR ? ptx::mapa(ptx::smem_u32(full_bar), 0) : ptx::smem_u32(full_bar);
      uint32_t issued = 0;
      bool ok = true;
      for (int t = cluster_id; t < p.num_tiles && ok; t += num_clusters) {
        int tm, tn;
        tile_coords(t, p, tm, tn);
        const int rot = kb_rotation(tm, tn, nkb);
        for (int i = 0; i < nkb; ++i) {
          const int kb = kb_begin + (i + rot < nkb ? i + rot : i + rot - nkb);
          const int s = issued % S_;
          const uint32_t ph = (issued / S_) & 1;
          if (!ptx::mbar_wait_bounded(&empty_bar[s], ph ^ 1, p.timeout_ns)) {
            record_error(kErrProducer);
            ok = false;
            break;
          }
          if constexpr (Cfg::kMcB) {
            // own 128 rows of A; half of B into both CTAs (each CTA's full
            // barrier counts its A, its own half and the peer's half)
            ptx::mbar_arrive_expect_tx(&full_bar[s], Cfg::kABytes + Cfg::kBBytes);
            ptx::tma_load_2d(smem_a + s * Cfg::kABytes, &tmap_a, &full_bar[s], kb * kBK, tm * TM + prank * kBM);
            ptx::tma_load_2d_mc(smem_b + s * Cfg::kBBytes + prank * (BN / 2) * kBK, &tmap_b, &full_bar[s], kb * kBK,
                                tn * BN + prank * (BN / 2), 0x3);
          } else if constexpr (PAIR) {
            // both CTAs' loads count on the leader's barrier
            if (leader) ptx::mbar_arrive_expect_tx(&full_bar[s], 2 * Cfg::kStageBytes);
            const uint32_t fb = full0 + 8u * static_cast<uint32_t>(s);
            ptx::tma_load_2d_pair(smem_a + s * Cfg::kABytes, &tmap_a, fb, kb * kBK, tm * TM + prank * kBM);
            ptx::tma_load_2d_pair(smem_b + s * Cfg::kBBytes, &tmap_b, fb, kb * kBK, tn * BN + prank * (BN / 2));
          } else if constexpr (Cfg::kFused) {
            // the activation in FP16/BF16 (FR rows, 128 columns = 256 bytes a
            // row) on a barrier of its own: the quantizer starts on it while
            // the weight tile is still in flight
            ptx::mbar_arrive_expect_tx(&xfull_bar[s], Cfg::kXBytes);
            ptx::tma_load_2d(smem_x + s * Cfg::kXBytes, &tmap_a, &xfull_bar[s], kb * kBK, tm * kBM);
            ptx::mbar_arrive_expect_tx(&full_bar[s], Cfg::kBBytes);
            ptx::tma_load_2d(smem_b + s * Cfg::kBBytes, &tmap_b, &full_bar[s], kb * kBK, tn * BN);
          } else {
            ptx::mbar_arrive_expect_tx(&full_bar[s], Cfg::kStageBytes);
            ptx::tma_load_2d(smem_a + s * Cfg::kABytes, &tmap_a, &full_bar[s], kb * kBK, tm * kBM);
            ptx::tma_load_2d(smem_b + s * Cfg::kBBytes, &tmap_b, &full_bar[s], kb * kBK, tn * BN);
          }
          ++issued;
        }
      }
      // Drain: every issued load has landed before the CTA may exit.  A pair
      // member waits until the MMA has consumed (and released) its last
      // stages, which also means the leader's multicast arrivals have landed.
      const uint32_t first = issued > S_ ? issued - S_ : 0;
      for (uint32_t j = first; j < issued; ++j) {
        const bool done = PAIR ? ptx::mbar_wait_bounded(&empty_bar[j % S_], (j / S_) & 1, p.timeout_ns)
                               : ptx::mbar_wait_bounded(&full_bar[j % S_], (j / S_) & 1, p.timeout_ns);
        if (!done) record_error(kErrProducer);
        if (Cfg::kFused && !ptx::mbar_wait_bounded(&xfull_bar[j % S_], (j / S_) & 1, p.timeout_ns))
          record_error(kErrProducer);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      // M of one MMA: 256 only for cta_group::2 pairs; B-multicast pairs
      // issue single-CTA MMAs over their own 128 rows
      constexpr int kMmaM = Cfg::kPairMma ? 2 * kBM : kBM;
      constexpr uint32_t idesc =
          Cfg::kUE8 ? ptx::idesc_mxf8_e4m3_ue8m0(kMmaM, BN) : ptx::idesc_e4m3_f32(kMmaM, BN);
      const uint32_t a0 = ptx::smem_u32(smem_a);
      const uint32_t b0 = ptx::smem_u32(smem_b);
      uint32_t consumed = 0, unit = 0;
      uint32_t sfg = 0, sf_tmem = 0;  // UE8M0: scale-factor groups consumed; TMEM columns of the current one
      bool ok = true;
      for (int t = cluster_id; t < p.num_tiles && ok; t += num_clusters) {
        for (int i = 0; i < nkb && ok; ++i) {  // i counts K blocks of the tile in issue order
          const bool new_unit = (MODE == kModeBlock) || i == 0;
          const uint32_t buf = unit % NBUF;
          if (new_unit) {
            const bool freed = Cfg::kPairMma
                                   ? ptx::mbar_wait_cluster_bounded(&tempty_bar[buf], ((unit / NBUF) & 1) ^ 1, p.timeout_ns)
                                   : ptx::mbar_wait_bounded(&tempty_bar[buf], ((unit / NBUF) & 1) ^ 1, p.timeout_ns);
            if (!freed) {
              record_error(kErrMma);
              ok = false;
              break;
            }
            ptx::tc_fence_after();
          }
          if constexpr (Cfg::kUE8) {
            if ((i & 3) == 0) {
              // the scale factors of this group of four K blocks: shared memory -> TMEM
              const uint32_t slot = sfg % Cfg::kSfSlots;
              if (!ptx::mbar_wait_bounded(&sf_full_bar[slot], (sfg / Cfg::kSfSlots) & 1, p.timeout_ns)) {
                record_error(kErrMma);
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              const uint32_t src = ptx::smem_u32(sf_smem + slot * Cfg::kSfSlotBytes);
              sf_tmem = tmem_base + Cfg::kTmemAccCols + slot * Cfg::kSfCols;
#pragma unroll
              for (int j = 0; j <= Cfg::kSfbTiles; ++j)
                ptx::tmem_cp_32x128b_warpx4(sf_tmem + 4 * j, ptx::smem_desc_rows16(src + 512 * j));
            }
          }
          const int s = consumed % S_;
          if (!ptx::mbar_wait_bounded(&full_bar[s], (consumed / S_) & 1, p.timeout_ns) ||
              (Cfg::kFused && !ptx::mbar_wait_bounded(&a8_ready_bar[s], (consumed / S_) & 1, p.timeout_ns))) {
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
            const uint32_t acc = (MODE == kModeBlock) ? (k > 0) : (i > 0 || k > 0);
            if constexpr (Cfg::kPairMma) ptx::mma_f8f6f4_pair(d, adesc + 2 * k, bdesc + 2 * k, idesc, acc);
            else if constexpr (Cfg::kUE8)
              // byte i % 4 of every scale word belongs to this K block (A's
              // words in the slot's first four columns, B's after them)
              ptx::mma_mxf8f6f4_bs(d, adesc + 2 * k, bdesc + 2 * k, ptx::idesc_sf_id(idesc, i & 3), sf_tmem,
                                   sf_tmem + 4, acc);
            else ptx::mma_f8f6f4(d, adesc + 2 * k, bdesc + 2 * k, idesc, acc);
          }
          if constexpr (Cfg::kPairMma) ptx::mma_commit_pair_mc(&empty_bar[s], 0x3);
          else if constexpr (Cfg::kMcB) ptx::mma_commit_mc(&empty_bar[s], 0x3);   // both CTAs' copies of B are read
          else ptx::mma_commit(&empty_bar[s]);
          if constexpr (Cfg::kUE8) {
            if ((i & 3) == 3 || i == nkb - 1) {  // the group's last MMA: its scale slot frees when they complete
              ptx::mma_commit(&sf_empty_bar[sfg % Cfg::kSfSlots]);
              ++sfg;
            }
          }
          ++consumed;
          const bool unit_done = (MODE == kModeBlock) || i == nkb - 1;
          if (unit_done) {
            if constexpr (Cfg::kPairMma) ptx::mma_commit_pair_mc(&tfull_bar[buf], 0x3);
            else ptx::mma_commit(&tfull_bar[buf]);
            ++unit;
          }
        }
      }
      // Drain: all issued MMAs complete before TMEM can be released.
      if constexpr (Cfg::kPairMma) ptx::mma_commit_pair_mc(mma_done_bar, 0x1);
      else ptx::mma_commit(mma_done_bar);
      if (!ptx::mbar_wait_bounded(mma_done_bar, 0, p.timeout_ns)) record_error(kErrMma);
    }
  } else if (Cfg::kFused && (warp == 2 || warp == 3)) {
    // ------------------------------------ fused activation quantizer
    // Per stage: the FR-row FP16/BF16 box of A has landed (its own barrier;
    // the weight tile may still be in flight).  Each row of the box is one
    // 1x128 token group ([P5] groups, [P2] s3 steps 2-4): a half-warp reads
    // its 256 bytes (8 elements a lane), the amax by shuffles, s =
    // fl32(amax / 448), and the E4M3 bytes go into the stage's A tile in the
    // MMA's 128-byte swizzled layout (16-byte unit u of row r at unit
    // u ^ (r % 8)), s into the slot of the scale ring that the epilogue reads
    // for this K block (quant_box16_rows, sixteen rows per call, one divide
    // for all of them); warp 2 takes rows 0-15, 32-47, ..., warp 3 rows
    // 16-31, 48-63, ...; rows past M are skipped (their bytes stay zero,
    // their scales 1).
    if constexpr (Cfg::kFused) {
      const int qwarp = warp - 2;
      uint32_t it = 0, u = 0;
      bool ok = true;
      for (int t = cluster_id; t < p.num_tiles && ok; t += num_clusters) {
        int tm, tn;
        tile_coords(t, p, tm, tn);
        const int rot = kb_rotation(tm, tn, nkb);
        const bool copy_out = p.qa_out != nullptr && tn == 0;
        for (int i = 0; i < nkb; ++i, ++it, ++u) {
          const int kb = kb_begin + (i + rot < nkb ? i + rot : i + rot - nkb);
          const int s = it % S_;
          const uint32_t slot = u % Cfg::kSaSlots;
          bool got = true;
          if (lane == 0)
            got = ptx::mbar_wait_bounded(&xfull_bar[s], (it / S_) & 1, p.timeout_ns) &&
                  ptx::mbar_wait_bounded(&sa_free_bar[slot], ((u / Cfg::kSaSlots) & 1) ^ 1, p.timeout_ns);
          if (!__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0)) {
            if (lane == 0) record_error(kErrProducer);
            ok = false;
            break;
          }
          const uint32_t xs = ptx::smem_u32(smem_x + s * Cfg::kXBytes);
          const uint32_t as = ptx::smem_u32(smem_a + s * Cfg::kABytes);
          float* sa_slot = sa_ring + slot * kBM;
          const int mrem = p.M - tm * kBM;   // rows of this tile that exist
          uint8_t* qo = copy_out ? p.qa_out + static_cast<int64_t>(tm * kBM) * p.K + kb * kBK : nullptr;
          float* so = copy_out ? p.sa_out + static_cast<int64_t>(kb) * p.M + tm * kBM : nullptr;
          for (int r0 = 16 * qwarp; r0 < FR && r0 < mrem; r0 += 32)
            quant_box16_rows<DT>(xs, as, r0, mrem < FR ? mrem : FR, lane, sa_slot, qo, p.K, so);
          ptx::fence_proxy_async_shared();  // the E4M3 bytes, before the MMA reads them
          __syncwarp();
          if (lane == 0) {
            ptx::mbar_arrive(&a8_ready_bar[s]);
            ptx::mbar_arrive(&sa_full_bar[slot]);
          }
        }
      }
    }
  } else if (Cfg::kUE8 && (warp == 2 || warp == 3)) {
    // ----------------------------------------- UE8M0 scale-factor stagers
    // Per tile and group of four K blocks (in the tile's issue order), warps
    // 2 and 3 taking alternate groups: lane l builds the scale words of rows
    // l, 32 + l, 64 + l, 96 + l of this CTA's 128 rows of A and of every 128
    // rows of B's BN (byte i = the code of the group's i-th K block; rows
    // past M or N and K blocks past the tile's range get 127, i.e. 2^0),
    // writes them as 16-byte rows of the slot's tiles and hands the slot to
    // the MMA issuer.  Every code load of a group is issued before any is
    // used; a 128-row block of the weight has one code per K block, loaded
    // once and shared by the warp.
    if constexpr (Cfg::kUE8) {
      const uint8_t* sa8 = reinterpret_cast<const uint8_t*>(p.sa);
      const uint8_t* sb8 = reinterpret_cast<const uint8_t*>(p.sb);
      const uint32_t me = static_cast<uint32_t>(warp - 2);
      uint32_t sfg = 0;
      bool ok = true;
      for (int t = cluster_id; t < p.num_tiles && ok; t += num_clusters) {
        int tm, tn;
        tile_coords(t, p, tm, tn);
        const int rot = kb_rotation(tm, tn, nkb);
        for (int g0 = 0; g0 < nkb; g0 += 4, ++sfg) {
          if ((sfg & 1u) != me) continue;   // the other stager's group
          const uint32_t slot = sfg % Cfg::kSfSlots;
          int kbs[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int idx = g0 + i;
            kbs[i] = idx < nkb ? kb_begin + (idx + rot < nkb ? idx + rot : idx + rot - nkb) : -1;
          }
          const int m0 = tm * Cfg::kTileM + static_cast<int>(prank) * kBM + lane;
          // Every load reads a valid address (K block and row clamped into
          // range) and the out-of-range ones are replaced by 127 afterwards,
          // so the loads carry no branches and all issue before any is used.
          int kbc[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) kbc[i] = kbs[i] >= 0 ? kbs[i] : kb_begin;
          // B: the weight block row of each 32-row chunk of the tile (a chunk
          // never straddles a 128-row block; a 192-wide tile's 128-row scale
          // tile can).  With BN a multiple of 128, or below 128, one block
          // row serves a whole scale tile.
          constexpr bool kOneBlockPerTile = BN % 128 == 0 || BN < 128;
          constexpr int kBJ = kOneBlockPerTile ? 1 : 4;
          uint32_t ca[4][4], cb[Cfg::kSfbTiles][kBJ][4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int m = min(m0 + 32 * j, p.M - 1);
#pragma unroll
            for (int i = 0; i < 4; ++i) ca[j][i] = __ldg(sa8 + static_cast<int64_t>(kbc[i]) * p.M + m);
          }
#pragma unroll
          for (int h = 0; h < Cfg::kSfbTiles; ++h)
#pragma unroll
            for (int jj = 0; jj < kBJ; ++jj) {
              const int nb = min(tn * BN + h * 128 + jj * 32, p.N - 1) / 128;
#pragma unroll
              for (int i = 0; i < 4; ++i) cb[h][jj][i] = __ldg(sb8 + static_cast<int64_t>(nb) * p.num_kb + kbc[i]);
            }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (kbs[i] < 0) {   // K blocks past the tile's range: 2^0
#pragma unroll
              for (int j = 0; j < 4; ++j) ca[j][i] = 127u;
#pragma unroll
              for (int h = 0; h < Cfg::kSfbTiles; ++h)
#pragma unroll
                for (int jj = 0; jj < kBJ; ++jj) cb[h][jj][i] = 127u;
            }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (m0 + 32 * j >= p.M) ca[j][0] = ca[j][1] = ca[j][2] = ca[j][3] = 127u;   // rows past M
          bool free_ok = true;
          if (lane == 0) free_ok = ptx::mbar_wait_bounded(&sf_empty_bar[slot], ((sfg / Cfg::kSfSlots) & 1) ^ 1,
                                                          p.timeout_ns);
          if (!__shfl_sync(0xFFFFFFFFu, free_ok ? 1 : 0, 0)) {
            if (lane == 0) record_error(kErrMma);
            ok = false;
            break;
          }
          const uint32_t dst = ptx::smem_u32(sf_smem + slot * Cfg::kSfSlotBytes) + static_cast<uint32_t>(lane * 16);
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) w[j] = ca[j][0] | (ca[j][1] << 8) | (ca[j][2] << 16) | (ca[j][3] << 24);
          ptx::sts128(dst, w[0], w[1], w[2], w[3]);
#pragma unroll
          for (int h = 0; h < Cfg::kSfbTiles; ++h) {
            // rows of this 128-row scale tile past N (or past the tile's BN) get 2^0
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t* c = cb[h][kOneBlockPerTile ? 0 : j];
              const uint32_t word = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
              const int n = tn * BN + h * 128 + j * 32 + lane;
              w[j] = (n < p.N && h * 128 + j * 32 + lane < BN) ? word : 0x7F7F7F7Fu;
            }
            ptx::sts128(dst + 512 * (h + 1), w[0], w[1], w[2], w[3]);
          }
          ptx::fence_proxy_async_shared();  // these stores, before tcgen05.cp reads them
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sf_full_bar[slot]);
        }
      }
    }
  } else if (warp >= 4) {
    // ----------------------------------------------------------- epilogue
    const int epi_tid = threadIdx.x - 128;
    const int epi_warp = warp - 4;
    const int quarter = warp & 3;   // TMEM lane quarter this warp may access
    const int wg = epi_warp >> 2;   // column slice of the tile
    const int row_local = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const bool vec_ok = (p.N % 8) == 0;
    uint16_t* C = reinterpret_cast<uint16_t*>(p.c);
    float* srow = staging + row_local * Cfg::kStagePitch + wg * CPT;  // split-K: this thread's partial row
    uint32_t unit = 0;
    bool ok = true;

    float pt_scale = 0.0f, pt_sa = 0.0f;
    if constexpr (MODE == kModePerTensor || MODE == kModePerChannel) {
      pt_sa = __ldg(p.sa);
      pt_scale = pt_sa * __ldg(p.sb);
    }

    for (int t = cluster_id; t < p.num_tiles && ok; t += num_clusters) {
      int tm, tn;
      tile_coords(t, p, tm, tn);
      const int row = tm * TM + static_cast<int>(prank) * kBM + row_local;
      // A warp whose 32 rows all lie past M (decode batches) skips the TMEM
      // loads and the promotion; it still waits for and hands back every
      // buffer, so the barrier phases stay in step.
      const bool live = tm * TM + static_cast<int>(prank) * kBM + quarter * 32 < p.M;
      const int n_base = tn * BN + wg * CPT;
      uint16_t* crow = C + static_cast<int64_t>(row) * p.N;

      if constexpr (MODE != kModeBlock) {
        const uint32_t buf = unit % NBUF;
        if (!ptx::mbar_wait_bounded(&tfull_bar[buf], (unit / NBUF) & 1, p.timeout_ns)) {
          record_error(kErrEpilogue);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if constexpr (SPLIT) {
          const bool staged_row = row_local < split_rows(p, tm, static_cast<int>(S)) * static_cast<int>(S);
#pragma unroll
          for (int c = 0; c < CPT / CW; ++c) {
            float v[CW];
            tmem_load_chunk<CW>(tmem_base + lane_off + buf * BN + wg * CPT + c * CW, v);
            scale_chunk<MODE, CW>(v, pt_scale, pt_sa, p, n_base + c * CW);
            if (staged_row) stage_row<CW>(srow + c * CW, v);
          }
          if (!cluster_waited) {  // peers' barriers are initialised from here on
            ptx::cluster_wait();
            cluster_waited = true;
          }
          if (!exchange_and_reduce<BN, OUT>(staged_bar, recv_bar, staging, recv, rank, S, epi_tid, Cfg::kEpiThreads,
                                            tm, tn, p))
            ok = false;
        } else if constexpr (Cfg::kUE8) {
          // The whole row slice is loaded before the buffer is handed back
          // (with one accumulator buffer, the next tile's MMAs wait for it),
          // then rounded and stored.
          uint32_t r[CPT];
          if (live) {
#pragma unroll
            for (int c = 0; c < CPT / CW; ++c) tmem_load_nowait<CW>(tmem_base + lane_off + buf * BN + wg * CPT + c * CW, &r[c * CW]);
            ptx::tmem_ld_wait();
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) release_tmem<Cfg::kPairMma>(&tempty_bar[buf]);
          if (row < p.M) {
#pragma unroll
            for (int c = 0; c < CPT / CW; ++c) {
              float v[CW];
#pragma unroll
              for (int j = 0; j < CW; ++j) v[j] = __uint_as_float(r[c * CW + j]);
              store_row<OUT, CW>(crow, n_base + c * CW, p.N, vec_ok, v);
            }
          }
          ++unit;
          continue;
        } else {
#pragma unroll
          for (int c = 0; c < CPT / CW; ++c) {
            float v[CW];
            tmem_load_chunk<CW>(tmem_base + lane_off + buf * BN + wg * CPT + c * CW, v);
            scale_chunk<MODE, CW>(v, pt_scale, pt_sa, p, n_base + c * CW);
            if (row < p.M) store_row<OUT, CW>(crow, n_base + c * CW, p.N, vec_ok, v);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) release_tmem<Cfg::kPairMma>(&tempty_bar[buf]);
        ++unit;
        if (!ok) break;
      } else {
        constexpr int KBT = Cfg::kBatch;
        float2 acc2[CPT / 2];
#pragma unroll
        for (int j = 0; j < CPT / 2; ++j) acc2[j] = make_float2(0.0f, 0.0f);
        // weight block row of this warpgroup's columns (clamped: a slice past
        // the last column of a ragged tile is computed but never stored)
        const int nb = (n_base < p.N ? n_base : p.N - 1) / 128;
        const float* sa_col = p.sa + (row < p.M ? row : 0);
        const float* sb_row = p.sb + static_cast<int64_t>(nb) * p.num_kb;
        const int rot = kb_rotation(tm, tn, nkb);
        if constexpr (Cfg::kSeqChunks) {
          // One K block at a time, kSeqLoadCols columns per wait: the
          // accumulators + the staged columns fit the register budget.  The
          // K block index walks the tile's rotated order incrementally and
          // the next block's scales are loaded one block ahead.
          constexpr int LC = Cfg::kSeqLoadCols;
          const int64_t sa_step = p.M;
          const int kb_stop = kb_begin + nkb;
          const uint32_t taddr0 = tmem_base + lane_off + static_cast<uint32_t>(wg * CPT);
          int kb = kb_begin + rot;
          float sa_c = Cfg::kFused ? 0.0f : __ldg(sa_col + kb * sa_step), sb_c = __ldg(sb_row + kb);
          for (int i = 0; i < nkb; ++i) {
            float sc = sa_c * sb_c;
            const float sb_now = sb_c;
            const int kn = kb + 1 == kb_stop ? kb_begin : kb + 1;
            if (i + 1 < nkb) {
              if constexpr (!Cfg::kFused) sa_c = __ldg(sa_col + kn * sa_step);
              sb_c = __ldg(sb_row + kn);
            }
            kb = kn;
            const uint32_t buf = unit % NBUF;
            if (!ptx::mbar_wait_bounded(&tfull_bar[buf], (unit / NBUF) & 1, p.timeout_ns)) {
              record_error(kErrEpilogue);
              ok = false;
              break;
            }
            if constexpr (Cfg::kFused) {
              // this K block's token scale, from the quantizer's ring
              const uint32_t slot = unit % Cfg::kSaSlots;
              bool got = true;
              if (lane == 0) got = ptx::mbar_wait_bounded(&sa_full_bar[slot], (unit / Cfg::kSaSlots) & 1, p.timeout_ns);
              if (!__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0)) {
                if (lane == 0) record_error(kErrEpilogue);
                ok = false;
                break;
              }
              __syncwarp();  // lane 0's acquire orders the other lanes' reads too
              sc = sa_ring[slot * kBM + row_local] * sb_now;
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(&sa_free_bar[slot]);
            }
            ptx::tc_fence_after();
            const uint32_t taddr = taddr0 + buf * BN;
            if (!live) {
              ptx::tc_fence_before();
              __syncwarp();
              if (lane == 0) release_tmem<Cfg::kPairMma>(&tempty_bar[buf]);
              unit += 1;
              continue;
            }
#pragma unroll
            for (int c0 = 0; c0 < CPT; c0 += LC) {
              uint32_t part[LC];
#pragma unroll
              for (int c = 0; c < LC; c += CW) tmem_load_nowait<CW>(taddr + c0 + c, &part[c]);
              ptx::tmem_ld_wait();
              if (c0 + LC == CPT) {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) release_tmem<Cfg::kPairMma>(&tempty_bar[buf]);
              }
#pragma unroll
              for (int j = 0; j < LC; j += 2) promote2(acc2[(c0 + j) / 2], part[j], part[j + 1], make_float2(sc, sc));
            }
            unit += 1;
          }
        } else {
        // global K block of the i-th K block issued for this tile
        auto kb_at = [&](int i) { return kb_begin + (i + rot < nkb ? i + rot : i + rot - nkb); };
        float sa_n[KBT], sb_n[KBT];
#pragma unroll
        for (int j = 0; j < KBT; ++j) {
          if constexpr (!Cfg::kFused) sa_n[j] = j < nkb ? __ldg(sa_col + static_cast<int64_t>(kb_at(j)) * p.M) : 0.0f;
          sb_n[j] = j < nkb ? __ldg(sb_row + kb_at(j)) : 0.0f;
        }
        for (int kb0 = 0; kb0 < nkb; kb0 += KBT) {
          const int nbat = min(KBT, nkb - kb0);
          float sc[KBT];
#pragma unroll
          for (int j = 0; j < KBT; ++j) {
            if constexpr (Cfg::kFused) sc[j] = sb_n[j];   // times the token scale, read below
            else sc[j] = sa_n[j] * sb_n[j];
            const int kn = kb0 + KBT + j;  // prefetch the next batch's scales
            if constexpr (!Cfg::kFused) sa_n[j] = kn < nkb ? __ldg(sa_col + static_cast<int64_t>(kb_at(kn)) * p.M) : 0.0f;
            sb_n[j] = kn < nkb ? __ldg(sb_row + kb_at(kn)) : 0.0f;
          }
          for (int j = 0; j < nbat && ok; ++j) {
            const uint32_t u = unit + j;
            if (!ptx::mbar_wait_bounded(&tfull_bar[u % NBUF], (u / NBUF) & 1, p.timeout_ns)) {
              record_error(kErrEpilogue);
              ok = false;
            }
          }
          if constexpr (Cfg::kFused) {
            // the token scales of these K blocks, from the quantizer's ring
            bool got = true;
            if (lane == 0)
              for (int j = 0; j < nbat && got && ok; ++j) {
                const uint32_t u = unit + j;
                got = ptx::mbar_wait_bounded(&sa_full_bar[u % Cfg::kSaSlots], (u / Cfg::kSaSlots) & 1, p.timeout_ns);
              }
            if (!__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0)) {
              if (lane == 0) record_error(kErrEpilogue);
              ok = false;
            }
            if (ok) {
              __syncwarp();  // lane 0's acquire orders the other lanes' reads too
#pragma unroll
              for (int j = 0; j < KBT; ++j)
                if (j < nbat) sc[j] *= sa_ring[((unit + j) % Cfg::kSaSlots) * kBM + row_local];
              __syncwarp();
              if (lane == 0)
                for (int j = 0; j < nbat; ++j) ptx::mbar_arrive(&sa_free_bar[(unit + j) % Cfg::kSaSlots]);
            }
          }
          if (!ok) break;
          ptx::tc_fence_after();
          if (!live) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
              for (int j = 0; j < nbat; ++j) release_tmem<Cfg::kPairMma>(&tempty_bar[(unit + j) % NBUF]);
            unit += nbat;
          } else {
            uint32_t part[KBT][CPT];
#pragma unroll
            for (int j = 0; j < KBT; ++j) {
              if (j < nbat) {
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
              for (int j = 0; j < nbat; ++j) release_tmem<Cfg::kPairMma>(&tempty_bar[(unit + j) % NBUF]);
            unit += nbat;
#pragma unroll
            for (int j = 0; j < KBT; ++j)
              if (j < nbat) {
#pragma unroll
                for (int c = 0; c < CPT; c += 2) promote2(acc2[c / 2], part[j][c], part[j][c + 1], make_float2(sc[j], sc[j]));
              }
          }
        }
        }
        if (!ok) break;
        if constexpr (SPLIT) {
          if (row_local < split_rows(p, tm, static_cast<int>(S)) * static_cast<int>(S)) stage_row2<CPT>(srow, acc2);
          if (!cluster_waited) {  // peers' barriers are initialised from here on
            ptx::cluster_wait();
            cluster_waited = true;
          }
          if (!exchange_and_reduce<BN, OUT>(staged_bar, recv_bar, staging, recv, rank, S, epi_tid, Cfg::kEpiThreads,
                                            tm, tn, p))
            ok = false;
          if (!ok) break;
        } else {
          if (row < p.M) {
#pragma unroll
            for (int c = 0; c < CPT / CW; ++c) store_row2<OUT, CW>(crow, n_base + c * CW, p.N, vec_ok, acc2 + c * CW / 2);
          }
        }
      }

    }
  }

  if (!cluster_waited) ptx::cluster_wait();  // every thread waits out its split-K arrival before the last barrier
  ptx::tc_fence_before();
  __syncthreads();
  // A pair frees its TMEM together, after both CTAs are done with it.
  if constexpr (PAIR) ptx::cluster_sync_all();
  if (warp == 2) {
    ptx::tc_fence_after();
    if constexpr (Cfg::kPairMma) ptx::tmem_dealloc_pair<Cfg::kTmemAlloc>(tmem_base);
    else ptx::tmem_dealloc<Cfg::kTmemAlloc>(tmem_base);
  }
  if constexpr (SPLIT || PAIR) ptx::cluster_sync_all();  // no CTA leaves while a peer may touch its shared memory
}

}  // namespace fp8s
