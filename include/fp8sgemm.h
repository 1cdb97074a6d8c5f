/*
 * fp8sgemm.h -- C ABI of the B300 (sm_103a) FP8 quantize + scaled-GEMM library
 * (libfp8sgemm.so).
 *
 * The path it implements, step by step, is the FP8 linear layer of
 *   [P2] "What is FP8 inference on H100 (Transformer Engine)?", s3 "How FP8
 *        inference works" (steps 2-6 and the pseudocode example fp8_gemm):
 *        amax = max|x|; scale = amax / 448; q = x / scale rounded to E4M3;
 *        C = (q_A . q_B accumulated in FP32) * scale_A * scale_B -> FP16;
 *   [P5] "FP8 chi tiet" (transformers fine-grained FP8 guide), opening
 *        bullets: weights quantized per 128x128 block, activations per token
 *        per group of 128 input channels.
 * [P1] "Technical assignment: implement FP8 inference on H100" (aivaro.ru,
 * practice 214), stage 3 steps 1-2, supplies the static/delayed-scaling
 * variant: a calibrated scale, or one derived from an amax history with a
 * margin (Transformer Engine's DelayedScaling recipe).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never frees or keeps them beyond the call (a host-side cache of TMA
 *    descriptors is keyed by pointer and shape; it holds no device memory).
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream) and returns once its kernels are enqueued.  Scales are written
 *    on the device; read them after synchronizing.
 *  - Arguments are checked on the host before anything is launched; a
 *    failing check returns its status and has no side effect.  No exception
 *    crosses the ABI and there is no CPU fallback.
 *  - The device must be compute capability 10.3 (B300); otherwise
 *    FP8S_ERR_UNSUPPORTED_DEVICE.  A launch failure gives FP8S_ERR_CUDA.
 *  - Matrices are row-major with K contiguous: activations A[M][K], weights
 *    W[N][K] (the nn.Linear layout; C = A * W^T), output C[M][N].
 *  - E4M3 is the "fn" variant (bias 7, max 448, no infinities); stored
 *    scales are dequantization factors s = fl32(amax / 448) (s = 1 when
 *    amax == 0); q = E4M3_rne_satfinite(fl32(x / s)).
 *  - Every pointer must be 16-byte aligned (FP8S_ERR_ALIGN), except the
 *    single floats and the amax history of the static/delayed-scaling
 *    calls, which need 4-byte alignment.
 */
#ifndef FP8SGEMM_H
#define FP8SGEMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define FP8S_API __attribute__((visibility("default")))
#else
#define FP8S_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st* fp8s_stream_t;

typedef enum {
  FP8S_OK = 0,
  FP8S_ERR_NULL = 1,               /* a required pointer is NULL */
  FP8S_ERR_SHAPE = 2,              /* a size is out of range or breaks a multiple-of rule */
  FP8S_ERR_ALIGN = 3,              /* a pointer is not 16-byte aligned */
  FP8S_ERR_DTYPE = 4,              /* unknown dtype or scale-mode value */
  FP8S_ERR_CUDA = 5,               /* a CUDA runtime/driver call or launch failed */
  FP8S_ERR_DEVICE_TIMEOUT = 6,     /* a kernel's bounded wait gave up (see fp8s_device_error) */
  FP8S_ERR_UNSUPPORTED_DEVICE = 7  /* current device is not compute capability 10.3 */
} fp8s_status;

typedef enum { FP8S_F16 = 0, FP8S_BF16 = 1 } fp8s_dtype;

typedef enum {
  FP8S_SCALE_PER_TENSOR = 0, /* sa, sb each point to one float */
  FP8S_SCALE_BLOCK = 1,      /* sa: [K/128][M] token-group scales, sb: [ceil(N/128)][K/128] block scales */
  FP8S_SCALE_PER_CHANNEL = 2, /* sa: one float (per-tensor activation), sb: [N] one scale per output channel */
  FP8S_SCALE_BLOCK_UE8M0 = 3  /* as FP8S_SCALE_BLOCK with UE8M0 codes (one byte each): sa [K/128][M], sb [ceil(N/128)][K/128] */
} fp8s_scale_mode;

/*
 * fp8_quantize_per_tensor -- [P2] s3 steps 2-4 with one scale per tensor.
 *   x      [numel] FP16/BF16 (xt), device.            numel >= 1.
 *   q      [numel] E4M3 bytes, device (output).
 *   scale  one float, device (output): s = fl32(max|x| / 448), 1 if all zero.
 * One kernel launch.  Up to 3 MB of input: one thread-block cluster whose
 * CTAs exchange their slice maxima through distributed shared memory.
 * Larger: one cooperative launch (its CTAs wait on each other, so all of them
 * are resident; the launch fails with FP8S_ERR_CUDA if the device cannot
 * hold them) whose CTAs exchange their slice maxima through `scale` (an
 * arrival count while the call runs; its final value is s) and the first
 * 4*G bytes of q (G = CTAs).  Up to ~29 MB of input (148 CTAs x 192 KB of
 * shared memory) is read from HBM once, a larger x twice.  Neither q nor
 * scale may be read or written by anything else while the call runs.
 */
FP8S_API fp8s_status fp8_quantize_per_tensor(const void* x, fp8s_dtype xt, int64_t numel,
                                    uint8_t* q, float* scale, fp8s_stream_t stream);

/*
 * fp8_quantize_per_tensor_static -- static or delayed per-tensor scaling:
 * [P2] s3 step 4 (q = x / scale rounded to E4M3) with a scale the caller
 * already holds, so steps 2-3 (amax, scale) leave the critical path and x is
 * read once.  The scale may come from calibration ([P1] stage 3 step 2,
 * "Calibrating the FP8 scales") or from an amax history as in the
 * Transformer Engine recipe DelayedScaling(margin, interval) of [P1] stage 3
 * step 1 (see fp8_scale_from_amax_history); [P5] "DeepGEMM fast path" names
 * static activation quantization beside the dynamic scheme.
 *   x      [numel] FP16/BF16 (xt), device, 16-byte aligned.   numel >= 1.
 *   scale  one float, device (input, 4-byte aligned): the dequant factor s,
 *          positive, finite and normal (other values give unspecified bytes,
 *          never a fault).
 *   q      [numel] E4M3 bytes, device (output, 16-byte aligned):
 *          q = E4M3_rne_satfinite(fl32(x / s)); |x / s| above 448 saturates.
 *   amax   NULL, or one float, device (output, 4-byte aligned): receives
 *          max|x| over the tensor (exact), e.g. one slot of a ring buffer of
 *          recorded amaxes.  It is zeroed on `stream` (by a one-thread
 *          kernel) before the quantize kernel folds in its CTAs' maxima, and
 *          must not overlap x, q or scale.
 * One kernel launch (two when amax is given), no memset: both keep
 * programmatic dependent launch with the stream's neighbouring kernels.
 */
FP8S_API fp8s_status fp8_quantize_per_tensor_static(const void* x, fp8s_dtype xt, int64_t numel,
                                           const float* scale, uint8_t* q, float* amax,
                                           fp8s_stream_t stream);

/*
 * fp8_scale_from_amax_history -- the scale update of delayed scaling ([P1]
 * stage 3 step 1, recipe.DelayedScaling(margin=0, interval=4)):
 *   s = fl32(max(history[0..H-1]) / 448) * 2^margin   (1 * 2^margin when the
 *   maximum is 0).
 *   history  [H] floats, device (input, 4-byte aligned), each >= 0 and
 *            finite: the amaxes of the last H steps, in any order (a ring
 *            buffer written by fp8_quantize_per_tensor_static's amax).
 *            1 <= H <= 2^24.
 *   margin   -64 <= margin <= 64: powers of two of headroom (a larger margin
 *            gives a larger dequant factor, so fewer values saturate).
 *   scale    one float, device (output, 4-byte aligned).
 * The caller decides how often to call it (the recipe's `interval`: every
 * interval-th step).  One single-CTA kernel launch.
 */
FP8S_API fp8s_status fp8_scale_from_amax_history(const float* history, int64_t H, int margin, float* scale,
                                        fp8s_stream_t stream);

/*
 * fp8_quantize_per_channel -- per-channel weight scaling ([P2] s5 "How to
 * minimize the losses": per-tensor scaling, or per-channel scaling for the
 * weights): one quantization unit per output channel, i.e. per row of W, each
 * quantized as in [P2] s3 steps 2-4.  One read of w.
 *   w   [N][K] FP16/BF16 (wt), device.   N >= 1, 8 <= K <= 65536, K % 8 == 0
 *       (the GEMM further needs K % 16 == 0).
 *   q   [N][K] E4M3 bytes, device (output).
 *   sb  [N] floats, device (output): sb[n] = fl32(max_k |w[n][k]| / 448)
 *       (1 for an all-zero row).
 * One kernel launch (persistent CTAs; a row is staged in K*2 bytes of
 * shared memory).
 */
FP8S_API fp8s_status fp8_quantize_per_channel(const void* w, fp8s_dtype wt, int64_t N, int64_t K,
                                     uint8_t* q, float* sb, fp8s_stream_t stream);

/*
 * fp8_quantize_token_group -- [P5] per-token 1x128 activation groups, each
 * group quantized as in [P2] s3 steps 2-4.  One read of x.
 *   x   [M][K] FP16/BF16 (xt), device.   M >= 1, K >= 128, K % 128 == 0.
 *   q   [M][K] E4M3 bytes, device (output).
 *   sa  [K/128][M] floats, device (output): sa[g*M + m] is the scale of
 *       x[m][128g .. 128g+127].  (Group-major so the GEMM reads 128
 *       consecutive token scales per K block.)
 */
FP8S_API fp8s_status fp8_quantize_token_group(const void* x, fp8s_dtype xt, int64_t M, int64_t K,
                                     uint8_t* q, float* sa, fp8s_stream_t stream);

/*
 * fp8_quantize_weight_block -- [P5] 128x128 weight blocks (weight_block_size
 * = (128, 128)), each quantized as in [P2] s3 steps 2-4.  One read of w.
 *   w   [N][K] FP16/BF16 (wt), device.   N >= 1, K >= 128, K % 128 == 0.
 *   q   [N][K] E4M3 bytes, device (output).
 *   sb  [ceil(N/128)][K/128] floats, device (output): sb[i*(K/128) + j] is the
 *       scale of rows 128i.. (the valid ones only, for a ragged last block)
 *       and columns 128j..128j+127.
 */
FP8S_API fp8s_status fp8_quantize_weight_block(const void* w, fp8s_dtype wt, int64_t N, int64_t K,
                                      uint8_t* q, float* sb, fp8s_stream_t stream);

/*
 * fp8_gemm_scaled -- [P2] s3 steps 5-6: C = (qa . qb^T, FP32 accumulation on
 * the tensor cores) rescaled by the operand scales, rounded to nearest-even
 * into FP16/BF16 (ct).
 *   qa  [M][K] E4M3, device.   qb [N][K] E4M3, device.   c [M][N] output, device.
 *   mode FP8S_SCALE_PER_TENSOR: sa, sb -> one float each;
 *        C[m][n] = RN(acc[m][n] * sa * sb).          K % 16 == 0.
 *   mode FP8S_SCALE_BLOCK ([P5] block geometry): sa [K/128][M], sb
 *        [ceil(N/128)][K/128]; each 128-wide K block's FP32 partial sum is
 *        multiplied by sa[kb][m] * sb[n/128][kb] and added into an FP32
 *        accumulator;  C[m][n] = RN(acc).             K % 128 == 0.
 *   mode FP8S_SCALE_PER_CHANNEL ([P2] s5 per-channel weight scaling): sa ->
 *        one float, sb [N] (from fp8_quantize_per_channel);
 *        C[m][n] = RN(acc[m][n] * (sa * sb[n])).       K % 16 == 0.
 *        The same kernels and tiles as per-tensor mode.
 *   mode FP8S_SCALE_BLOCK_UE8M0 ([P5] block geometry, "UE8M0 scale format"):
 *        sa [K/128][M] and sb [ceil(N/128)][K/128] UE8M0 codes (bytes, value
 *        2^(code-127); from the *_ue8m0 quantizers).  The tensor core applies
 *        them itself (tcgen05.mma kind::mxf8f6f4.block_scale, one scale per
 *        row per 32-wide K slice, each code repeated over its 128-wide K
 *        block): C[m][n] = RN(sum_k dec(qa)*2^(ca-127) * dec(qb)*2^(cb-127))
 *        accumulated in FP32.  K % 128 == 0.  Codes of 255 (NaN) are not
 *        accepted.
 *   M, N >= 1, K >= 16.  N need not be a multiple of anything.
 * Block mode with M <= 32 (and no tile override) runs a decode kernel that
 * computes C^T = qb . qa^T: each 128-row weight tile is the MMA's 128-row
 * operand and the M tokens its 16 or 32 columns, the tile's K range split
 * over a thread-block cluster (partials exchanged through distributed
 * shared memory and summed in rank order, so results are deterministic).
 */
FP8S_API fp8s_status fp8_gemm_scaled(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                            void* c, fp8s_dtype ct, int64_t M, int64_t N, int64_t K,
                            fp8s_scale_mode mode, fp8s_stream_t stream);

/*
 * fp8_quantize_token_group_ue8m0 / fp8_quantize_weight_block_ue8m0 -- the
 * two block quantizers with power-of-two scales stored as UE8M0 codes
 * ([P5] "UE8M0 scale format": checkpoints that keep each scale as an 8-bit
 * biased exponent, float8_e8m0fnu; the format Blackwell's block-scaled
 * tensor-core MMA takes).  Units as in fp8_quantize_token_group (1x128
 * activation groups) and fp8_quantize_weight_block (128x128 weight blocks).
 * Per unit: s32 = fl32(amax / 448) (1 when amax == 0), rounded UP to the
 * nearest power of two 2^k (k >= -127); code = k + 127 (value 2^(code-127));
 * q = E4M3_rne_satfinite(x / 2^k) (the division is exact), so |x / 2^k| <=
 * 448 still holds and the amax element may land below 448.
 *   token group:  x [M][K] -> q [M][K], sa_code [K/128][M] bytes (layout of
 *                 the FP32 sa).  M >= 1, K >= 128, K % 128 == 0.
 *   weight block: w [N][K] -> q [N][K], sb_code [ceil(N/128)][K/128] bytes.
 * All pointers device, 16-byte aligned.  One kernel launch each (the same
 * kernels as the FP32-scale quantizers, with the scale rounded up).
 */
FP8S_API fp8s_status fp8_quantize_token_group_ue8m0(const void* x, fp8s_dtype xt, int64_t M, int64_t K,
                                                    uint8_t* q, uint8_t* sa_code, fp8s_stream_t stream);
FP8S_API fp8s_status fp8_quantize_weight_block_ue8m0(const void* w, fp8s_dtype wt, int64_t N, int64_t K,
                                                     uint8_t* q, uint8_t* sb_code, fp8s_stream_t stream);

/*
 * fp8_e5m2_encode / fp8_e5m2_decode -- the E5M2 format (5 exponent + 2
 * mantissa bits: [P2] s2 "FP8 formats", [P3] s2), the FP8 variant with the
 * wider range and coarser steps that the pages name beside E4M3.  Reading
 * taken where the pages give only the bit split: bias 15, S.11111.00 =
 * +-infinity, S.11111.xx (xx != 0) = NaN, largest finite value 57344.
 *   encode: x [numel] FP16/BF16 (xt), device -> q [numel] E5M2 bytes, device:
 *           round to nearest even; finite values beyond 57344 and
 *           +-infinity saturate to +-57344; a NaN gives S.11111.11 with the
 *           input's sign; the sign of zero is kept.  No scaling.
 *   decode: q [numel] E5M2 bytes, device -> y [numel] FP16/BF16 (yt), device:
 *           exact (every E5M2 value is an FP16 and a BF16 value); the
 *           infinity codes give infinities, the NaN codes NaNs.
 * numel >= 1; all pointers 16-byte aligned.  One kernel launch each (an
 * HBM-bound stream, 3 bytes of traffic per element).
 */
FP8S_API fp8s_status fp8_e5m2_encode(const void* x, fp8s_dtype xt, int64_t numel, uint8_t* q,
                                     fp8s_stream_t stream);
FP8S_API fp8s_status fp8_e5m2_decode(const uint8_t* q, int64_t numel, void* y, fp8s_dtype yt,
                                     fp8s_stream_t stream);

/*
 * fp8_linear_token_group -- the fused FP8 linear layer: [P2] s3 steps 2-6
 * with [P5]'s 1x128 token groups on the activation, in ONE kernel.  The
 * activation arrives unquantized; each CTA of the block-scaled GEMM loads
 * its FP16/BF16 tiles of x, quantizes every 1x128 group in shared memory
 * (amax, s = fl32(amax / 448), E4M3(fl32(x / s)), exactly as
 * fp8_quantize_token_group) and feeds the E4M3 tile to the tensor core,
 * so the quantized activation never makes a round trip through HBM and the
 * quantize launch disappears.  The weight is pre-quantized per 128x128 block
 * (fp8_quantize_weight_block).
 *   x   [M][K] FP16/BF16 (xt), device.          K >= 128, K % 128 == 0, M, N >= 1.
 *   qw  [N][K] E4M3, sw [ceil(N/128)][K/128] FP32: the block-quantized weight.
 *   c   [M][N] output in the activation's type xt, device:
 *       C = the FP8S_SCALE_BLOCK GEMM of (token-group quantized x, qw, sw).
 *   qa, sa  both NULL, or qa [M][K] E4M3 and sa [K/128][M] FP32 outputs that
 *       receive the quantized activation and its scales (byte- and
 *       bit-identical to fp8_quantize_token_group's).
 * M <= 32 without a tile override runs the transposed decode kernel (the
 * weight tile as the MMA's 128-row operand, the M tokens as its 16 or 32
 * columns); larger M, or a call with an override, runs the general kernel
 * on 128-row activation boxes.  Any M is correct.  Every CTA quantizes the
 * activation of its own K range, so a row of output tiles repeats that
 * work.  Measured on a B300 against the two-call path
 * (fp8_quantize_token_group, then fp8_gemm_scaled), Llama-2-7B linears:
 * on par at M = 1 for qkv and down, slower for o and gate/up, ~1.4x its
 * time at M = 16 and several times at M = 128.  Tile overrides
 * (fp8s_gemm_override) apply with bn 64 or 128 (any split), or bn 192
 * (split only for M <= 16), and no pair; others give FP8S_ERR_SHAPE.
 * All pointers 16-byte aligned.  One kernel launch.
 */
FP8S_API fp8s_status fp8_linear_token_group(const void* x, fp8s_dtype xt, int64_t M, int64_t K, const uint8_t* qw,
                                            const float* sw, int64_t N, void* c, uint8_t* qa, float* sa,
                                            fp8s_stream_t stream);

/*
 * fp8s_gemm_override -- tuning aid: makes every later fp8_gemm_scaled call on
 * any device use output tiles of 128 x bn and split each tile's K range over
 * `splits` CTAs of a thread-block cluster, or (pair != 0, splits == 1, bn >=
 * 64) tiles of 256 x bn shared by a pair of CTAs, instead of the library's
 * own choice.  bn in {32, 64, 128, 192, 256}; splits in {1, 2, 4, 8}, with
 * splits > 1 only for bn <= 192.  With splits > 1 every cluster must own a
 * single output tile; a later call whose
 * K has fewer 128-wide blocks than `splits`, or with more 128 x bn output
 * tiles than the device can hold clusters of `splits` CTAs at once, fails
 * with FP8S_ERR_SHAPE.  bn = 0 restores the automatic choice.
 * Results stay within the documented tolerance for every setting; only
 * speed changes.  Not thread-safe against concurrent GEMM calls.
 */
FP8S_API fp8s_status fp8s_gemm_override(int bn, int splits, int pair);

/*
 * fp8s_gemm_plan -- the tile configuration fp8_gemm_scaled picks for a
 * shape on a device with `sms` streaming multiprocessors (148 on the B300),
 * from a time model whose constants were measured on the B300: *bn (output
 * tile 128 x bn, or 256 x bn when *pair), *splits (CTAs of a cluster sharing
 * one tile's K range; 1 = none) and *pair (1 when two CTAs share a 256-row
 * tile through tcgen05 cta_group::2).  Host-only and side-effect free; no
 * GPU is needed.  Same shape rules and status codes as fp8_gemm_scaled.  (At
 * run time a split that the device cannot hold falls back to splits = 1.)
 * For FP8S_SCALE_BLOCK with M <= 32 it describes the decode kernel:
 * *bn = 128 output columns per tile, *splits its split-K, *pair = 0.
 */
FP8S_API fp8s_status fp8s_gemm_plan(int64_t M, int64_t N, int64_t K, fp8s_scale_mode mode, int sms, int* bn,
                                    int* splits, int* pair);

/* Human-readable name of a status code (static storage, never NULL). */
FP8S_API const char* fp8s_status_string(fp8s_status status);

/*
 * fp8s_last_cuda_error -- the CUDA runtime's description of the error behind
 * the calling host thread's most recent FP8S_ERR_CUDA (static storage, never
 * NULL; "" before any).  Diagnostic only: no method step stands behind it.
 */
FP8S_API const char* fp8s_last_cuda_error(void);

/*
 * fp8s_device_error -- synchronizes `stream`, then reads and clears the
 * current device's error word, which a kernel sets when one of its bounded
 * waits gives up (the kernel then exits without finishing its output).
 * *where (if not NULL) receives the word: 0 if no wait gave up, else
 * 1 = GEMM TMA producer, 2 = GEMM MMA issuer, 3 = GEMM epilogue,
 * 4 = quantizer.  Returns FP8S_OK,
 * FP8S_ERR_DEVICE_TIMEOUT or FP8S_ERR_CUDA.
 */
FP8S_API fp8s_status fp8s_device_error(fp8s_stream_t stream, int* where);

/*
 * fp8s_set_exchange_timeout_ns -- test aid for the failure path of the
 * bounded waits: sets the wall-time limit (ns) of the grid-wide exchange
 * spin of fp8_quantize_per_tensor for inputs above ~29 MB (whose CTAs stream
 * their slices, so no asynchronous copy is in flight while they wait);
 * 0 restores the default of 2 s.  A spin that runs out records 4 in the
 * device error word (fp8s_device_error) and its CTA carries on, so the call
 * ends with unspecified output bytes and no hang.  Every other wait keeps
 * its 2 s limit.  Process-wide; not for production use.  Diagnostic only:
 * no method step stands behind it.
 */
FP8S_API fp8s_status fp8s_set_exchange_timeout_ns(unsigned long long ns);

/* Library version, major*10000 + minor*100 + patch. */
FP8S_API int fp8s_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8SGEMM_H */
