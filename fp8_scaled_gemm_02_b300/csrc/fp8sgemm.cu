// fp8sgemm.cu -- the C ABI of libfp8sgemm.so (declared in include/fp8sgemm.h).
//
// One translation unit: the kernels (quantize.cuh, gemm.cuh) are included
// here so the device error word is a single symbol without relocatable
// device code.  Host code validates arguments, checks the device, encodes
// (and caches) TMA descriptors, picks a tile configuration and launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>
#include <unordered_map>

#include "../../include/fp8sgemm.h"
#include "codec.cuh"
#include "decode.cuh"
#include "gemm.cuh"
#include "quantize.cuh"

namespace fp8s {
namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s per mbarrier wait
// Limit of the per-tensor quantizer's grid-wide exchange spin when it
// streams its slices (no bulk copy in flight): the default, or the value a
// test set with fp8s_set_exchange_timeout_ns to make the spin run out.
std::atomic<unsigned long long> g_exchange_timeout_ns{kWaitTimeoutNs};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline cudaStream_t as_stream(fp8s_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Text behind the calling thread's latest FP8S_ERR_CUDA (fp8s_last_cuda_error).
thread_local const char* t_cuda_msg = "";

fp8s_status cuda_fail(const char* msg) {
  t_cuda_msg = msg;
  return FP8S_ERR_CUDA;
}

// Reports a runtime error (and clears it from cudaGetLastError).
fp8s_status cuda_fail(cudaError_t e) {
  cudaGetLastError();
  return cuda_fail(cudaGetErrorString(e));
}

// ---------------------------------------------------------------- device
struct DeviceInfo {
  bool ok = false;
  bool checked = false;
  int sms = 0;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

fp8s_status current_device(int* dev_out, DeviceInfo* info_out) {
  int dev = 0;
  if (const cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return FP8S_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      return cuda_fail(cudaGetLastError());
    }
    d.ok = (major == 10 && minor == 3);
    d.sms = sms;
    d.checked = true;
  }
  if (!d.ok) return FP8S_ERR_UNSUPPORTED_DEVICE;
  *dev_out = dev;
  *info_out = d;
  return FP8S_OK;
}

fp8s_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FP8S_OK : cuda_fail(cudaGetErrorString(e));
}

// ------------------------------------------------------ TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

struct MapKey {
  const void* ptr;
  int64_t rows, cols;
  int box_rows, box_cols, elem_bytes, swizzle;
  int dev;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && cols == o.cols && box_rows == o.box_rows && box_cols == o.box_cols &&
           elem_bytes == o.elem_bytes && swizzle == o.swizzle && dev == o.dev;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    size_t h = std::hash<const void*>()(k.ptr);
    auto mix = [&h](size_t v) { h ^= v + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2); };
    mix(std::hash<int64_t>()(k.rows));
    mix(std::hash<int64_t>()(k.cols));
    mix(static_cast<size_t>(k.box_rows) * 1000003u + static_cast<size_t>(k.box_cols) * 131u +
        static_cast<size_t>(k.elem_bytes) * 7u + static_cast<size_t>(k.swizzle) + static_cast<size_t>(k.dev) * 65537u);
    return h;
  }
};
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;
std::mutex g_maps_mu;

// Row-major [rows][cols] matrix of 1- or 2-byte elements; box of
// box_cols x box_rows elements; out-of-range elements read as zero.
fp8s_status tensor_map_2d(const void* ptr, int64_t rows, int64_t cols, int elem_bytes, int box_rows, int box_cols,
                          bool swizzle128, int dev, CUtensorMap* out) {
  MapKey key{ptr, rows, cols, box_rows, box_cols, elem_bytes, swizzle128 ? 1 : 0, dev};
  {
    std::lock_guard<std::mutex> lk(g_maps_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *out = it->second;
      return FP8S_OK;
    }
  }
  auto fn = encode_fn();
  if (!fn) return cuda_fail("cuTensorMapEncodeTiled is not available from the driver");
  CUtensorMap m;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * elem_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  CUresult r = fn(&m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail("cuTensorMapEncodeTiled rejected the tensor map");
  {
    std::lock_guard<std::mutex> lk(g_maps_mu);
    if (g_maps.size() > 4096) g_maps.clear();
    g_maps.emplace(key, m);
  }
  *out = m;
  return FP8S_OK;
}

// E4M3 operand of the GEMM: boxes of one 128-byte K block x box_rows rows,
// 128-byte swizzle (the layout the MMA's shared-memory descriptors expect).
fp8s_status tensor_map_e4m3(const uint8_t* ptr, int64_t rows, int64_t cols, int box_rows, int dev, CUtensorMap* out) {
  return tensor_map_2d(ptr, rows, cols, 1, box_rows, kBK, true, dev, out);
}

// Launches `kern` with programmatic stream serialization (it may start while
// the previous kernel of the stream finishes; every kernel of this library
// waits for it before touching global memory) and, for cluster > 1, a 1-D
// cluster dimension.
template <typename... KArgs, typename... Args>
fp8s_status launch_ex(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t st, int cluster,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  if (const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...); e != cudaSuccess)
    return cuda_fail(e);
  return FP8S_OK;
}

template <typename KernelT>
fp8s_status ensure_smem_attr(KernelT kern, int bytes, bool* done_per_device) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return launch_status(), FP8S_ERR_CUDA;
  if (!done_per_device[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
      return launch_status(), FP8S_ERR_CUDA;
    done_per_device[dev] = true;
  }
  return FP8S_OK;
}

// ------------------------------------------------------------ quantizers
template <int DT, int GPW, bool UE8>
fp8s_status launch_token_group_gpw(const void* x, int64_t M, int64_t G, uint8_t* q, void* sa, cudaStream_t st,
                                   const DeviceInfo& info) {
  static bool attr_done[kMaxDevices] = {};
  auto kern = quant_token_group_kernel<DT, GPW, UE8>;
  constexpr int kSmem = tg_smem_bytes(GPW);
  if (fp8s_status s = ensure_smem_attr(kern, kSmem, attr_done)) return s;
  const int64_t groups = M * G;
  const int64_t chunks = (groups + 8 * GPW - 1) / (8 * GPW);
  const int64_t cap = 2LL * info.sms;
  const unsigned grid = static_cast<unsigned>(chunks < cap ? chunks : cap);
  return launch_ex(kern, grid, 288, kSmem, st, 1, static_cast<const uint8_t*>(x), reinterpret_cast<uint2*>(q), sa,
                   static_cast<uint32_t>(M), static_cast<uint32_t>(G), static_cast<uint32_t>(groups), kWaitTimeoutNs);
}

// Groups per consumer warp: the largest that still gives every SM two chunks.
// `sa` receives FP32 scales, or UE8M0 codes when UE8.
template <int DT, bool UE8 = false>
fp8s_status launch_token_group(const void* x, int64_t M, int64_t K, uint8_t* q, void* sa, cudaStream_t st,
                               const DeviceInfo& info) {
  const int64_t G = K / 128;
  const int64_t groups = M * G;
  const int64_t want = 2LL * info.sms;
  if (groups >= want * 8 * 16) return launch_token_group_gpw<DT, 16, UE8>(x, M, G, q, sa, st, info);
  if (groups >= want * 8 * 8) return launch_token_group_gpw<DT, 8, UE8>(x, M, G, q, sa, st, info);
  if (groups >= want * 8 * 4) return launch_token_group_gpw<DT, 4, UE8>(x, M, G, q, sa, st, info);
  return launch_token_group_gpw<DT, 2, UE8>(x, M, G, q, sa, st, info);
}

template <int DT, bool UE8 = false>
fp8s_status launch_weight_block(const void* w, int64_t N, int64_t K, uint8_t* q, void* sb, cudaStream_t st,
                                const DeviceInfo& info, int dev) {
  CUtensorMap mw;
  if (fp8s_status s = tensor_map_2d(w, N, K, 2, 128, 128, false, dev, &mw)) return s;
  static bool attr_done[kMaxDevices] = {};
  auto kern = quant_weight_block_tma_kernel<DT, UE8>;
  if (fp8s_status s = ensure_smem_attr(kern, kWbSmemBytes, attr_done)) return s;
  const int64_t nblocks = ((N + 127) / 128) * (K / 128);
  const int64_t cap = info.sms;  // one CTA per SM
  const unsigned grid = static_cast<unsigned>(nblocks < cap ? nblocks : cap);
  return launch_ex(kern, grid, kWbThreads, kWbSmemBytes, st, 1, mw, reinterpret_cast<uint2*>(q), sb, static_cast<int>(N),
                   static_cast<int>(K / 128), static_cast<int>(nblocks), kWaitTimeoutNs);
}

// CTAs of the cooperative per-tensor kernel that fit on the device at once.
int pt_capacity(int dev, int sms) {
  static std::mutex mu;
  static int cap[kMaxDevices] = {};
  std::lock_guard<std::mutex> lk(mu);
  if (cap[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quant_per_tensor_kernel<kInF16>, kPtThreads, kPtSmemBytes) !=
            cudaSuccess ||
        n < 1) {
      cudaGetLastError();
      n = 1;
    }
    cap[dev] = n * sms;
  }
  return cap[dev];
}

// Largest cluster (16, else 8) of the small-tensor per-tensor kernel the
// device can schedule.
template <int DT>
int pt_cluster_max(int dev) {
  static std::mutex mu;
  static int cmax[kMaxDevices] = {};
  std::lock_guard<std::mutex> lk(mu);
  if (cmax[dev] == 0) {
    auto kern = quant_per_tensor_cluster_kernel<DT>;
    int c = 8;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16, 1, 1);
      cfg.blockDim = dim3(kPtThreads, 1, 1);
      cfg.dynamicSmemBytes = kPtSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 16;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= 1) c = 16;
    }
    cudaGetLastError();
    cmax[dev] = c;
  }
  return cmax[dev];
}

// Per-tensor quantization in one launch: a tensor that fits in one cluster's
// shared memory goes to the cluster kernel (no memset, no cooperative
// launch); a larger one to the cooperative kernel, whose CTAs wait on each
// other, so all of them must be resident (the launch fails otherwise).
template <int DT>
fp8s_status launch_per_tensor(const void* x, int64_t numel, uint8_t* q, float* scale, cudaStream_t st,
                              const DeviceInfo& info, int dev) {
  const int64_t nvec = numel / 8;
  const int ntail = static_cast<int>(numel - nvec * 8);
  const uint16_t* tail = static_cast<const uint16_t*>(x) + nvec * 8;
  const int64_t bytes = nvec * 16;
  {
    auto ckern = quant_per_tensor_cluster_kernel<DT>;
    static bool cattr_done[kMaxDevices] = {};
    if (fp8s_status s = ensure_smem_attr(ckern, kPtSmemBytes, cattr_done)) return s;
    const int64_t cmax = pt_cluster_max<DT>(dev);
    if (bytes <= cmax * kPtSliceBytes) {
      // ~64 KB of input per CTA, at least enough CTAs to hold every slice
      const int64_t g_res = (bytes + kPtSliceBytes - 1) / kPtSliceBytes;
      const int64_t G = std::max(g_res, std::min(cmax, std::max<int64_t>(1, (bytes + 65535) / 65536)));
      return launch_ex(ckern, static_cast<unsigned>(G), kPtThreads, kPtSmemBytes, st, static_cast<int>(G),
                       static_cast<const uint4*>(x), nvec, tail, ntail, reinterpret_cast<uint2*>(q), q + nvec * 8,
                       scale, kWaitTimeoutNs);
    }
  }
  auto kern = quant_per_tensor_kernel<DT>;
  static bool attr_done[kMaxDevices] = {};
  if (fp8s_status s = ensure_smem_attr(kern, kPtSmemBytes, attr_done)) return s;
  const int64_t gmax = pt_capacity(dev, info.sms);
  // CTAs: at least 16 KB of input each (for small tensors fewer CTAs mean a
  // cheaper exchange), enough to keep every slice in shared memory when the
  // whole tensor fits on chip, and few enough that CTA 0's slice covers the
  // slot words (G * (G + 1) <= 2 * nvec).
  const int64_t g_res = (bytes + kPtSliceBytes - 1) / kPtSliceBytes;
  int64_t G = std::min<int64_t>(gmax, std::max<int64_t>(1, (bytes + 16383) / 16384));
  bool resident = g_res <= gmax;
  if (resident) G = std::max(G, g_res);
  while (G > 1 && G * (G + 1) > 2 * nvec) --G;
  if (G < g_res) resident = false;
  unsigned int* word = reinterpret_cast<unsigned int*>(scale);
  if (const cudaError_t e = cudaMemsetAsync(word, 0, sizeof(unsigned int), st); e != cudaSuccess) return cuda_fail(e);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(G), 1, 1);
  cfg.blockDim = dim3(kPtThreads, 1, 1);
  cfg.dynamicSmemBytes = kPtSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Streamed slices: the kernel's only waits are the exchange spins.
  const unsigned long long tmo = resident ? kWaitTimeoutNs : g_exchange_timeout_ns.load();
  if (const cudaError_t e =
          cudaLaunchKernelEx(&cfg, kern, static_cast<const uint4*>(x), nvec, tail, ntail, reinterpret_cast<uint2*>(q),
                             q + nvec * 8, word, resident ? 1 : 0, tmo);
      e != cudaSuccess)
    return cuda_fail(e);
  return FP8S_OK;
}

// Per-tensor quantization with a given scale: a grid-stride stream over x,
// one wave of CTAs (as many as the device holds at once), each thread with
// kPsUnroll 32-byte units (eight 16-byte loads) in flight.  The amax slot is
// zeroed first by a one-thread kernel when requested.
template <int DT>
fp8s_status launch_static(const void* x, int64_t numel, const float* scale, uint8_t* q, float* amax,
                          cudaStream_t st, const DeviceInfo& info, int dev) {
  static std::mutex mu;
  static int per_sm[kMaxDevices] = {};
  int resident;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (per_sm[dev] == 0) {
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quant_static_kernel<DT>, kPsThreads, 0) != cudaSuccess ||
          n < 1) {
        cudaGetLastError();
        n = 1;
      }
      per_sm[dev] = n;
    }
    resident = per_sm[dev] * info.sms;
  }
  const int64_t nvec = numel / 8;
  const int ntail = static_cast<int>(numel - nvec * 8);
  const uint16_t* tail = static_cast<const uint16_t*>(x) + nvec * 8;
  if (amax) {
    if (fp8s_status r = launch_ex(zero_word_kernel, 1, 32, 0, st, 1, reinterpret_cast<unsigned int*>(amax))) return r;
  }
  const int64_t per_cta = static_cast<int64_t>(kPsThreads) * kPsUnroll * 2;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((nvec + per_cta - 1) / per_cta, resident));
  return launch_ex(quant_static_kernel<DT>, static_cast<unsigned>(grid), kPsThreads, 0, st, 1,
                   static_cast<const uint4*>(x), nvec, tail, ntail, scale, reinterpret_cast<uint2*>(q), q + nvec * 8,
                   reinterpret_cast<unsigned int*>(amax));
}

// Per-channel weight quantization: persistent CTAs over the rows, each row
// staged in kvec * 16 bytes of shared memory.
template <int DT>
fp8s_status launch_per_channel(const void* w, int64_t N, int64_t K, uint8_t* q, float* sb, cudaStream_t st,
                               const DeviceInfo& info, int dev) {
  auto kern = quant_per_channel_kernel<DT>;
  const int64_t kvec = K / 8;
  const int smem = static_cast<int>(kvec * 16);
  static std::mutex mu;
  static bool attr_done[kMaxDevices] = {};
  int resident;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (smem > 48 * 1024 && !attr_done[dev]) {
      if (const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 128 * 1024);
          e != cudaSuccess)
        return cuda_fail(e);
      attr_done[dev] = true;
    }
    // CTAs per SM depend on the row's shared memory, so this is asked per call
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kPcThreads, smem) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 1;
    }
    resident = n * info.sms;
  }
  const int64_t grid = std::min<int64_t>(N, resident);
  return launch_ex(kern, static_cast<unsigned>(grid), kPcThreads, smem, st, 1, static_cast<const uint4*>(w), N, kvec,
                   reinterpret_cast<uint2*>(q), sb);
}

// ---------------------------------------------------------------- E5M2
// One wave of 256-thread CTAs (8 per SM), fewer for small inputs.
unsigned codec_grid(int64_t units, const DeviceInfo& info) {
  const int64_t want = (units + kCodecThreads - 1) / kCodecThreads;
  const int64_t cap = 8LL * info.sms;
  return static_cast<unsigned>(std::max<int64_t>(1, std::min(want, cap)));
}

template <int DT>
fp8s_status launch_e5m2_encode(const void* x, int64_t numel, uint8_t* q, cudaStream_t st, const DeviceInfo& info) {
  const int64_t nvec = numel / 8;
  const int ntail = static_cast<int>(numel - nvec * 8);
  return launch_ex(e5m2_encode_kernel<DT>, codec_grid(nvec, info), kCodecThreads, 0, st, 1,
                   static_cast<const uint4*>(x), nvec, static_cast<const uint16_t*>(x) + nvec * 8, ntail,
                   reinterpret_cast<uint2*>(q), q + nvec * 8);
}

template <int DT>
fp8s_status launch_e5m2_decode(const uint8_t* q, int64_t numel, void* y, cudaStream_t st, const DeviceInfo& info) {
  const int64_t nvec = numel / 16;
  const int ntail = static_cast<int>(numel - nvec * 16);
  return launch_ex(e5m2_decode_kernel<DT>, codec_grid(nvec, info), kCodecThreads, 0, st, 1,
                   reinterpret_cast<const uint4*>(q), nvec, q + nvec * 16, ntail, static_cast<uint4*>(y),
                   static_cast<uint16_t*>(y) + nvec * 16);
}

// ------------------------------------------------------------------ GEMM
struct GemmChoice {
  int bn = 128;
  int splits = 1;     // CTAs of a cluster sharing one output tile (split-K)
  bool pair = false;  // CTA pairs sharing 256 x bn tiles (tcgen05 cta_group::2)
};

// Tile/split override for tuning sweeps (0 = automatic).
int g_force_bn = 0;
int g_force_splits = 0;
int g_force_pair = 0;

// Most clusters of `splits` CTAs of this kernel the device can hold at once
// (cached per kernel, cluster size and device).
template <typename KernelT>
int max_active_clusters(KernelT kern, int threads, int smem, int splits, int dev, int sms) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, int> cache;
  const uint64_t key = (reinterpret_cast<uint64_t>(reinterpret_cast<const void*>(kern)) << 8) ^
                       (static_cast<uint64_t>(splits) << 4) ^ static_cast<uint64_t>(dev);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  // a grid of one cluster per SM: the count is not capped below what a
  // kernel with several CTAs per SM can hold
  cfg.gridDim = dim3(static_cast<unsigned>(splits * sms), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
  if (e != cudaSuccess || n < 1) {
    cudaGetLastError();
    t_cuda_msg = e != cudaSuccess ? cudaGetErrorString(e) : "no thread-block cluster of this kernel fits on the device";
    n = 0;
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = n;
  return n;
}

template <int BN, int MODE, int OUT, bool SPLIT, bool PAIR, int FR = 0>
fp8s_status launch_gemm_cfg(const CUtensorMap& ma, const CUtensorMap& mb, const GemmParams& p, int splits,
                            const DeviceInfo& info, int dev, cudaStream_t st) {
  using Cfg = GemmCfg<BN, MODE, SPLIT, PAIR, FR>;
  auto kern = fp8_gemm_kernel<BN, MODE, OUT, SPLIT, PAIR, FR>;
  static bool attr_set[kMaxDevices] = {};
  if (fp8s_status s = ensure_smem_attr(kern, Cfg::kSmemBytes, attr_set)) return s;
  if constexpr (PAIR) {
    const int cmax = max_active_clusters(kern, Cfg::kThreads, Cfg::kSmemBytes, 2, dev, info.sms);
    if (cmax < 1) return cuda_fail("no thread-block cluster of this kernel fits on the device");
    const int clusters = p.num_tiles < cmax ? p.num_tiles : cmax;
    return launch_ex(kern, static_cast<unsigned>(clusters * 2), Cfg::kThreads, Cfg::kSmemBytes, st, 2, ma, mb, p);
  } else if constexpr (!SPLIT) {
    const int grid = p.num_tiles < info.sms ? p.num_tiles : info.sms;
    return launch_ex(kern, static_cast<unsigned>(grid), Cfg::kThreads, Cfg::kSmemBytes, st, 1, ma, mb, p);
  } else {
    const int cmax = max_active_clusters(kern, Cfg::kThreads, Cfg::kSmemBytes, splits, dev, info.sms);
    if (cmax < 1) return cuda_fail("no thread-block cluster of this kernel fits on the device");
    // one tile per cluster: the kernel stages its split-K partials in the
    // operand ring, which only drains for good after a cluster's last tile
    if (p.num_tiles > cmax) return FP8S_ERR_SHAPE;
    return launch_ex(kern, static_cast<unsigned>(p.num_tiles * splits), Cfg::kThreads, Cfg::kSmemBytes, st, splits, ma,
                     mb, p);
  }
}

// Time model for choosing the tile width, split-K factor and CTA pairing,
// in microseconds, with constants measured on the B300 (sweeps of every
// configuration over the workloads' shapes, inputs rotated past L2):
//  - a CTA's time per 128-wide K block of its tile is the larger of the
//    tensor-pipe-and-epilogue time (per width, mode and pairing; narrow
//    tiles are bound by shared-memory operand traffic, block mode by the
//    per-K-block promotion in the epilogue) and the time to stream the
//    block's operands at ~85 GB/s per SM;
//  - the whole grid is bound below by the L2 -> SM traffic at ~10.5 TB/s
//    and by HBM traffic at ~6.2 TB/s;
//  - a launch costs ~2.5 us of fixed time (prologue, first loads, tail), a
//    split-K exchange ~4 us more and a CTA pair's start-up ~0.7 us more.
double kb_compute_us(int bn, int mode, bool pair) {
  if (mode == FP8S_SCALE_BLOCK) {
    if (pair) return 1e9;  // a per-K-block hand-off across the pair stalls the MMA
    return bn == 256 ? 0.684 : bn == 192 ? 0.5625 : bn == 128 ? 0.458 : bn == 64 ? 0.415 : 0.39;
  }
  if (pair) return bn == 256 ? 0.43 : bn == 192 ? 0.40 : 0.35;
  return bn == 256 ? 0.475 : bn == 192 ? 0.40 : bn == 128 ? 0.343 : 0.33;
}

// Tensor-core time of one K block of a 128 x bn tile: four MMAs of
// 128 clocks per 256 columns, never below 64 clocks each (measured), ~1.9 GHz.
double kb_mma_us(int bn) { return 4.0 * std::max(64.0, 128.0 * bn / 256.0) / 1.9e3; }

double estimate_us(int64_t M, int64_t N, int64_t KB, int mode, int sms, int bn, int s, bool pair) {
  const int64_t tile_m = pair ? 2 * kBM : kBM;
  const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + bn - 1) / bn);
  const int64_t csize = pair ? 2 : s;
  const int64_t clusters = sms / csize;
  const int64_t waves = (tiles + clusters - 1) / clusters;
  const int64_t nkb = (KB + s - 1) / s;
  const double kb_bytes = 16384.0 + (pair ? bn * 64.0 : bn * 128.0);  // per CTA per K block
  double compute = kb_compute_us(bn, mode, pair);
  if (mode == FP8S_SCALE_BLOCK && M < kBM) {
    // the promotion runs only in the warps whose 32 rows hold a row of M
    const double live = static_cast<double>((M + 31) / 32) / 4.0;
    compute = std::max(kb_mma_us(bn), compute * live);
  }
  const double kb_us = std::max(compute, kb_bytes / 85e3);
  double t = static_cast<double>(waves) * static_cast<double>(nkb) * kb_us;
  const double l2_bytes = static_cast<double>(tiles) * csize * static_cast<double>(nkb) * kb_bytes;
  const double hbm_bytes = static_cast<double>(M) * KB * 128 + static_cast<double>(N) * KB * 128 + 2.0 * M * N;
  t = std::max(t, std::max(l2_bytes / 10.5e6, hbm_bytes / 6.2e6));
  return t + 2.5 + (s > 1 ? 4.0 : 0.0) + (pair ? 0.7 : 0.0);  // a pair also waits on a cluster barrier to start
}

GemmChoice choose_gemm(int64_t M, int64_t N, int64_t KB, int mode, int sms, int max_bn = 256, int min_bn = 32,
                       int max_split_bn = 192) {
  GemmChoice best;
  double best_t = 1e300;
  const int bns[] = {256, 192, 128, 64, 32};
  const int64_t tm = (M + kBM - 1) / kBM;
  for (int bn : bns) {
    if (bn > max_bn || bn < min_bn) continue;
    for (int s = 1; s <= 8; s *= 2) {
      if (s > KB || (s > 1 && bn > max_split_bn)) continue;
      const int64_t tiles = tm * ((N + bn - 1) / bn);
      // split-K needs one tile per cluster (with slack for GPC packing)
      if (s > 1 && tiles > (sms / s) * 7 / 8) continue;
      for (int pr = 0; pr < 2; ++pr) {
        const bool pair = pr != 0;
        // pairs pay off from M = 1024 up (at M = 512, per-tensor 512x11264x2048:
        // 19.8 us paired vs 17.7 us single-CTA 128x192 tiles)
        if (pair && (s > 1 || bn < 64 || M < 1024 || mode == FP8S_SCALE_BLOCK_UE8M0)) continue;
        const double t = estimate_us(M, N, KB, mode, sms, bn, s, pair);
        if (t < best_t * 0.999) {
          best_t = t;
          best.bn = bn;
          best.splits = s;
          best.pair = pair;
        }
      }
    }
  }
  return best;
}

template <int MODE, int OUT>
fp8s_status dispatch_gemm(const GemmChoice& ch, const CUtensorMap& ma, const CUtensorMap& mb, const GemmParams& p,
                          const DeviceInfo& info, int dev, cudaStream_t st) {
  if (ch.pair) {
    if constexpr (MODE == kModeBlock || MODE == kModeUE8) {
      // the block modes' pairs share B by multicast and keep single-CTA MMAs: 256-wide tiles only
      if (ch.bn != 256) return FP8S_ERR_SHAPE;
      return launch_gemm_cfg<256, MODE, OUT, false, true>(ma, mb, p, 2, info, dev, st);
    } else {
      switch (ch.bn) {
        case 64: return launch_gemm_cfg<64, MODE, OUT, false, true>(ma, mb, p, 2, info, dev, st);
        case 128: return launch_gemm_cfg<128, MODE, OUT, false, true>(ma, mb, p, 2, info, dev, st);
        case 192: return launch_gemm_cfg<192, MODE, OUT, false, true>(ma, mb, p, 2, info, dev, st);
        case 256: return launch_gemm_cfg<256, MODE, OUT, false, true>(ma, mb, p, 2, info, dev, st);
        default: return FP8S_ERR_SHAPE;
      }
    }
  }
  if (ch.splits > 1) {
    switch (ch.bn) {
      case 32: return launch_gemm_cfg<32, MODE, OUT, true, false>(ma, mb, p, ch.splits, info, dev, st);
      case 64: return launch_gemm_cfg<64, MODE, OUT, true, false>(ma, mb, p, ch.splits, info, dev, st);
      case 128: return launch_gemm_cfg<128, MODE, OUT, true, false>(ma, mb, p, ch.splits, info, dev, st);
      case 192: return launch_gemm_cfg<192, MODE, OUT, true, false>(ma, mb, p, ch.splits, info, dev, st);
      default: return FP8S_ERR_SHAPE;
    }
  }
  switch (ch.bn) {
    case 32: return launch_gemm_cfg<32, MODE, OUT, false, false>(ma, mb, p, 1, info, dev, st);
    case 64: return launch_gemm_cfg<64, MODE, OUT, false, false>(ma, mb, p, 1, info, dev, st);
    case 128: return launch_gemm_cfg<128, MODE, OUT, false, false>(ma, mb, p, 1, info, dev, st);
    case 192: return launch_gemm_cfg<192, MODE, OUT, false, false>(ma, mb, p, 1, info, dev, st);
    case 256: return launch_gemm_cfg<256, MODE, OUT, false, false>(ma, mb, p, 1, info, dev, st);
    default: return FP8S_ERR_SHAPE;
  }
}

// ---------------------------------------------------------- decode GEMM
// Block-scaled GEMMs of up to 32 tokens run transposed (decode.cuh): one
// cluster of S CTAs per 128-row weight tile, S the largest power of two up to
// 8 with at least one K block per CTA and a grid the SMs hold in one wave
// (two CTAs per SM where the kernel's ~100 KB of shared memory and <= 128
// registers let the hardware place two, else one).  The occupancy
// query reports one CTA per SM for any kernel that allocates tensor memory,
// so it is not asked: the clusters do not depend on one another, and a grid
// larger than the SMs hold still completes.
constexpr int kDecodeMaxM = 32;

// Splits of the decode kernel's K range: the largest power of two up to 8
// with at least one K block per CTA and tiles * S <= slots (CTAs the SMs
// hold at once).
int decode_splits(int64_t tiles, int num_kb, int64_t slots) {
  int s = 8;
  while (s > 1 && (s > num_kb || tiles * s > slots)) s /= 2;
  return s;
}

template <int MT, int OUT, bool SPLIT, int FUSED>
fp8s_status launch_decode_cfg(const CUtensorMap& mw, const CUtensorMap& mx, const GemmParams& p, int splits,
                              const DeviceInfo& info, int dev, cudaStream_t st) {
  using Cfg = DecCfg<MT, SPLIT, FUSED>;
  auto kern = fp8_decode_kernel<MT, OUT, SPLIT, FUSED>;
  static bool attr_set[kMaxDevices] = {};
  if (fp8s_status s = ensure_smem_attr(kern, Cfg::kSmemBytes, attr_set)) return s;
  (void)info;
  (void)dev;
  return launch_ex(kern, static_cast<unsigned>(p.tiles_n * splits), Cfg::kThreads, Cfg::kSmemBytes, st,
                   SPLIT ? splits : 1, mw, mx, p);
}

// s: the split-K (1, 2, 4 or 8); 0 = decode_splits' choice for this kernel.
template <int MT, int OUT, int FUSED>
fp8s_status dispatch_decode(const CUtensorMap& mw, const CUtensorMap& mx, const GemmParams& p, const DeviceInfo& info,
                            int dev, cudaStream_t st, int s = 0) {
  if (s == 0)
    s = decode_splits(p.tiles_n, p.num_kb, DecCfg<MT, true, FUSED>::kCtasPerSm * static_cast<int64_t>(info.sms));
  switch (s) {
    case 8: return launch_decode_cfg<MT, OUT, true, FUSED>(mw, mx, p, 8, info, dev, st);
    case 4: return launch_decode_cfg<MT, OUT, true, FUSED>(mw, mx, p, 4, info, dev, st);
    case 2: return launch_decode_cfg<MT, OUT, true, FUSED>(mw, mx, p, 2, info, dev, st);
    default: return launch_decode_cfg<MT, OUT, false, FUSED>(mw, mx, p, 1, info, dev, st);
  }
}

// qa/x: the E4M3 activation (unfused) or the FP16/BF16 one (fused).
template <bool FUSED>
fp8s_status run_decode(const void* act, const uint8_t* qw, const float* sa, const float* sw, void* c, fp8s_dtype ct,
                       int64_t M, int64_t N, int64_t K, uint8_t* qa_out, float* sa_out, const DeviceInfo& info,
                       int dev, cudaStream_t st) {
  const int mt = M <= 16 ? 16 : 32;
  CUtensorMap mw, mx;
  if (fp8s_status s = tensor_map_e4m3(qw, N, K, kBM, dev, &mw)) return s;
  if constexpr (FUSED) {
    // the box covers the M token rows only (the kernel expects M * 256 bytes)
    if (fp8s_status s = tensor_map_2d(act, M, K, 2, static_cast<int>(M), kBK, false, dev, &mx)) return s;
  } else {
    if (fp8s_status s = tensor_map_e4m3(static_cast<const uint8_t*>(act), M, K, mt, dev, &mx)) return s;
  }
  GemmParams p{};
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.num_kb = static_cast<int>(K / kBK);
  p.tiles_m = 1;
  p.tiles_n = static_cast<int>((N + kBM - 1) / kBM);
  p.num_tiles = p.tiles_n;
  p.group_m = 1;
  p.sa = sa;
  p.sb = sw;
  p.c = c;
  p.timeout_ns = kWaitTimeoutNs;
  p.qa_out = qa_out;
  p.sa_out = sa_out;
  p.x = FUSED ? act : nullptr;
  if constexpr (FUSED) {
    // The resident form (the CTA's whole K range quantized up front) when
    // that range fits its activation buffer, with K split further if needed,
    // one round of its quantizer lanes covers it (2 * M * K blocks <= the
    // 192 lanes of warps 2-7) and M < 16; else the ring form.  (Measured on
    // the Llama-2-7B linears: the resident form is faster up to M = 8, the
    // ring from M = 16.)
    const int act_kb = mt == 16 ? DecCfg<16, true, 2>::kActKb : DecCfg<32, true, 2>::kActKb;
    int s = decode_splits(p.tiles_n, p.num_kb, DecCfg<16, true, 2>::kCtasPerSm * static_cast<int64_t>(info.sms));
    while (s < 8 && 2 * s <= p.num_kb && (p.num_kb + s - 1) / s > act_kb) s *= 2;
    const int kb_per_cta = (p.num_kb + s - 1) / s;
    const bool res = kb_per_cta <= act_kb && 2 * M * kb_per_cta <= 6 * 32 && M < 16;
    if (ct == FP8S_F16) {
      if (mt == 16)
        return res ? dispatch_decode<16, kOutF16, 2>(mw, mx, p, info, dev, st, s)
                   : dispatch_decode<16, kOutF16, 1>(mw, mx, p, info, dev, st);
      return res ? dispatch_decode<32, kOutF16, 2>(mw, mx, p, info, dev, st, s)
                 : dispatch_decode<32, kOutF16, 1>(mw, mx, p, info, dev, st);
    }
    if (mt == 16)
      return res ? dispatch_decode<16, kOutBF16, 2>(mw, mx, p, info, dev, st, s)
                 : dispatch_decode<16, kOutBF16, 1>(mw, mx, p, info, dev, st);
    return res ? dispatch_decode<32, kOutBF16, 2>(mw, mx, p, info, dev, st, s)
               : dispatch_decode<32, kOutBF16, 1>(mw, mx, p, info, dev, st);
  } else {
    if (ct == FP8S_F16)
      return mt == 16 ? dispatch_decode<16, kOutF16, 0>(mw, mx, p, info, dev, st)
                      : dispatch_decode<32, kOutF16, 0>(mw, mx, p, info, dev, st);
    return mt == 16 ? dispatch_decode<16, kOutBF16, 0>(mw, mx, p, info, dev, st)
                    : dispatch_decode<32, kOutBF16, 0>(mw, mx, p, info, dev, st);
  }
}

// The fused linear: block mode, single-CTA tiles of 64 or 128 columns (with
// or without split-K) or 192 columns (split-K only with 16-row boxes);
// FR-row activation boxes.
template <int OUT, int FR>
fp8s_status dispatch_fused(const GemmChoice& ch, const CUtensorMap& mx, const CUtensorMap& mb, const GemmParams& p,
                           const DeviceInfo& info, int dev, cudaStream_t st) {
  if (ch.splits > 1) {
    switch (ch.bn) {
      case 64: return launch_gemm_cfg<64, kModeBlock, OUT, true, false, FR>(mx, mb, p, ch.splits, info, dev, st);
      case 128: return launch_gemm_cfg<128, kModeBlock, OUT, true, false, FR>(mx, mb, p, ch.splits, info, dev, st);
      case 192:
        if constexpr (FR == 16) return launch_gemm_cfg<192, kModeBlock, OUT, true, false, FR>(mx, mb, p, ch.splits, info, dev, st);
        return FP8S_ERR_SHAPE;
      default: return FP8S_ERR_SHAPE;
    }
  }
  switch (ch.bn) {
    case 64: return launch_gemm_cfg<64, kModeBlock, OUT, false, false, FR>(mx, mb, p, 1, info, dev, st);
    case 128: return launch_gemm_cfg<128, kModeBlock, OUT, false, false, FR>(mx, mb, p, 1, info, dev, st);
    case 192: return launch_gemm_cfg<192, kModeBlock, OUT, false, false, FR>(mx, mb, p, 1, info, dev, st);
    default: return FP8S_ERR_SHAPE;
  }
}

}  // namespace
}  // namespace fp8s

using namespace fp8s;

extern "C" {

fp8s_status fp8_quantize_per_tensor(const void* x, fp8s_dtype xt, int64_t numel, uint8_t* q, float* scale,
                                    fp8s_stream_t stream) {
  if (xt != FP8S_F16 && xt != FP8S_BF16) return FP8S_ERR_DTYPE;
  if (!x || !q || !scale) return FP8S_ERR_NULL;
  if (numel < 1) return FP8S_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(q) || !aligned16(scale)) return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  cudaStream_t st = as_stream(stream);
  return xt == FP8S_F16 ? launch_per_tensor<kInF16>(x, numel, q, scale, st, info, dev)
                        : launch_per_tensor<kInBF16>(x, numel, q, scale, st, info, dev);
}

fp8s_status fp8_quantize_per_tensor_static(const void* x, fp8s_dtype xt, int64_t numel, const float* scale,
                                           uint8_t* q, float* amax, fp8s_stream_t stream) {
  if (xt != FP8S_F16 && xt != FP8S_BF16) return FP8S_ERR_DTYPE;
  if (!x || !q || !scale) return FP8S_ERR_NULL;
  if (numel < 1) return FP8S_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(q) || !aligned4(scale) || !aligned4(amax)) return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  cudaStream_t st = as_stream(stream);
  return xt == FP8S_F16 ? launch_static<kInF16>(x, numel, scale, q, amax, st, info, dev)
                        : launch_static<kInBF16>(x, numel, scale, q, amax, st, info, dev);
}

fp8s_status fp8_scale_from_amax_history(const float* history, int64_t H, int margin, float* scale,
                                        fp8s_stream_t stream) {
  if (!history || !scale) return FP8S_ERR_NULL;
  if (H < 1 || H > (1LL << 24) || margin < -64 || margin > 64) return FP8S_ERR_SHAPE;
  if (!aligned4(history) || !aligned4(scale)) return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  return launch_ex(scale_from_history_kernel, 1, kHsThreads, 0, as_stream(stream), 1, history, H, margin, scale);
}

fp8s_status fp8_quantize_token_group(const void* x, fp8s_dtype xt, int64_t M, int64_t K, uint8_t* q, float* sa,
                                     fp8s_stream_t stream) {
  if (xt != FP8S_F16 && xt != FP8S_BF16) return FP8S_ERR_DTYPE;
  if (!x || !q || !sa) return FP8S_ERR_NULL;
  if (M < 1 || K < 128 || K % 128 != 0 || M > (1LL << 31) - 1 || M * (K / 128) > (1LL << 31) - 1)
    return FP8S_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sa)) return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  cudaStream_t st = as_stream(stream);
  return xt == FP8S_F16 ? launch_token_group<kInF16>(x, M, K, q, sa, st, info)
                        : launch_token_group<kInBF16>(x, M, K, q, sa, st, info);
}

fp8s_status fp8_quantize_weight_block(const void* w, fp8s_dtype wt, int64_t N, int64_t K, uint8_t* q, float* sb,
                                      fp8s_stream_t stream) {
  if (wt != FP8S_F16 && wt != FP8S_BF16) return FP8S_ERR_DTYPE;
  if (!w || !q || !sb) return FP8S_ERR_NULL;
  if (N < 1 || K < 128 || K % 128 != 0 || K / 128 > 65535 || N > (1LL << 31) - 128 ||
      ((N + 127) / 128) * (K / 128) > (1LL << 31) - 1)
    return FP8S_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(q) || !aligned16(sb)) return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  cudaStream_t st = as_stream(stream);
  return wt == FP8S_F16 ? launch_weight_block<kInF16>(w, N, K, q, sb, st, info, dev)
                        : launch_weight_block<kInBF16>(w, N, K, q, sb, st, info, dev);
}

fp8s_status fp8_quantize_token_group_ue8m0(const void* x, fp8s_dtype xt, int64_t M, int64_t K, uint8_t* q,
                                           uint8_t* sa_code, fp8s_stream_t stream) {
  if (xt != FP8S_F16 && xt != FP8S_BF16) return FP8S_ERR_DTYPE;
  if (!x || !q || !sa_code) return FP8S_ERR_NULL;
  if (M < 1 || K < 128 || K % 128 != 0 || M > (1LL << 31) - 1 || M * (K / 128) > (1LL << 31) - 1)
    return FP8S_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sa_code)) return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  cudaStream_t st = as_stream(stream);
  return xt == FP8S_F16 ? launch_token_group<kInF16, true>(x, M, K, q, sa_code, st, info)
                        : launch_token_group<kInBF16, true>(x, M, K, q, sa_code, st, info);
}

fp8s_status fp8_quantize_weight_block_ue8m0(const void* w, fp8s_dtype wt, int64_t N, int64_t K, uint8_t* q,
                                            uint8_t* sb_code, fp8s_stream_t stream) {
  if (wt != FP8S_F16 && wt != FP8S_BF16) return FP8S_ERR_DTYPE;
  if (!w || !q || !sb_code) return FP8S_ERR_NULL;
  if (N < 1 || K < 128 || K % 128 != 0 || K / 128 > 65535 || N > (1LL << 31) - 128 ||
      ((N + 127) / 128) * (K / 128) > (1LL << 31) - 1)
    return FP8S_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(q) || !aligned16(sb_code)) return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  cudaStream_t st = as_stream(stream);
  return wt == FP8S_F16 ? launch_weight_block<kInF16, true>(w, N, K, q, sb_code, st, info, dev)
                        : launch_weight_block<kInBF16, true>(w, N, K, q, sb_code, st, info, dev);
}

fp8s_status fp8_quantize_per_channel(const void* w, fp8s_dtype wt, int64_t N, int64_t K, uint8_t* q, float* sb,
                                     fp8s_stream_t stream) {
  if (wt != FP8S_F16 && wt != FP8S_BF16) return FP8S_ERR_DTYPE;
  if (!w || !q || !sb) return FP8S_ERR_NULL;
  if (N < 1 || K < 8 || K % 8 != 0 || K > 65536 || N > (1LL << 31) - 1) return FP8S_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(q) || !aligned16(sb)) return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  cudaStream_t st = as_stream(stream);
  return wt == FP8S_F16 ? launch_per_channel<kInF16>(w, N, K, q, sb, st, info, dev)
                        : launch_per_channel<kInBF16>(w, N, K, q, sb, st, info, dev);
}

fp8s_status fp8_e5m2_encode(const void* x, fp8s_dtype xt, int64_t numel, uint8_t* q, fp8s_stream_t stream) {
  if (xt != FP8S_F16 && xt != FP8S_BF16) return FP8S_ERR_DTYPE;
  if (!x || !q) return FP8S_ERR_NULL;
  if (numel < 1) return FP8S_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(q)) return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  cudaStream_t st = as_stream(stream);
  return xt == FP8S_F16 ? launch_e5m2_encode<kInF16>(x, numel, q, st, info)
                        : launch_e5m2_encode<kInBF16>(x, numel, q, st, info);
}

fp8s_status fp8_e5m2_decode(const uint8_t* q, int64_t numel, void* y, fp8s_dtype yt, fp8s_stream_t stream) {
  if (yt != FP8S_F16 && yt != FP8S_BF16) return FP8S_ERR_DTYPE;
  if (!q || !y) return FP8S_ERR_NULL;
  if (numel < 1) return FP8S_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(y)) return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  cudaStream_t st = as_stream(stream);
  return yt == FP8S_F16 ? launch_e5m2_decode<kInF16>(q, numel, y, st, info)
                        : launch_e5m2_decode<kInBF16>(q, numel, y, st, info);
}

fp8s_status fp8_gemm_scaled(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb, void* c,
                            fp8s_dtype ct, int64_t M, int64_t N, int64_t K, fp8s_scale_mode mode_in,
                            fp8s_stream_t stream) {
  if (ct != FP8S_F16 && ct != FP8S_BF16) return FP8S_ERR_DTYPE;
  if (mode_in != FP8S_SCALE_PER_TENSOR && mode_in != FP8S_SCALE_BLOCK && mode_in != FP8S_SCALE_PER_CHANNEL &&
      mode_in != FP8S_SCALE_BLOCK_UE8M0)
    return FP8S_ERR_DTYPE;
  // per-channel weights run the per-tensor kernels with a per-column sB
  const bool per_col = mode_in == FP8S_SCALE_PER_CHANNEL;
  const fp8s_scale_mode mode = per_col ? FP8S_SCALE_PER_TENSOR : mode_in;
  if (!qa || !sa || !qb || !sb || !c) return FP8S_ERR_NULL;
  if (M < 1 || N < 1 || K < 16 || K % 16 != 0) return FP8S_ERR_SHAPE;
  if ((mode == FP8S_SCALE_BLOCK || mode == FP8S_SCALE_BLOCK_UE8M0) && K % 128 != 0) return FP8S_ERR_SHAPE;
  if (M > (1LL << 31) - 256 || N > (1LL << 31) - 256 || K > (1LL << 31) - 256 || M * N > (1LL << 40))
    return FP8S_ERR_SHAPE;
  if (!aligned16(qa) || !aligned16(sa) || !aligned16(qb) || !aligned16(sb) || !aligned16(c)) return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  cudaStream_t st = as_stream(stream);

  const int64_t KB = (K + kBK - 1) / kBK;
  if (mode == FP8S_SCALE_BLOCK && !per_col && M <= kDecodeMaxM && !g_force_bn)
    return run_decode<false>(qa, qb, sa, sb, c, ct, M, N, K, nullptr, nullptr, info, dev, st);
  GemmChoice ch = choose_gemm(M, N, KB, mode, info.sms);
  if (g_force_bn) {
    ch.bn = g_force_bn;
    ch.splits = g_force_splits > 0 ? g_force_splits : 1;
    ch.pair = g_force_pair != 0;
    if (ch.splits > KB) return FP8S_ERR_SHAPE;

  }
  const int bn = ch.bn;
  const int tile_m = ch.pair ? 2 * kBM : kBM;
  CUtensorMap ma, mb;
  if (fp8s_status s = tensor_map_e4m3(qa, M, K, kBM, dev, &ma)) return s;
  if (fp8s_status s = tensor_map_e4m3(qb, N, K, ch.pair ? bn / 2 : bn, dev, &mb)) return s;

  GemmParams p{};
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.num_kb = static_cast<int>(KB);
  p.tiles_m = static_cast<int>((M + tile_m - 1) / tile_m);
  p.tiles_n = static_cast<int>((N + bn - 1) / bn);
  const int64_t tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
  if (tiles > (1LL << 31) - 1) return FP8S_ERR_SHAPE;
  p.num_tiles = static_cast<int>(tiles);
  p.group_m = p.tiles_m < 16 ? p.tiles_m : 16;
  p.sa = sa;
  p.sb = sb;
  p.c = c;
  p.timeout_ns = kWaitTimeoutNs;

  auto run = [&](const GemmChoice& c) {
    if (per_col)
      return ct == FP8S_F16 ? dispatch_gemm<kModePerChannel, kOutF16>(c, ma, mb, p, info, dev, st)
                            : dispatch_gemm<kModePerChannel, kOutBF16>(c, ma, mb, p, info, dev, st);
    if (mode == FP8S_SCALE_PER_TENSOR)
      return ct == FP8S_F16 ? dispatch_gemm<kModePerTensor, kOutF16>(c, ma, mb, p, info, dev, st)
                            : dispatch_gemm<kModePerTensor, kOutBF16>(c, ma, mb, p, info, dev, st);
    if (mode == FP8S_SCALE_BLOCK_UE8M0)
      return ct == FP8S_F16 ? dispatch_gemm<kModeUE8, kOutF16>(c, ma, mb, p, info, dev, st)
                            : dispatch_gemm<kModeUE8, kOutBF16>(c, ma, mb, p, info, dev, st);
    return ct == FP8S_F16 ? dispatch_gemm<kModeBlock, kOutF16>(c, ma, mb, p, info, dev, st)
                          : dispatch_gemm<kModeBlock, kOutBF16>(c, ma, mb, p, info, dev, st);
  };
  fp8s_status r = run(ch);
  if (r == FP8S_ERR_SHAPE && ch.splits > 1 && !g_force_bn) {
    // the device holds fewer clusters than the estimate assumed: no split
    ch.splits = 1;
    r = run(ch);
  }
  return r;
}

fp8s_status fp8_linear_token_group(const void* x, fp8s_dtype xt, int64_t M, int64_t K, const uint8_t* qw,
                                   const float* sw, int64_t N, void* c, uint8_t* qa, float* sa, fp8s_stream_t stream) {
  if (xt != FP8S_F16 && xt != FP8S_BF16) return FP8S_ERR_DTYPE;
  if (!x || !qw || !sw || !c || (!qa) != (!sa)) return FP8S_ERR_NULL;
  if (M < 1 || N < 1 || K < 128 || K % 128 != 0) return FP8S_ERR_SHAPE;
  if (M > (1LL << 31) - 256 || N > (1LL << 31) - 256 || K > (1LL << 31) - 256 || M * N > (1LL << 40) ||
      M * (K / 128) > (1LL << 31) - 1)
    return FP8S_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(qw) || !aligned16(sw) || !aligned16(c) || (qa && (!aligned16(qa) || !aligned16(sa))))
    return FP8S_ERR_ALIGN;
  int dev;
  DeviceInfo info;
  if (fp8s_status s = current_device(&dev, &info)) return s;
  cudaStream_t st = as_stream(stream);

  const int64_t KB = K / kBK;
  if (M <= kDecodeMaxM && !g_force_bn)
    return run_decode<true>(x, qw, nullptr, sw, c, xt, M, N, K, qa, sa, info, dev, st);
  // the fused kernel's tile widths: 64, 128 and 192 (split-K at 192 only with
  // 16-row activation boxes, M <= 16)
  const int fr = M <= 16 ? 16 : 128;   // rows of the activation box: M <= 16 needs only 16
  GemmChoice ch = choose_gemm(M, N, KB, FP8S_SCALE_BLOCK, info.sms, 192, 64, fr == 16 ? 192 : 128);
  if (g_force_bn) {
    ch.bn = g_force_bn;
    ch.splits = g_force_splits > 0 ? g_force_splits : 1;
    if (g_force_pair || (ch.bn != 64 && ch.bn != 128 && ch.bn != 192) || (ch.bn == 192 && ch.splits > 1 && fr != 16) ||
        ch.splits > KB)
      return FP8S_ERR_SHAPE;
  }
  CUtensorMap mx, mb;
  if (fp8s_status s = tensor_map_2d(x, M, K, 2, fr, kBK, false, dev, &mx)) return s;
  if (fp8s_status s = tensor_map_e4m3(qw, N, K, ch.bn, dev, &mb)) return s;

  GemmParams p{};
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.num_kb = static_cast<int>(KB);
  p.tiles_m = static_cast<int>((M + kBM - 1) / kBM);
  p.tiles_n = static_cast<int>((N + ch.bn - 1) / ch.bn);
  const int64_t tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
  if (tiles > (1LL << 31) - 1) return FP8S_ERR_SHAPE;
  p.num_tiles = static_cast<int>(tiles);
  p.group_m = p.tiles_m < 16 ? p.tiles_m : 16;
  p.sa = nullptr;
  p.sb = sw;
  p.c = c;
  p.timeout_ns = kWaitTimeoutNs;
  p.qa_out = qa;
  p.sa_out = sa;
  auto run = [&](const GemmChoice& cc) {
    if (xt == FP8S_F16)
      return fr == 16 ? dispatch_fused<kOutF16, 16>(cc, mx, mb, p, info, dev, st)
                      : dispatch_fused<kOutF16, 128>(cc, mx, mb, p, info, dev, st);
    return fr == 16 ? dispatch_fused<kOutBF16, 16>(cc, mx, mb, p, info, dev, st)
                    : dispatch_fused<kOutBF16, 128>(cc, mx, mb, p, info, dev, st);
  };
  fp8s_status r = run(ch);
  if (r == FP8S_ERR_SHAPE && ch.splits > 1 && !g_force_bn) {
    ch.splits = 1;   // the device holds fewer clusters than the estimate assumed: no split
    r = run(ch);
  }
  return r;
}

fp8s_status fp8s_gemm_plan(int64_t M, int64_t N, int64_t K, fp8s_scale_mode mode_in, int sms, int* bn, int* splits,
                           int* pair) {
  if (mode_in != FP8S_SCALE_PER_TENSOR && mode_in != FP8S_SCALE_BLOCK && mode_in != FP8S_SCALE_PER_CHANNEL &&
      mode_in != FP8S_SCALE_BLOCK_UE8M0)
    return FP8S_ERR_DTYPE;
  const fp8s_scale_mode mode = mode_in == FP8S_SCALE_PER_CHANNEL ? FP8S_SCALE_PER_TENSOR : mode_in;
  if (!bn || !splits || !pair) return FP8S_ERR_NULL;
  if (M < 1 || N < 1 || K < 16 || K % 16 != 0 || sms < 1) return FP8S_ERR_SHAPE;
  if ((mode == FP8S_SCALE_BLOCK || mode == FP8S_SCALE_BLOCK_UE8M0) && K % 128 != 0) return FP8S_ERR_SHAPE;
  if (mode == FP8S_SCALE_BLOCK && M <= kDecodeMaxM) {
    // the transposed decode kernel: 128 output columns a tile, split-K
    *bn = kBM;
    *splits = decode_splits((N + kBM - 1) / kBM, static_cast<int>(K / kBK),
                            DecCfg<16, true, 0>::kCtasPerSm * static_cast<int64_t>(sms));
    *pair = 0;
    return FP8S_OK;
  }
  const GemmChoice ch = choose_gemm(M, N, (K + kBK - 1) / kBK, mode, sms);
  *bn = ch.bn;
  *splits = ch.splits;
  *pair = ch.pair ? 1 : 0;
  return FP8S_OK;
}

fp8s_status fp8s_gemm_override(int bn, int splits, int pair) {
  if (bn == 0) {
    g_force_bn = 0;
    g_force_splits = 0;
    g_force_pair = 0;
    return FP8S_OK;
  }
  if ((bn != 32 && bn != 64 && bn != 128 && bn != 192 && bn != 256) ||
      (splits != 1 && splits != 2 && splits != 4 && splits != 8))
    return FP8S_ERR_SHAPE;
  if (pair && (splits != 1 || bn < 64)) return FP8S_ERR_SHAPE;
  if (splits > 1 && bn > 192) return FP8S_ERR_SHAPE;  // split-K exchanges the partial tile in one pass
  g_force_bn = bn;
  g_force_splits = splits;
  g_force_pair = pair ? 1 : 0;
  return FP8S_OK;
}

const char* fp8s_status_string(fp8s_status status) {
  switch (status) {
    case FP8S_OK: return "ok";
    case FP8S_ERR_NULL: return "null pointer argument";
    case FP8S_ERR_SHAPE: return "size out of range or not a required multiple";
    case FP8S_ERR_ALIGN: return "pointer not 16-byte aligned";
    case FP8S_ERR_DTYPE: return "unknown dtype or scale mode";
    case FP8S_ERR_CUDA: return "CUDA call or kernel launch failed";
    case FP8S_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait expired";
    case FP8S_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (B300)";
  }
  return "unknown status";
}

fp8s_status fp8s_device_error(fp8s_stream_t stream, int* where) {
  if (const cudaError_t e = cudaStreamSynchronize(as_stream(stream)); e != cudaSuccess) return cuda_fail(e);
  unsigned int word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_fp8s_error, sizeof word) != cudaSuccess ||
      cudaMemcpyToSymbol(g_fp8s_error, &zero, sizeof zero) != cudaSuccess) {
    return cuda_fail(cudaGetLastError());
  }
  if (where) *where = static_cast<int>(word);
  return word ? FP8S_ERR_DEVICE_TIMEOUT : FP8S_OK;
}

fp8s_status fp8s_set_exchange_timeout_ns(unsigned long long ns) {
  g_exchange_timeout_ns.store(ns == 0 ? kWaitTimeoutNs : ns);
  return FP8S_OK;
}

int fp8s_version(void) { return kVersion; }

const char* fp8s_last_cuda_error(void) { return t_cuda_msg; }

}  // extern "C"
