// C ABI entry points: argument checks, the arch witness, the tile-fill gate,
// the whole-product call, launch counters and the device error word.
//
// Sources: page "fix(qtip): gate the trellis grouped GEMM on m-tile occupancy,
// not token count" ("The cause is a threshold", "The fix", post-merge note:
// the closed form, the predicate, the n <= 8 floor and the GEMV pin; the
// once-per-process engagement log line), and page "perf(qtip): arch-specialise
// the trellis grouped GEMM (D16) + close the silent-failure holes (D18)" ("D18",
// "The arch witness": statuses on every launcher, empty grids refused, the
// witness compiled under the same guard as the kernel, not taken during
// capture, only a successful answer cached).
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kMaxDevices = 64;

__device__ int g_error_word[2];     // code, where
__device__ int g_witness_arch;      // written by the witness kernel

// Compiled under the same guard as the tensor-core kernels: an image without
// sm_103a device code leaves g_witness_arch at the sentinel.
__global__ void arch_witness_kernel() {
#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 1000) && defined(__CUDA_ARCH_FEAT_SM103_ALL)
  g_witness_arch = __CUDA_ARCH__;
#elif defined(__CUDA_ARCH__)
  g_witness_arch = -__CUDA_ARCH__;
#endif
}

std::atomic<int> g_witness_ok[kMaxDevices];   // 0 unknown, 1 ok (only success is cached)
std::atomic<int> g_witness_val[kMaxDevices];
std::atomic<int*> g_err_ptr[kMaxDevices];
std::atomic<int> g_sms[kMaxDevices];
std::atomic<long long> g_counts[kCntNum];
std::once_flag g_log_once;

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  if (*dev < 0 || *dev >= kMaxDevices) return TQ_ERR_CUDA;
  return TQ_OK;
}

bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();
    return true;  // cannot tell: treat as capturing (decline rather than guess)
  }
  return cs != cudaStreamCaptureStatusNone;
}

int take_witness(int dev, int* arch_out) {
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  if (!(prop.major == 10 && prop.minor == 3)) return TQ_ERR_UNSUPPORTED_ARCH;
  if (stream_capturing(cudaStreamLegacy) || stream_capturing(cudaStreamPerThread)) return TQ_ERR_CAPTURING;
  cudaStream_t s;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  int rc = TQ_OK;
  const int sentinel = 0;
  int arch = 0;
  if (cudaMemcpyToSymbolAsync(g_witness_arch, &sentinel, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
      cudaSuccess) {
    rc = TQ_ERR_CUDA;
  } else {
    arch_witness_kernel<<<1, 1, 0, s>>>();
    if (cudaGetLastError() != cudaSuccess) {
      rc = TQ_ERR_UNSUPPORTED_ARCH;  // no loadable image for this device
    } else if (cudaMemcpyFromSymbolAsync(&arch, g_witness_arch, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
                   cudaSuccess ||
               cudaStreamSynchronize(s) != cudaSuccess) {
      rc = TQ_ERR_CUDA;
    }
  }
  cudaGetLastError();
  cudaStreamDestroy(s);
  if (rc != TQ_OK) return rc;
  if (arch_out) *arch_out = arch;
  if (arch < 1030) return TQ_ERR_UNSUPPORTED_ARCH;  // sentinel or another architecture's body
  g_witness_val[dev].store(arch);
  g_witness_ok[dev].store(1);
  return TQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool bad_shape(int top_k, int E) { return E < 1 || top_k < 1 || top_k > E; }

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

}  // namespace

int* error_word(int* status) {
  int dev;
  *status = current_device(&dev);
  if (*status != TQ_OK) return nullptr;
  int* p = g_err_ptr[dev].load();
  if (!p) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_error_word) != cudaSuccess) {
      cudaGetLastError();
      *status = TQ_ERR_CUDA;
      return nullptr;
    }
    p = static_cast<int*>(a);
    g_err_ptr[dev].store(p);
  }
  return p;
}

int require_sm103(cudaStream_t stream) {
  int dev;
  int rc = current_device(&dev);
  if (rc != TQ_OK) return rc;
  if (g_witness_ok[dev].load()) return TQ_OK;
  if (stream_capturing(stream)) return TQ_ERR_CAPTURING;
  return take_witness(dev, nullptr);
}

int launch_status() {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return TQ_OK;
  if (e == cudaErrorInvalidConfiguration || e == cudaErrorLaunchOutOfResources) return TQ_ERR_LAUNCH;
  if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction) return TQ_ERR_UNSUPPORTED_ARCH;
  return TQ_ERR_LAUNCH;
}

void count_launch(Counter c) { g_counts[c].fetch_add(1); }

int sm_count() {
  int dev = 0;
  if (current_device(&dev) != TQ_OK) return 1;
  int v = g_sms[dev].load();
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
      cudaGetLastError();
      v = 1;
    }
    g_sms[dev].store(v);
  }
  return v;
}

// TQ_TILE_M=<1..256>: the kernel m-tile of whole-product calls made with
// TQ_TILE_NATIVE (0 or unset: the native tile; anything else is ignored with
// one warning).
static int env_tile_m() {
  const char* v = std::getenv("TQ_TILE_M");
  if (!v || !*v) return 0;
  char* endp = nullptr;
  const long t = std::strtol(v, &endp, 10);
  if (endp && *endp == '\0' && t >= 0 && t <= 256) return static_cast<int>(t);
  static std::once_flag warned;
  std::call_once(warned, [v] {
    std::fprintf(stderr, "tqmoe: ignoring TQ_TILE_M=%s (expected 0..256)\n", v);
  });
  return 0;
}

bool resolve_tile(int64_t n, int top_k, int E, int tile_m, int* kernel_tile, int* gate_tile) {
  if (tile_m == TQ_TILE_NATIVE) {
    const int t = tq_native_tile_m(n, top_k, E);
    if (t < 0) return false;
    const int forced = env_tile_m();
    *kernel_tile = forced > 0 ? forced : t;
    *gate_tile = TQ_GATE_TILE_M;
    return true;
  }
  if (tile_m < 1 || tile_m > 256) return false;
  *kernel_tile = *gate_tile = tile_m;
  return true;
}

// Every region is 256-byte aligned and sized as in tq_moe_workspace_size.
MoeScratch carve_moe_scratch(void* workspace, int64_t n, int top_k, int E, int K, int N, int64_t cap,
                             int kernel_tile_m) {
  const size_t P = static_cast<size_t>(n) * top_k;
  MoeScratch m{};
  uint8_t* w = static_cast<uint8_t*>(workspace);
  m.counts = reinterpret_cast<int32_t*>(w);        w += align256(sizeof(int32_t) * E);
  m.offsets = reinterpret_cast<int32_t*>(w);       w += align256(sizeof(int32_t) * (E + 1));
  m.sorted_pairs = reinterpret_cast<int32_t*>(w);  w += align256(sizeof(int32_t) * std::max<size_t>(P, 1));
  m.tiles = reinterpret_cast<int32_t*>(w);         w += align256(sizeof(int32_t) * 3 * std::max<int64_t>(cap, 1));
  m.num_tiles = reinterpret_cast<int32_t*>(w);     w += align256(sizeof(int32_t));
  m.y32 = reinterpret_cast<float*>(w);             w += align256(sizeof(float) * static_cast<size_t>(n) * N);
  m.x_sorted = nullptr;
  m.slot_of = nullptr;
  if (!gathers_in_kernel(kernel_tile_m)) {
    m.x_sorted = reinterpret_cast<uint16_t*>(w);   w += align256(sizeof(uint16_t) * P * K);
    m.slot_of = reinterpret_cast<int32_t*>(w);     w += align256(sizeof(int32_t) * std::max<size_t>(P, 1));
  }
  m.end = w;
  return m;
}

int env_pin(int pin) {
  if (pin != TQ_ARM_AUTO) return pin;
  const char* v = std::getenv("TQ_FORCE_ARM");
  if (!v || !*v || !std::strcmp(v, "auto")) return TQ_ARM_AUTO;
  if (!std::strcmp(v, "gemv")) return TQ_ARM_GEMV;
  if (!std::strcmp(v, "grouped")) return TQ_ARM_GROUPED;
  if (!std::strcmp(v, "measured")) return TQ_ARM_MEASURED;
  static std::once_flag warned;
  std::call_once(warned, [v] {
    std::fprintf(stderr, "tqmoe: unknown TQ_FORCE_ARM=%s (expected auto|gemv|grouped|measured); keeping auto\n", v);
  });
  return TQ_ARM_AUTO;
}

}  // namespace tq

using namespace tq;

extern "C" {

const char* tq_status_string(int status) {
  switch (status) {
    case TQ_OK: return "TQ_OK";
    case TQ_ERR_INVALID_ARG: return "TQ_ERR_INVALID_ARG: invalid argument";
    case TQ_ERR_UNSUPPORTED_ARCH: return "TQ_ERR_UNSUPPORTED_ARCH: device or binary lacks sm_103a code";
    case TQ_ERR_CAPACITY: return "TQ_ERR_CAPACITY: tile map over capacity";
    case TQ_ERR_LAUNCH: return "TQ_ERR_LAUNCH: kernel launch failed";
    case TQ_ERR_CAPTURING: return "TQ_ERR_CAPTURING: arch witness cannot be taken during capture";
    case TQ_ERR_DEVICE_TIMEOUT: return "TQ_ERR_DEVICE_TIMEOUT: a device-side wait gave up";
    case TQ_ERR_CUDA: return "TQ_ERR_CUDA: CUDA runtime error";
    case TQ_ERR_WORKSPACE: return "TQ_ERR_WORKSPACE: workspace too small or misaligned";
    default: return "unknown tq status";
  }
}

int tq_init(int device) {
  if (device < 0 || device >= kMaxDevices) return TQ_ERR_INVALID_ARG;
  if (cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  if (g_witness_ok[device].load()) return TQ_OK;
  return take_witness(device, nullptr);
}

int tq_arch_witness(int device, int* arch_out) {
  if (device < 0 || device >= kMaxDevices) return TQ_ERR_INVALID_ARG;
  if (cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  if (g_witness_ok[device].load()) {
    if (arch_out) *arch_out = g_witness_val[device].load();
    return TQ_OK;
  }
  return take_witness(device, arch_out);
}

double tq_pairs_per_woken_expert(int64_t n, int top_k, int E) {
  if (bad_shape(top_k, E) || n < 0) return std::nan("");
  if (n == 0) return 0.0;
  const double nd = static_cast<double>(n);
  const double woken = static_cast<double>(E) * (1.0 - std::pow(1.0 - static_cast<double>(top_k) / E, nd));
  return nd * top_k / woken;
}

int tq_tiles_amortize(int64_t n, int top_k, int E, int tile_m) {
  if (bad_shape(top_k, E) || tile_m < 1 || n < 0) return TQ_ERR_INVALID_ARG;
  if (n == 0) return 0;
  return tq_pairs_per_woken_expert(n, top_k, E) >= static_cast<double>(tile_m) ? 1 : 0;
}

int64_t tq_grouped_min_tokens(int top_k, int E, int tile_m) {
  if (bad_shape(top_k, E) || tile_m < 1) return TQ_ERR_INVALID_ARG;
  // pairs per woken expert is increasing in n and reaches tile_m by
  // n = ceil(tile_m * E / top_k): bisect on [1, that], then confirm the flip.
  int64_t lo = 0, hi = (static_cast<int64_t>(tile_m) * E + top_k - 1) / top_k;
  if (hi < 1) hi = 1;
  while (tq_tiles_amortize(hi, top_k, E, tile_m) != 1) hi *= 2;
  while (hi - lo > 1) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (tq_tiles_amortize(mid, top_k, E, tile_m) == 1) hi = mid; else lo = mid;
  }
  return hi;
}

int64_t tq_tile_map_capacity(int64_t n, int top_k, int E, int tile_m) {
  if (bad_shape(top_k, E) || tile_m < 1 || n < 0) return TQ_ERR_INVALID_ARG;
  const int64_t P = n * top_k;
  const int64_t bound = P / tile_m + std::min<int64_t>(E, P);
  return std::min<int64_t>(P, bound);
}

int tq_select_arm(int64_t n, int top_k, int E, int tile_m, int pin) {
  if (bad_shape(top_k, E) || tile_m < 1 || n < 0) return TQ_ERR_INVALID_ARG;
  if (pin == TQ_ARM_GEMV || pin == TQ_ARM_GROUPED) return pin;
  if (pin == TQ_ARM_MEASURED)
    return (n > 0 && tq_pairs_per_woken_expert(n, top_k, E) >= TQ_MEASURED_CROSSOVER_PPW) ? TQ_ARM_GROUPED
                                                                                         : TQ_ARM_GEMV;
  if (pin != TQ_ARM_AUTO) return TQ_ERR_INVALID_ARG;
  if (n <= TQ_DECODE_REGIME_MAX_TOKENS) return TQ_ARM_GEMV;
  return tq_tiles_amortize(n, top_k, E, tile_m) == 1 ? TQ_ARM_GROUPED : TQ_ARM_GEMV;
}

int tq_route(const int32_t* topk_ids, int64_t n, int top_k, int E, int32_t* counts, int32_t* offsets,
             int32_t* sorted_pairs, tq_stream_t stream) {
  if (bad_shape(top_k, E) || E > 1024 || n < 0) return TQ_ERR_INVALID_ARG;
  const int64_t P = n * top_k;
  if (P >= (static_cast<int64_t>(1) << 31)) return TQ_ERR_INVALID_ARG;
  if (!counts || !offsets || (P > 0 && (!topk_ids || !sorted_pairs))) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  int* err = error_word(&rc);
  if (!err) return rc;
  return launch_route(topk_ids, static_cast<int>(P), E, counts, offsets, sorted_pairs, err, s);
}

int tq_router_topk(const float* logits, int64_t n, int E, int top_k, int32_t* topk_ids, float* topk_w,
                   tq_stream_t stream) {
  if (bad_shape(top_k, E) || E > 1024 || top_k > 32 || n < 0 || n >= (static_cast<int64_t>(1) << 31))
    return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!logits || !topk_ids || !topk_w)) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  return launch_router(logits, static_cast<int>(n), E, top_k, topk_ids, topk_w, s);
}

int tq_route_logits(const float* logits, int64_t n, int E, int top_k, int32_t* topk_ids, float* topk_w,
                    int32_t* counts, int32_t* offsets, int32_t* sorted_pairs, tq_stream_t stream) {
  int rc = tq_router_topk(logits, n, E, top_k, topk_ids, topk_w, stream);
  if (rc != TQ_OK) return rc;
  return tq_route(topk_ids, n, top_k, E, counts, offsets, sorted_pairs, stream);
}

int tq_build_tile_map(const int32_t* offsets, int E, int tile_m, int32_t* tiles, int32_t* num_tiles,
                      int64_t cap, tq_stream_t stream) {
  if (E < 1 || E > 1024 || tile_m < 1 || tile_m > 256 || cap < 1 || cap >= (static_cast<int64_t>(1) << 31))
    return TQ_ERR_INVALID_ARG;
  if (!offsets || !tiles || !num_tiles) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  int* err = error_word(&rc);
  if (!err) return rc;
  return launch_tile_map(offsets, E, tile_m, tiles, num_tiles, cap, err, s);
}

static int check_gemm_common(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L,
                             const float* topk_w, int64_t n, int top_k, int E, int K, int N,
                             const void* out) {
  if (bad_shape(top_k, E) || n < 0 || K < 64 || K % 64 != 0 || N < 1) return TQ_ERR_INVALID_ARG;
  if (L < 2 || L > 16 || (L & 1)) return TQ_ERR_INVALID_ARG;
  if (n * top_k >= (static_cast<int64_t>(1) << 31)) return TQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(E) * N >= (static_cast<int64_t>(1) << 31)) return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!x || !packed || !lut || !topk_w || !out)) return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!aligned16(x) || !aligned16(packed) || !aligned16(lut))) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

int tq_gather_rows(const uint16_t* x, const int32_t* sorted_pairs, int64_t n, int top_k, int K,
                   uint16_t* x_sorted, tq_stream_t stream) {
  if (n < 0 || top_k < 1 || K < 8 || K % 8 != 0) return TQ_ERR_INVALID_ARG;
  const int64_t P = n * top_k;
  if (P >= (static_cast<int64_t>(1) << 31)) return TQ_ERR_INVALID_ARG;
  if (P > 0 && (!x || !sorted_pairs || !x_sorted || !aligned16(x) || !aligned16(x_sorted)))
    return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  int* err = error_word(&rc);
  if (!err) return rc;
  return launch_gather(x, sorted_pairs, static_cast<int>(P), top_k, K, x_sorted, err, s);
}

int tq_prepare(const int32_t* topk_ids, const uint16_t* x, int64_t n, int top_k, int E, int K, int tile_m,
               int32_t* counts, int32_t* offsets, int32_t* sorted_pairs, int32_t* tiles, int32_t* num_tiles,
               int64_t cap, uint16_t* x_sorted, float* y32, int64_t y32_count, tq_stream_t stream) {
  if (bad_shape(top_k, E) || E > 1024 || n < 0 || tile_m < 1 || K < 8 || K % 8 != 0 || y32_count < 0)
    return TQ_ERR_INVALID_ARG;
  if (cap < 1 || cap >= (static_cast<int64_t>(1) << 31)) return TQ_ERR_INVALID_ARG;
  const int64_t P = n * top_k;
  if (P >= (static_cast<int64_t>(1) << 31)) return TQ_ERR_INVALID_ARG;
  if (!counts || !offsets || !tiles || !num_tiles) return TQ_ERR_INVALID_ARG;
  if (P > 0 && (!topk_ids || !sorted_pairs)) return TQ_ERR_INVALID_ARG;
  if (P > 0 && x_sorted && (!x || !aligned16(x) || !aligned16(x_sorted))) return TQ_ERR_INVALID_ARG;
  if (y32_count > 0 && !y32) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  int* err = error_word(&rc);
  if (!err) return rc;
  rc = launch_route_tile_map(topk_ids, static_cast<int>(P), E, tile_m, counts, offsets, sorted_pairs, tiles,
                             num_tiles, cap, err, s, y32, y32_count);
  if (rc != TQ_OK || !x_sorted || P == 0) return rc;
  return launch_gather(x, sorted_pairs, static_cast<int>(P), top_k, K, x_sorted, err, s);
}

int tq_grouped_gemm(const uint16_t* x, int x_layout, const uint8_t* packed, const uint16_t* lut, int L,
                    const int32_t* sorted_pairs, const float* topk_w, const int32_t* tiles,
                    const int32_t* num_tiles, int64_t cap, int64_t n, int top_k, int E, int K, int N,
                    int tile_m, float* y32, tq_stream_t stream) {
  int rc = check_gemm_common(x, packed, lut, L, topk_w, n, top_k, E, K, N, y32);
  if (rc != TQ_OK) return rc;
  if (x_layout != TQ_X_TOKENS && x_layout != TQ_X_PAIR_SORTED) return TQ_ERR_INVALID_ARG;
  if (N % 128 != 0 || tile_m < 1 || tile_m > 256 || cap < 1 || cap >= (static_cast<int64_t>(1) << 31))
    return TQ_ERR_INVALID_ARG;
  if (n > 0 && !aligned16(y32)) return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!sorted_pairs || !tiles || !num_tiles)) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  if (n == 0) return TQ_OK;
  int* err = error_word(&rc);
  if (!err) return rc;
  return launch_grouped(x, packed, lut, L, sorted_pairs, topk_w, tiles, num_tiles, cap, n, top_k, E, K, N, tile_m,
                        y32, err, s, 0, nullptr, false, false, x_layout == TQ_X_PAIR_SORTED);
}

int tq_gemv(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L, const int32_t* topk_ids,
            const float* topk_w, int64_t n, int top_k, int E, int K, int N, float* y32, tq_stream_t stream) {
  int rc = check_gemm_common(x, packed, lut, L, topk_w, n, top_k, E, K, N, y32);
  if (rc != TQ_OK) return rc;
  if (K > 8192) return TQ_ERR_INVALID_ARG;
  if (n > 0 && !topk_ids) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  if (n == 0) return TQ_OK;
  int* err = error_word(&rc);
  if (!err) return rc;
  return launch_gemv(x, packed, lut, L, topk_ids, topk_w, n, top_k, E, K, N, y32, err, s);
}

int tq_combine(const float* y32, uint16_t* y, int64_t count, tq_stream_t stream) {
  if (count < 0 || (count > 0 && (!y32 || !y))) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  return launch_combine(y32, y, count, s);
}

int tq_native_tile_m(int64_t n, int top_k, int E) {
  if (bad_shape(top_k, E) || n < 0) return TQ_ERR_INVALID_ARG;
  const double ppw = n > 0 ? tq_pairs_per_woken_expert(n, top_k, E) : 0.0;
  if (ppw >= 128.0) return 256;
  return ppw > 4.0 ? 128 : 16;
}

size_t tq_moe_workspace_size(int64_t n, int top_k, int E, int K, int N, int tile_m) {
  int kt, gt;
  if (!resolve_tile(n, top_k, E, tile_m, &kt, &gt)) return 0;
  const int64_t cap = tq_tile_map_capacity(n, top_k, E, kt);
  if (cap < 0 || N < 1 || K < 1) return 0;
  const size_t P = static_cast<size_t>(n) * top_k;
  size_t b = 0;
  b += align256(sizeof(int32_t) * E);                               // counts
  b += align256(sizeof(int32_t) * (E + 1));                         // offsets
  b += align256(sizeof(int32_t) * std::max<size_t>(P, 1));          // sorted pairs
  b += align256(sizeof(int32_t) * 3 * std::max<int64_t>(cap, 1));   // tiles
  b += align256(sizeof(int32_t));                                   // num_tiles
  b += align256(sizeof(float) * static_cast<size_t>(n) * N);        // y32
  if (!gathers_in_kernel(kt)) {
    b += align256(sizeof(uint16_t) * P * K);                        // pair-sorted activations
    b += align256(sizeof(int32_t) * std::max<size_t>(P, 1));        // pair -> sorted slot
  }
  return b;
}


int tq_moe_forward(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L, const int32_t* topk_ids,
                   const float* topk_w, int64_t n, int top_k, int E, int K, int N, int tile_m, int pin,
                   void* workspace, size_t workspace_bytes, uint16_t* y, int* arm_used, tq_stream_t stream) {
  int rc = check_gemm_common(x, packed, lut, L, topk_w, n, top_k, E, K, N, y);
  if (rc != TQ_OK) return rc;
  int gate_tile = 0;
  if (E > 1024 || !resolve_tile(n, top_k, E, tile_m, &tile_m, &gate_tile)) return TQ_ERR_INVALID_ARG;
  if (n > 0 && !topk_ids) return TQ_ERR_INVALID_ARG;
  const int arm = tq_select_arm(n, top_k, E, gate_tile, env_pin(pin));
  if (arm < 0) return arm;
  if (arm == TQ_ARM_GROUPED && N % 128 != 0) return TQ_ERR_INVALID_ARG;
  if (arm == TQ_ARM_GEMV && K > 8192) return TQ_ERR_INVALID_ARG;
  const size_t need = tq_moe_workspace_size(n, top_k, E, K, N, tile_m);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return TQ_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  if (arm_used) *arm_used = arm;
  if (n == 0) return TQ_OK;
  int* err = error_word(&rc);
  if (!err) return rc;

  const int64_t cap = tq_tile_map_capacity(n, top_k, E, tile_m);
  const size_t P = static_cast<size_t>(n) * top_k;
  const MoeScratch ws = carve_moe_scratch(workspace, n, top_k, E, K, N, cap, tile_m);
  int32_t* counts = ws.counts;
  int32_t* offsets = ws.offsets;
  int32_t* sorted_pairs = ws.sorted_pairs;
  int32_t* tiles = ws.tiles;
  int32_t* num_tiles = ws.num_tiles;
  float* y32 = ws.y32;

  if (arm == TQ_ARM_GROUPED) {
    // route + tile map in one launch (its other blocks clear y32); for large
    // m-tiles the pair-sorted copy of x; then the grouped kernel as a
    // programmatic dependent (its prologue overlaps the previous launch's tail)
    rc = launch_route_tile_map(topk_ids, static_cast<int>(P), E, tile_m, counts, offsets, sorted_pairs, tiles,
                               num_tiles, cap, err, s, y32, static_cast<int64_t>(n) * N, ws.slot_of);
    if (rc != TQ_OK) return rc;
    if (ws.x_sorted) {
      rc = launch_gather_tokens(x, ws.slot_of, n, top_k, K, ws.x_sorted, s);
      if (rc != TQ_OK) return rc;
    }
    rc = launch_grouped(ws.x_sorted ? ws.x_sorted : x, packed, lut, L, sorted_pairs, topk_w, tiles, num_tiles, cap,
                        n, top_k, E, K, N, tile_m, y32, err, s, 0, nullptr, true, false, ws.x_sorted != nullptr);
    if (rc != TQ_OK) return rc;
    std::call_once(g_log_once, [&] {
      const char* q = std::getenv("TQ_QUIET");
      if (q && !std::strcmp(q, "1")) return;
      const double ppw = tq_pairs_per_woken_expert(n, top_k, E);
      std::fprintf(stderr,
                   "tqmoe: trellis grouped GEMM engaged at %lld tokens x top-%d of %d experts - m-tiles %.0f%% "
                   "full (%.2f pairs per woken expert against TILE_M=%d); the amortization boundary for this "
                   "routing shape is %lld tokens; kernel m-tile %d\n",
                   static_cast<long long>(n), top_k, E, 100.0 * ppw / gate_tile, ppw, gate_tile,
                   static_cast<long long>(tq_grouped_min_tokens(top_k, E, gate_tile)), tile_m);
    });
    return launch_combine(y32, y, static_cast<int64_t>(n) * N, s);
  }
  // The GEMV arm in one launch: each warp sums a token's top_k pairs for its
  // output rows in registers and writes the bf16 product (y32 is not used).
  // Its predecessor on the stream is the caller's, which may have written
  // the inputs, so the kernel waits for it before staging anything.
  return launch_gemv(x, packed, lut, L, topk_ids, topk_w, n, top_k, E, K, N, nullptr, err, s, 0, 0, false, y);
}

int tq_device_error(int* code, int* where) {
  if (!code) return TQ_ERR_INVALID_ARG;
  int rc;
  int* err = error_word(&rc);
  if (!err) return rc;
  int h[2] = {0, 0};
  const int z[2] = {0, 0};
  if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(h, err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(err, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  *code = h[0];
  if (where) *where = h[1];
  return TQ_OK;
}

void tq_launch_counts(int64_t out[TQ_NUM_LAUNCH_COUNTERS]) {
  if (!out) return;
  for (int i = 0; i < kCntNum; ++i) out[i] = g_counts[i].load();
}

}  // extern "C"
