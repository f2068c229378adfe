// tq_moe_forward_static: the whole routed-expert product without a caller
// workspace and without allocating anything.
//
// Who needs it: callers that cannot allocate device memory — for example a
// plugin to which a host framework passes only its input and output buffers
// (that framework owns every allocation), or a serving loop that forbids
// allocation after start-up because cudaMalloc can block and synchronize the
// device.  They still pass inputs and outputs; the scratch this call needs
// (counts, offsets, sorted pairs, tile map, fp32 accumulator, and for large
// m-tiles the pair-sorted activations) lives in one file-scope device array
// of fixed size, which
// every GPU that loads this library holds until the process exits.
#include <cuda_runtime.h>

#include <atomic>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kMaxDevicesStatic = 64;

// The shared scratch.  In host code this name is a host-side stand-in, not a
// device address: only the pointer returned by cudaGetSymbolAddress may be
// passed to a kernel.
static __device__ __align__(256) unsigned char g_static_scratch[TQ_STATIC_SCRATCH_BYTES];

std::atomic<void*> g_static_ptr[kMaxDevicesStatic];

// Device address of the scratch on the current device; looked up once per
// device (with that device current) and cached.
int static_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevicesStatic) return TQ_ERR_CUDA;
  void* p = g_static_ptr[dev].load();
  if (!p) {
    const cudaError_t rc = cudaGetSymbolAddress(&p, g_static_scratch);
    if (rc != cudaSuccess || !p) {
      cudaGetLastError();
      return TQ_ERR_CUDA;
    }
    g_static_ptr[dev].store(p);
  }
  *out = p;
  return TQ_OK;
}

}  // namespace
}  // namespace tq

extern "C" int tq_moe_forward_static(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L,
                                     const int32_t* topk_ids, const float* topk_w, int64_t n, int top_k, int E,
                                     int K, int N, int tile_m, int pin, uint16_t* y, int* arm_used,
                                     tq_stream_t stream) {
  if (n < 0 || N < 1) return TQ_ERR_INVALID_ARG;
  const size_t need = tq_moe_workspace_size(n, top_k, E, K, N, tile_m);
  if (need == 0) return TQ_ERR_INVALID_ARG;
  if (need > static_cast<size_t>(TQ_STATIC_SCRATCH_BYTES)) return TQ_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = tq::static_scratch(&scratch);
  if (rc != TQ_OK) return rc;
  // The regular entry point zeroes the fp32 accumulator on the stream and
  // overwrites every other scratch region before reading it.
  return tq_moe_forward(x, packed, lut, L, topk_ids, topk_w, n, top_k, E, K, N, tile_m, pin, scratch,
                        static_cast<size_t>(TQ_STATIC_SCRATCH_BYTES), y, arm_used, stream);
}
