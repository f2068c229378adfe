// Measurement of the resource that bounds the trellis decode: random 16-bit
// lookups in a 2^16-entry table held in shared memory.  Every staged weight of
// the grouped GEMM and of the GEMV arm costs one such lookup; the rate this
// probe reaches is the ceiling the decode is reported against.
#include <cuda_runtime.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kProbeUnroll = 16;

// Each thread walks kProbeUnroll independent pseudo-random 16-bit indices (a
// 32-bit LCG per index) and loads table[index] from shared memory; the loads
// are summed so none is dead.
__global__ void lut_probe_kernel(const uint16_t* __restrict__ table, int iters, uint32_t* __restrict__ sink,
                                 unsigned long long* __restrict__ cycles) {
  extern __shared__ __align__(16) uint16_t lut[];
  for (int i = threadIdx.x; i < 65536 / 8; i += blockDim.x)
    reinterpret_cast<uint4*>(lut)[i] = __ldg(reinterpret_cast<const uint4*>(table) + i);
  __syncthreads();
  const uint32_t base = smem_u32(lut);
  uint32_t st[kProbeUnroll];
#pragma unroll
  for (int u = 0; u < kProbeUnroll; ++u)
    st[u] = (threadIdx.x * 2654435761u) ^ (blockIdx.x * 40503u) ^ (static_cast<uint32_t>(u) * 0x9E3779B9u);
  uint32_t acc = 0;
  __syncthreads();
  const unsigned long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    uint32_t v[kProbeUnroll];
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) {
      st[u] = st[u] * 1664525u + 1013904223u;
      const uint32_t addr = base + ((st[u] >> 15) & 0x1FFFEu);   // byte offset of entry (st >> 16)
      asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v[u]) : "r"(addr));
    }
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) acc += v[u];
  }
  const unsigned long long t1 = clock64();
  sink[static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x] = acc;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// One thread waits, through the bounded wait of the pipelined kernels, on a
// barrier that nothing arrives on: the wait gives up after timeout_ns, records
// TQ_ERR_DEVICE_TIMEOUT in the device error word, and the kernel returns.
// out[0] = 1 if the wait completed (it cannot), out[1] = microseconds waited.
__global__ void wait_timeout_probe_kernel(uint64_t timeout_ns, int* __restrict__ err, int* __restrict__ out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  abort_flag = 0;
  mbar_init(b, 1);
  mbar_fence_init();
  const uint64_t t0 = globaltimer();
  const bool done = mbar_wait(b, 0, &abort_flag, err, kWhereProbe, timeout_ns);
  const uint64_t us = (globaltimer() - t0) / 1000u;
  out[0] = done ? 1 : 0;
  out[1] = static_cast<int>(us < 0x7fffffffull ? us : 0x7fffffffull);
}

}  // namespace
}  // namespace tq

extern "C" int tq_probe_wait_timeout(int64_t timeout_ns, int* out, tq_stream_t stream) {
  if (!out || (reinterpret_cast<uintptr_t>(out) & 3u) != 0 || timeout_ns < 1000 ||
      timeout_ns > static_cast<int64_t>(tq::kWaitTimeoutNs))
    return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = tq::require_sm103(s);
  if (rc != TQ_OK) return rc;
  int* err = tq::error_word(&rc);
  if (rc != TQ_OK) return rc;
  tq::wait_timeout_probe_kernel<<<1, 1, 0, s>>>(static_cast<uint64_t>(timeout_ns), err, out);
  return tq::launch_status();
}

extern "C" int tq_probe_lut_rate(const uint16_t* table, int warps_per_sm, int iters, uint32_t* sink,
                                 unsigned long long* cycles, tq_stream_t stream) {
  if (!table || !sink || !cycles || warps_per_sm < 1 || warps_per_sm > 32 || iters < 1) return TQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(table) & 15u) != 0) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = tq::require_sm103(s);
  if (rc != TQ_OK) return rc;
  if (cudaFuncSetAttribute(tq::lut_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 131072) !=
      cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  tq::lut_probe_kernel<<<tq::sm_count(), warps_per_sm * 32, 131072, s>>>(table, iters, sink, cycles);
  return tq::launch_status();
}
