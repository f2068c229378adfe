// The dequantize-materialize comparator: the path the fused kernel replaces.
//
// The first page ("fix(qtip): gate the trellis grouped GEMM on m-tile
// occupancy, not token count", section "Tests") names a dequantize-materialize
// path that dispatch falls through to outside the fused arms' token ranges:
// expert weights are decoded to a dense matrix in device memory and an
// ordinary GEMM multiplies them.  The second page ("perf(qtip): arch-specialise
// the trellis grouped GEMM", "The two changes") states what the fused design
// avoids: full-size decoded weights never exist.  This file builds that
// avoided path so the two can be measured against each other on the same
// inputs:
//
//   dequant_kernel  packed bitstreams -> bf16 W_e [N][K] for every woken expert
//                   (the same window-identity decode and fp16 -> bf16 rounding
//                   as the fused kernels)
//   grouped kernel in dense mode (tq_grouped.cu): the same m-tiles, pipeline
//                   and epilogue, with A read by TMA from the dense matrix.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kDqThreads = 1024;
constexpr int kDqChunk = 16;   // passes whose stream words are loaded before any is decoded

// One warp per weight row.  Lane l of pass i takes the row's 16-bit stream
// word wi = 32i + l (symbols 8wi .. 8wi + 7) and the word before it (from lane
// l - 1, or lane 31 of the previous pass; zero before the row start), so every
// state of its 8 symbols is one shift and mask of a 32-bit window (bits
// [16wi - 16, 16wi + 16) of the stream).  The 8 bf16 values leave as one
// 16-byte store: a warp writes 512 contiguous bytes per pass.  The words of
// kDqChunk passes are loaded first (that many loads in flight per lane), so
// the HBM latency is paid once per chunk, not once per pass.
template <int L>
__global__ void __launch_bounds__(kDqThreads)
dequant_kernel(const uint8_t* __restrict__ packed, const uint16_t* __restrict__ lut,
               const int32_t* __restrict__ expert_ids, const int32_t* __restrict__ counts, int m, int E, int N,
               int K, uint16_t* __restrict__ out, int* __restrict__ err) {
  extern __shared__ __align__(16) uint16_t lut_s[];
  constexpr int kEntries = 1 << L;
  constexpr uint32_t kMask = (1u << L) - 1u;
  if constexpr (kEntries >= 8) {
    // fp16 table in by asynchronous copies, then converted in place
    stage_to_smem(smem_u32(lut_s), lut, kEntries * 2);
    __syncthreads();
    for (int i = threadIdx.x; i < kEntries / 2; i += blockDim.x) {
      uint32_t* w = reinterpret_cast<uint32_t*>(lut_s) + i;
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(w));
      const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
      *w = *reinterpret_cast<const uint32_t*>(&b);
    }
  } else {
    for (int i = threadIdx.x; i < kEntries; i += blockDim.x) {
      const __nv_bfloat16 b = __float2bfloat16_rn(__half2float(__ushort_as_half(__ldg(lut + i))));
      lut_s[i] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  const long long rows = static_cast<long long>(m) * N;
  const int words = K / 8;
  for (long long gr = static_cast<long long>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5); gr < rows;
       gr += static_cast<long long>(gridDim.x) * warps_per_block) {
    const int slot = static_cast<int>(gr / N);
    const int r = static_cast<int>(gr - static_cast<long long>(slot) * N);
    const int e = expert_ids ? __ldg(expert_ids + slot) : slot;
    if (e < 0) continue;
    if (e >= E) {
      if (lane == 0) record_error(err, TQ_ERR_INVALID_ARG, kWhereDequant);
      continue;
    }
    if (counts && __ldg(counts + e) == 0) continue;
    const uint16_t* src =
        reinterpret_cast<const uint16_t*>(packed + (static_cast<size_t>(e) * N + r) * static_cast<size_t>(K / 4));
    uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(slot) * N + r) * static_cast<size_t>(K));
    uint32_t carry = 0;
    for (int c0 = 0; c0 < words; c0 += 32 * kDqChunk) {
      uint32_t cw[kDqChunk];
#pragma unroll
      for (int j = 0; j < kDqChunk; ++j) {
        const int wi = c0 + 32 * j + lane;
        cw[j] = wi < words ? static_cast<uint32_t>(__ldg(src + wi)) : 0u;
      }
#pragma unroll
      for (int j = 0; j < kDqChunk; ++j) {
        const int wi = c0 + 32 * j + lane;
        if (c0 + 32 * j >= words) break;   // uniform across the warp
        const uint32_t cur = cw[j];
        uint32_t prev = __shfl_up_sync(0xffffffffu, cur, 1);
        if (lane == 0) prev = carry;
        carry = __shfl_sync(0xffffffffu, cur, 31);
        if (wi < words) {
          const uint32_t win = prev | (cur << 16);
          uint32_t v[4];
#pragma unroll
          for (int t = 0; t < 8; t += 2) {
            // symbol 8wi + t: bits [2t + 18 - L, 2t + 18) of the window
            const uint32_t s0 = (win >> (2 * t + 18 - L)) & kMask;
            const uint32_t s1 = (win >> (2 * t + 20 - L)) & kMask;
            v[t / 2] = static_cast<uint32_t>(lut_s[s0]) | (static_cast<uint32_t>(lut_s[s1]) << 16);
          }
          dst[wi] = make_uint4(v[0], v[1], v[2], v[3]);
        }
      }
    }
  }
}

template <int L>
int launch_dequant_l(const uint8_t* packed, const uint16_t* lut, const int32_t* expert_ids, const int32_t* counts,
                     int m, int E, int N, int K, uint16_t* out, int* err, cudaStream_t s) {
  const int smem = std::max(16, 2 << L);
  auto kfn = dequant_kernel<L>;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, kDqThreads, smem) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  const long long rows = static_cast<long long>(m) * N;   // one warp per row
  const int grid = static_cast<int>(
      std::max<long long>(1, std::min<long long>(static_cast<long long>(per_sm) * sm_count(),
                                                 (rows + kDqThreads / 32 - 1) / (kDqThreads / 32))));
  kfn<<<grid, kDqThreads, smem, s>>>(packed, lut, expert_ids, counts, m, E, N, K, out, err);
  const int st = launch_status();
  if (st == TQ_OK) count_launch(kCntDequant);
  return st;
}

}  // namespace

int launch_dequant(const uint8_t* packed, const uint16_t* lut, int L, const int32_t* expert_ids,
                   const int32_t* counts, int m, int E, int N, int K, uint16_t* out, int* err, cudaStream_t s) {
  switch (L) {
    case 2: return launch_dequant_l<2>(packed, lut, expert_ids, counts, m, E, N, K, out, err, s);
    case 4: return launch_dequant_l<4>(packed, lut, expert_ids, counts, m, E, N, K, out, err, s);
    case 6: return launch_dequant_l<6>(packed, lut, expert_ids, counts, m, E, N, K, out, err, s);
    case 8: return launch_dequant_l<8>(packed, lut, expert_ids, counts, m, E, N, K, out, err, s);
    case 10: return launch_dequant_l<10>(packed, lut, expert_ids, counts, m, E, N, K, out, err, s);
    case 12: return launch_dequant_l<12>(packed, lut, expert_ids, counts, m, E, N, K, out, err, s);
    case 14: return launch_dequant_l<14>(packed, lut, expert_ids, counts, m, E, N, K, out, err, s);
    case 16: return launch_dequant_l<16>(packed, lut, expert_ids, counts, m, E, N, K, out, err, s);
    default: return TQ_ERR_INVALID_ARG;
  }
}

}  // namespace tq

using namespace tq;

namespace {
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t al256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
}  // namespace

extern "C" {

int tq_dequantize(const uint8_t* packed, const uint16_t* lut, int L, const int32_t* expert_ids, int m, int E,
                  int N, int K, uint16_t* w_out, tq_stream_t stream) {
  if (m < 0 || E < 1 || N < 1 || K < 8 || K % 8 != 0 || L < 2 || L > 16 || (L & 1)) return TQ_ERR_INVALID_ARG;
  if (!expert_ids && m > E) return TQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(m) * N >= (static_cast<int64_t>(1) << 40)) return TQ_ERR_INVALID_ARG;
  if (m > 0 && (!packed || !lut || !w_out || !al16(packed) || !al16(lut) || !al16(w_out)))
    return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  if (m == 0) return TQ_OK;
  int* err = error_word(&rc);
  if (!err) return rc;
  return launch_dequant(packed, lut, L, expert_ids, nullptr, m, E, N, K, w_out, err, s);
}

int tq_grouped_gemm_dense(const uint16_t* x, int x_layout, const uint16_t* w_dense, const int32_t* sorted_pairs,
                          const float* topk_w, const int32_t* tiles, const int32_t* num_tiles, int64_t cap,
                          int64_t n, int top_k, int E, int K, int N, int tile_m, float* y32, tq_stream_t stream) {
  if (E < 1 || top_k < 1 || top_k > E || n < 0 || K < 64 || K % 64 != 0 || N < 128 || N % 128 != 0)
    return TQ_ERR_INVALID_ARG;
  if (tile_m < 1 || tile_m > 256 || cap < 1 || cap >= (static_cast<int64_t>(1) << 31)) return TQ_ERR_INVALID_ARG;
  if (n * top_k >= (static_cast<int64_t>(1) << 31) || static_cast<int64_t>(E) * N >= (static_cast<int64_t>(1) << 31))
    return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!x || !w_dense || !sorted_pairs || !topk_w || !tiles || !num_tiles || !y32))
    return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!al16(x) || !al16(w_dense) || !al16(y32))) return TQ_ERR_INVALID_ARG;
  if (x_layout != TQ_X_TOKENS && x_layout != TQ_X_PAIR_SORTED) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  if (n == 0) return TQ_OK;
  int* err = error_word(&rc);
  if (!err) return rc;
  return launch_grouped(x, nullptr, nullptr, 2, sorted_pairs, topk_w, tiles, num_tiles, cap, n, top_k, E, K, N,
                        tile_m, y32, err, s, 0, w_dense, false, false, x_layout == TQ_X_PAIR_SORTED);
}

size_t tq_moe_dequant_workspace_size(int64_t n, int top_k, int E, int K, int N, int tile_m) {
  const size_t base = tq_moe_workspace_size(n, top_k, E, K, N, tile_m);   // resolves TQ_TILE_NATIVE
  if (base == 0) return 0;
  return base + al256(sizeof(uint16_t) * static_cast<size_t>(E) * N * K);
}

int tq_moe_forward_dequant(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L,
                           const int32_t* topk_ids, const float* topk_w, int64_t n, int top_k, int E, int K, int N,
                           int tile_m, void* workspace, size_t workspace_bytes, uint16_t* y, tq_stream_t stream) {
  if (E < 1 || top_k < 1 || top_k > E || E > 1024 || n < 0 || K < 64 || K % 64 != 0 || N < 128 || N % 128 != 0)
    return TQ_ERR_INVALID_ARG;
  const int tile_arg = tile_m;
  int gate_tile = 0;
  if (L < 2 || L > 16 || (L & 1) || !resolve_tile(n, top_k, E, tile_arg, &tile_m, &gate_tile))
    return TQ_ERR_INVALID_ARG;
  (void)gate_tile;   // the comparator has no arm selection
  if (n * top_k >= (static_cast<int64_t>(1) << 31) || static_cast<int64_t>(E) * N >= (static_cast<int64_t>(1) << 31))
    return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!x || !packed || !lut || !topk_ids || !topk_w || !y)) return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!al16(x) || !al16(packed) || !al16(lut))) return TQ_ERR_INVALID_ARG;
  const size_t need = tq_moe_dequant_workspace_size(n, top_k, E, K, N, tile_arg);
  if (need == 0) return TQ_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return TQ_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  if (n == 0) return TQ_OK;
  int* err = error_word(&rc);
  if (!err) return rc;

  const int64_t cap = tq_tile_map_capacity(n, top_k, E, tile_m);
  const int P = static_cast<int>(n * top_k);
  const MoeScratch ws = carve_moe_scratch(workspace, n, top_k, E, K, N, cap, tile_m);
  uint16_t* w_dense = reinterpret_cast<uint16_t*>(ws.end);   // [E][N][K]; slot e = expert e
  if ((rc = launch_route_tile_map(topk_ids, P, E, tile_m, ws.counts, ws.offsets, ws.sorted_pairs, ws.tiles,
                                  ws.num_tiles, cap, err, s, ws.y32, static_cast<int64_t>(n) * N, ws.slot_of)) !=
      TQ_OK)
    return rc;
  if (ws.x_sorted && (rc = launch_gather_tokens(x, ws.slot_of, n, top_k, K, ws.x_sorted, s)) != TQ_OK) return rc;
  // Materialize every woken expert (experts no pair routes to are skipped).
  if ((rc = launch_dequant(packed, lut, L, nullptr, ws.counts, E, E, N, K, w_dense, err, s)) != TQ_OK) return rc;
  if ((rc = launch_grouped(ws.x_sorted ? ws.x_sorted : x, nullptr, nullptr, 2, ws.sorted_pairs, topk_w, ws.tiles,
                           ws.num_tiles, cap, n, top_k, E, K, N, tile_m, ws.y32, err, s, 0, w_dense, false, false,
                           ws.x_sorted != nullptr)) != TQ_OK)
    return rc;
  return launch_combine(ws.y32, y, static_cast<int64_t>(n) * N, s);
}

}  // extern "C"
