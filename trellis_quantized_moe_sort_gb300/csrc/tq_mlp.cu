// The whole routed-expert MLP of a SwiGLU expert on top of the grouped GEMM:
//   gate|up = W_gu,e x_t  (one grouped GEMM, outputs kept per pair),
//   h       = silu(gate) * up  (bf16, rows in sorted-pair order),
//   y_t     = sum_j w_tj W_down,e h_(t,j)  (grouped GEMM, combined per token).
// The per-pair activations of the down projection are already in the order
// the grouped kernel reads them, so no second gather is needed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

// h[s][i] = bf16(silu(g) * u), g = gate_up[s][i], u = gate_up[s][I + i],
// silu(g) = g / (1 + e^-g); four elements per thread step.
__global__ void swiglu_kernel(const float4* __restrict__ gate_up, long long P, int I4, uint2* __restrict__ h) {
  pdl_wait();
  pdl_trigger();
  const long long total = P * I4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long s = i / I4;
    const int c = static_cast<int>(i - s * I4);
    const float4 g = gate_up[s * 2 * I4 + c];
    const float4 u = gate_up[s * 2 * I4 + I4 + c];
    const float a = g.x / (1.f + expf(-g.x)) * u.x;
    const float b = g.y / (1.f + expf(-g.y)) * u.y;
    const float d = g.z / (1.f + expf(-g.z)) * u.z;
    const float e = g.w / (1.f + expf(-g.w)) * u.w;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(d, e);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&lo);
    o.y = *reinterpret_cast<const uint32_t*>(&hi);
    h[i] = o;
  }
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int launch_swiglu(const float* gate_up, int64_t P, int I, uint16_t* h, cudaStream_t s) {
  if (P == 0) return TQ_OK;
  const int I4 = I / 4;
  const long long total = static_cast<long long>(P) * I4;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<long long>((total + threads - 1) / threads, sm_count() * 8));
  int st = launch_pdl(swiglu_kernel, dim3(blocks), dim3(threads), 0, s, reinterpret_cast<const float4*>(gate_up), P,
                      I4, reinterpret_cast<uint2*>(h));
  if (st == TQ_OK) st = launch_status();
  if (st == TQ_OK) count_launch(kCntSwiglu);
  return st;
}

}  // namespace tq

using namespace tq;

extern "C" {

int tq_grouped_gemm_pairs(const uint16_t* x_sorted, const uint8_t* packed, const uint16_t* lut, int L,
                          const int32_t* sorted_pairs, const int32_t* tiles, const int32_t* num_tiles, int64_t cap,
                          int64_t n, int top_k, int E, int K, int N, int tile_m, float* out32,
                          tq_stream_t stream) {
  if (E < 1 || top_k < 1 || top_k > E || n < 0 || K < 64 || K % 64 != 0 || N % 128 != 0 || N < 128)
    return TQ_ERR_INVALID_ARG;
  if (L < 2 || L > 16 || (L & 1) || tile_m < 1 || tile_m > 256 || cap < 1 || cap >= (1ll << 31))
    return TQ_ERR_INVALID_ARG;
  if (n * top_k >= (1ll << 31) || static_cast<int64_t>(E) * N >= (1ll << 31)) return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!x_sorted || !packed || !lut || !sorted_pairs || !tiles || !num_tiles || !out32))
    return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!aligned16(x_sorted) || !aligned16(packed) || !aligned16(lut) || !aligned16(out32)))
    return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  if (n == 0) return TQ_OK;
  int* err = error_word(&rc);
  if (!err) return rc;
  return launch_grouped(x_sorted, packed, lut, L, sorted_pairs, nullptr, tiles, num_tiles, cap, n, top_k, E, K, N,
                        tile_m, out32, err, s, /*pair_out=*/1, nullptr, false, false, /*x_pair_sorted=*/true);
}

int tq_swiglu(const float* gate_up, int64_t P, int I, uint16_t* h, tq_stream_t stream) {
  if (P < 0 || I < 4 || I % 4 != 0 || (P > 0 && (!gate_up || !h || !aligned16(gate_up))) ||
      (P > 0 && (reinterpret_cast<uintptr_t>(h) & 7u)))
    return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  return launch_swiglu(gate_up, P, I, h, s);
}

size_t tq_moe_mlp_workspace_size(int64_t n, int top_k, int E, int H, int I, int tile_m) {
  int kt, gt;
  if (!resolve_tile(n, top_k, E, tile_m, &kt, &gt)) return 0;
  const int64_t cap = tq_tile_map_capacity(n, top_k, E, kt);
  if (cap < 0 || H < 1 || I < 1) return 0;
  const size_t P = static_cast<size_t>(n) * top_k;
  size_t b = 0;
  b += align256(sizeof(int32_t) * E);                              // counts
  b += align256(sizeof(int32_t) * (E + 1));                        // offsets
  b += align256(sizeof(int32_t) * std::max<size_t>(P, 1));         // sorted pairs
  b += align256(sizeof(int32_t) * 3 * std::max<int64_t>(cap, 1));  // tiles
  b += align256(sizeof(int32_t));                                  // num_tiles
  if (!gathers_in_kernel(kt)) {
    b += align256(sizeof(uint16_t) * P * H);                       // x, pair-sorted
    b += align256(sizeof(int32_t) * std::max<size_t>(P, 1));       // pair -> sorted slot
  }
  b += align256(sizeof(float) * P * 2 * I);                        // gate|up per pair
  b += align256(sizeof(uint16_t) * P * I);                         // h per pair
  b += align256(sizeof(float) * static_cast<size_t>(n) * H);       // y32
  return b;
}

int tq_moe_mlp_forward(const uint16_t* x, const uint8_t* packed_gu, const uint16_t* lut_gu,
                       const uint8_t* packed_down, const uint16_t* lut_down, int L, const int32_t* topk_ids,
                       const float* topk_w, int64_t n, int top_k, int E, int H, int I, int tile_m, int pin,
                       void* workspace, size_t workspace_bytes, uint16_t* y, int* arm_used, tq_stream_t stream) {
  const int tile_arg = tile_m;
  int gate_tile = 0;
  if (E < 1 || E > 1024 || top_k < 1 || top_k > E || n < 0) return TQ_ERR_INVALID_ARG;
  if (!resolve_tile(n, top_k, E, tile_arg, &tile_m, &gate_tile)) return TQ_ERR_INVALID_ARG;
  const int arm = tq_select_arm(n, top_k, E, gate_tile, env_pin(pin));
  if (arm < 0) return arm;
  if (H < 128 || H % 128 != 0 || I < 64 || I % 64 != 0 || (2 * I) % 128 != 0) return TQ_ERR_INVALID_ARG;
  if (L < 2 || L > 16 || (L & 1)) return TQ_ERR_INVALID_ARG;
  if (n * top_k >= (1ll << 31)) return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!x || !packed_gu || !lut_gu || !packed_down || !lut_down || !topk_ids || !topk_w || !y))
    return TQ_ERR_INVALID_ARG;
  if (n > 0 && (!aligned16(x) || !aligned16(packed_gu) || !aligned16(lut_gu) || !aligned16(packed_down) ||
                !aligned16(lut_down)))
    return TQ_ERR_INVALID_ARG;
  const size_t need = tq_moe_mlp_workspace_size(n, top_k, E, H, I, tile_arg);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return TQ_ERR_WORKSPACE;
  if (arm == TQ_ARM_GEMV && (H > 8192 || I > 8192)) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = require_sm103(s);
  if (rc != TQ_OK) return rc;
  if (arm_used) *arm_used = arm;
  if (n == 0) return TQ_OK;
  int* err = error_word(&rc);
  if (!err) return rc;

  const int64_t cap = tq_tile_map_capacity(n, top_k, E, tile_m);
  const size_t P = static_cast<size_t>(n) * top_k;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  int32_t* counts = reinterpret_cast<int32_t*>(w);      w += align256(sizeof(int32_t) * E);
  int32_t* offsets = reinterpret_cast<int32_t*>(w);     w += align256(sizeof(int32_t) * (E + 1));
  int32_t* sorted_pairs = reinterpret_cast<int32_t*>(w); w += align256(sizeof(int32_t) * P);
  int32_t* tiles = reinterpret_cast<int32_t*>(w);       w += align256(sizeof(int32_t) * 3 * cap);
  int32_t* num_tiles = reinterpret_cast<int32_t*>(w);   w += align256(sizeof(int32_t));
  uint16_t* x_sorted = nullptr;   // large m-tiles: the gate|up input in pair-sorted order
  int32_t* slot_of = nullptr;     // and the sort's inverse, to write it in token order
  if (!gathers_in_kernel(tile_m)) {
    x_sorted = reinterpret_cast<uint16_t*>(w);          w += align256(sizeof(uint16_t) * P * H);
    slot_of = reinterpret_cast<int32_t*>(w);            w += align256(sizeof(int32_t) * std::max<size_t>(P, 1));
  }
  float* gate_up = reinterpret_cast<float*>(w);         w += align256(sizeof(float) * P * 2 * I);
  uint16_t* h = reinterpret_cast<uint16_t*>(w);         w += align256(sizeof(uint16_t) * P * I);
  float* y32 = reinterpret_cast<float*>(w);

  if (arm == TQ_ARM_GEMV) {
    // per-pair GEMVs: gate|up per pair (plain stores), SwiGLU, down per pair
    // with the router weights into y32 (no routing sort, no tile map)
    rc = launch_clear(y32, static_cast<int64_t>(n) * H, s);
    if (rc == TQ_OK)
      rc = launch_gemv(x, packed_gu, lut_gu, L, topk_ids, nullptr, n, top_k, E, H, 2 * I, gate_up, err, s,
                       /*pair_in=*/0, /*pair_out=*/1, /*early_prologue=*/true);
    if (rc == TQ_OK) rc = launch_swiglu(gate_up, static_cast<int64_t>(P), I, h, s);
    if (rc == TQ_OK)
      rc = launch_gemv(h, packed_down, lut_down, L, topk_ids, topk_w, n, top_k, E, I, H, y32, err, s,
                       /*pair_in=*/1, /*pair_out=*/0);
    if (rc == TQ_OK) rc = launch_combine(y32, y, static_cast<int64_t>(n) * H, s);
    return rc;
  }
  // route + tile map (its other blocks clear y32), gate|up (token rows of x
  // gathered by the kernel, or copied into pair-sorted order first for large
  // m-tiles), SwiGLU, down reading h in sorted order, combine
  rc = launch_route_tile_map(topk_ids, static_cast<int>(P), E, tile_m, counts, offsets, sorted_pairs, tiles,
                             num_tiles, cap, err, s, y32, static_cast<int64_t>(n) * H, slot_of);
  if (rc == TQ_OK && x_sorted) rc = launch_gather_tokens(x, slot_of, n, top_k, H, x_sorted, s);
  if (rc == TQ_OK)
    rc = launch_grouped(x_sorted ? x_sorted : x, packed_gu, lut_gu, L, sorted_pairs, nullptr, tiles, num_tiles, cap,
                        n, top_k, E, H, 2 * I, tile_m, gate_up, err, s, /*pair_out=*/1, nullptr, true,
                        /*store_out=*/true,    // every gate|up element written once: no clear needed
                        x_sorted != nullptr);
  if (rc == TQ_OK) rc = launch_swiglu(gate_up, static_cast<int64_t>(P), I, h, s);
  if (rc == TQ_OK)
    rc = launch_grouped(h, packed_down, lut_down, L, sorted_pairs, topk_w, tiles, num_tiles, cap, n, top_k, E, I,
                        H, tile_m, y32, err, s, /*pair_out=*/0, nullptr, false, false, /*x_pair_sorted=*/true);
  if (rc == TQ_OK) rc = launch_combine(y32, y, static_cast<int64_t>(n) * H, s);
  return rc;
}

}  // extern "C"
