// Host-side internals shared by the library's translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "tqmoe.h"

namespace tq {

// Device address of the current device's error word (int[2]: code, where),
// or nullptr with *status set on failure.
int* error_word(int* status);

// Checks (and on first use takes) the arch witness for the current device.
// Refuses during capture of `stream` if the witness has not been cached yet.
int require_sm103(cudaStream_t stream);

// Converts the last launch error into a status and clears it.
int launch_status();

enum Counter {
  kCntRoute = 0, kCntTileMap, kCntGrouped, kCntGemv, kCntCombine, kCntGather, kCntRouter, kCntDequant,
  kCntRouteTileMap, kCntClear, kCntSwiglu, kCntNum
};
static_assert(kCntNum == TQ_NUM_LAUNCH_COUNTERS, "counter layout of tq_launch_counts");
void count_launch(Counter c);

// Number of SMs of the current device (cached per device).
int sm_count();

// Launches `kernel` with programmatic stream serialization: it may begin while
// the previous kernel on the stream finishes, so it must call pdl_wait()
// before touching anything that kernel writes.  Returns the launch status.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_LAUNCH;
  }
  return TQ_OK;
}

// Kernel launchers (defined in their own translation units).  Arguments are
// validated by the caller; these only configure and launch.
int launch_route(const int32_t* topk_ids, int P, int E, int32_t* counts, int32_t* offsets,
                 int32_t* sorted_pairs, int* err, cudaStream_t s);
int launch_tile_map(const int32_t* offsets, int E, int tile_m, int32_t* tiles, int32_t* num_tiles,
                    int64_t cap, int* err, cudaStream_t s);
int launch_combine(const float* y32, uint16_t* y, int64_t count, cudaStream_t s);
// y[0 .. count) = 0 (fp32), as a programmatic dependent of the previous kernel.
int launch_clear(float* y, int64_t count, cudaStream_t s);
int launch_router(const float* logits, int n, int E, int top_k, int32_t* ids, float* w, cudaStream_t s);
int launch_gather(const uint16_t* x, const int32_t* sorted_pairs, int P, int top_k, int K,
                  uint16_t* x_sorted, int* err, cudaStream_t s);
// Route and tile map in one launch, also clearing y32[0 .. y32_count) (in
// extra blocks of the same launch, or by a separate memset when y32 is not
// 16-byte aligned or y32_count % 4 != 0).
// With slot_of (device, [P]) the sort also writes its inverse: slot_of[p] =
// the sorted slot of pair p, -1 for a pair whose expert is out of range.
int launch_route_tile_map(const int32_t* topk_ids, int P, int E, int tile_m, int32_t* counts, int32_t* offsets,
                          int32_t* sorted_pairs, int32_t* tiles, int32_t* num_tiles, int64_t cap, int* err,
                          cudaStream_t s, float* y32 = nullptr, int64_t y32_count = 0,
                          int32_t* slot_of = nullptr);
// x_sorted[slot_of[t * top_k + j]] = x[t]: the pair-sorted copy written in
// token order (each row of x read once); slot -1 is skipped.
int launch_gather_tokens(const uint16_t* x, const int32_t* slot_of, int64_t n, int top_k, int K, uint16_t* x_sorted,
                         cudaStream_t s);
// x: token rows [n][K], gathered by sorted pair inside the kernel; or, with
// x_pair_sorted, the pair-sorted rows [n*top_k][K] (row = sorted slot).
int launch_grouped(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L,
                   const int32_t* sorted_pairs, const float* topk_w, const int32_t* tiles,
                   const int32_t* num_tiles, int64_t cap, int64_t n, int top_k, int E, int K, int N,
                   int tile_m, float* y32, int* err, cudaStream_t s, int pair_out = 0,
                   const uint16_t* dense_w = nullptr, bool pdl = false, bool store_out = false,
                   bool x_pair_sorted = false);
// Materializes weights: out[i] = bf16(W_{e_i}) [N][K] for slot i < m, e_i =
// expert_ids[i] (or i when expert_ids is null); a slot whose expert has
// counts[e_i] == 0 (when counts is given) or e_i < 0 is skipped.
int launch_dequant(const uint8_t* packed, const uint16_t* lut, int L, const int32_t* expert_ids,
                   const int32_t* counts, int m, int E, int N, int K, uint16_t* out, int* err, cudaStream_t s);

// True when the whole-product calls let the grouped kernel gather the token
// rows itself (kernel m-tile <= TQ_GATHER_MAX_TILE_M); above it they copy the
// rows into pair-sorted order first (tq_gather_rows), which is faster there.
inline bool gathers_in_kernel(int kernel_tile_m) { return kernel_tile_m <= TQ_GATHER_MAX_TILE_M; }

// The scratch regions of tq_moe_forward inside a caller workspace (layout of
// tq_moe_workspace_size: counts, offsets, sorted pairs, tiles, num_tiles, y32,
// then x_sorted [P][K] only when the kernel m-tile does not gather in the
// kernel, each 256-byte aligned); `end` is the first byte after them.
struct MoeScratch {
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_pairs;
  int32_t* tiles;
  int32_t* num_tiles;
  float* y32;
  uint16_t* x_sorted;   // nullptr when the kernel gathers
  int32_t* slot_of;     // pair -> sorted slot, with x_sorted
  uint8_t* end;
};
MoeScratch carve_moe_scratch(void* workspace, int64_t n, int top_k, int E, int K, int N, int64_t cap,
                             int kernel_tile_m);

// tile_m of the whole-product calls: 1..256 for both the arm selection and the
// kernel, or TQ_TILE_NATIVE (the kernel's native tile or TQ_TILE_M from the
// environment, the pages' TILE_M for the selection).  Returns false on an
// invalid value.
bool resolve_tile(int64_t n, int top_k, int E, int tile_m, int* kernel_tile, int* gate_tile);
int launch_swiglu(const float* gate_up, int64_t P, int I, uint16_t* h, cudaStream_t s);
// pair_in: x holds one row per pair (x[pair]) instead of per token;
// pair_out: out[pair][row] = the row's dot product (plain store, no router
// weight) instead of y32[token][row] += w * dot; y_tok (x per token, neither
// pair_in nor pair_out): y_tok[token][row] = bf16(sum_j w_j dot_j) written
// once per element, y32 unused.  Launched as a programmatic dependent of the
// previous kernel; early_prologue: that kernel writes none of x, topk_ids,
// the LUT or packed, so the kernel stages them (and loads its first row)
// before waiting for it.
int launch_gemv(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L,
                const int32_t* topk_ids, const float* topk_w, int64_t n, int top_k, int E, int K,
                int N, float* y32, int* err, cudaStream_t s, int pair_in = 0, int pair_out = 0,
                bool early_prologue = false, uint16_t* y_tok = nullptr);
// TQ_FORCE_ARM (auto|gemv|grouped|measured) applied to an automatic pin.
int env_pin(int pin);

}  // namespace tq
