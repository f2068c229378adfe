// Routing sort, m-tile map and the bf16 combine.
//
// Routing: the grouped GEMM works on pairs sorted by expert and visits
// sum_e ceil(count_e / TILE_M) m-tiles (page "fix(qtip): gate the trellis
// grouped GEMM on m-tile occupancy, not token count", section "The cause is a
// threshold, not a kernel defect").  The sort here is a stable counting sort
// done by one thread block: each warp owns a contiguous slice of the pair
// list, so ranking lanes with equal experts (match.any) inside a warp and
// offsetting by the counts of lower warps keeps ascending pair order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kBlock = 1024;
constexpr int kWarps = kBlock / 32;

// Exclusive scan of one int per thread over the whole 1024-thread block.
// Returns the exclusive prefix; *total receives the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total) {
  __shared__ int warp_sums[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += t;
    }
    warp_sums[lane] = si - s;  // exclusive prefix of warp sums
    __syncwarp();
  }
  __syncthreads();
  const int excl = warp_sums[warp] + incl - v;
  // block total: last thread's inclusive value
  __shared__ int blk_total;
  if (threadIdx.x == kBlock - 1) blk_total = excl + v;
  __syncthreads();
  *total = blk_total;
  __syncthreads();
  return excl;
}

// The routing sort, by `sorters` blocks (block b of them handles the
// contiguous pairs [P*b/sorters, P*(b+1)/sorters)); thread e < E of every
// sorting block returns expert e's first sorted slot in *first and its pair
// count in *count.  Each block counts its own chunk per warp (match.any
// leaders), and with more than one block also counts every pair by shared
// atomics: the totals per expert (every block derives the same offsets) and
// the pairs before its chunk (its base inside each expert's range).  Ranks
// follow (chunk, warp, lane) order, i.e. ascending pair ids: a stable sort.
__device__ __forceinline__ void route_chunk(const int32_t* __restrict__ ids, int P, int E, int sorters,
                                            int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                            int32_t* __restrict__ sorted_pairs, int* err, int* first,
                                            int* count, int32_t* __restrict__ slot_of = nullptr) {
  // [kWarps][E] per-warp count, then per-warp base; [E] totals; [E] pairs before the chunk
  extern __shared__ int32_t wcnt[];
  int32_t* tot = wcnt + kWarps * E;
  int32_t* pre = tot + E;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (kWarps + 2) * E; i += kBlock) wcnt[i] = 0;
  __syncthreads();

  const int b = blockIdx.x;
  const int c0 = static_cast<int>(static_cast<long long>(P) * b / sorters);
  const int c1 = static_cast<int>(static_cast<long long>(P) * (b + 1) / sorters);
  const int per_warp = ((((c1 - c0) + kWarps - 1) / kWarps) + 31) & ~31;
  const int beg = min(c1, c0 + warp * per_warp);
  const int end = min(c1, beg + per_warp);
  int32_t* mine = wcnt + warp * E;

  // Expert ids, kBatch rows of 32 at a time: all of a batch's loads are in
  // flight before the first is used.
  constexpr int kBatch = 8;
  // (positions are 64-bit: a batch may run past 2^31 - 1 at the end of the list)
  auto load_batch = [&](long long base, int lim, int (&eb)[kBatch]) {
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const long long p = base + 32 * i + lane;
      eb[i] = p < lim ? ids[p] : -1;
    }
  };

  // 0. (several blocks) totals and the prefix over all pairs
  if (sorters > 1) {
    for (long long base = warp * 32; base < P; base += kBlock * kBatch) {
      int eb[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const long long p = base + kBlock * i + lane;
        eb[i] = p < P ? ids[p] : -1;
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const long long p = base + kBlock * i + lane;
        const int e = eb[i];
        if (e >= 0 && e < E) {
          atomicAdd(&tot[e], 1);
          if (p < c0) atomicAdd(&pre[e], 1);
        }
      }
    }
  }

  // 1. per-warp histogram of its slice of the chunk
  for (long long base = beg; base < end; base += 32 * kBatch) {
    int eb[kBatch];
    load_batch(base, end, eb);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      int e = eb[i];
      if (base + 32 * i + lane < end && (e < 0 || e >= E)) {   // past the slice: loaded as -1
        record_error(err, TQ_ERR_INVALID_ARG, kWhereRoute);
        e = -1;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();

  // 2. per expert: exclusive counts over this block's warps, the totals and
  // their exclusive scan over experts, per-warp bases
  const int e = threadIdx.x;
  int own = 0;
  if (e < E) {
    for (int w = 0; w < kWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = own;
      own += c;
    }
  }
  const int total = sorters > 1 ? (e < E ? tot[e] : 0) : own;
  const int before = sorters > 1 && e < E ? pre[e] : 0;
  int all = 0;
  const int excl = block_exclusive_scan(total, &all);
  if (e < E) {
    if (b == 0) {
      counts[e] = total;
      offsets[e] = excl;
    }
    for (int w = 0; w < kWarps; ++w) wcnt[w * E + e] += excl + before;
  }
  if (b == 0 && threadIdx.x == 0) offsets[E] = all;
  *first = excl;
  *count = e < E ? total : 0;
  __syncthreads();

  // 3. stable scatter: rank among equal experts of lower lanes, then advance
  const unsigned lower = (1u << lane) - 1u;
  for (long long base = beg; base < end; base += 32 * kBatch) {
    int eb[kBatch];
    load_batch(base, end, eb);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const long long p = base + 32 * i + lane;
      const int ex = (eb[i] < 0 || eb[i] >= E) ? -1 : eb[i];
      const unsigned peers = __match_any_sync(0xffffffffu, ex);
      int slot = 0;
      if (ex >= 0) slot = mine[ex] + __popc(peers & lower);
      __syncwarp();
      if (ex >= 0) {
        sorted_pairs[slot] = static_cast<int32_t>(p);   // p < end <= P < 2^31
        if (lane == __ffs(peers) - 1) mine[ex] += __popc(peers);
      }
      // the inverse (pair -> sorted slot; -1 for a pair whose expert is out of range)
      if (slot_of && p < end) slot_of[p] = ex >= 0 ? slot : -1;
      __syncwarp();
    }
  }
}

__global__ void __launch_bounds__(kBlock, 1)
route_kernel(const int32_t* __restrict__ ids, int P, int E, int sorters, int32_t* __restrict__ counts,
             int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_pairs, int* err) {
  pdl_wait();
  pdl_trigger();
  int first, count;
  route_chunk(ids, P, E, sorters, counts, offsets, sorted_pairs, err, &first, &count);
}

// The m-tile map of one block from expert e's (first slot, count) in thread e.
__device__ __forceinline__ void tile_map_block(int E, int off, int cnt, int tile_m, int32_t* __restrict__ tiles,
                                               int32_t* __restrict__ num_tiles, long long cap, int* err) {
  const int e = threadIdx.x;
  const int nt = e < E ? (cnt + tile_m - 1) / tile_m : 0;
  int total = 0;
  const int start = block_exclusive_scan(nt, &total);
  for (int i = 0; i < nt; ++i) {
    const long long idx = static_cast<long long>(start) + i;
    if (idx >= cap) break;
    int32_t* t = tiles + 3 * idx;
    t[0] = e;
    t[1] = off + i * tile_m;
    t[2] = min(tile_m, cnt - i * tile_m);
  }
  if (threadIdx.x == 0) {
    if (total > cap) {
      record_error(err, TQ_ERR_CAPACITY, kWhereTileMap);
      *num_tiles = static_cast<int32_t>(cap);
    } else {
      *num_tiles = total;
    }
  }
}

__global__ void __launch_bounds__(kBlock, 1)
tile_map_kernel(const int32_t* __restrict__ offsets, int E, int tile_m, int32_t* __restrict__ tiles,
                int32_t* __restrict__ num_tiles, long long cap, int* err) {
  pdl_wait();
  pdl_trigger();
  const int e = threadIdx.x;
  int off = 0, cnt = 0;
  if (e < E) {
    off = offsets[e];
    cnt = offsets[e + 1] - off;
  }
  tile_map_block(E, off, cnt, tile_m, tiles, num_tiles, cap, err);
}

// Route and tile map in one launch: the first `sorters` blocks sort, block 0
// then builds the tile map from each expert's slot range held in registers;
// the blocks after them clear zero4[0 .. zero_n4) (the fp32 accumulator of
// the grouped GEMM that follows) meanwhile.
__global__ void __launch_bounds__(kBlock, 1)
route_tile_map_kernel(const int32_t* __restrict__ ids, int P, int E, int sorters, int tile_m,
                      int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                      int32_t* __restrict__ sorted_pairs, int32_t* __restrict__ tiles,
                      int32_t* __restrict__ num_tiles, long long cap, int* err, float4* __restrict__ zero4,
                      long long zero_n4, int32_t* __restrict__ slot_of) {
  pdl_wait();
  pdl_trigger();
  if (static_cast<int>(blockIdx.x) >= sorters) {
    const long long stride = static_cast<long long>(gridDim.x - sorters) * kBlock;
    for (long long i = static_cast<long long>(blockIdx.x - sorters) * kBlock + threadIdx.x; i < zero_n4;
         i += stride)
      zero4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  int first, count;
  route_chunk(ids, P, E, sorters, counts, offsets, sorted_pairs, err, &first, &count, slot_of);
  if (blockIdx.x == 0) tile_map_block(E, first, count, tile_m, tiles, num_tiles, cap, err);
}

// y[0 .. n) = 0: float4 stores over the 16-byte aligned middle, scalar
// stores over the ragged head and tail.
__global__ void clear_kernel(float* __restrict__ y, long long n) {
  pdl_wait();
  pdl_trigger();
  const long long head = min(n, static_cast<long long>(((16 - (reinterpret_cast<uintptr_t>(y) & 15)) & 15) / 4));
  const long long n4 = (n - head) / 4;
  float4* y4 = reinterpret_cast<float4*>(y + head);
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = tid; i < n4; i += stride) y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = tid; i < head; i += stride) y[i] = 0.f;
  for (long long i = head + 4 * n4 + tid; i < n; i += stride) y[i] = 0.f;
}

__global__ void combine_kernel_v4(const float4* __restrict__ y32, uint2* __restrict__ y, long long n4) {
  pdl_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = y32[i];
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&a);
    o.y = *reinterpret_cast<const uint32_t*>(&b);
    y[i] = o;
  }
}

__global__ void combine_kernel_scalar(const float* __restrict__ y32, uint16_t* __restrict__ y,
                                      long long n) {
  pdl_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const __nv_bfloat16 b = __float2bfloat16_rn(y32[i]);
    y[i] = *reinterpret_cast<const uint16_t*>(&b);
  }
}

// x_sorted[slot] = x[sorted_pairs[slot] / top_k]: the activations in pair-sorted
// order.  One warp per slot; each lane has eight 16-byte loads in flight
// before it stores them (row_vecs = K / 8 vectors per row), and the stores
// are marked streaming so that the copy, read once later, does not push x
// (read top_k times) out of L2.  An out-of-range pair id yields a zero row
// and is reported.
__global__ void gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ sorted_pairs,
                                   int P, int top_k, int row_vecs, uint4* __restrict__ x_sorted, int* err) {
  pdl_wait();
  pdl_trigger();
  constexpr int kUnroll = 8;
  const int lane = threadIdx.x & 31;
  const long long warp = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long slot = warp; slot < P; slot += nwarps) {
    const int pair = sorted_pairs[slot];
    const bool ok = pair >= 0 && pair < P;
    if (!ok && lane == 0) record_error(err, TQ_ERR_INVALID_ARG, kWhereRoute);
    const uint4* src = x + static_cast<size_t>(ok ? pair / top_k : 0) * row_vecs;
    uint4* dst = x_sorted + static_cast<size_t>(slot) * row_vecs;
    for (int v0 = 0; v0 < row_vecs; v0 += 32 * kUnroll) {
      uint4 t[kUnroll];
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) {
        const int v = v0 + 32 * j + lane;
        t[j] = (ok && v < row_vecs) ? __ldg(src + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) {
        const int v = v0 + 32 * j + lane;
        if (v < row_vecs) __stcs(dst + v, t[j]);
      }
    }
  }
}

// The same copy in token order: x_sorted[slot_of[t * top_k + j]] = x[t] for
// every j.  One warp per token reads the row once (eight 16-byte loads per
// lane in flight) and stores it into the sorted slots of the token's pairs;
// slot -1 (a pair whose expert is out of range, reported by the route) is
// skipped.  Read in sorted order instead, a row is fetched top_k times, far
// apart, and the streaming writes push it out of L2 in between.
__global__ void gather_tokens_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ slot_of, int n,
                                     int top_k, int row_vecs, uint4* __restrict__ x_sorted) {
  pdl_wait();
  pdl_trigger();
  constexpr int kUnroll = 8;
  const int lane = threadIdx.x & 31;
  const long long warp = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long t = warp; t < n; t += nwarps) {
    const uint4* src = x + static_cast<size_t>(t) * row_vecs;
    for (int v0 = 0; v0 < row_vecs; v0 += 32 * kUnroll) {
      uint4 q[kUnroll];
#pragma unroll
      for (int i = 0; i < kUnroll; ++i) {
        const int v = v0 + 32 * i + lane;
        q[i] = v < row_vecs ? __ldg(src + v) : make_uint4(0u, 0u, 0u, 0u);
      }
      for (int j = 0; j < top_k; ++j) {
        const int slot = __ldg(slot_of + t * top_k + j);
        if (slot < 0) continue;
        uint4* dst = x_sorted + static_cast<size_t>(slot) * row_vecs;
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
          const int v = v0 + 32 * i + lane;
          if (v < row_vecs) __stcs(dst + v, q[i]);
        }
      }
    }
  }
}

// Router top-k: one warp per token.  Lane l holds logits l, l+32, ... ;
// top_k rounds of a warp arg-max (larger logit wins, equal logits go to the
// lower expert id, taken experts are skipped) pick the experts in descending
// order; the weights are a softmax over the picked logits in fp32.
// Non-finite logits count as -infinity; a row with no finite logit gets
// equal weights.
template <int PER_LANE>
__global__ void router_topk_kernel(const float* __restrict__ logits, int n, int E, int top_k,
                                   int32_t* __restrict__ ids, float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < n; t += gridDim.x * warps) {
    float v[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const int e = lane + 32 * i;
      const float x = (e < E) ? logits[static_cast<size_t>(t) * E + e] : -INFINITY;
      v[i] = (x == x && x != INFINITY) ? x : -INFINITY;
    }
    uint32_t taken = 0;
    float top0 = 0.f, sum = 0.f, mine = 0.f;
    int mine_e = 0;
    for (int j = 0; j < top_k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i) {
        const int e = lane + 32 * i;
        const bool free = e < E && !((taken >> i) & 1u);
        if (free && (v[i] > bv || (v[i] == bv && e < be))) {
          bv = v[i];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (j == 0) top0 = bv;
      const float ex = (top0 == -INFINITY) ? 1.f : expf(bv - top0);
      sum += ex;
      if (j == lane) {
        mine = ex;
        mine_e = be;
      }
    }
    if (lane < top_k) {
      ids[static_cast<size_t>(t) * top_k + lane] = mine_e;
      w[static_cast<size_t>(t) * top_k + lane] = mine / sum;
    }
  }
}

}  // namespace

int launch_router(const float* logits, int n, int E, int top_k, int32_t* ids, float* w, cudaStream_t s) {
  if (n == 0) return TQ_OK;
  const int threads = 256, warps = threads / 32;
  const int blocks = std::max(1, std::min((n + warps - 1) / warps, sm_count() * 8));
  if (E <= 256)
    router_topk_kernel<8><<<blocks, threads, 0, s>>>(logits, n, E, top_k, ids, w);
  else
    router_topk_kernel<32><<<blocks, threads, 0, s>>>(logits, n, E, top_k, ids, w);
  const int st = launch_status();
  if (st == TQ_OK) count_launch(kCntRouter);
  return st;
}

int launch_gather(const uint16_t* x, const int32_t* sorted_pairs, int P, int top_k, int K, uint16_t* x_sorted,
                  int* err, cudaStream_t s) {
  if (P == 0) return TQ_OK;
  const int row_vecs = K / 8;
  const int threads = 256;   // 8 warps, one slot each per pass
  const int blocks = static_cast<int>(std::max<long long>(
      1, std::min<long long>((static_cast<long long>(P) + 7) / 8, sm_count() * 8ll)));
  int st = launch_pdl(gather_rows_kernel, dim3(blocks), dim3(threads), 0, s, reinterpret_cast<const uint4*>(x),
                      sorted_pairs, P, top_k, row_vecs, reinterpret_cast<uint4*>(x_sorted), err);
  if (st == TQ_OK) st = launch_status();
  if (st == TQ_OK) count_launch(kCntGather);
  return st;
}

int launch_gather_tokens(const uint16_t* x, const int32_t* slot_of, int64_t n, int top_k, int K, uint16_t* x_sorted,
                         cudaStream_t s) {
  if (n == 0) return TQ_OK;
  const int row_vecs = K / 8;
  const int threads = 256;   // 8 warps, one token each per pass
  const int blocks = static_cast<int>(std::max<long long>(1, std::min<long long>((n + 7) / 8, sm_count() * 8ll)));
  int st = launch_pdl(gather_tokens_kernel, dim3(blocks), dim3(threads), 0, s, reinterpret_cast<const uint4*>(x),
                      slot_of, static_cast<int>(n), top_k, row_vecs, reinterpret_cast<uint4*>(x_sorted));
  if (st == TQ_OK) st = launch_status();
  if (st == TQ_OK) count_launch(kCntGather);
  return st;
}

// Blocks sharing the routing sort: one up to 8192 pairs (a block's own
// histogram is all it needs), else one per 2048 pairs, at most 64.
static int route_sorters(int P) {
  if (P <= 8192) return 1;
  return static_cast<int>(std::min<long long>(64, (static_cast<long long>(P) + 2047) / 2048));
}

static size_t route_smem(int E) { return sizeof(int32_t) * (kWarps + 2) * static_cast<size_t>(E); }

int launch_route_tile_map(const int32_t* topk_ids, int P, int E, int tile_m, int32_t* counts, int32_t* offsets,
                          int32_t* sorted_pairs, int32_t* tiles, int32_t* num_tiles, int64_t cap, int* err,
                          cudaStream_t s, float* y32, int64_t y32_count, int32_t* slot_of) {
  const size_t smem = route_smem(E);
  if (cudaFuncSetAttribute(route_tile_map_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(route_smem(1024))) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  long long z4 = 0;
  if (y32_count > 0) {
    if (y32_count % 4 != 0 || (reinterpret_cast<uintptr_t>(y32) & 15u) != 0) {
      // not clearable in 16-byte steps: a separate clear
      if (cudaMemsetAsync(y32, 0, sizeof(float) * static_cast<size_t>(y32_count), s) != cudaSuccess) {
        cudaGetLastError();
        return TQ_ERR_CUDA;
      }
    } else {
      z4 = y32_count / 4;
    }
  }
  // one routing block, plus clearing blocks (16 float4 stores per thread, at
  // most two per SM)
  const long long clear_blocks = std::min<long long>((z4 + 16ll * kBlock - 1) / (16ll * kBlock), 2ll * sm_count());
  const int sorters = route_sorters(P);
  int st = launch_pdl(route_tile_map_kernel, dim3(static_cast<unsigned>(sorters + clear_blocks)), dim3(kBlock), smem,
                      s, topk_ids, P, E, sorters, tile_m, counts, offsets, sorted_pairs, tiles, num_tiles,
                      static_cast<long long>(cap), err, reinterpret_cast<float4*>(y32), z4, slot_of);
  if (st == TQ_OK) st = launch_status();
  if (st == TQ_OK) count_launch(kCntRouteTileMap);
  return st;
}

int launch_route(const int32_t* topk_ids, int P, int E, int32_t* counts, int32_t* offsets,
                 int32_t* sorted_pairs, int* err, cudaStream_t s) {
  const size_t smem = route_smem(E);
  if (cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(route_smem(1024))) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  const int sorters = route_sorters(P);
  int st = launch_pdl(route_kernel, dim3(sorters), dim3(kBlock), smem, s, topk_ids, P, E, sorters, counts, offsets,
                      sorted_pairs, err);
  if (st == TQ_OK) st = launch_status();
  if (st == TQ_OK) count_launch(kCntRoute);
  return st;
}

int launch_tile_map(const int32_t* offsets, int E, int tile_m, int32_t* tiles, int32_t* num_tiles,
                    int64_t cap, int* err, cudaStream_t s) {
  int st = launch_pdl(tile_map_kernel, dim3(1), dim3(kBlock), 0, s, offsets, E, tile_m, tiles, num_tiles,
                      static_cast<long long>(cap), err);
  if (st == TQ_OK) st = launch_status();
  if (st == TQ_OK) count_launch(kCntTileMap);
  return st;
}

int launch_clear(float* y, int64_t count, cudaStream_t s) {
  if (count <= 0) return TQ_OK;
  const int threads = 256;
  const long long per_block = 4ll * threads * 4;   // four float4 stores per thread
  const int blocks = static_cast<int>(std::max<long long>(
      1, std::min<long long>((count + per_block - 1) / per_block, 4ll * sm_count())));
  int st = launch_pdl(clear_kernel, dim3(blocks), dim3(threads), 0, s, y, static_cast<long long>(count));
  if (st == TQ_OK) st = launch_status();
  if (st == TQ_OK) count_launch(kCntClear);
  return st;
}

int launch_combine(const float* y32, uint16_t* y, int64_t count, cudaStream_t s) {
  if (count == 0) return TQ_OK;
  const int threads = 256;
  const int max_blocks = sm_count() * 8;
  const bool vec = (count % 4 == 0) && (reinterpret_cast<uintptr_t>(y32) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(y) % 8 == 0);
  if (vec) {
    const long long n4 = count / 4;
    const int blocks = static_cast<int>(std::min<long long>((n4 + threads - 1) / threads, max_blocks));
    const int st = launch_pdl(combine_kernel_v4, dim3(blocks), dim3(threads), 0, s,
                              reinterpret_cast<const float4*>(y32), reinterpret_cast<uint2*>(y), n4);
    if (st != TQ_OK) return st;
  } else {
    const int blocks = static_cast<int>(std::min<long long>((count + threads - 1) / threads, max_blocks));
    const int st = launch_pdl(combine_kernel_scalar, dim3(blocks), dim3(threads), 0, s, y32, y,
                              static_cast<long long>(count));
    if (st != TQ_OK) return st;
  }
  const int st = launch_status();
  if (st == TQ_OK) count_launch(kCntCombine);
  return st;
}

}  // namespace tq
