// Per-pair GEMV arm over 2-bit bitshift-trellis experts.
//
// Page "fix(qtip): gate the trellis grouped GEMM on m-tile occupancy, not token
// count", section "The regression" and the post-merge note: below the
// amortization boundary (and always for n <= 8) each (token, expert) pair runs
// its own GEMV, re-reading and re-decoding the expert once per pair (no
// de-duplication across pairs).
//
// GB300 design: one CTA per SM holds the fp16 LUT (and, for small batches,
// every token's activations) in shared memory.  A warp takes a contiguous
// range of (pair, weight row) items, or, when the output is the per-token
// bf16 product itself, of (token, weight row) items whose top_k pairs it
// walks in order, summing w_j times each pair's partial dot product in
// registers and writing the rounded sum once (no fp32 accumulator to clear,
// no atomics, no separate combine launch).  It keeps the current token's
// activations in registers (lane l holds the 64-element chunks l, l+32, ...
// of x[t]) and, for each row, loads the row's packed bytes with coalesced
// 16-byte loads (lane l takes bytes [16c, 16c+16) of chunk c) one row ahead,
// gets the 4 bytes before its chunk from the neighbour lane by shuffle (lane 0
// from lane 31 of the previous pass, zero at the row start), decodes its 64
// symbols by window identity, multiplies in fp32 (fp16 weights widened
// exactly) and reduces the row over the warp with xor shuffles.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kChunkSyms = 64;  // symbols per lane per pass (16 packed bytes)

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

template <int L, int CPL, int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
gemv_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ packed,
            const uint16_t* __restrict__ lut, const int32_t* __restrict__ topk_ids,
            const float* __restrict__ topk_w, int P, int top_k, int E, int K, int N, int x_in_smem,
            int pair_in, int pair_out, int early_prologue, float* __restrict__ y32, uint16_t* __restrict__ y_tok,
            int* err, int bar_off) {
  extern __shared__ __align__(16) uint16_t lut_s[];
  constexpr int kEntries = 1 << L;
  constexpr int kLutBytes = (kEntries * 2 + 15) & ~15;
  // Launched as a programmatic dependent of the previous kernel: with
  // early_prologue (that kernel writes none of the inputs, only the output)
  // the staging and the first row's loads below run while it finishes, and
  // the wait comes before the first output write.
  if (!early_prologue) pdl_wait();

  const int lane = threadIdx.x & 31;
  const int warps_per_block = THREADS / 32;
  const long long gwarp = static_cast<long long>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5);
  const long long nwarps = static_cast<long long>(gridDim.x) * warps_per_block;
  const int nchunks = K / kChunkSyms;
  const size_t row_bytes = static_cast<size_t>(K / 4);
  // This warp's contiguous range of items: (pair, row), consecutive rows of
  // one pair sharing the token's activations; or, with y_tok, (token, row),
  // each walked as its top_k (pair, row) steps.
  const bool tok_out = y_tok != nullptr;
  const long long items = static_cast<long long>(tok_out ? P / top_k : P) * N;
  const long long i0 = items * gwarp / nwarps, i1 = items * (gwarp + 1) / nwarps;

  // packed bytes of row r of the pair's expert (zeros for a bad expert id,
  // which process() reports)
  auto load_row = [&](int pair, int r, uint4 (&q)[CPL]) {
    const int e = __ldg(topk_ids + pair);
    const bool ok = e >= 0 && e < E;
    const uint4* rp = reinterpret_cast<const uint4*>(packed + (static_cast<size_t>(ok ? e : 0) * N + r) * row_bytes);
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      q[i] = (ok && c < nchunks) ? __ldg(rp + c) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // The warp walks its range in order: only the first item's (pair, row) is
  // found by division, the others step a counter.
  int p0 = 0, r0 = 0;
  if (i0 < i1) {
    p0 = static_cast<int>(i0 / N);
    r0 = static_cast<int>(i0 - static_cast<long long>(p0) * N);
    if (tok_out) p0 *= top_k;   // the token's first pair
  }
  // the (pair, row) step after (p, r)
  auto next = [&](int& p, int& r) {
    if (tok_out) {
      if (++p % top_k == 0) {   // past the token's last pair: next row, same token
        p -= top_k;
        if (++r == N) {
          r = 0;
          p += top_k;
        }
      }
    } else if (++r == N) {
      r = 0;
      ++p;
    }
  };
  const long long steps = (i1 - i0) * (tok_out ? top_k : 1);
  // The first row's bytes are in flight while the tables are staged.
  uint4 qa[CPL], qb[CPL];
  if (i0 < i1) load_row(p0, r0, qa);

  // The table by the bulk copy engine (one thread; the barrier sits after
  // the table and the activations), waited for after the activations.
  __shared__ int abort_flag;
  const uint32_t bar = smem_u32(lut_s) + static_cast<uint32_t>(bar_off);
  if constexpr (kEntries >= 8) {
    if (threadIdx.x == 0) {
      abort_flag = 0;
      mbar_init(bar, 1);
      mbar_fence_init();
      bulk_stage_to_smem(smem_u32(lut_s), lut, kEntries * 2, bar);
    }
  } else {
    for (int i = threadIdx.x; i < kEntries; i += THREADS) lut_s[i] = lut[i];
  }
  // Small batches: every token's activations staged once per CTA (after the
  // LUT), so a warp that moves to another pair refills its registers from
  // shared memory instead of waiting on global memory.
  const int n_tok = P / top_k;
  const int x_rows = pair_in ? P : n_tok;   // x is per pair (sorted by pair id) or per token
  uint4* xs = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(lut_s) + kLutBytes);
  if (x_in_smem) {
    // 16-byte piece v of 128-byte chunk c goes to piece v ^ (c & 7) of the chunk
    const uint32_t xs_base = smem_u32(xs);
    const int pieces = x_rows * K / 8;
    for (int q = threadIdx.x; q < pieces; q += THREADS) {
      const int g = q >> 3, v = q & 7;   // global chunk (8 pieces each; K is a multiple of 64)
      const int c = g % (K / kChunkSyms);  // chunk within its token: the reader's swizzle key
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(xs_base + 16u * static_cast<uint32_t>(8 * g + (v ^ (c & 7)))),
                   "l"(reinterpret_cast<const uint4*>(x) + q)
                   : "memory");
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  }
  __syncthreads();
  if constexpr (kEntries >= 8) {
    if (!mbar_wait(bar, 0, &abort_flag, err, kWhereTableStage)) return;
  }
  const uint32_t lut_base = smem_u32(lut_s);
  if (early_prologue) pdl_wait();
  pdl_trigger();

  int cur_pair = -1, cur_tok = -1;
  float wt = 0.f;
  bool pair_ok = false;
  uint32_t xr[CPL][32];
  // this lane's share of pair . row (fp32, not yet reduced over the warp)
  auto process = [&](bool first_item, int pair, int r, const uint4 (&qv)[CPL]) -> float {
    if (pair != cur_pair) {
      cur_pair = pair;
      const int e = __ldg(topk_ids + pair);
      pair_ok = e >= 0 && e < E;
      if (!pair_ok && lane == 0 && (r == 0 || first_item)) record_error(err, TQ_ERR_INVALID_ARG, kWhereRoute);
      wt = pair_out ? 1.f : __ldg(topk_w + pair);   // per-pair outputs carry no router weight
    }
    const int tok = pair_in ? pair : pair / top_k;   // the row of x this pair multiplies
    if (tok != cur_tok) {
      cur_tok = tok;
      // activations of this token: chunk c = lane + 32 i, 64 bf16 = 32 words
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c < nchunks) {
          const size_t off16 = (static_cast<size_t>(tok) * K + static_cast<size_t>(c) * kChunkSyms) / 8;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            // shared copy: piece v of chunk c sits at piece v ^ (c & 7), so
            // the 32 lanes (chunks 32 apart) spread over all banks
            const uint4 q = x_in_smem ? xs[off16 + (v ^ (c & 7))]
                                      : __ldg(reinterpret_cast<const uint4*>(x) + off16 + v);
            xr[i][4 * v] = q.x;
            xr[i][4 * v + 1] = q.y;
            xr[i][4 * v + 2] = q.z;
            xr[i][4 * v + 3] = q.w;
          }
        } else {
#pragma unroll
          for (int v = 0; v < 32; ++v) xr[i][v] = 0u;
        }
      }
    }
    if (!pair_ok) return 0.f;
    float acc = 0.f;
    uint32_t carry = 0u;  // last word of chunk (32 i - 1), held by lane 31
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      const uint4 q = qv[i];
      uint32_t prev = __shfl_up_sync(0xffffffffu, q.w, 1);
      if (lane == 0) prev = carry;
      carry = __shfl_sync(0xffffffffu, q.w, 31);
      if (c < nchunks) {
        const uint32_t words[5] = {prev, q.x, q.y, q.z, q.w};
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
          const uint64_t lo64 = static_cast<uint64_t>(words[wi]) | (static_cast<uint64_t>(words[wi + 1]) << 32);
#pragma unroll
          for (int m = 0; m < 16; m += 2) {
            const uint32_t o0 = static_cast<uint32_t>(lo64 >> (33 + 2 * m - L)) & ((1u << (L + 1)) - 2u);
            const uint32_t o1 = static_cast<uint32_t>(lo64 >> (35 + 2 * m - L)) & ((1u << (L + 1)) - 2u);
            uint32_t h0, h1;
            asm volatile("ld.shared.u16 %0, [%1];" : "=r"(h0) : "r"(lut_base + o0));
            asm volatile("ld.shared.u16 %0, [%1];" : "=r"(h1) : "r"(lut_base + o1));
            const uint32_t xv = xr[i][wi * 8 + m / 2];
            acc = fmaf(__half2float(__ushort_as_half(static_cast<unsigned short>(h0))), bf16lo(xv), acc);
            acc = fmaf(__half2float(__ushort_as_half(static_cast<unsigned short>(h1))), bf16hi(xv), acc);
          }
        }
      }
    }
    return acc;
  };
  // fold one (pair, row) step into the output
  float item_acc = 0.f;   // tok_out: this lane's share of sum_j w_j (pair_j . row)
  // (a pair with an out-of-range expert id adds nothing and writes nothing)
  auto finish = [&](int pair, int r, float acc) {
    if (tok_out) {
      if (pair_ok) item_acc = fmaf(wt, acc, item_acc);
      if ((pair + 1) % top_k != 0) return;   // more pairs of this token to come
      acc = item_acc;
      item_acc = 0.f;
    } else if (!pair_ok) {
      return;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      if (tok_out) {
        const __nv_bfloat16 b = __float2bfloat16_rn(acc);
        y_tok[static_cast<size_t>(pair / top_k) * N + r] = __bfloat16_as_ushort(b);   // one writer per (token, row)
      } else if (pair_out) {
        y32[static_cast<size_t>(pair) * N + r] = acc;   // one writer per (pair, row)
      } else {
        atomicAdd(y32 + static_cast<size_t>(pair / top_k) * N + r, acc * wt);
      }
    }
  };

  // The next row's bytes are in flight while this row decodes (two register
  // sets used in turn, so no copy waits for a load).
  int pa = p0, ra = r0;
  for (long long it = 0; it < steps; it += 2) {
    int pb = pa, rb = ra;
    next(pb, rb);
    if (it + 1 < steps) load_row(pb, rb, qb);
    finish(pa, ra, process(it == 0, pa, ra, qa));
    if (it + 1 >= steps) break;
    pa = pb;
    ra = rb;
    next(pa, ra);
    if (it + 2 < steps) load_row(pa, ra, qa);
    finish(pb, rb, process(false, pb, rb, qb));
  }
}

template <int L, int CPL>
int launch_one(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, const int32_t* ids,
               const float* w, int P, int top_k, int E, int K, int N, float* y32, uint16_t* y_tok, int* err,
               cudaStream_t s, int pair_in, int pair_out, int early) {
  constexpr int kThreads = (CPL >= 4) ? 256 : 512;
  auto kfn = gemv_kernel<L, CPL, kThreads>;
  const size_t lut_bytes = ((sizeof(uint16_t) << L) + 15) & ~static_cast<size_t>(15);
  const size_t x_bytes = static_cast<size_t>(pair_in ? P : P / top_k) * K * 2;
  // activations go to shared memory when they fit beside the LUT (small batches)
  const int x_in_smem = (lut_bytes + x_bytes <= 200u * 1024u) ? 1 : 0;
  const size_t bar_off = lut_bytes + (x_in_smem ? x_bytes : 0);   // a multiple of 16
  const size_t smem = bar_off + 16;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  const int sms = sm_count();
  const long long items = static_cast<long long>(P) * N;
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(sms, (items + kThreads / 32 - 1) / (kThreads / 32))));
  const int st = launch_pdl(kfn, dim3(grid), dim3(kThreads), smem, s, x, packed, lut, ids, w, P, top_k, E, K, N,
                            x_in_smem, pair_in, pair_out, early, y32, y_tok, err, static_cast<int>(bar_off));
  return st == TQ_OK ? launch_status() : st;
}

template <int L>
int launch_L(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, const int32_t* ids,
             const float* w, int P, int top_k, int E, int K, int N, float* y32, uint16_t* yt, int* err,
             cudaStream_t s, int pi, int po, int early) {
  const int nchunks = K / kChunkSyms;
  if (nchunks <= 32) return launch_one<L, 1>(x, packed, lut, ids, w, P, top_k, E, K, N, y32, yt, err, s, pi, po, early);
  if (nchunks <= 64) return launch_one<L, 2>(x, packed, lut, ids, w, P, top_k, E, K, N, y32, yt, err, s, pi, po, early);
  return launch_one<L, 4>(x, packed, lut, ids, w, P, top_k, E, K, N, y32, yt, err, s, pi, po, early);
}

}  // namespace

int launch_gemv(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L,
                const int32_t* topk_ids, const float* topk_w, int64_t n, int top_k, int E, int K,
                int N, float* y32, int* err, cudaStream_t s, int pair_in, int pair_out, bool early_prologue,
                uint16_t* y_tok) {
  const int P = static_cast<int>(n * top_k);
  if (P == 0) return TQ_OK;
  if (y_tok && (pair_in || pair_out)) return TQ_ERR_INVALID_ARG;   // per-token output: x per token
  const int early = early_prologue ? 1 : 0;
  int st;
  switch (L) {
    case 2: st = launch_L<2>(x, packed, lut, topk_ids, topk_w, P, top_k, E, K, N, y32, y_tok, err, s, pair_in, pair_out, early); break;
    case 4: st = launch_L<4>(x, packed, lut, topk_ids, topk_w, P, top_k, E, K, N, y32, y_tok, err, s, pair_in, pair_out, early); break;
    case 6: st = launch_L<6>(x, packed, lut, topk_ids, topk_w, P, top_k, E, K, N, y32, y_tok, err, s, pair_in, pair_out, early); break;
    case 8: st = launch_L<8>(x, packed, lut, topk_ids, topk_w, P, top_k, E, K, N, y32, y_tok, err, s, pair_in, pair_out, early); break;
    case 10: st = launch_L<10>(x, packed, lut, topk_ids, topk_w, P, top_k, E, K, N, y32, y_tok, err, s, pair_in, pair_out, early); break;
    case 12: st = launch_L<12>(x, packed, lut, topk_ids, topk_w, P, top_k, E, K, N, y32, y_tok, err, s, pair_in, pair_out, early); break;
    case 14: st = launch_L<14>(x, packed, lut, topk_ids, topk_w, P, top_k, E, K, N, y32, y_tok, err, s, pair_in, pair_out, early); break;
    case 16: st = launch_L<16>(x, packed, lut, topk_ids, topk_w, P, top_k, E, K, N, y32, y_tok, err, s, pair_in, pair_out, early); break;
    default: return TQ_ERR_INVALID_ARG;
  }
  if (st == TQ_OK) count_launch(kCntGemv);
  return st;
}

}  // namespace tq
