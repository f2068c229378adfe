// Grouped GEMM over 2-bit bitshift-trellis experts with the decode fused into
// the multiply, for sm_103a (tcgen05 tensor cores, tensor memory, TMA).
//
// What it computes (page "fix(qtip): gate the trellis grouped GEMM on m-tile
// occupancy, not token count", section "The cause is a threshold, not a kernel
// defect"): pairs are sorted by expert and grouped into m-tiles; for each
// m-tile the expert's packed bytes are staged once and every pair of the tile
// is multiplied against them.  Page "perf(qtip): arch-specialise the trellis
// grouped GEMM (D16) + close the silent-failure holes (D18)", item 2 and "The
// two changes": a thread owns a run of 32 symbols of one weight row, seeds the
// trellis state from the window identity; only packed 2-bit bytes cross HBM
// and full-size weights never materialise.
//
// GB300 design (one persistent CTA per SM, warp-specialised):
//   warp 0      TMA producer.  Packed bytes: one 2-D box of the expert's 128
//               rows x 128 bytes (512 symbols = 8 k-steps of 64) per
//               "super-stage", 128B-swizzled; wide rows keep the TMA unit's
//               per-row cost low.
//   (with E epilogue warps, 4 or 8: the decode warps start at 2 + E and the
//   activation producer follows them; the numbers below are for E = 4)
//   warp 14     TMA producer for activations, 64 columns per k-step into the
//               MMA's 128B-swizzled B layout: gathered from the token rows of
//               x, four rows per copy (small m-tiles), or, from the
//               pair-sorted copy of x, one box of (tile_m rounded up to 16)
//               consecutive rows.
//   warp 1      MMA issuer: tcgen05.mma kind::f16, A = decoded weights in tensor
//               memory (M = 128 rows), B = activations in shared memory
//               (N = pairs of the tile padded to 16), fp32 accumulator in
//               tensor memory.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, scale by the router
//               weight, 16-byte fp32 vector reductions into y32[token][rows];
//               eight warps (2-9, two per lane quarter) when the m-tiles span
//               both accumulator slots.
//   warps 6-13  decode: thread (quarter q, half h) owns weight row 32q + lane
//               and symbols [32h, 32h + 32) of each k-step; the state of each
//               symbol is a shift + mask of a 64-bit window of the staged
//               bytes (window identity), looked up in a bf16 copy of the LUT
//               held in shared memory, and the 32 bf16 weights go to tensor
//               memory with tcgen05.st.
// Work: units = (m-tile, 128-row block of N) x super-stages, split into equal
// contiguous ranges per CTA (a unit may be shared by two CTAs; the epilogue
// adds partial sums atomically), or, when every CTA has many units and the
// output is large, whole units dealt round-robin (see Walk).
// Modes: pair_out (per-pair outputs, no router weight: the MLP's gate|up),
// store_out (with pair_out: whole units and plain stores), kDense (A read from
// materialized bf16 weights: the dequantize-materialize comparator).
// Launched with programmatic stream serialization: the kernel waits for its
// predecessor at its start, or after its prologue (LUT staging, tensor memory)
// when the caller knows the predecessor writes nothing the prologue reads.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kBlockRows = 128;                      // weight rows per unit (MMA M)
constexpr int kKStep = 64;                           // symbols per MMA step (4 x K16)
constexpr int kKStepBytes = kKStep / 4;              // 16 packed bytes per row per k-step
constexpr int kSSBytes = 128;                        // packed bytes per row per super-stage
constexpr int kSSSteps = kSSBytes / kKStepBytes;     // 8 k-steps per super-stage
constexpr int kPkStageBytes = kBlockRows * kSSBytes; // 16 KiB
constexpr int kActRowBytes = kKStep * 2;             // one 128-byte swizzle row per pair
constexpr int kATmemCols = kKStep / 2;               // bf16x2 columns per A stage
constexpr int kNumAStages = 8;
constexpr int kNumDecodeWarps = 8;
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpEpi0 = 2;
constexpr int kMaxPkStages = 6;
constexpr int kActPrefetch = 8;                       // k-steps of activations asked into L2 ahead
constexpr int kMaxActStages = 8;
constexpr int kSmemLimit = 232448;                   // 227 KiB opt-in per block
constexpr int kNumBars = 2 * kMaxPkStages + 2 * kMaxActStages + 2 * kNumAStages + 2 + 2 + 1 + 1;
static_assert(kNumDecodeWarps == 8, "decode mapping assumes 2 warps per TMEM lane quarter");
// Warp roles for kEpi epilogue warps (4: one per lane quarter; 8, used when
// the units span both accumulator slots: two per quarter, each draining half
// of the columns, so a drain the next large unit waits for takes half as long).
// Four: 480 threads; eight: 608.
template <int kEpi>
struct Roles {
  static constexpr int dec0 = kWarpEpi0 + kEpi;
  static constexpr int act = dec0 + kNumDecodeWarps;
  static constexpr int threads = 32 * (act + 1);
  static_assert(kEpi % 4 == 0 && dec0 % 4 == 2, "role warps must cover all four quarters");
};

struct Params {
  const int32_t* sorted_pairs;
  const float* topk_w;
  const int32_t* tiles;
  const int32_t* num_tiles;
  const uint16_t* lut;
  const uint8_t* packed;
  float* y32;
  int* err;
  long long cap;
  int P, E, tile_m;
  int top_k, N, K;
  int row_blocks;
  int rb_group;     // row blocks per ordering group (row_blocks = plain tile-major order)
  int pair_out;     // 0: y32[token] += w * D (combine); 1: y32[sorted slot] += D (per pair)
  int allow_interleave;  // whole units round-robin over CTAs when there are many (blocked order only)
  int store_out;         // whole units always, and plain stores: every output element has one writer
  int early_prologue;    // the previous kernel writes nothing the prologue reads (LUT): overlap it
  int act_gather;        // activations: 1 = x holds token rows, gathered by sorted pair; 0 = x holds
                         // the pair-sorted rows themselves
  int n_mma_max;    // largest MMA N (tile_m rounded up to 16)
  int pk_stages;    // packed super-stage buffers
  int act_stages;   // activation k-step buffers
  int nacc;         // accumulator buffers of n_mma_max columns in tensor memory (1 or 2)
  int acc_slots;    // 1: no room for two buffers; two 128-column slots instead (see AccSlots)
  int acol0;        // first tensor-memory column of the A stages
  int tmem_cols;    // allocated tensor-memory columns
  uint32_t off_pk, off_lut, off_bar;  // byte offsets from the 1024-aligned base
};

struct Pipe {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void advance(int n) {
    if (++stage == n) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

// Accumulator slots, for m-tiles above 128 pairs, where two accumulators of
// n_mma_max columns do not fit beside the 8 A stages: the 256 accumulator
// columns are two slots of 128.  A unit of at most 128 pairs takes one slot,
// alternating, so consecutive small units are double-buffered; a larger unit
// takes both (one MMA of N = n_mma at column 0), and the epilogue frees slot 0
// as soon as it has drained the first 128 columns, so a small unit after it can
// start while the rest drains.  The MMA warp and the epilogue walk the same
// units and step this state alike.
struct AccSlots {
  int next = 0;           // slot of the next small unit
  uint32_t full_ph = 0;   // bit k: phase of slot k's full barrier (epilogue)
  uint32_t empty_ph = 0;  // bit k: phase of slot k's empty barrier (MMA warp)
  __device__ __forceinline__ static bool big(uint32_t n_mma) { return n_mma > 128u; }
  __device__ __forceinline__ int first(uint32_t n_mma) const { return big(n_mma) ? 0 : next; }
  __device__ __forceinline__ void step(uint32_t n_mma) { next = big(n_mma) ? 0 : (next ^ 1); }
};

// A tile entry is used only if it describes 1..tile_m consecutive sorted slots
// of an existing expert; anything else (a map built for another tile_m, a
// stale buffer) is skipped by every role alike and reported.
struct Tile {
  int e, slot0, rows;
  bool ok;
};
__device__ __forceinline__ Tile read_tile(const Params& p, int tile) {
  Tile t;
  const int32_t* const entry = p.tiles + 3ll * tile;
  t.e = entry[0];
  t.slot0 = entry[1];
  t.rows = entry[2];
  t.ok = t.e >= 0 && t.e < p.E && t.rows >= 1 && t.rows <= p.tile_m && t.slot0 >= 0 &&
         t.slot0 <= p.P - t.rows;
  return t;
}

// A run of super-stages [ss0, ss1) of one work unit (m-tile `tile`, row block
// `rb`) starting at flattened position g and ending no later than g_end.
// Units are ordered by groups of `rb_group` row blocks, then m-tile, then row
// block: CTAs running at the same time touch one slice of the output (which
// stays in L2 for the atomic adds) while each tile's activations are reused
// across the group's row blocks.
struct Segment {
  int tile, rb, ss0, ss1;
};
__device__ __forceinline__ Segment segment_at(long long g, long long g_end, int n_ss, int num_tiles,
                                              int rb_group) {
  Segment sg;
  const long long u = g / n_ss;
  sg.ss0 = static_cast<int>(g - u * n_ss);
  sg.ss1 = static_cast<int>(min(static_cast<long long>(n_ss), sg.ss0 + (g_end - g)));
  const long long per_group = static_cast<long long>(num_tiles) * rb_group;
  const long long grp = u / per_group;
  const long long r = u - grp * per_group;
  sg.tile = static_cast<int>(r / rb_group);
  sg.rb = static_cast<int>(grp * rb_group + (r - static_cast<long long>(sg.tile) * rb_group));
  return sg;
}

// A CTA's walk over its work.  Contiguous (step == 0): an equal share of the
// flattened (unit, super-stage) positions, split at any super-stage, so every
// CTA gets the same number of super-stages.  Interleaved (step == grid): whole
// units blockIdx.x, blockIdx.x + grid, ...: the CTAs running at one time take
// consecutive units, i.e. the row blocks of the same few m-tiles, so a tile's
// activations are read from L2 by all of them instead of from DRAM once per
// row block; used when every CTA has many units (the imbalance is at most one
// unit in many).
struct Walk {
  long long g, g_end, step;
};
__device__ __forceinline__ Walk walk_begin(long long units, int n_ss, bool interleave) {
  Walk w;
  if (interleave) {
    w.g = blockIdx.x;
    w.g_end = units;
    w.step = gridDim.x;
  } else {
    const long long total = units * n_ss;
    w.g = total * blockIdx.x / gridDim.x;
    w.g_end = total * (blockIdx.x + 1) / gridDim.x;
    w.step = 0;
  }
  return w;
}
__device__ __forceinline__ bool walk_next(Walk& w, int n_ss, int num_tiles, int rb_group, Segment& sg) {
  if (w.g >= w.g_end) return false;
  if (w.step == 0) {
    sg = segment_at(w.g, w.g_end, n_ss, num_tiles, rb_group);
    w.g += sg.ss1 - sg.ss0;
  } else {
    sg = segment_at(w.g * n_ss, (w.g + 1) * n_ss, n_ss, num_tiles, rb_group);
    w.g += w.step;
  }
  return true;
}

// Byte offset of logical byte b of staged row r (128-byte pitch) in the
// 128B-swizzled super-stage: the 16-byte chunk index is XORed with r mod 8.
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t b) {
  return r * kSSBytes + (b ^ ((r & 7u) << 4));
}

template <int L>
__device__ __forceinline__ uint32_t lut_byte_offset_lo(uint64_t lo64, int m) {
  // state of run symbol m (< 16): bits [34 + 2m - L, 34 + 2m) of lo64; times 2
  return static_cast<uint32_t>(lo64 >> (33 + 2 * m - L)) & ((1u << (L + 1)) - 2u);
}
template <int L>
__device__ __forceinline__ uint32_t lut_byte_offset_hi(uint64_t cur, int m) {
  // state of run symbol m (>= 16): bits [2 + 2m - L, 2 + 2m) of the 8 run bytes
  return static_cast<uint32_t>(cur >> (1 + 2 * m - L)) & ((1u << (L + 1)) - 2u);
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds_u128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
// The 32 bf16 weights of one run: window states of the 4 bytes before the run
// (prev) and the run's 8 bytes (cur), looked up in the shared-memory LUT and
// packed two per 32-bit word (even symbol in the low half).
template <int L>
__device__ __forceinline__ void lookup_run(uint32_t lut_s, uint32_t prev, uint64_t cur, uint32_t (&w)[16]) {
  const uint64_t lo64 = static_cast<uint64_t>(prev) | (cur << 32);
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const uint32_t a = lds_u16(lut_s + lut_byte_offset_lo<L>(lo64, 2 * m));
    const uint32_t b = lds_u16(lut_s + lut_byte_offset_lo<L>(lo64, 2 * m + 1));
    w[m] = a | (b << 16);
  }
#pragma unroll
  for (int m = 8; m < 16; ++m) {
    const uint32_t a = lds_u16(lut_s + lut_byte_offset_hi<L>(cur, 2 * m));
    const uint32_t b = lds_u16(lut_s + lut_byte_offset_hi<L>(cur, 2 * m + 1));
    w[m] = a | (b << 16);
  }
}

// Waits (bounded, ignoring the abort flag) for the last `pending` phases of a
// ring of full barriers to complete: copies in flight must land before exit.
__device__ __forceinline__ void drain_ring(uint32_t bar0, Pipe pipe, int nstages, long long issued, int* err) {
  const long long pending = min(issued, static_cast<long long>(nstages));
  for (long long k = 1; k <= pending; ++k) {
    int st = pipe.stage - static_cast<int>(k);
    uint32_t ph = pipe.phase;
    if (st < 0) {
      st += nstages;
      ph ^= 1u;
    }
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar0 + 8 * st, ph)) {
      if (globaltimer() - t0 > kWaitTimeoutNs) {
        record_error(err, TQ_ERR_DEVICE_TIMEOUT, kWhereGroupedTeardown);
        break;
      }
    }
  }
}

// kDense: the comparator mode.  A comes from materialized bf16 weights
// [E][N][K] through TMA (one 128 x 64 box per k-step into the same ring the
// packed bytes use) and the MMA reads it from shared memory; the decode warps
// and the LUT stay idle.
template <int L, bool kDense, int kEpi>
__global__ void __launch_bounds__(Roles<kEpi>::threads, 1)
grouped_kernel(const __grid_constant__ CUtensorMap tm_packed, const __grid_constant__ CUtensorMap tm_xs,
               const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  if (!p.early_prologue) pdl_wait();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int SP = p.pk_stages;
  const int SA = p.act_stages;

  const uint32_t act0 = base;                                  // SA x n_mma_max x 128 B
  const uint32_t pk0 = base + p.off_pk;                        // SP x 16 KiB
  const uint32_t lut_s = base + p.off_lut;                     // 2^L bf16
  const uint32_t bar_pkfull = base + p.off_bar;
  const uint32_t bar_pkempty = bar_pkfull + 8 * kMaxPkStages;
  const uint32_t bar_actfull = bar_pkempty + 8 * kMaxPkStages;
  const uint32_t bar_actempty = bar_actfull + 8 * kMaxActStages;
  const uint32_t bar_afull = bar_actempty + 8 * kMaxActStages;
  const uint32_t bar_aempty = bar_afull + 8 * kNumAStages;
  const uint32_t bar_accfull = bar_aempty + 8 * kNumAStages;
  // When the activation ring and the A ring have the same depth they advance
  // in lockstep (one stage of each per k-step): the MMA's one commit on the
  // activation stage then also releases the A stage of the same index.
  const uint32_t bar_arel = (SA == kNumAStages) ? bar_actempty : bar_aempty;
  const uint32_t bar_accempty = bar_accfull + 16;
  const uint32_t bar_drain = bar_accempty + 16;
  const uint32_t bar_lut = bar_drain + 8;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + p.off_bar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SP; ++s) {
      mbar_init(bar_pkfull + 8 * s, 1);
      mbar_init(bar_pkempty + 8 * s, kDense ? 1 : kNumDecodeWarps);
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(bar_actfull + 8 * s, 1);
      mbar_init(bar_actempty + 8 * s, 1);
    }
    for (int a = 0; a < kNumAStages; ++a) {
      mbar_init(bar_afull + 8 * a, kNumDecodeWarps);
      mbar_init(bar_aempty + 8 * a, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_accfull + 8 * b, 1);
      mbar_init(bar_accempty + 8 * b, kEpi);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_lut, 1);
    *abort_flag = 0;
    mbar_fence_init();
    // the fp16 table by the bulk copy engine, converted below once it is in
    if constexpr (!kDense && (1 << L) >= 8) bulk_stage_to_smem(lut_s, p.lut, (1u << L) * 2u, bar_lut);
  }
  if (warp == kWarpProducer) tmem_alloc(smem_u32(tmem_holder), static_cast<uint32_t>(p.tmem_cols));

  // LUT: fp16 (global) -> bf16 (shared), nearest-even.
  if constexpr (!kDense) {
    constexpr int kEntries = 1 << L;
    uint16_t* lut_dst = reinterpret_cast<uint16_t*>(gbase + p.off_lut);
    if constexpr (kEntries >= 8) {
      // the bulk copy issued with the barrier inits, then converted in place,
      // 8 entries per step (a timed-out wait raises the abort flag, which
      // every role's next wait sees)
      __syncthreads();
      const bool in = mbar_wait(bar_lut, 0, abort_flag, p.err, kWhereTableStage);
      uint4* dst = reinterpret_cast<uint4*>(lut_dst);
      for (int i = threadIdx.x; in && i < kEntries / 8; i += Roles<kEpi>::threads) {
        uint4 v = dst[i];
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
          const float2 f = __half22float2(h);
          const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
          w[j] = *reinterpret_cast<const uint32_t*>(&b);
        }
        dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
      for (int i = threadIdx.x; i < kEntries; i += Roles<kEpi>::threads) {
        const __nv_bfloat16 b = __float2bfloat16_rn(__half2float(__ushort_as_half(p.lut[i])));
        lut_dst[i] = *reinterpret_cast<const uint16_t*>(&b);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
  // Launched as a programmatic dependent of the kernel before it on the
  // stream: with early_prologue the prologue above (which reads only the
  // LUT) ran while that kernel finished; everything below may depend on it.
  pdl_wait();

  const int num_tiles = static_cast<int>(min(static_cast<long long>(*p.num_tiles), p.cap));
  const int ksteps = p.K / kKStep;
  const int n_ss = (ksteps + kSSSteps - 1) / kSSSteps;
  const uint32_t acol0 = static_cast<uint32_t>(p.acol0);
  const int rb_group = p.rb_group;
  // This CTA's share of the (unit, super-stage) work; every role walks it in
  // the same order, one segment at a time.
  const long long units = static_cast<long long>(num_tiles) * p.row_blocks;
  const Walk walk0 = walk_begin(units, n_ss, p.store_out || (p.allow_interleave && units >= 16ll * gridDim.x));

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ packed-byte producer
    if (lane == 0) tma_prefetch_desc(&tm_packed);
    // Packed bytes are read once per m-tile: mark them first to leave L2, so
    // that the fp32 output slice the atomics add into stays resident (prefill
    // DRAM traffic 1.774 -> 1.692 GB at the down projection, time unchanged).
    const uint64_t pk_policy = l2_evict_first_policy();
    Pipe pk;
    long long pk_issued = 0;
    bool ok = true;
    Walk w = walk0;
    Segment sg;
    while (ok && walk_next(w, n_ss, num_tiles, rb_group, sg)) {
      const Tile tl = read_tile(p, sg.tile);
      if (!tl.ok) {
        if (lane == 0) record_error(p.err, TQ_ERR_INVALID_ARG, kWhereGroupedProducer);
        continue;
      }
      const int row_g = tl.e * p.N + sg.rb * kBlockRows;
      // One ring slot per super-stage of packed bytes, or per k-step of dense
      // bf16 weights (128 rows x 64 values = the same 16 KiB).
      const int i0 = kDense ? sg.ss0 * kSSSteps : sg.ss0;
      const int i1 = kDense ? min(ksteps, sg.ss1 * kSSSteps) : sg.ss1;
      for (int i = i0; i < i1; ++i) {
        if (!mbar_wait(bar_pkempty + 8 * pk.stage, pk.phase ^ 1u, abort_flag, p.err, kWhereGroupedProducer)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full = bar_pkfull + 8 * pk.stage;
          mbar_arrive_expect_tx(full, kPkStageBytes);
          tma_load_2d_hint(pk0 + pk.stage * kPkStageBytes, &tm_packed, kDense ? i * kKStep : i * kSSBytes, row_g,
                           full, pk_policy);
        }
        ++pk_issued;
        pk.advance(SP);
      }
    }
    // Teardown: every copy issued must have landed before the CTA exits.
    __syncwarp();
    drain_ring(bar_pkfull, pk, SP, pk_issued, p.err);
  } else if (warp == Roles<kEpi>::act) {
    // ------------------------------------------------------------ activation producer
    // Gathered (act_gather): the tile's rows are token rows of x, four per
    // gather copy; lane l copies row groups l and l + 32 (rows 4g .. 4g+3)
    // of the tile's n_mma rows, rows past the tile repeating its last pair.
    // Pair-sorted: the rows are consecutive, one box of n_mma_max rows per
    // k-step (rows past the tile are never read back by the epilogue).
    if (lane == 0) tma_prefetch_desc(&tm_xs);
    Pipe act;
    long long act_issued = 0;
    bool ok = true;
    Walk w = walk0;
    Segment sg;
    while (ok && walk_next(w, n_ss, num_tiles, rb_group, sg)) {
      const Tile tl = read_tile(p, sg.tile);
      if (!tl.ok) continue;
      const int ks0 = sg.ss0 * kSSSteps, ks1 = min(ksteps, sg.ss1 * kSSSteps);
      const int n_mma = (tl.rows + 15) & ~15;
      int tok[2][4];   // gathered: x rows of this lane's two row groups
      if (p.act_gather) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int row = min(4 * (lane + 32 * j) + r, tl.rows - 1);
            const int pair = __ldg(p.sorted_pairs + tl.slot0 + row);
            // a pair id out of range is reported by the epilogue, which
            // discards its column; copy a valid row in its place
            tok[j][r] = (pair >= 0 && pair < p.P) ? pair / p.top_k : 0;
          }
        }
      } else if (lane == 0) {
        // Activations of a tile are read by several CTAs at different times
        // and may have left L2: ask for them kActPrefetch k-steps before the
        // copy into shared memory needs them.
        for (int j = ks0; j < min(ks1, ks0 + kActPrefetch); ++j) tma_prefetch_l2_2d(&tm_xs, j * kKStep, tl.slot0);
      }
      const uint32_t act_tx = static_cast<uint32_t>(p.act_gather ? n_mma : p.n_mma_max) * kActRowBytes;
      for (int ks = ks0; ks < ks1; ++ks) {
        if (!mbar_wait(bar_actempty + 8 * act.stage, act.phase ^ 1u, abort_flag, p.err,
                       kWhereGroupedProducer)) {
          ok = false;
          break;
        }
        const uint32_t full = bar_actfull + 8 * act.stage;
        const uint32_t dst = act0 + static_cast<uint32_t>(act.stage * p.n_mma_max * kActRowBytes);
        if (lane == 0) mbar_arrive_expect_tx(full, act_tx);
        if (p.act_gather) {
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int g = lane + 32 * j;
            if (4 * g < n_mma)
              tma_gather4_2d(dst + static_cast<uint32_t>(g * 4 * kActRowBytes), &tm_xs, ks * kKStep, tok[j][0],
                             tok[j][1], tok[j][2], tok[j][3], full);
          }
        } else if (lane == 0) {
          tma_load_2d(dst, &tm_xs, ks * kKStep, tl.slot0, full);
          if (ks + kActPrefetch < ks1) tma_prefetch_l2_2d(&tm_xs, (ks + kActPrefetch) * kKStep, tl.slot0);
        }
        ++act_issued;
        act.advance(SA);
      }
    }
    __syncwarp();
    drain_ring(bar_actfull, act, SA, act_issued, p.err);
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    Pipe act, apipe, accp;
    AccSlots slots;
    Pipe& wpipe = apipe;   // kDense: the A ring is the packed-byte ring
    bool ok = true;
    Walk w = walk0;
    Segment sg;
    while (ok && walk_next(w, n_ss, num_tiles, rb_group, sg)) {
      const Tile tl = read_tile(p, sg.tile);
      if (!tl.ok) continue;
      const uint32_t n_mma = static_cast<uint32_t>((tl.rows + 15) & ~15);
      const uint32_t idesc = idesc_bf16_f32(kBlockRows, n_mma);
      uint32_t d_tmem;
      int acc_bar;   // the full barrier this unit's commit arrives on
      if (p.acc_slots) {
        const int first = slots.first(n_mma);
        const int last = AccSlots::big(n_mma) ? 1 : first;
        for (int k = first; k <= last && ok; ++k) {
          if (!mbar_wait(bar_accempty + 8 * k, ((slots.empty_ph >> k) & 1u) ^ 1u, abort_flag, p.err,
                         kWhereGroupedMma))
            ok = false;
          slots.empty_ph ^= 1u << k;
        }
        if (!ok) break;
        d_tmem = tmem_base + static_cast<uint32_t>(128 * first);
        acc_bar = first;
        slots.step(n_mma);
      } else {
        if (!mbar_wait(bar_accempty + 8 * accp.stage, accp.phase ^ 1u, abort_flag, p.err, kWhereGroupedMma)) {
          ok = false;
          break;
        }
        d_tmem = tmem_base + static_cast<uint32_t>(accp.stage * p.n_mma_max);
        acc_bar = accp.stage;
        accp.advance(p.nacc);
      }
      tc_fence_after();
      const int ks0 = sg.ss0 * kSSSteps, ks1 = min(ksteps, sg.ss1 * kSSSteps);
      for (int ks = ks0; ks < ks1; ++ks) {
        const uint32_t bar_wfull = kDense ? bar_pkfull : bar_afull;
        if (!mbar_wait(bar_actfull + 8 * act.stage, act.phase, abort_flag, p.err, kWhereGroupedMma) ||
            !mbar_wait(bar_wfull + 8 * wpipe.stage, wpipe.phase, abort_flag, p.err, kWhereGroupedMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t b_smem = act0 + static_cast<uint32_t>(act.stage * p.n_mma_max * kActRowBytes);
          if constexpr (kDense) {
            const uint32_t a_smem = pk0 + wpipe.stage * kPkStageBytes;
#pragma unroll
            for (int kk = 0; kk < kKStep / 16; ++kk) {
              mma_bf16_ss(d_tmem, smem_desc_sw128(a_smem + kk * 32), smem_desc_sw128(b_smem + kk * 32), idesc,
                          (ks != ks0 || kk != 0) ? 1u : 0u);
            }
            mma_commit(bar_actempty + 8 * act.stage);
            mma_commit(bar_pkempty + 8 * wpipe.stage);
          } else {
            const uint32_t a_tmem = tmem_base + acol0 + static_cast<uint32_t>(apipe.stage * kATmemCols);
#pragma unroll
            for (int kk = 0; kk < kKStep / 16; ++kk) {
              mma_bf16_ts(d_tmem, a_tmem + kk * 8, smem_desc_sw128(b_smem + kk * 32), idesc,
                          (ks != ks0 || kk != 0) ? 1u : 0u);
            }
            mma_commit(bar_actempty + 8 * act.stage);
            if (SA != kNumAStages) mma_commit(bar_aempty + 8 * apipe.stage);
          }
        }
        __syncwarp();
        act.advance(SA);
        wpipe.advance(kDense ? SP : kNumAStages);
      }
      if (!ok) break;
      if (lane == 0) mma_commit(bar_accfull + 8 * acc_bar);
      __syncwarp();
    }
    // Drain: every MMA issued by this warp has completed before teardown.
    if (lane == 0) {
      mma_commit(bar_drain);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar_drain, 0)) {
        if (globaltimer() - t0 > kWaitTimeoutNs) {
          record_error(p.err, TQ_ERR_DEVICE_TIMEOUT, kWhereGroupedTeardown);
          break;
        }
      }
    }
    __syncwarp();
  } else if (warp < Roles<kEpi>::dec0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int eh = (warp - kWarpEpi0) >> 2;   // with 8 epilogue warps: which half of the columns
    Pipe accp;
    AccSlots slots;
    Walk w = walk0;
    Segment sg;
    while (walk_next(w, n_ss, num_tiles, rb_group, sg)) {
      const Tile tl = read_tile(p, sg.tile);
      if (!tl.ok) continue;
      const int slot0 = tl.slot0, rows = tl.rows;
      const uint32_t n_mma = static_cast<uint32_t>((rows + 15) & ~15);
      const bool two_slots = p.acc_slots && AccSlots::big(n_mma);
      // the 32-column blocks this warp drains: all (4 warps); with 8, one slot
      // each for a unit spanning both slots, else alternate blocks
      auto mine = [&](int b) { return kEpi == 4 || (two_slots ? (b >> 2) == eh : (b & 1) == eh); };
      // Output row and weight of every column of the tile, loaded while the
      // MMAs run: lane j holds columns j + 32i (i < 8; tile_m <= 256), and the
      // drain below takes them by shuffle.  -1 = no output (past the tile, or
      // a pair id out of range, which is reported).
      int orow[8];
      float owt[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int col = lane + 32 * i;
        orow[i] = -1;
        owt[i] = 0.f;
        if (col < rows && mine(i)) {
          if (p.pair_out) {
            orow[i] = slot0 + col;
            owt[i] = 1.f;
          } else {
            const int pair = __ldg(p.sorted_pairs + slot0 + col);
            if (pair < 0 || pair >= p.P) {
              record_error(p.err, TQ_ERR_INVALID_ARG, kWhereGroupedEpilogue);
            } else {
              orow[i] = pair / p.top_k;
              owt[i] = __ldg(p.topk_w + pair);
            }
          }
        }
      }
      int acc_first, acc_done;   // full barrier to wait on; empty barrier to arrive on at the end
      uint32_t acc_ph;
      if (p.acc_slots) {
        acc_first = slots.first(n_mma);
        acc_ph = (slots.full_ph >> acc_first) & 1u;
        slots.full_ph ^= 1u << acc_first;
        acc_done = two_slots ? 1 : acc_first;
        slots.step(n_mma);
      } else {
        acc_first = acc_done = accp.stage;
        acc_ph = accp.phase;
        accp.advance(p.nacc);
      }
      if (!mbar_wait(bar_accfull + 8 * acc_first, acc_ph, abort_flag, p.err, kWhereGroupedEpilogue)) break;
      tc_fence_after();
      if (kEpi == 8 && two_slots && eh == 1) {
        // this half reads only the second slot: the first is free as far as it goes
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_accempty);
      }
      const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(p.acc_slots ? 128 * acc_first : acc_first * p.n_mma_max);
      // Each 4x4 block (4 lanes = 4 consecutive rows, 4 pair columns) is
      // transposed by shuffles so that a lane holds 4 consecutive rows of one
      // pair and adds them with one 16-byte vector reduction.
      const int qa = lane >> 2, qb = lane & 3;
      float* const yrow = p.y32 + static_cast<size_t>(sg.rb) * kBlockRows + 32 * q + 4 * qa;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if (32 * b >= rows) break;
        if (!mine(b)) continue;
        // both 16-column halves of the block in flight before one wait
        uint32_t v2[2][16];
        tmem_ld16(t_acc + 32 * b, v2[0]);
        if (32 * b + 16 < rows) tmem_ld16(t_acc + 32 * b + 16, v2[1]);
        tmem_wait_ld();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int c0 = 32 * b + 16 * hf;
          if (c0 >= rows) break;
          const uint32_t (&v)[16] = v2[hf];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (c0 + 4 * k >= rows) break;
            float x0 = __uint_as_float(v[4 * k]), x1 = __uint_as_float(v[4 * k + 1]);
            float x2 = __uint_as_float(v[4 * k + 2]), x3 = __uint_as_float(v[4 * k + 3]);
            float t = __shfl_xor_sync(0xffffffffu, (qb & 1) ? x0 : x1, 1);
            if (qb & 1) x0 = t; else x1 = t;
            t = __shfl_xor_sync(0xffffffffu, (qb & 1) ? x2 : x3, 1);
            if (qb & 1) x2 = t; else x3 = t;
            t = __shfl_xor_sync(0xffffffffu, (qb & 2) ? x0 : x2, 2);
            if (qb & 2) x0 = t; else x2 = t;
            t = __shfl_xor_sync(0xffffffffu, (qb & 2) ? x1 : x3, 2);
            if (qb & 2) x1 = t; else x3 = t;
            const int src = (c0 & 31) + 4 * k + qb;   // lane holding this column's metadata
            const int out_row = __shfl_sync(0xffffffffu, orow[b], src);
            const float wt = __shfl_sync(0xffffffffu, owt[b], src);
            if (out_row >= 0) {
              float* dst = yrow + static_cast<size_t>(out_row) * p.N;
              if (p.store_out)
                asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(x0 * wt), "f"(x1 * wt),
                             "f"(x2 * wt), "f"(x3 * wt)
                             : "memory");
              else
                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(x0 * wt),
                             "f"(x1 * wt), "f"(x2 * wt), "f"(x3 * wt)
                             : "memory");
            }
          }
        }
        if (two_slots && b == 3) {
          // the first 128 columns are read: slot 0 is free for the next unit
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_accempty);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_accempty + 8 * acc_done);
    }
  } else if constexpr (!kDense) {
    // ------------------------------------------------------------ decode
    const int dw = warp - Roles<kEpi>::dec0;
    const int q = warp & 3;
    const int h = dw >> 2;
    const uint32_t row = static_cast<uint32_t>(32 * q + lane);
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acol0 +
                            static_cast<uint32_t>(16 * h);
    const size_t row_bytes = static_cast<size_t>(p.K / 4);
    Pipe pk, apipe;
    int pending_afull = -1;   // A stage stored but not yet handed to the MMA
    bool ok = true;
    Walk w = walk0;
    Segment sg;
    while (ok && walk_next(w, n_ss, num_tiles, rb_group, sg)) {
      const Tile tl = read_tile(p, sg.tile);
      if (!tl.ok) continue;
      // 4 stream bytes before the first symbol of the segment (zero at the
      // row start): symbols of the window that lie in an earlier super-stage.
      uint32_t carry = 0;
      if (h == 0 && sg.ss0 > 0) {
        const uint8_t* rp = p.packed + (static_cast<size_t>(tl.e) * p.N + sg.rb * kBlockRows + row) * row_bytes;
        carry = __ldg(reinterpret_cast<const uint32_t*>(rp + sg.ss0 * kSSBytes - 4));
      }
      for (int ss = sg.ss0; ss < sg.ss1 && ok; ++ss) {
        if (!mbar_wait(bar_pkfull + 8 * pk.stage, pk.phase, abort_flag, p.err, kWhereGroupedDecode)) {
          ok = false;
          break;
        }
        const uint32_t buf = pk0 + pk.stage * kPkStageBytes;
        const int nks = min(kSSSteps, ksteps - ss * kSSSteps);
        // k-step i's 16 stream bytes per row (one conflict-free 16-byte load,
        // one k-step ahead): half h decodes bytes [8h, 8h + 8); the 4 bytes
        // before them are bytes 4..7 of the same chunk (h = 1) or bytes
        // 12..15 of the previous chunk (h = 0; `carry` before a super-stage).
        uint4 chunk_n = lds_u128(buf + sw128(row, 0));
        uint32_t last = carry;
        for (int i = 0; i < nks && ok; ++i) {
          const uint4 chunk = chunk_n;
          const uint64_t cur = h ? (static_cast<uint64_t>(chunk.w) << 32 | chunk.z)
                                 : (static_cast<uint64_t>(chunk.y) << 32 | chunk.x);
          const uint32_t prev = h ? chunk.y : last;
          last = chunk.w;
          // issue this k-step's LUT loads first, then the next k-step's packed words
          uint32_t w[16];
          lookup_run<L>(lut_s, prev, cur, w);
          if (i + 1 < nks) chunk_n = lds_u128(buf + sw128(row, 16 * (i + 1)));
          // while the loads are in flight: hand the previous k-step's weights to the MMA
          if (pending_afull >= 0) {
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_afull + 8 * pending_afull);
            pending_afull = -1;
          }
          if (!mbar_wait(bar_arel + 8 * apipe.stage, apipe.phase ^ 1u, abort_flag, p.err, kWhereGroupedDecode)) {
            ok = false;
            break;
          }
          tc_fence_after();
          tmem_st16(t_lane + static_cast<uint32_t>(apipe.stage * kATmemCols), w);
          pending_afull = apipe.stage;
          apipe.advance(kNumAStages);
        }
        carry = last;   // bytes 124..127 of this super-stage, the next one's history
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pkempty + 8 * pk.stage);
        pk.advance(SP);
      }
    }
    if (pending_afull >= 0) {
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_afull + 8 * pending_afull);
    }
  }

  pdl_trigger();   // the next kernel (the combine) may launch while this grid tears down
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpProducer) {
    tc_fence_after();
    tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
  }
}

template <int L>
void* kernel_ptr(bool epi8) {
  return epi8 ? reinterpret_cast<void*>(&grouped_kernel<L, false, 8>)
              : reinterpret_cast<void*>(&grouped_kernel<L, false, 4>);
}

void* grouped_kernel_for(int L, bool epi8) {
  switch (L) {
    case 2: return kernel_ptr<2>(epi8);
    case 4: return kernel_ptr<4>(epi8);
    case 6: return kernel_ptr<6>(epi8);
    case 8: return kernel_ptr<8>(epi8);
    case 10: return kernel_ptr<10>(epi8);
    case 12: return kernel_ptr<12>(epi8);
    case 14: return kernel_ptr<14>(epi8);
    case 16: return kernel_ptr<16>(epi8);
    default: return nullptr;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

int launch_grouped(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L,
                   const int32_t* sorted_pairs, const float* topk_w, const int32_t* tiles,
                   const int32_t* num_tiles, int64_t cap, int64_t n, int top_k, int E, int K, int N,
                   int tile_m, float* y32, int* err, cudaStream_t s, int pair_out, const uint16_t* dense_w,
                   bool pdl, bool store_out, bool x_pair_sorted) {
  auto encode = encode_fn();
  if (!encode) return TQ_ERR_CUDA;
  const bool dense = dense_w != nullptr;
  if (!dense && !grouped_kernel_for(L, false)) return TQ_ERR_INVALID_ARG;

  Params p{};
  p.sorted_pairs = sorted_pairs;
  p.topk_w = topk_w;
  p.tiles = tiles;
  p.num_tiles = num_tiles;
  p.lut = lut;
  p.packed = packed;
  p.y32 = y32;
  p.err = err;
  p.cap = cap;
  p.P = static_cast<int>(n * top_k);
  p.E = E;
  p.tile_m = tile_m;
  p.top_k = top_k;
  p.N = N;
  p.K = K;
  p.row_blocks = N / kBlockRows;
  // Order by row-block groups only when the fp32 output is too large to stay
  // in L2 while six scattered partial sums per element arrive.
  p.pair_out = pair_out;
  p.early_prologue = pdl ? 1 : 0;
  p.act_gather = x_pair_sorted ? 0 : 1;
  // Per-pair outputs written once each: whole units (never split between
  // CTAs) and plain stores, so the caller need not clear the output first.
  p.store_out = (store_out && pair_out) ? 1 : 0;
  p.rb_group = p.row_blocks;
  const long long out_rows = pair_out ? n * static_cast<long long>(top_k) : n;
  if (out_rows * N * 4 > (24ll << 20)) {
    // The largest group of row blocks whose slice of the fp32 output (which the
    // CTAs running together add into) stays within 64 MiB of L2: fewer groups
    // mean fewer passes over the tiles' activations (each group reads them
    // once from DRAM).  At least one row block; a divisor of row_blocks.
    // Plain stores (store_out) write each output once and need no slice in
    // L2: one group.
    const long long slice_per_rb = out_rows * kBlockRows * 4;
    p.rb_group = 1;
    for (int g = p.row_blocks; g >= 1; --g) {
      if (p.row_blocks % g == 0 && (slice_per_rb * g <= (64ll << 20) || (store_out && pair_out))) {
        p.rb_group = g;
        break;
      }
    }
    p.allow_interleave = 1;
  }
  p.n_mma_max = (tile_m + 15) & ~15;
  const int a_cols = dense ? 0 : kNumAStages * kATmemCols;   // decoded A stages in tensor memory
  p.nacc = (2 * p.n_mma_max + a_cols <= 512) ? 2 : 1;
  // m-tiles above 128 pairs beside the 8 A stages: two 128-column slots
  p.acc_slots = (!dense && p.nacc == 1) ? 1 : 0;
  p.acol0 = p.acc_slots ? 256 : p.nacc * p.n_mma_max;
  // units above 128 pairs (both accumulator slots): eight epilogue warps
  const bool epi8 = !dense && p.acc_slots;
  void* kfn = dense ? reinterpret_cast<void*>(&grouped_kernel<2, true, 4>) : grouped_kernel_for(L, epi8);
  const int threads = epi8 ? Roles<8>::threads : Roles<4>::threads;
  const int cols_needed = p.acol0 + a_cols;
  int cols = 32;
  while (cols < cols_needed) cols <<= 1;
  p.tmem_cols = cols;

  // Shared memory: activation stages, packed super-stages, LUT, barriers.
  // Prefer 3 packed buffers and up to 8 activation stages; shrink to fit.
  const uint32_t act_stage = static_cast<uint32_t>(p.n_mma_max * kActRowBytes);
  const uint32_t lut_bytes = dense ? 16u : std::max<uint32_t>(16u, 2u << L);
  const uint32_t bar_bytes = 8 * kNumBars + 16;
  auto total_for = [&](int sp, int sa) {
    return 1024u + sa * act_stage + sp * kPkStageBytes + lut_bytes + bar_bytes;
  };
  int SP = 0, SA = 0;
  for (int sp = kMaxPkStages; sp >= 2 && SP == 0; --sp) {
    for (int sa = kMaxActStages; sa >= 2; --sa) {
      if (total_for(sp, sa) <= static_cast<uint32_t>(kSmemLimit)) {
        SP = sp;
        SA = sa;
        break;
      }
    }
  }
  if (SP == 0) return TQ_ERR_INVALID_ARG;
  p.pk_stages = SP;
  p.act_stages = SA;
  p.off_pk = SA * act_stage;
  p.off_lut = p.off_pk + SP * kPkStageBytes;
  p.off_bar = (p.off_lut + lut_bytes + 15u) & ~15u;
  // Ask for more than half of the SM's shared memory so that exactly one CTA
  // (and one tensor-memory allocation) sits on each SM.
  const uint32_t smem = std::max<uint32_t>(total_for(SP, SA), 120u * 1024u);

  CUtensorMap tm_packed, tm_xs;
  if (dense) {
    // Materialized weights: bf16 [E*N][K], one 64 x 128 box per k-step.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(E) * N};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {kKStep, kBlockRows};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tm_packed, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(dense_w), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TQ_ERR_INVALID_ARG;
  } else {
    // Box wider than a short row (K/4 < 128) reads zeros past the row end.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 4), static_cast<cuuint64_t>(E) * N};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 4)};
    const cuuint32_t box[2] = {kSSBytes, kBlockRows};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tm_packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(packed), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TQ_ERR_INVALID_ARG;
  }
  {
    // Token rows [n][K] copied four rows at a time by gather (a box one row
    // high), or pair-sorted rows [P][K] one n_mma_max-row box per k-step.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(p.act_gather ? n : p.P)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {kKStep, p.act_gather ? 1u : static_cast<cuuint32_t>(p.n_mma_max)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tm_xs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TQ_ERR_INVALID_ARG;
  }

  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  const int n_ss = (K / kKStep + kSSSteps - 1) / kSSSteps;
  const long long work = cap * static_cast<long long>(p.row_blocks) * n_ss;
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(work, sm_count())));
  void* args[] = {&tm_packed, &tm_xs, &p};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // The kernel may start while the previous kernel on the stream finishes; it
  // waits for it (pdl_wait) at its start, or after its prologue when the
  // caller knows that kernel does not write the LUT (early_prologue).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelExC(&cfg, kfn, args) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_LAUNCH;
  }
  const int st = launch_status();
  if (st == TQ_OK) count_launch(kCntGrouped);
  return st;
}

}  // namespace tq
