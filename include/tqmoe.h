/*
 * tqmoe.h — C ABI of the trellis-quantized MoE grouped GEMM for GB300 (sm_103a).
 *
 * The routed-expert (MoE) product over expert weights stored as 2-bit
 * bitshift-trellis bitstreams, with the trellis decode fused into the multiply.
 *
 * Sources (pages; cited by title and section):
 *  [P1] "fix(qtip): gate the trellis grouped GEMM on m-tile occupancy, not token
 *       count" — "The cause is a threshold, not a kernel defect" (pairs sorted
 *       by expert, sum_e ceil(count_e / TILE_M) m-tiles, each woken expert's
 *       packed bytes staged once per m-tile; the tile-fill closed form), "The
 *       fix" (the amortization predicate), "Tests", post-merge note (the
 *       n <= 8 floor, the GEMV pin).
 *  [P2] "perf(qtip): arch-specialise the trellis grouped GEMM (D16) + close the
 *       silent-failure holes (D18)" — items 1 and 2 of the commit message
 *       (m-tile size; contiguous-run decode seeded by the window identity),
 *       "The two changes" (packed 2-bit bytes cross HBM, decode lands in a
 *       shared-memory tile, full-size weights never materialise), "D18" (every
 *       launcher returns a status, empty grids are errors, unsupported arch is
 *       refused), "The arch witness".
 *  [P3] "fix(ArcLab/ArcQuant): make prefill measurable, then ship the two
 *       kernels it proves were switched off" — launch counters prove which
 *       kernel ran; unknown environment values warn and keep the default.
 *
 * Data model (the pages leave the decode constants open; this library fixes):
 *  - Pair p = t * top_k + j is token t's j-th routed expert topk_ids[t][j].
 *  - Expert e's weight row r (0 <= r < N) is a bitstream of K 2-bit symbols in
 *    packed[e][r][0 .. K/4): symbol i is bits [2(i%4), 2(i%4)+2) of byte i/4.
 *  - The trellis state of symbol i is the L-bit window of the stream ending
 *    with symbol i (bits [2i+2-L, 2i+2), zeros before the row start), i.e.
 *    s_i = (s_{i-1} >> 2) | (c_i << (L-2)), s_{-1} = 0.  The weight is
 *    W_e[r][i] = lut[s_i], lut an fp16 table of 2^L entries.
 *  - Y[t][r] = sum_j topk_w[t][j] * sum_i W_{topk_ids[t][j]}[r][i] * x[t][i].
 *
 * Conventions for every call below:
 *  - Pointers marked (device) are device memory owned by the caller; no call
 *    allocates device memory or keeps a pointer after returning (the one fixed
 *    device array the library holds is described at tq_moe_forward_static).
 *  - Calls taking a stream enqueue work on it and return without waiting;
 *    they never synchronize the device.  The route, tile map, gather,
 *    grouped GEMM and combine kernels are launched as programmatic dependents
 *    of the previous kernel on the stream (they may start while it drains)
 *    and wait for it to finish before touching memory, so stream order holds
 *    as for ordinary launches.  (Inside tq_moe_forward and the grouped arm
 *    of tq_moe_mlp_forward, the first grouped kernel sets up its tensor
 *    memory and stages its LUT before that wait.  Its predecessor there is
 *    always one of this library's own launches, and neither writes the LUT:
 *    the fused route / tile-map launch when the kernel m-tile is at most
 *    TQ_GATHER_MAX_TILE_M, the activation gather above it.)  Status codes
 *    report argument and launch errors only; device-side faults of the data
 *    (an expert id out of range, a tile map over capacity, a wait that timed
 *    out) are recorded in a device error word read by tq_device_error().
 *  - Return value: TQ_OK (0) or a negative TQ_ERR_* code.  A failed call has
 *    launched nothing or reports the launch failure; outputs are then
 *    undefined and must not be read as results.
 *  - Layouts are row-major and dense.  bf16/fp16 values are passed as their
 *    16-bit patterns (uint16_t).
 */
#ifndef TQMOE_H
#define TQMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without the CUDA headers; NULL is the legacy default stream. */
typedef struct CUstream_st* tq_stream_t;

enum tq_status {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = -1,      /* null pointer, bad size or alignment          */
  TQ_ERR_UNSUPPORTED_ARCH = -2, /* device or binary lacks sm_103a device code    */
  TQ_ERR_CAPACITY = -3,         /* tile map larger than the caller's capacity    */
  TQ_ERR_LAUNCH = -4,           /* kernel launch failed (cudaGetLastError)       */
  TQ_ERR_CAPTURING = -5,        /* arch witness cannot be taken during capture   */
  TQ_ERR_DEVICE_TIMEOUT = -6,   /* a device-side wait gave up (device error word)*/
  TQ_ERR_CUDA = -7,             /* another CUDA runtime error                     */
  TQ_ERR_WORKSPACE = -8         /* workspace too small or misaligned             */
};

/* Human-readable name of a status code.  Never NULL. */
const char* tq_status_string(int status);

/* ---------------------------------------------------------------------------
 * Arch witness  ([P2] "The arch witness", D18 #12)
 *
 * Launches a one-thread kernel compiled under the same architecture guard as
 * the grouped GEMM and reads back the architecture the running binary carries.
 * Succeeds only if the device is compute capability 10.3 and the binary holds
 * sm_103a device code.  Only a successful answer is cached (per device); the
 * witness is not taken while the calling thread's legacy stream or the given
 * stream is capturing, in which case TQ_ERR_CAPTURING is returned and the
 * next call retries.  Every launcher below checks the cached witness first and
 * takes it if missing.  `device` is a CUDA ordinal; it becomes current.
 * arch_out (host, may be NULL) receives __CUDA_ARCH__ of the device code.
 * ------------------------------------------------------------------------- */
int tq_init(int device);
int tq_arch_witness(int device, int* arch_out);

/* ---------------------------------------------------------------------------
 * Tile fill and the amortization gate  ([P1] "The cause is a threshold",
 * "The fix", post-merge note).  Host-only closed forms in three scalars: safe
 * inside CUDA-graph capture.  All evaluated in fp64.
 * ------------------------------------------------------------------------- */

/* n*k / (E * (1 - (1 - k/E)^n)); 0 for n == 0; NaN on invalid arguments
 * (k < 1, k > E, n < 0). */
double tq_pairs_per_woken_expert(int64_t n, int top_k, int E);

/* 1 if pairs per woken expert >= tile_m (an average m-tile is full), 0 if
 * not or n == 0, TQ_ERR_INVALID_ARG if k < 1, k > E, tile_m < 1 or n < 0. */
int tq_tiles_amortize(int64_t n, int top_k, int E, int tile_m);

/* Smallest n with tq_tiles_amortize(n, ...) == 1 (683 for top-6 of 256 at
 * tile_m 16).  Negative TQ_ERR_INVALID_ARG on invalid arguments. */
int64_t tq_grouped_min_tokens(int top_k, int E, int tile_m);

/* Native m-tile size of the grouped kernel on sm_103a for a routing shape,
 * by the expected pairs per woken expert (ppw, tq_pairs_per_woken_expert):
 * 256 when ppw >= 128 (prefill sizes, where one decode per 256 pairs beats
 * one per 128); 16 when ppw <= 4 (almost no expert has more than 16 pairs,
 * so the m-tiles are the woken experts either way, and at 16 the kernel
 * gathers the token rows itself, saving the pair-sorted copy); else 128
 * (fewer m-tiles, hence fewer decodes, than 16 once experts share more
 * pairs).  Measured on GB300 at 32, 128, 512, 1024 and 8192 tokens of top-6
 * of 256.  The whole-product calls below take tile_m = TQ_TILE_NATIVE to use
 * it: their kernels then run with this tile while the arm selection keeps the
 * pages' TILE_M (TQ_GATE_TILE_M).  Negative on invalid arguments. */
#define TQ_TILE_NATIVE 0
#define TQ_GATE_TILE_M 16
/* Environment (read at each call):
 *   TQ_FORCE_ARM=auto|gemv|grouped|measured  replaces pin = TQ_ARM_AUTO in the
 *       whole-product calls (the pages' env pin of the GEMV arm).
 *   TQ_TILE_M=1..256  the kernel m-tile of whole-product calls made with
 *       tile_m = TQ_TILE_NATIVE (the arm selection keeps TQ_GATE_TILE_M).
 *   TQ_QUIET=1  no engagement log line.
 * An unrecognised value is ignored with one warning on stderr. */
int tq_native_tile_m(int64_t n, int top_k, int E);

/* Upper bound on the number of m-tiles sum_e ceil(count_e / tile_m) for ANY
 * routing of n*top_k pairs: min(P, floor(P / tile_m) + min(E, P)).  Size the
 * tile map with it.  Negative on invalid arguments. */
int64_t tq_tile_map_capacity(int64_t n, int top_k, int E, int tile_m);

/* Arm selection ([P1] post-merge note): TQ_ARM_GEMV when n <= 8 or the tiles
 * do not amortize, TQ_ARM_GROUPED otherwise; `pin` forces an arm.  Negative
 * on invalid arguments.
 * pin = TQ_ARM_MEASURED selects by the crossover measured on GB300 instead
 * ([P3] "Two things that were built, correct, and switched off": the tile-fill
 * gate does not reproduce): this library's grouped kernel decodes each woken
 * expert once per m-tile whatever the tile's fill, so it wins as soon as
 * experts are shared enough; the arms tie near 1.16 pairs per woken expert
 * (V4 up shape, n ~ 14) and the grouped arm is chosen from there on, with no
 * token floor.
 * tq_moe_forward reports TQ_ARM_GEMV or TQ_ARM_GROUPED as the arm used. */
enum tq_arm { TQ_ARM_AUTO = 0, TQ_ARM_GEMV = 1, TQ_ARM_GROUPED = 2, TQ_ARM_MEASURED = 3 };
#define TQ_DECODE_REGIME_MAX_TOKENS 8
#define TQ_MEASURED_CROSSOVER_PPW 1.16
int tq_select_arm(int64_t n, int top_k, int E, int tile_m, int pin);

/* ---------------------------------------------------------------------------
 * Routing sort  ([P1] "The cause is a threshold": the grouped GEMM sorts pairs
 * by expert)
 *
 * topk_ids    (device) int32 [n][top_k], expert ids in [0, E).
 * counts      (device) int32 [E]       out: pairs per expert.
 * offsets     (device) int32 [E + 1]   out: exclusive prefix sum of counts.
 * sorted_pairs(device) int32 [n*top_k] out: pair ids p ordered by expert,
 *             ascending p within an expert (a stable sort).
 * Limits: 1 <= top_k <= E <= 1024, 0 <= n*top_k < 2^31.  An expert id out of
 * range is skipped and sets TQ_ERR_INVALID_ARG in the device error word.
 * One thread block up to 8192 pairs; above that one block per 2048 pairs
 * (at most 64), each sorting a contiguous chunk after counting every pair
 * itself, so no block waits for another.  No scratch memory.
 * ------------------------------------------------------------------------- */
int tq_route(const int32_t* topk_ids, int64_t n, int top_k, int E,
             int32_t* counts, int32_t* offsets, int32_t* sorted_pairs,
             tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Device router: per token the top_k experts by fp32 logit (descending;
 * equal logits go to the lower expert id) and their weights, a softmax over
 * the picked logits computed in fp32.  The router GEMM that produces the
 * logits is not part of this library.  Page "The 794 ms decode step,
 * itemised", list of un-owned items: the router runs in fp32.
 *
 * logits   (device) fp32 [n][E]; non-finite values count as -infinity (a row
 *          with no finite logit gets equal weights).
 * topk_ids (device) int32 [n][top_k] out; topk_w (device) fp32 [n][top_k] out.
 * Limits: 1 <= top_k <= min(E, 32), E <= 1024.
 * tq_route_logits = tq_router_topk then tq_route on the ids it wrote.
 * ------------------------------------------------------------------------- */
int tq_router_topk(const float* logits, int64_t n, int E, int top_k,
                   int32_t* topk_ids, float* topk_w, tq_stream_t stream);
int tq_route_logits(const float* logits, int64_t n, int E, int top_k,
                    int32_t* topk_ids, float* topk_w,
                    int32_t* counts, int32_t* offsets, int32_t* sorted_pairs,
                    tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * m-tile map  ([P1] "The cause is a threshold"; [P2] D18: route and GEMM must
 * agree on tile_m)
 *
 * For experts e ascending with count_e > 0 and i < ceil(count_e / tile_m):
 *   tiles[t] = { e, offsets[e] + i*tile_m, min(tile_m, count_e - i*tile_m) }.
 * offsets   (device) int32 [E + 1] from tq_route.
 * tiles     (device) int32 [cap][3]  out.
 * num_tiles (device) int32 [1]       out: number of tiles written (<= cap).
 * cap: capacity of `tiles` in tiles, >= 1; tq_tile_map_capacity() is always
 * enough.  If the map would exceed cap, only cap tiles are written,
 * *num_tiles = cap and TQ_ERR_CAPACITY is set in the device error word.
 * 1 <= tile_m <= 256 (the grouped kernel's largest m-tile).
 * ------------------------------------------------------------------------- */
int tq_build_tile_map(const int32_t* offsets, int E, int tile_m,
                      int32_t* tiles, int32_t* num_tiles, int64_t cap,
                      tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Activation gather: x_sorted[s][:] = x[sorted_pairs[s] / top_k][:] for every
 * sorted slot s < n*top_k, so that the rows of an m-tile are consecutive
 * (TQ_X_PAIR_SORTED input of tq_grouped_gemm; tq_grouped_gemm_pairs input).
 * x (device) bf16 [n][K]; x_sorted (device) bf16 [n*top_k][K]; both 16-byte
 * aligned; K % 8 == 0.  A pair id out of range gives a zero row and sets
 * TQ_ERR_INVALID_ARG in the device error word.
 * ------------------------------------------------------------------------- */
int tq_gather_rows(const uint16_t* x, const int32_t* sorted_pairs, int64_t n, int top_k, int K,
                   uint16_t* x_sorted, tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Everything the grouped GEMM needs, in one launch: tq_route and
 * tq_build_tile_map fused (one block sorts; the tile map takes each expert's
 * slot range from the sort's registers) while the launch's other blocks
 * clear y32[0 .. y32_count) (the fp32 accumulator; 16-byte aligned and
 * y32_count % 4 == 0 for the fused clear, otherwise it is cleared by a
 * separate memset).  x_sorted may be NULL: when given, tq_gather_rows also
 * runs (a second launch; x is unused otherwise).  Results are those of the separate calls.  Arguments as in
 * tq_route, tq_build_tile_map and tq_gather_rows; y32 may be NULL when
 * y32_count == 0.
 * ------------------------------------------------------------------------- */
int tq_prepare(const int32_t* topk_ids, const uint16_t* x, int64_t n, int top_k, int E, int K, int tile_m,
               int32_t* counts, int32_t* offsets, int32_t* sorted_pairs, int32_t* tiles, int32_t* num_tiles,
               int64_t cap, uint16_t* x_sorted, float* y32, int64_t y32_count, tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Grouped GEMM  ([P1] m-tiles; [P2] contiguous-run decode, decode fused into
 * the multiply)
 *
 * For every m-tile and every 128-row block of N: TMA stages the expert's
 * packed rows once, warps decode runs of 32 symbols (seeded by the window
 * identity, then stepped) into a bf16 weight tile in tensor memory, TMA
 * copies the tile's activation rows into shared memory, tcgen05 MMAs
 * contract the two (fp32 accumulate), and the epilogue scales by the router
 * weight and adds into y32.
 *
 * x_layout   TQ_X_TOKENS: x (device) bf16 [n][K], the token activations; the
 *            kernel gathers row sorted_pairs[slot] / top_k of each m-tile
 *            slot, four rows per copy.  TQ_X_PAIR_SORTED: x (device) bf16
 *            [n*top_k][K] from tq_gather_rows (row = sorted slot), one box
 *            copy per m-tile and k-step.  Results are identical; the row
 *            gathers cost one copy per four pairs, so for m-tiles above
 *            TQ_GATHER_MAX_TILE_M the separate tq_gather_rows pass is faster
 *            (the whole-product calls choose by that rule).
 * x          16-byte aligned.
 * packed     (device) uint8 [E][N][K/4]; 16-byte aligned.
 * lut        (device) fp16 [2^L] (converted to bf16, nearest-even, on chip).
 * sorted_pairs, tiles, num_tiles: from tq_route / tq_build_tile_map with the
 *            same tile_m.  cap = capacity of `tiles`.
 * topk_w     (device) fp32 [n][top_k] router weights.
 * y32        (device) fp32 [n][N], 16-byte aligned: ACCUMULATED into (y32 += ...); zero it
 *            first for a plain product.  Additions are fp32 atomics, so the
 *            summation order (and the last bits) vary between runs.
 * Requires: K % 64 == 0, N % 128 == 0, L even in [2, 16], 1 <= tile_m <= 256,
 * 1 <= top_k <= E.  Device: compute capability 10.3.
 * ------------------------------------------------------------------------- */
#define TQ_X_TOKENS 0
#define TQ_X_PAIR_SORTED 1
#define TQ_GATHER_MAX_TILE_M 16
int tq_grouped_gemm(const uint16_t* x, int x_layout, const uint8_t* packed, const uint16_t* lut, int L,
                    const int32_t* sorted_pairs, const float* topk_w,
                    const int32_t* tiles, const int32_t* num_tiles, int64_t cap,
                    int64_t n, int top_k, int E, int K, int N, int tile_m,
                    float* y32, tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Per-pair GEMV arm  ([P1] "The regression": the per-pair gather GEMV; no
 * de-duplication of experts across pairs)
 *
 * For every pair p (token t = p / top_k, expert e = topk_ids[p]) and every
 * row r: y32[t][r] += topk_w[p] * sum_i W_e[r][i] * x[t][i], fp32 accumulate,
 * fp16 weights widened exactly.  Same layouts as tq_grouped_gemm; needs no
 * routing sort.  Requires K % 64 == 0, K <= 8192, L even in [2, 16].
 * ------------------------------------------------------------------------- */
int tq_gemv(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L,
            const int32_t* topk_ids, const float* topk_w,
            int64_t n, int top_k, int E, int K, int N,
            float* y32, tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Combine: y[i] = bf16(y32[i]), round to nearest even, for i < count.  The
 * stated numerics of the product: fp32 accumulation, bf16 output (the routed
 * outputs are summed per token in fp32 by the arms above; this call rounds
 * the sum once).  [P1] "The cause is a threshold": the grouped GEMM's output
 * is the per-token combined projection.
 * y32 (device) fp32 [count]; y (device) bf16 [count].
 * ------------------------------------------------------------------------- */
int tq_combine(const float* y32, uint16_t* y, int64_t count, tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Whole routed-expert product: arm selection (tq_select_arm with `pin`),
 * then on the grouped arm route + tile map (clearing the fp32 accumulator),
 * the grouped kernel and the combine to bf16 y [n][N]; on the GEMV arm one
 * launch that sums each token's top_k pairs in fp32 registers and writes
 * bf16 y [n][N] directly (the workspace is not touched).
 *
 * workspace (device): caller-owned scratch of at least
 *   tq_moe_workspace_size(n, top_k, E, K, N, tile_m) bytes, 256-byte aligned.
 *   It holds counts, offsets, sorted pairs, the tile map, the fp32
 *   accumulator and, for a kernel m-tile above TQ_GATHER_MAX_TILE_M, the
 *   pair-sorted activations and the sort's inverse (the sorted slot of each
 *   pair, written by the routing launch, through which the activations are
 *   copied in token order: each row of x read once); its contents are
 *   undefined after the call.
 * tile_m: 1..256, the m-tile of both the arm selection and the kernel, or
 *   TQ_TILE_NATIVE (tq_native_tile_m for the kernel, TQ_GATE_TILE_M for the
 *   selection).
 * arm_used (host, may be NULL): receives TQ_ARM_GEMV or TQ_ARM_GROUPED.
 * The first grouped engagement in a process logs the tile fill and the
 * amortization boundary to stderr once (unless TQ_QUIET=1).
 * ------------------------------------------------------------------------- */
size_t tq_moe_workspace_size(int64_t n, int top_k, int E, int K, int N, int tile_m);
int tq_moe_forward(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L,
                   const int32_t* topk_ids, const float* topk_w,
                   int64_t n, int top_k, int E, int K, int N, int tile_m, int pin,
                   void* workspace, size_t workspace_bytes,
                   uint16_t* y, int* arm_used, tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Whole routed-expert product without allocating: tq_moe_forward with its
 * scratch in a fixed device array inside the library instead of a caller
 * workspace.  The pages have no counterpart; this exists for callers that
 * cannot allocate device memory — e.g. a plugin to which a host framework
 * passes only input and output buffers, or a serving loop that forbids
 * allocation after start-up because cudaMalloc can block and synchronize.
 *
 * Arguments, layouts and results are those of tq_moe_forward minus the
 * workspace.  The scratch is a file-scope device array of
 * TQ_STATIC_SCRATCH_BYTES (16 MiB) that every GPU loading this library holds
 * until the process exits; a shape whose tq_moe_workspace_size() exceeds it
 * is rejected with TQ_ERR_WORKSPACE before anything is launched (at
 * K = 4096, N = 2048, top-6 that is n > 2040 tokens at tile_m 16, where the kernel gathers its own
 * rows, and n > 292 with larger m-tiles, which add the pair-sorted copy of x).  The call allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library routine).
 *
 * The first call on a device does one-time set-up there: it looks up the
 * array's device address with that device current (cudaGetSymbolAddress) and
 * caches it, and, unless tq_init(device) ran first, takes the arch witness
 * (which creates a private stream, launches one tiny kernel, synchronizes
 * that stream and destroys it) and looks up the driver's tensor-map encoder.
 * That first call can therefore stall the host; make it (or tq_init) at
 * start-up, before any stream capture.  Later calls only enqueue.  Every call on a device shares the one array and
 * it keeps the last call's contents (each call zeroes what must start at
 * zero): calls that overlap on the GPU — on different streams or threads —
 * race and corrupt each other's results; serialize them.
 * ------------------------------------------------------------------------- */
#define TQ_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
int tq_moe_forward_static(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L,
                          const int32_t* topk_ids, const float* topk_w,
                          int64_t n, int top_k, int E, int K, int N, int tile_m, int pin,
                          uint16_t* y, int* arm_used, tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * The whole expert MLP (SwiGLU experts).  The routed-expert grouped GEMM
 * above is one of an expert's three projections; these calls chain them:
 *   gate|up_p = W_gu,e x_t,  h_p = silu(gate_p) * up_p,
 *   y_t = sum_j w_tj W_down,e h_(t,j).
 * packed_gu (device) uint8 [E][2I][H/4]: rows 0..I-1 the gate, I..2I-1 the
 * up projection; packed_down (device) uint8 [E][H][I/4]; one LUT each
 * (fp16 [2^L]); the same L.
 *
 * tq_grouped_gemm_pairs: the grouped GEMM with per-pair outputs and no
 *   router weight: out32[slot][:] += W_e x_sorted[slot] for every sorted
 *   slot (out32 (device) fp32 [n*top_k][N], 16-byte aligned, zero it first).
 * tq_swiglu: h[s][i] = bf16(silu(g) * u), g = gate_up[s][i],
 *   u = gate_up[s][I + i]; gate_up (device) fp32 [P][2I], h (device) bf16
 *   [P][I]; I % 4 == 0.
 * tq_moe_mlp_forward: the arm chosen as in tq_moe_forward (tq_select_arm with
 *   `pin`, the gate's TILE_M from `tile_m`; arm_used (host, may be NULL)
 *   receives it).  Grouped arm: route + tile map, gate|up (per pair; token
 *   rows gathered in the kernel, or, above TQ_GATHER_MAX_TILE_M, copied into
 *   pair-sorted order in token order through the sort's inverse, as in
 *   tq_moe_forward), SwiGLU, down (combined per token with the router
 *   weights).  GEMV arm:
 *   gate|up by per-pair GEMVs, SwiGLU, down by per-pair GEMVs on h combined
 *   per token.  Output bf16 y [n][H].  H % 128 == 0, I % 64 == 0 (and
 *   H, I <= 8192 for the GEMV arm).  workspace (device) >=
 *   tq_moe_mlp_workspace_size(...) bytes, 256-byte aligned.
 * ------------------------------------------------------------------------- */
int tq_grouped_gemm_pairs(const uint16_t* x_sorted, const uint8_t* packed, const uint16_t* lut, int L,
                          const int32_t* sorted_pairs, const int32_t* tiles, const int32_t* num_tiles,
                          int64_t cap, int64_t n, int top_k, int E, int K, int N, int tile_m,
                          float* out32, tq_stream_t stream);
int tq_swiglu(const float* gate_up, int64_t P, int I, uint16_t* h, tq_stream_t stream);
size_t tq_moe_mlp_workspace_size(int64_t n, int top_k, int E, int H, int I, int tile_m);
int tq_moe_mlp_forward(const uint16_t* x, const uint8_t* packed_gu, const uint16_t* lut_gu,
                       const uint8_t* packed_down, const uint16_t* lut_down, int L,
                       const int32_t* topk_ids, const float* topk_w,
                       int64_t n, int top_k, int E, int H, int I, int tile_m, int pin,
                       void* workspace, size_t workspace_bytes, uint16_t* y, int* arm_used,
                       tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Dequantize-materialize comparator  ([P1] "Tests": the dequantize path that
 * dispatch falls through to outside the fused arms' ranges; [P2] "The two
 * changes": the fused design never materialises full-size weights).  These
 * calls build that path so it can be measured against the fused arms; the
 * selection of tq_select_arm never picks it.
 *
 * tq_dequantize: w_out[i] = bf16(W_{expert_ids[i]}) for i < m, each a dense
 *   row-major [N][K] matrix: the trellis decode of the bitstreams above and
 *   fp16 -> bf16 nearest-even, bit-identical to the values the fused kernels
 *   feed their MMAs.  expert_ids (device) int32 [m], or NULL for experts
 *   0..m-1 (then m <= E); an id < 0 leaves its slot untouched; an id >= E
 *   leaves it untouched and sets TQ_ERR_INVALID_ARG in the device error word.
 *   packed, lut, w_out (device) 16-byte aligned; K % 8 == 0; L even in
 *   [2, 16].  w_out holds m*N*K bf16 values (16 MiB per expert at
 *   4096 x 2048).
 * tq_grouped_gemm_dense: tq_grouped_gemm with dense bf16 weights
 *   w_dense (device) [E][N][K] (16-byte aligned) in place of packed + lut;
 *   same m-tiles, activation layouts (x, x_layout), MMA and epilogue
 *   (y32 += w * W_e x).
 * tq_moe_forward_dequant: zero y32, route, tile map, dequantize every
 *   expert with at least one pair into slot e of an [E][N][K] bf16 buffer in
 *   the workspace, tq_grouped_gemm_dense, combine to bf16 y [n][N].
 *   workspace (device) >= tq_moe_dequant_workspace_size(...) bytes (the
 *   tq_moe_workspace_size regions followed by E*N*K*2 bytes), 256-byte
 *   aligned.  Requires K % 64 == 0, N % 128 == 0, E <= 1024.
 * ------------------------------------------------------------------------- */
int tq_dequantize(const uint8_t* packed, const uint16_t* lut, int L, const int32_t* expert_ids, int m,
                  int E, int N, int K, uint16_t* w_out, tq_stream_t stream);
int tq_grouped_gemm_dense(const uint16_t* x, int x_layout, const uint16_t* w_dense, const int32_t* sorted_pairs,
                          const float* topk_w, const int32_t* tiles, const int32_t* num_tiles, int64_t cap,
                          int64_t n, int top_k, int E, int K, int N, int tile_m, float* y32,
                          tq_stream_t stream);
size_t tq_moe_dequant_workspace_size(int64_t n, int top_k, int E, int K, int N, int tile_m);
int tq_moe_forward_dequant(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, int L,
                           const int32_t* topk_ids, const float* topk_w,
                           int64_t n, int top_k, int E, int K, int N, int tile_m,
                           void* workspace, size_t workspace_bytes, uint16_t* y, tq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Diagnostics
 * ------------------------------------------------------------------------- */

/* Reads and clears the current device's error word (synchronizes the device).
 * *code (host) receives 0 or the first TQ_ERR_* recorded by a kernel since the
 * last read; *where (host, may be NULL) a kernel-specific location tag. */
int tq_device_error(int* code, int* where);

/* Rate of the resource that bounds the trellis decode: every SM loads the
 * 65536-entry fp16/bf16 `table` (device, 16-byte aligned) into shared memory
 * and its `warps_per_sm` (1..32) warps each perform iters x 16 random 16-bit
 * lookups in it.  cycles (device) [SM count] receives each SM's clock cycles
 * for the lookups; sink (device) [SM count x warps_per_sm x 32] receives one
 * word per thread so no load is dead.  Lookups per clock per SM =
 * warps_per_sm * 32 * iters * 16 / cycles. */
int tq_probe_lut_rate(const uint16_t* table, int warps_per_sm, int iters, uint32_t* sink,
                      unsigned long long* cycles, tq_stream_t stream);

/* The bounded device-side wait ([P2] "The two changes": a failed or stuck
 * launch must surface as an error, never as a silent result): launches one
 * kernel whose single thread waits, through the same bounded mbarrier wait the
 * pipelined kernels use, on a barrier that nothing arrives on, with a limit of
 * timeout_ns (1e3 .. 2e9).  The wait gives up, records TQ_ERR_DEVICE_TIMEOUT
 * (location tag 10) in the device error word and the kernel returns, leaving
 * the context usable.  out (device) int[2], 4-byte aligned: out[0] = 1 if the
 * wait completed (0 expected), out[1] = microseconds waited.  Returns
 * TQ_ERR_INVALID_ARG on a bad argument, else the launch status. */
int tq_probe_wait_timeout(int64_t timeout_ns, int* out, tq_stream_t stream);

/* Host-side counts of successful launches since process start, per kernel:
 * out[0] route, out[1] tile map, out[2] grouped GEMM (trellis or dense),
 * out[3] GEMV, out[4] combine, out[5] activation gather, out[6] router
 * top-k, out[7] dequantize, out[8] route and tile map fused in one launch
 * (clearing y32 in its other blocks), out[9] accumulator clear (the GEMV
 * arms), out[10] SwiGLU ([P3]: counters prove which arm ran). */
#define TQ_NUM_LAUNCH_COUNTERS 11
void tq_launch_counts(int64_t out[TQ_NUM_LAUNCH_COUNTERS]);

#ifdef __cplusplus
}
#endif
#endif /* TQMOE_H */
