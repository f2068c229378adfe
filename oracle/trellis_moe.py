"""Plain CPU oracle for the routed-expert grouped GEMM over 2-bit bitshift-trellis
weights.  TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Everything here is numpy on the CPU, floating point in fp64.  Each function
states the passage it follows.  Page titles used in the citations:

* [P1] "fix(qtip): gate the trellis grouped GEMM on m-tile occupancy, not token
  count" — sections "The cause is a threshold, not a kernel defect" (tile-fill
  closed form and its table), "The fix" (the amortization predicate),
  "Tests" (flip-point tests), and the post-merge note (the n <= 8 floor).
* [P2] "perf(qtip): arch-specialise the trellis grouped GEMM (D16) + close the
  silent-failure holes (D18)" — commit message items 1 (m-tile) and 2
  (contiguous-run decode seeded by the window identity, runs independent of
  each other), and
  "The two changes" (packed 2-bit bytes cross HBM; decode fused into the
  multiply).

Readings where the pages leave a step open:

R1  Bitstream.  Each (expert e, output row r) owns one stream of K 2-bit
    symbols; symbol j is bits [2(j%4), 2(j%4)+2) of byte j//4 of the row
    (least significant first).
R2  Trellis state.  The state of symbol j is the L-bit window of the stream
    that ends with symbol j: s_j = sum_{i=0}^{L/2-1} c_{j-i} * 4^(L/2-1-i),
    with c_{j} = 0 for j < 0 (a zero warm-up region before the row).  The
    stepped form s_j = (s_{j-1} >> 2) | (c_j << (L-2)), s_{-1} = 0, gives the
    same value; [P2] seeds a run from the window and then steps.
R3  Value.  w = LUT[s_j], one fp16 table of 2^L entries per projection shared
    by all experts; the oracle widens fp16 exactly (the GPU path rounds it to
    bf16 for the tensor cores; that error is inside the output tolerance).
R4  Pairs.  Pair p = t * top_k + j for token t and its j-th routed expert.
    Routing sorts pairs by expert, stably (equal experts keep ascending p).
R5  Tile map.  For experts in ascending order with count_e > 0, tiles
    (e, offsets[e] + i*T, min(T, count_e - i*T)) for i < ceil(count_e / T)
    ([P1]: the kernel visits sum_e ceil(count_e / TILE_M) m-tiles).
R6  Output.  Y[t, r] = sum_j w[t,j] * sum_i W_{e(t,j)}[r, i] * x[t, i], x read
    exactly from bf16, w as fp32; the library then rounds to bf16.
R7  Gate.  tiles_amortize(n,k,E,T) := n > 0 and
    n*k / (E * (1 - (1 - k/E)^n)) >= T, evaluated in fp64 ([P1] "The fix").
    The dispatcher adds the n <= 8 floor ([P1] post-merge note).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "symbols", "states_window", "run_states", "lut_values", "decode_rows",
    "bf16_bits_to_f64", "route", "tile_map", "expected_woken_experts",
    "pairs_per_woken_expert", "tile_fill", "tiles_amortize", "grouped_min_tokens",
    "tile_map_capacity", "dispatch_arm", "moe_forward", "bf16_rne_bits", "router_topk",
    "silu", "moe_mlp",
    "DECODE_REGIME_MAX_TOKENS",
]

# [P1] "The cause is a threshold": the old gate was n_tokens > 8; the post-merge
# note keeps n <= 8 as a floor that always takes the per-pair GEMV.
DECODE_REGIME_MAX_TOKENS = 8


# ---------------------------------------------------------------------------
# Trellis decode  ([P2] item 2, "Contiguous-run decode"; readings R1-R3)
# ---------------------------------------------------------------------------

def symbols(packed_rows: np.ndarray) -> np.ndarray:
    """2-bit symbols c_j of each row (R1).  packed_rows: uint8 [..., K/4] ->
    int64 [..., K]."""
    b = np.asarray(packed_rows).astype(np.int64)
    parts = [(b >> (2 * q)) & 3 for q in range(4)]          # symbol 4*byte + q
    return np.stack(parts, axis=-1).reshape(*b.shape[:-1], b.shape[-1] * 4)


def states_window(c: np.ndarray, L: int) -> np.ndarray:
    """Window identity (R2): s_j = sum_{i<L/2} c_{j-i} 4^(L/2-1-i), c_{<0}=0."""
    if L % 2 or not 2 <= L <= 16:
        raise ValueError("L must be even and in [2, 16]")
    h = L // 2
    K = c.shape[-1]
    s = np.zeros_like(c)
    for i in range(min(h, K)):
        lagged = np.zeros_like(c)                           # lagged[..., j] = c[..., j-i]
        lagged[..., i:] = c[..., :K - i]
        s += lagged * (4 ** (h - 1 - i))
    return s


def run_states(c: np.ndarray, L: int, run_start: int, run_len: int) -> np.ndarray:
    """[P2] contiguous-run decode: seed the state of symbol ``run_start`` from
    the window identity, then step s <- (s >> 2) | (c << (L-2)) through the
    rest of the run.  Returns the run's states [..., run_len]."""
    seed = states_window(c[..., :run_start + 1], L)[..., run_start]
    out = np.empty(c.shape[:-1] + (run_len,), dtype=np.int64)
    s = seed
    out[..., 0] = s
    for m in range(1, run_len):
        s = (s >> 2) | (c[..., run_start + m] << (L - 2))
        out[..., m] = s
    return out


def lut_values(lut_bits: np.ndarray) -> np.ndarray:
    """fp16 table (bit patterns) -> exact fp64 values (R3)."""
    return np.asarray(lut_bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def decode_rows(packed_rows: np.ndarray, lut_bits: np.ndarray, L: int) -> np.ndarray:
    """Decoded weights W[r, j] = LUT[s_j(r)] in fp64 for the given rows
    (uint8 [R, K/4] -> float64 [R, K])."""
    lut = lut_values(lut_bits)
    if lut.shape[0] != (1 << L):
        raise ValueError("LUT must have 2^L entries")
    return lut[states_window(symbols(packed_rows), L)]


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 (bf16 is the top half of an fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Routing sort and tile map  ([P1] "The cause is a threshold"; R4, R5)
# ---------------------------------------------------------------------------

def route(topk_ids: np.ndarray, E: int):
    """Sort the (token, expert) pairs by expert (R4).

    Returns counts int32[E], offsets int32[E+1], sorted_pairs int32[P]."""
    flat = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    sorted_pairs = np.argsort(flat, kind="stable")
    return counts.astype(np.int32), offsets.astype(np.int32), sorted_pairs.astype(np.int32)


def tile_map(offsets: np.ndarray, tile_m: int) -> np.ndarray:
    """m-tiles (R5): int32 [num_tiles, 3] rows (expert, first sorted slot, rows)."""
    if tile_m < 1:
        raise ValueError("tile_m must be >= 1")
    tiles = []
    for e in range(len(offsets) - 1):
        start, count = int(offsets[e]), int(offsets[e + 1] - offsets[e])
        for i in range(-(-count // tile_m)):
            tiles.append((e, start + i * tile_m, min(tile_m, count - i * tile_m)))
    return np.asarray(tiles, dtype=np.int32).reshape(-1, 3)


# ---------------------------------------------------------------------------
# Tile fill and the amortization gate  ([P1] "The cause is a threshold",
# "The fix", "Tests"; R7)
# ---------------------------------------------------------------------------

def _check_shape(top_k: int, E: int, tile_m: int | None = None):
    if E < 1 or top_k < 1 or top_k > E:
        raise ValueError("need 1 <= top_k <= E")
    if tile_m is not None and tile_m < 1:
        raise ValueError("tile_m must be >= 1")


def expected_woken_experts(n: int, top_k: int, E: int) -> float:
    """E * (1 - (1 - k/E)^n): expected distinct experts under uniform routing."""
    _check_shape(top_k, E)
    return E * (1 - (1 - top_k / E) ** n)


def pairs_per_woken_expert(n: int, top_k: int, E: int) -> float:
    """[P1]: pairs per woken expert = n*k / (E * (1 - (1 - k/E)^n))."""
    _check_shape(top_k, E)
    if n <= 0:
        return 0.0
    return n * top_k / (E * (1 - (1 - top_k / E) ** n))


def tile_fill(n: int, top_k: int, E: int, tile_m: int) -> float:
    """[P1]: fill = pairs per woken expert / GROUPED_TILE_M."""
    return pairs_per_woken_expert(n, top_k, E) / tile_m


def tiles_amortize(n: int, top_k: int, E: int, tile_m: int) -> bool:
    """[P1] "The fix": grouped arm iff pairs per woken expert >= TILE_M."""
    _check_shape(top_k, E, tile_m)
    if n < 0:
        raise ValueError("n must be >= 0")
    return n > 0 and pairs_per_woken_expert(n, top_k, E) >= tile_m


def grouped_min_tokens(top_k: int, E: int, tile_m: int, limit: int = 1 << 26) -> int:
    """Smallest n with tiles_amortize true, by linear scan ([P1] "Tests":
    the reported boundary is the exact flip point).  -1 if none below limit."""
    _check_shape(top_k, E, tile_m)
    for n in range(1, limit):
        if tiles_amortize(n, top_k, E, tile_m):
            return n
    return -1


def tile_map_capacity(n: int, top_k: int, E: int, tile_m: int) -> int:
    """An upper bound on sum_e ceil(count_e / T) over every routing of n*k pairs:
    min(P, floor(P/T) + min(E, P))."""
    _check_shape(top_k, E, tile_m)
    P = n * top_k
    return min(P, P // tile_m + min(E, P))


def dispatch_arm(n: int, top_k: int, E: int, tile_m: int, pin: str = "auto") -> str:
    """[P1] post-merge note: n <= 8 or not amortized -> per-pair GEMV, else the
    grouped GEMM; ``pin`` forces an arm (the pages' A/B knob)."""
    if pin in ("gemv", "grouped"):
        return pin
    if pin != "auto":
        raise ValueError(f"unknown pin {pin!r}")
    if n <= DECODE_REGIME_MAX_TOKENS or not tiles_amortize(n, top_k, E, tile_m):
        return "gemv"
    return "grouped"


# ---------------------------------------------------------------------------
# Router top-k  (reading R13: each token's top_k experts by logit, weighted by
# a softmax over the picked logits; page "The 794 ms decode step, itemised",
# list of un-owned items, notes that the router runs in fp32)
# ---------------------------------------------------------------------------

def router_topk(logits: np.ndarray, top_k: int):
    """Per token: the top_k experts by logit, descending, ties to the lower
    expert id; weights = softmax over those top_k logits (fp64).  Non-finite
    logits count as -infinity; a row with no finite logit gets equal weights.
    logits float32 [n, E] -> (ids int32 [n, k], weights float64 [n, k])."""
    lg = np.asarray(logits, dtype=np.float32).astype(np.float64)
    lg = np.where(np.isnan(lg) | (lg == np.inf), -np.inf, lg)
    n, E = lg.shape
    if not 1 <= top_k <= E:
        raise ValueError("need 1 <= top_k <= E")
    order = np.lexsort((np.broadcast_to(np.arange(E), (n, E)), -lg), axis=1)[:, :top_k]
    sel = np.take_along_axis(lg, order, axis=1)
    top = sel[:, :1]
    with np.errstate(invalid="ignore"):
        z = np.where(np.isfinite(top), np.exp(sel - np.where(np.isfinite(top), top, 0.0)), 1.0)
    return order.astype(np.int32), z / z.sum(axis=1, keepdims=True)


# ---------------------------------------------------------------------------
# The MoE product  (R6)
# ---------------------------------------------------------------------------

def moe_forward(x_bits, topk_ids, topk_w, packed, lut_bits, L, rows=None):
    """Y[t, r] = sum_j w[t,j] sum_i W_{e(t,j)}[r,i] x[t,i] in fp64.

    ``rows`` restricts the output to those rows of every expert (sampled
    parity at full size); default all N rows.  Returns float64 [n, len(rows)].
    Experts are decoded one at a time (only those some token routes to); the
    per-expert product is a fp64 matmul.
    """
    x = bf16_bits_to_f64(x_bits)
    ids = np.asarray(topk_ids)
    w = np.asarray(topk_w, dtype=np.float32).astype(np.float64)
    n, k = ids.shape
    N = packed.shape[1]
    rows = np.arange(N) if rows is None else np.asarray(rows)
    Y = np.zeros((n, len(rows)), dtype=np.float64)
    for e in np.unique(ids):
        W = decode_rows(packed[e][rows], lut_bits, L)        # [R, K]
        t_idx, j_idx = np.nonzero(ids == e)
        partial = x[t_idx] @ W.T                              # [m, R]
        for m in range(len(t_idx)):
            Y[t_idx[m]] += w[t_idx[m], j_idx[m]] * partial[m]
    return Y


def bf16_rne_bits(y32: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16, nearest with ties to even (bit patterns).

    Written from the definition: of the two bf16 values that bracket y (the
    truncation and the next one away from zero), take the nearer; on a tie
    take the one with an even last mantissa bit."""
    y = np.ascontiguousarray(y32, dtype=np.float32)
    if not np.all(np.isfinite(y)):
        raise ValueError("finite inputs only")
    u = y.view(np.uint32)
    lo = (u >> 16).astype(np.uint32)                         # truncated toward zero
    hi = lo + 1                                              # next bf16 away from zero
    mag_lo = np.abs((lo << 16).astype(np.uint32).view(np.float32).astype(np.float64))
    expf = (lo >> 7) & 0xFF                                  # biased exponent of lo
    ulp = np.ldexp(1.0, np.maximum(expf, 1).astype(np.int64) - 127 - 7)
    mag_hi = mag_lo + ulp                                    # 2^128 past the largest finite
    mag = np.abs(y.astype(np.float64))
    dl, dh = mag - mag_lo, mag_hi - mag
    pick_hi = (dh < dl) | ((dh == dl) & ((lo & 1) == 1))
    return np.where(pick_hi, hi, lo).astype(np.uint16)


# ---------------------------------------------------------------------------
# The whole expert MLP  (reading R14: the routed-expert GEMM is one of three
# projections of a SwiGLU expert; gate and up share the input, down takes
# silu(gate) * up of the same pair)
# ---------------------------------------------------------------------------

def silu(v):
    """x * sigmoid(x) = x / (1 + e^-x)."""
    return v / (1.0 + np.exp(-v))


def moe_mlp(x_bits, topk_ids, topk_w, packed_gu, lut_gu, packed_down, lut_down, L, tokens=None):
    """Y[t] = sum_j w[t,j] * W_down,e (silu(W_gate,e x_t) * (W_up,e x_t)), fp64.

    packed_gu [E, 2I, H/4] holds each expert's gate rows (0..I-1) then up rows
    (I..2I-1); packed_down [E, H, I/4].  ``tokens`` restricts the output to
    those tokens (only their experts are decoded).  Returns [len(tokens), H]."""
    x = bf16_bits_to_f64(x_bits)
    ids = np.asarray(topk_ids)
    w = np.asarray(topk_w, dtype=np.float32).astype(np.float64)
    tokens = np.arange(ids.shape[0]) if tokens is None else np.asarray(tokens)
    I = packed_gu.shape[1] // 2
    H = packed_down.shape[1]
    Y = np.zeros((len(tokens), H), dtype=np.float64)
    sub = ids[tokens]
    for e in np.unique(sub):
        Wgu = decode_rows(packed_gu[e], lut_gu, L)            # [2I, H]
        Wd = decode_rows(packed_down[e], lut_down, L)         # [H, I]
        ti, ji = np.nonzero(sub == e)
        gu = x[tokens[ti]] @ Wgu.T                            # [m, 2I]
        h = silu(gu[:, :I]) * gu[:, I:]
        out = h @ Wd.T                                        # [m, H]
        for m in range(len(ti)):
            Y[ti[m]] += w[tokens[ti[m]], ji[m]] * out[m]
    return Y
