"""Seeded synthetic inputs for the trellis-quantized MoE grouped GEMM.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no trellis decode, no routing sort, no GEMM).  Both the CPU
oracle and the CUDA library are fed from here, so that the two sides see the
same bytes.

What one problem holds (one projection of one MoE layer):

* ``x_bits``     uint16 [n, K]     activations, bf16 bit patterns, drawn N(0,1)
                                   in fp32 and rounded to bf16 (nearest-even).
* ``topk_ids``   int32  [n, k]     the router's expert choice per token, in
                                   descending score order (column 0 = best).
* ``topk_w``     float32[n, k]     router weights: softmax over the k selected
                                   scores.
* ``packed``     uint8  [E, N, K/4] 2-bit trellis bitstreams, uniform random
                                   bytes (trained weights are not available;
                                   a trained bitstream is also close to uniform).
* ``lut_bits``   uint16 [2^L]      fp16 bit patterns of the state-to-value table,
                                   drawn N(0, 1/K) and rounded to fp16.

Routing recipes:

* ``uniform``: per-token logits ~ N(0,1) over the E experts, top-k of the
  logits (ties to the lower expert id), weights = softmax of the k selected
  logits.  By symmetry every k-subset of experts is equally likely.
* ``zipf``: expert popularity p_e proportional to (e+1)^-s; each token draws k
  distinct experts without replacement with probability proportional to p_e
  (Gumbel-top-k on log p_e), weights = softmax of the selected perturbed scores.

Seeds: one ``SeedSequence`` per problem (``base_seed + config_index`` mixed with
the projection and layer ids), spawned into four independent PCG64 streams
(x, routing, packed, LUT).
"""
from __future__ import annotations

from dataclasses import dataclass, field
import numpy as np

BASE_SEED = 20261202


@dataclass(frozen=True)
class Shape:
    """One projection's shapes and routing recipe."""
    name: str
    E: int          # experts
    top_k: int      # experts per token
    n: int          # tokens
    K: int          # input features (symbols per bitstream row)
    N: int          # output features (bitstream rows per expert)
    L: int          # trellis window bits
    tile_m: int = 16
    routing: str = "uniform"   # "uniform" | "zipf"
    zipf_s: float = 1.1

    @property
    def pairs(self) -> int:
        return self.n * self.top_k


# The five workloads, by what they are.  Two-projection workloads list both.
WORKLOADS: dict[str, list[Shape]] = {
    # Tiny MoE: E=8, top-2, 16 tokens, 256 -> 128, L=12 (4096-entry LUT).
    "tiny_e8_k2_n16": [Shape("tiny_e8_k2_n16", 8, 2, 16, 256, 128, 12)],
    # DeepSeek-V4-shaped decode: 32 tokens x top-6 of 256, 4096 -> 2048, L=16.
    "v4_decode_n32": [Shape("v4_decode_n32", 256, 6, 32, 4096, 2048, 16)],
    # Same expert shapes at 128 tokens, up (4096->2048) and down (2048->4096).
    "v4_n128_up": [Shape("v4_n128_up", 256, 6, 128, 4096, 2048, 16)],
    "v4_n128_down": [Shape("v4_n128_down", 256, 6, 128, 2048, 4096, 16)],
    # Tile-fill boundary sweep (75% / 100% / 150% fill at TILE_M=16).
    "v4_fill_n512": [Shape("v4_fill_n512", 256, 6, 512, 4096, 2048, 16)],
    "v4_fill_n683": [Shape("v4_fill_n683", 256, 6, 683, 4096, 2048, 16)],
    "v4_fill_n1024": [Shape("v4_fill_n1024", 256, 6, 1024, 4096, 2048, 16)],
    # Prefill: 8192 tokens, Zipf(1.1) expert popularity, up and down.
    "v4_prefill_n8192_up": [Shape("v4_prefill_n8192_up", 256, 6, 8192, 4096, 2048, 16,
                                  routing="zipf")],
    "v4_prefill_n8192_down": [Shape("v4_prefill_n8192_down", 256, 6, 8192, 2048, 4096, 16,
                                    routing="zipf")],
    # The same prefill with the popularity ranks shuffled over the expert ids
    # (the heavy experts anywhere in id order); appended last so the others
    # keep their seeds.
    "v4_prefill_n8192_up_zipf_perm": [Shape("v4_prefill_n8192_up_zipf_perm", 256, 6, 8192, 4096, 2048, 16,
                                            routing="zipf_perm")],
}

# Stable numeric id per workload (enters the seed).
_WORKLOAD_ID = {name: i for i, name in enumerate(WORKLOADS)}


def shape(name: str) -> Shape:
    return WORKLOADS[name][0]


def _streams(seed_key: tuple[int, ...]) -> list[np.random.Generator]:
    ss = np.random.SeedSequence(list(seed_key))
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(4)]


def fp32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even); return bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def draw_x(rng: np.random.Generator, n: int, K: int) -> np.ndarray:
    return fp32_to_bf16_bits(rng.standard_normal((n, K), dtype=np.float32))


def draw_routing(rng: np.random.Generator, n: int, E: int, k: int, routing: str = "uniform",
                 zipf_s: float = 1.1) -> tuple[np.ndarray, np.ndarray]:
    """Return (topk_ids int32 [n,k], topk_w float32 [n,k])."""
    if routing == "uniform":
        scores = rng.standard_normal((n, E)).astype(np.float32).astype(np.float64)
    elif routing in ("zipf", "zipf_perm"):
        # popularity rank r (0 = most popular) has p ~ (r + 1)^-s; "zipf" gives
        # expert e rank e, "zipf_perm" a random bijection of experts to ranks
        rank = np.arange(E) if routing == "zipf" else rng.permutation(E)
        logp = -zipf_s * np.log(rank.astype(np.float64) + 1.0)
        scores = logp[None, :] + rng.gumbel(size=(n, E))
    else:
        raise ValueError(f"unknown routing {routing!r}")
    # descending score, ties to the lower expert id (stable sort of -score)
    order = np.argsort(-scores, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(scores, order, axis=1)
    z = np.exp(sel - sel.max(axis=1, keepdims=True))
    w = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return order.astype(np.int32), w


def draw_packed(rng: np.random.Generator, E: int, N: int, K: int) -> np.ndarray:
    if K % 4:
        raise ValueError("K must be a multiple of 4 (four 2-bit symbols per byte)")
    nbytes = E * N * (K // 4)
    return np.frombuffer(rng.bytes(nbytes), dtype=np.uint8).reshape(E, N, K // 4)


def draw_lut(rng: np.random.Generator, L: int, K: int) -> np.ndarray:
    v = rng.standard_normal(1 << L) / np.sqrt(K)
    return v.astype(np.float16).view(np.uint16)


@dataclass
class Problem:
    shape: Shape
    x_bits: np.ndarray
    topk_ids: np.ndarray
    topk_w: np.ndarray
    packed: np.ndarray
    lut_bits: np.ndarray
    seed_key: tuple = field(default=())


def make_problem(name: str, layer: int = 0, n: int | None = None,
                 with_packed: bool = True) -> Problem:
    """Draw the named workload.  ``layer`` selects an independent weight set
    (same shapes, different bitstreams/LUT/activations/routing); ``n`` overrides
    the token count (sweeps)."""
    shp = shape(name)
    if n is not None:
        shp = Shape(**{**shp.__dict__, "n": n})
    key = (BASE_SEED + _WORKLOAD_ID[name], layer, shp.n)
    rx, rr, rp, rl = _streams(key)
    x = draw_x(rx, shp.n, shp.K)
    ids, w = draw_routing(rr, shp.n, shp.E, shp.top_k, shp.routing, shp.zipf_s)
    packed = draw_packed(rp, shp.E, shp.N, shp.K) if with_packed else None
    lut = draw_lut(rl, shp.L, shp.K)
    return Problem(shp, x, ids, w, packed, lut, key)


def make_custom(E: int, top_k: int, n: int, K: int, N: int, L: int, seed: int,
                routing: str = "uniform") -> Problem:
    """Small ad-hoc problem for edge-case tests."""
    rx, rr, rp, rl = _streams((BASE_SEED, 999, seed, E, top_k, n, K, N, L))
    shp = Shape(f"custom_{seed}", E, top_k, n, K, N, L, routing=routing)
    x = draw_x(rx, n, K)
    ids, w = draw_routing(rr, n, E, top_k, routing)
    return Problem(shp, x, ids, w, draw_packed(rp, E, N, K), draw_lut(rl, L, K),
                   (seed,))


# ---------------------------------------------------------------------------
# Whole expert MLP: y = sum_j w_j * W_down,e (silu(W_gate,e x) * (W_up,e x)).
# The gate and up matrices of an expert are stored as one [2I, H] bitstream
# block (rows 0..I-1 gate, I..2I-1 up), the down matrix as [H, I].
# ---------------------------------------------------------------------------

@dataclass
class MLPProblem:
    name: str
    E: int
    top_k: int
    n: int
    H: int          # hidden size (gate/up input, down output)
    I: int          # expert intermediate size
    L: int
    x_bits: np.ndarray
    topk_ids: np.ndarray
    topk_w: np.ndarray
    packed_gu: np.ndarray      # uint8 [E, 2I, H/4]
    lut_gu: np.ndarray         # fp16 bits [2^L], N(0, 1/H)
    packed_down: np.ndarray    # uint8 [E, H, I/4]
    lut_down: np.ndarray       # fp16 bits [2^L], N(0, 1/I)


MLP_WORKLOADS = {
    # name: (E, top_k, n, H, I, L, routing)
    "tiny_mlp_e8_k2_n16": (8, 2, 16, 256, 128, 12, "uniform"),
    "v4_mlp_n32": (256, 6, 32, 4096, 2048, 16, "uniform"),
    "v4_mlp_n128": (256, 6, 128, 4096, 2048, 16, "uniform"),
    "v4_mlp_prefill_n8192": (256, 6, 8192, 4096, 2048, 16, "zipf"),
    # one token (batch-1 decode), appended last so earlier workloads keep their seeds
    "v4_mlp_n1": (256, 6, 1, 4096, 2048, 16, "uniform"),
}


def make_mlp_custom(E: int, top_k: int, n: int, H: int, I: int, L: int, seed: int,
                    routing: str = "uniform") -> MLPProblem:
    """Small ad-hoc expert-MLP problem for edge-case tests."""
    ss = np.random.SeedSequence([BASE_SEED, 778, seed, E, top_k, n, H, I, L])
    rx, rr, rg, rlg, rd, rld = [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(6)]
    x = draw_x(rx, n, H)
    ids, w = draw_routing(rr, n, E, top_k, routing)
    return MLPProblem(f"mlp_custom_{seed}", E, top_k, n, H, I, L, x, ids, w,
                      draw_packed(rg, E, 2 * I, H), draw_lut(rlg, L, H),
                      draw_packed(rd, E, H, I), draw_lut(rld, L, I))


def make_mlp_problem(name: str, n: int | None = None, layer: int = 0) -> MLPProblem:
    E, k, n0, H, I, L, routing = MLP_WORKLOADS[name]
    n = n0 if n is None else n
    ss = np.random.SeedSequence([BASE_SEED, 777, list(MLP_WORKLOADS).index(name), layer, n])
    rx, rr, rg, rlg, rd, rld = [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(6)]
    x = draw_x(rx, n, H)
    ids, w = draw_routing(rr, n, E, k, routing)
    return MLPProblem(name, E, k, n, H, I, L, x, ids, w,
                      draw_packed(rg, E, 2 * I, H), draw_lut(rlg, L, H),
                      draw_packed(rd, E, H, I), draw_lut(rld, L, I))
