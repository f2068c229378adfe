"""Pins for the CPU oracle: checks of oracle.trellis_moe against facts that do
not come from the oracle itself — numbers printed on the pages (tests/golden),
closed forms, brute force written differently (big-integer bit slicing,
pure-Python loops with exact sums), and library routines (torch's bf16 cast).

Each pin is a plain function that raises AssertionError on a mismatch.  The
oracle module is looked up at call time (``T.<name>``) so that the mutation
tests can plant a mistake in one oracle function and check that some pin
catches it.
"""
from __future__ import annotations

import math
import os
import struct

import numpy as np

import oracle.trellis_moe as T
import moe_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split("\t"))
    return rows


# ---------------------------------------------------------------------------
# tile fill and gate
# ---------------------------------------------------------------------------

def pin_fill_table():
    """The pages' tile-fill table (top-6 of 256, TILE_M=16)."""
    rows = _golden_rows("tile_fill_v4.txt")
    assert len(rows) == 5
    for n, pairs, woken, ppe, fill in rows:
        n = int(n)
        assert n * 6 == int(pairs)
        assert f"{T.expected_woken_experts(n, 6, 256):.1f}" == woken, (n, woken)
        assert f"{T.pairs_per_woken_expert(n, 6, 256):.2f}" == ppe, (n, ppe)
        assert f"{100 * T.tile_fill(n, 6, 256, 16):.1f}" == fill, (n, fill)


def pin_gate_points():
    """Flip point, engagement line and selections printed on the pages."""
    for k, E, tm, n, fact, val in _golden_rows("gate_points.txt"):
        k, E, tm, n = int(k), int(E), int(tm), int(n)
        if fact == "pairs_per_woken_2dp":
            assert f"{T.pairs_per_woken_expert(n, k, E):.2f}" == val
        elif fact == "pairs_per_woken_1dp":
            assert f"{T.pairs_per_woken_expert(n, k, E):.1f}" == val
        elif fact == "fill_percent_int":
            assert f"{100 * T.tile_fill(n, k, E, tm):.0f}" == val
        elif fact == "min_tokens":
            assert T.grouped_min_tokens(k, E, tm) == int(val)
        elif fact == "amortize":
            assert T.tiles_amortize(n, k, E, tm) == bool(int(val)), (k, E, tm, n)
        elif fact == "dispatch":
            assert T.dispatch_arm(n, k, E, tm) == val
        else:
            raise AssertionError(f"unknown fact {fact}")
    # the pages' test: the grouped arm is not selected for 9 <= n <= 682, and is from 683 on
    assert not any(T.tiles_amortize(n, 6, 256, 16) for n in range(9, 683))
    assert all(T.tiles_amortize(n, 6, 256, 16) for n in range(683, 4000))
    assert all(T.dispatch_arm(n, 6, 256, 16) == "gemv" for n in range(0, 683))
    assert all(T.dispatch_arm(n, 6, 256, 16) == "grouped" for n in range(683, 1200))
    assert T.dispatch_arm(1, 6, 256, 16, pin="grouped") == "grouped"
    assert T.dispatch_arm(5000, 6, 256, 16, pin="gemv") == "gemv"
    # the post-merge note's decode floor at its edge: up to 8 tokens the
    # per-pair GEMV runs even where the tiles amortize (TILE_M 1; and k = E,
    # where pairs per woken expert = n reaches TILE_M 8 exactly at n = 8);
    # from 9 tokens the predicate decides
    for k, E, tm in ((6, 256, 1), (8, 8, 8)):
        assert T.tiles_amortize(8, k, E, tm)
        assert [T.dispatch_arm(n, k, E, tm) for n in range(1, 10)] == ["gemv"] * 8 + ["grouped"]


def pin_gate_closed_forms():
    """Special cases with exact answers.  k == E wakes every expert for every
    token, so pairs per woken expert is exactly n and the gate is n >= T (the
    boundary itself must select: the predicate is '>=').  n == 1 wakes exactly
    k experts with one pair each.  n == 0 never selects."""
    for E in (1, 4, 8, 64):
        for tm in (1, 16, 64):
            for n in range(1, 3 * tm):
                assert T.pairs_per_woken_expert(n, E, E) == n
                assert T.tiles_amortize(n, E, E, tm) == (n >= tm), (E, tm, n)
    for k, E in ((1, 8), (6, 256), (2, 3)):
        assert abs(T.pairs_per_woken_expert(1, k, E) - 1.0) < 1e-12
        assert abs(T.expected_woken_experts(1, k, E) - k) < 1e-9
        assert not T.tiles_amortize(0, k, E, 1)
    # large n: every expert woken, pairs per expert -> n*k/E
    assert abs(T.pairs_per_woken_expert(100000, 6, 256) - 100000 * 6 / 256) < 1e-9


def pin_min_tokens_flip():
    """The reported boundary is the exact flip point across 30 routing shapes,
    and agrees with a bisection on the real-valued closed form written with
    log1p/expm1 (a different evaluation of the same formula)."""
    shapes = [(k, E, tm) for (k, E) in ((1, 8), (2, 8), (6, 8), (2, 16), (4, 32),
                                       (6, 64), (8, 128), (6, 256), (8, 256), (2, 256))
              for tm in (16, 64, 4)]
    assert len(shapes) == 30
    for k, E, tm in shapes:
        n = T.grouped_min_tokens(k, E, tm)
        assert n >= 1
        assert T.tiles_amortize(n, k, E, tm)
        assert not T.tiles_amortize(n - 1, k, E, tm)

        def f(x):
            return x * k / (E * -math.expm1(x * math.log1p(-k / E))) - tm if k < E else x - tm
        lo, hi = 1e-9, float(max(n, 1) * 4 + 10)
        if f(hi) < 0:
            raise AssertionError("bisection bracket")
        for _ in range(200):
            mid = 0.5 * (lo + hi)
            if f(mid) >= 0:
                hi = mid
            else:
                lo = mid
        assert abs(n - math.ceil(hi - 1e-7)) <= 1, (k, E, tm, n, hi)
    assert T.grouped_min_tokens(6, 256, 64) == 2731       # TILE_M = 64 (sm_90+ m-tile)
    assert T.grouped_min_tokens(2, 8, 16) == 64
    assert T.grouped_min_tokens(6, 8, 16) == 22


def pin_closed_form_empirical(seeds: int = 200):
    """E[woken] = E(1-(1-k/E)^n) against uniform routing drawn by the input
    generator (means over seeds within 1%); pairs per woken = P / mean woken."""
    for (n, k, E) in ((32, 6, 256), (128, 6, 256), (16, 2, 8), (512, 6, 256)):
        woken = []
        for s in range(seeds):
            rng = np.random.Generator(np.random.PCG64(1000 + s))
            ids, _ = moe_inputs.draw_routing(rng, n, E, k)
            assert all(len(set(r)) == k for r in ids.tolist())
            woken.append(len(np.unique(ids)))
        mw = float(np.mean(woken))
        assert abs(mw / T.expected_woken_experts(n, k, E) - 1) < 0.01, (n, mw)
        assert abs((n * k / mw) / T.pairs_per_woken_expert(n, k, E) - 1) < 0.01


def pin_capacity_bound():
    """Sum of ceil(count_e/T) never exceeds tile_map_capacity, including
    adversarial routings that put count = 1 mod T on every expert."""
    rng = np.random.Generator(np.random.PCG64(7))
    for (n, k, E, tm) in ((16, 2, 8, 16), (32, 6, 256, 16), (683, 6, 256, 16),
                          (100, 4, 16, 4), (7, 3, 3, 2), (1, 1, 1, 1)):
        cap = T.tile_map_capacity(n, k, E, tm)
        for trial in range(50):
            if trial == 0:                 # as many experts at count 1 (mod T) as possible
                P = n * k
                counts = np.zeros(E, int)
                for p in range(P):
                    counts[p % E] += 1
            else:
                ids, _ = moe_inputs.draw_routing(rng, n, E, k)
                counts = np.bincount(ids.reshape(-1), minlength=E)
            assert sum(-(-int(c) // tm) for c in counts) <= cap
    assert T.tile_map_capacity(32, 6, 256, 16) == min(192, 12 + 192)


# ---------------------------------------------------------------------------
# trellis decode
# ---------------------------------------------------------------------------

def _bitfield_states(row: bytes, L: int):
    """State of symbol j read directly as bits [2j+2-L, 2j+2) of the row taken
    as one little-endian integer, with zeros below bit 0."""
    S = int.from_bytes(row, "little") << L          # stream bit b -> bit b + L
    mask = (1 << L) - 1
    return [(S >> (2 * j + 2)) & mask for j in range(4 * len(row))]


def _python_symbols(row: bytes):
    return [(row[j // 4] >> (2 * (j % 4))) & 3 for j in range(4 * len(row))]


def pin_decode_bitfield():
    """Window states equal bit-field slices of the stream (every symbol,
    every row, warm-up region included) for L in {2,...,16}."""
    rng = np.random.Generator(np.random.PCG64(11))
    for L in (2, 4, 6, 8, 10, 12, 14, 16):
        rows = rng.integers(0, 256, size=(6, 40), dtype=np.uint8)
        got = T.states_window(T.symbols(rows), L)
        for r in range(rows.shape[0]):
            want = _bitfield_states(rows[r].tobytes(), L)
            assert got[r].tolist() == want, (L, r)
    # symbols themselves: per-symbol byte/bit arithmetic in plain Python
    rows = rng.integers(0, 256, size=(3, 17), dtype=np.uint8)
    for r in range(3):
        assert T.symbols(rows[r]).tolist() == _python_symbols(rows[r].tobytes())


def pin_run_decode_identity():
    """Seeding a run from the window and stepping the recurrence gives the
    window state at every position, for every run start (runs of 32 at
    multiples of 32 as the pages' kernels use, and every other start)."""
    rng = np.random.Generator(np.random.PCG64(12))
    for L in (2, 8, 12, 16):
        rows = rng.integers(0, 256, size=(4, 64), dtype=np.uint8)     # K = 256
        c = T.symbols(rows)
        win = T.states_window(c, L)
        for start in range(0, 256 - 32 + 1):
            got = T.run_states(c, L, start, 32)
            assert np.array_equal(got, win[:, start:start + 32]), (L, start)


def pin_special_luts():
    """LUTs with known decodes.  (a) LUT[s] = s (exact in fp16 for L <= 10):
    W equals the bit-field states.  (b) LUT[s] = f(newest symbol) = f(s >> (L-2)):
    W[j] = f(c_j).  (c) LUT[s] = f(oldest symbol) = f(s & 3): W[j] =
    f(c_{j-L/2+1}), and f(0) inside the warm-up region."""
    rng = np.random.Generator(np.random.PCG64(13))
    f = np.array([0.5, -1.25, 2.0, -3.0])
    for L in (4, 8, 10):
        lut = np.arange(1 << L).astype(np.float16).view(np.uint16)
        rows = rng.integers(0, 256, size=(3, 16), dtype=np.uint8)
        W = T.decode_rows(rows, lut, L)
        for r in range(3):
            assert W[r].tolist() == [float(s) for s in _bitfield_states(rows[r].tobytes(), L)]
    for L in (4, 12, 16):
        s = np.arange(1 << L)
        rows = rng.integers(0, 256, size=(3, 16), dtype=np.uint8)
        newest = T.decode_rows(rows, f[s >> (L - 2)].astype(np.float16).view(np.uint16), L)
        oldest = T.decode_rows(rows, f[s & 3].astype(np.float16).view(np.uint16), L)
        for r in range(3):
            c = _python_symbols(rows[r].tobytes())
            assert newest[r].tolist() == [f[cj] for cj in c]
            lag = L // 2 - 1
            assert oldest[r].tolist() == [f[c[j - lag]] if j >= lag else f[0]
                                          for j in range(len(c))], (L, r)


# ---------------------------------------------------------------------------
# the MoE product
# ---------------------------------------------------------------------------

def _fp16(bits):
    return struct.unpack("<e", int(bits).to_bytes(2, "little"))[0]


def _bf16(bits):
    return struct.unpack("<f", (int(bits) << 16).to_bytes(4, "little"))[0]


def _bruteforce_y(prob, rows=None):
    """Pure-Python triple loop: decode each weight by bit slicing, multiply
    exactly (fp16 x bf16 x fp32 products fit in fp64) and sum with fsum."""
    ids, w, x, packed, lut, L = (prob.topk_ids, prob.topk_w, prob.x_bits, prob.packed,
                                 prob.lut_bits, prob.shape.L)
    n, k = ids.shape
    N = packed.shape[1]
    rows = range(N) if rows is None else rows
    out = np.zeros((n, len(rows)))
    for t in range(n):
        xs = [_bf16(b) for b in x[t]]
        for ri, r in enumerate(rows):
            terms = []
            for j in range(k):
                e = int(ids[t, j])
                wt = float(np.float32(w[t, j]))
                st = _bitfield_states(packed[e, r].tobytes(), L)
                terms.extend(wt * _fp16(lut[s]) * xi for s, xi in zip(st, xs))
            out[t, ri] = math.fsum(terms)
    return out


def pin_bruteforce_tiny():
    """Oracle Y equals the brute force on tiny problems (E=2..4, n<=4)."""
    for (E, k, n, K, N, L, seed) in ((2, 1, 3, 64, 8, 8, 1), (2, 2, 4, 64, 8, 12, 2),
                                     (4, 2, 3, 32, 5, 16, 3), (3, 3, 2, 16, 4, 6, 4)):
        prob = moe_inputs.make_custom(E, k, n, K, N, L, seed)
        got = T.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed,
                            prob.lut_bits, L)
        want = _bruteforce_y(prob)
        scale = max(np.abs(want).max(), 1e-30)
        assert np.abs(got - want).max() / scale < 1e-12, (E, k, n)
    # sampled rows equal the matching columns of the full product
    prob = moe_inputs.make_custom(4, 2, 3, 64, 16, 12, 5)
    full = T.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, 12)
    sub = T.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, 12,
                        rows=[3, 0, 15])
    assert np.array_equal(sub, full[:, [3, 0, 15]])


def pin_constant_lut():
    """Constant LUT c: Y[t, r] = c * sum_j w[t,j] * sum_i x[t,i] for every r."""
    prob = moe_inputs.make_custom(8, 2, 16, 256, 32, 12, 21)
    c = 0.375
    lut = np.full(1 << 12, c, dtype=np.float16).view(np.uint16)
    Y = T.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, lut, 12)
    xs = np.array([[_bf16(b) for b in row] for row in prob.x_bits])
    ws = prob.topk_w.astype(np.float64).sum(axis=1)
    want = c * ws * np.array([math.fsum(r) for r in xs])
    assert np.allclose(Y, want[:, None], rtol=1e-12, atol=1e-12)


def pin_onehot_x():
    """x[t] = e_i (bf16 1.0 at column i): Y[t, r] = sum_j w[t,j] W_{e(t,j)}[r, i],
    the weights read by bit slicing."""
    prob = moe_inputs.make_custom(4, 2, 4, 64, 8, 16, 31)
    x = np.zeros_like(prob.x_bits)
    cols = [0, 7, 33, 63]
    for t, i in enumerate(cols):
        x[t, i] = 0x3F80                      # bf16 1.0
    Y = T.moe_forward(x, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, 16)
    for t, i in enumerate(cols):
        for r in range(8):
            want = 0.0
            for j in range(2):
                e = int(prob.topk_ids[t, j])
                s = _bitfield_states(prob.packed[e, r].tobytes(), 16)[i]
                want += float(np.float32(prob.topk_w[t, j])) * _fp16(prob.lut_bits[s])
            assert abs(Y[t, r] - want) <= 1e-12 * max(1.0, abs(want)), (t, r)


# ---------------------------------------------------------------------------
# routing sort and tile map
# ---------------------------------------------------------------------------

def pin_route_bruteforce():
    """Stable sort by expert equals Python's sorted() on (expert, pair) keys;
    counts and offsets equal direct counting."""
    rng = np.random.Generator(np.random.PCG64(41))
    cases = [moe_inputs.draw_routing(rng, 16, 8, 2)[0],
             moe_inputs.draw_routing(rng, 32, 256, 6)[0],
             moe_inputs.draw_routing(rng, 64, 256, 6, "zipf")[0],
             np.zeros((5, 1), np.int32),                     # one expert takes all
             np.array([[3, 1], [1, 3], [3, 0]], np.int32)]
    for ids in cases:
        E = int(max(ids.max() + 1, 8))
        flat = ids.reshape(-1).tolist()
        counts, offsets, sp = T.route(ids, E)
        assert sp.tolist() == sorted(range(len(flat)), key=lambda p: (flat[p], p))
        assert counts.tolist() == [flat.count(e) for e in range(E)]
        assert offsets.tolist() == [sum(1 for v in flat if v < e) for e in range(E + 1)]
    c, o, sp = T.route(np.zeros((0, 6), np.int32), 256)
    assert c.sum() == 0 and o.tolist() == [0] * 257 and sp.size == 0


def pin_tile_map():
    """Tile map equals a walk over the sorted slots that opens a new tile when
    the expert changes or the tile is full; invariants hold."""
    rng = np.random.Generator(np.random.PCG64(42))
    for (n, k, E, tm, routing) in ((16, 2, 8, 16, "uniform"), (32, 6, 256, 16, "uniform"),
                                   (300, 6, 256, 16, "zipf"), (300, 6, 256, 64, "zipf"),
                                   (50, 3, 7, 1, "uniform"), (40, 4, 16, 5, "uniform")):
        ids, _ = moe_inputs.draw_routing(rng, n, E, k, routing)
        counts, offsets, sp = T.route(ids, E)
        tiles = T.tile_map(offsets, tm)
        flat = ids.reshape(-1)
        walk = []
        for slot, p in enumerate(sp.tolist()):
            e = int(flat[p])
            if walk and walk[-1][0] == e and walk[-1][2] < tm:
                walk[-1][2] += 1
            else:
                walk.append([e, slot, 1])
        assert tiles.tolist() == walk
        assert tiles[:, 2].sum() == n * k
        assert (tiles[:, 2] >= 1).all() and (tiles[:, 2] <= tm).all()
        assert len(tiles) == sum(-(-int(c) // tm) for c in counts)
        assert len(tiles) <= T.tile_map_capacity(n, k, E, tm)


def pin_bf16_rne():
    """Round-to-nearest-even fp32 -> bf16 equals torch's CPU cast, on random
    values, exact ties, near-overflow and subnormals."""
    import torch
    rng = np.random.Generator(np.random.PCG64(43))
    v = [rng.standard_normal(5000).astype(np.float32),
         (rng.standard_normal(2000) * 1e30).astype(np.float32),
         (rng.standard_normal(2000) * 1e-39).astype(np.float32)]
    u = rng.integers(0, 1 << 16, 3000, dtype=np.uint32)
    ties = ((u << 16) | 0x8000).astype(np.uint32).view(np.float32)           # exact halfway
    v.append(ties[np.isfinite(ties)])
    v.append(np.array([3.3895e38, 3.40282e38, -3.4e38, 0.0, -0.0, 1.0, 1.00390625], np.float32))
    y = np.concatenate(v)
    got = T.bf16_rne_bits(y)
    want = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def pin_router_topk():
    """Top-k by a Python sort on (-logit, expert) and softmax by math.exp and
    fsum; ties to the lower expert id; weights sum to one; k = E keeps every
    expert; a constant row picks experts 0..k-1 with equal weights."""
    rng = np.random.Generator(np.random.PCG64(44))
    for (n, E, k) in ((5, 8, 2), (7, 256, 6), (3, 16, 16), (4, 33, 5)):
        lg = rng.standard_normal((n, E)).astype(np.float32)
        lg[0, 3] = lg[0, 5] = lg[0].max() + 1.0           # an exact tie at the top
        ids, w = T.router_topk(lg, k)
        for t in range(n):
            want = sorted(range(E), key=lambda e: (-float(lg[t, e]), e))[:k]
            assert ids[t].tolist() == want, (n, E, k, t)
            ex = [math.exp(float(lg[t, e]) - float(lg[t, want[0]])) for e in want]
            tot = math.fsum(ex)
            assert np.allclose(w[t], [v / tot for v in ex], rtol=1e-12, atol=0)
            assert abs(w[t].sum() - 1) < 1e-12
        assert ids[0, 0] == 3 and ids[0, 1] == 5
    ids, w = T.router_topk(np.zeros((2, 8), np.float32), 3)
    assert ids.tolist() == [[0, 1, 2]] * 2 and np.allclose(w, 1 / 3)
    bad = np.array([[np.nan, 1.0, -np.inf, np.inf, 0.5], [np.nan] * 5], np.float32)
    ids, w = T.router_topk(bad, 3)
    assert ids[0].tolist() == [1, 4, 0] and abs(w[0, 2]) == 0.0
    assert ids[1].tolist() == [0, 1, 2] and np.allclose(w[1], 1 / 3)


def pin_mlp_bruteforce():
    """The MLP oracle against pure-Python loops (bit-sliced weights, math.exp
    silu, fsum) on a tiny problem, and its token subset against the full."""
    rng = np.random.Generator(np.random.PCG64(66))
    E, k, n, H, I, L = 3, 2, 3, 16, 8, 8
    ids = np.array([[0, 2], [1, 0], [2, 1]], np.int32)
    w = rng.random((n, k)).astype(np.float32)
    x = moe_inputs.fp32_to_bf16_bits(rng.standard_normal((n, H)).astype(np.float32))
    pgu = rng.integers(0, 256, (E, 2 * I, H // 4), dtype=np.uint8)
    pd = rng.integers(0, 256, (E, H, I // 4), dtype=np.uint8)
    lgu = (rng.standard_normal(1 << L) / 4).astype(np.float16).view(np.uint16)
    ld = (rng.standard_normal(1 << L) / 3).astype(np.float16).view(np.uint16)
    got = T.moe_mlp(x, ids, w, pgu, lgu, pd, ld, L)
    xs = [[_bf16(b) for b in row] for row in x]
    for t in range(n):
        for r in range(H):
            terms = []
            for j in range(k):
                e = int(ids[t, j])
                h = []
                for i in range(I):
                    g = math.fsum(_fp16(lgu[s]) * xv for s, xv in zip(_bitfield_states(pgu[e, i].tobytes(), L), xs[t]))
                    u = math.fsum(_fp16(lgu[s]) * xv for s, xv in zip(_bitfield_states(pgu[e, I + i].tobytes(), L), xs[t]))
                    h.append(g / (1.0 + math.exp(-g)) * u)
                d = math.fsum(_fp16(ld[s]) * hv for s, hv in zip(_bitfield_states(pd[e, r].tobytes(), L), h))
                terms.append(float(np.float32(w[t, j])) * d)
            want = math.fsum(terms)
            assert abs(got[t, r] - want) <= 1e-9 * max(1.0, abs(want)), (t, r, got[t, r], want)
    sub = T.moe_mlp(x, ids, w, pgu, lgu, pd, ld, L, tokens=[2, 0])
    assert np.allclose(sub, got[[2, 0]], rtol=1e-12, atol=1e-12)


ALL_PINS = [pin_fill_table, pin_gate_points, pin_gate_closed_forms, pin_min_tokens_flip,
            pin_capacity_bound, pin_decode_bitfield, pin_run_decode_identity,
            pin_special_luts, pin_bruteforce_tiny, pin_constant_lut, pin_onehot_x,
            pin_route_bruteforce, pin_tile_map, pin_bf16_rne, pin_router_topk,
            pin_mlp_bruteforce]
