"""Plant plausible mistakes in the oracle (on the CPU) and check that some pin
catches each one: off-by-one symbol, wrong state mask, off-by-one seed,
shift-by-1 (the four mutation classes the arch-specialisation page reports),
plus reversed window order, dropped router weight, wrong token index, unstable
route, tile-map off-by-one, '>' for '>=', a wrong exponent in the fill, an
undersized capacity bound, a late flip, a strict decode floor, the
with-replacement woken-expert formula, reversed symbol order, an unweighted
MLP, activations read as fp16, the wrong expert and reversed output rows."""
import numpy as np
import pytest

import oracle.trellis_moe as T
import oracle_pins as P

orig = {name: getattr(T, name) for name in dir(T) if not name.startswith("_")}


def _symbols_off_by_one(packed_rows):
    c = orig["symbols"](packed_rows)
    return np.concatenate([c[..., 1:], np.zeros_like(c[..., :1])], axis=-1)


def _window_wrong_mask(c, L):
    return orig["states_window"](c, L) & ((1 << (L - 2)) - 1)


def _window_too_wide(c, L):
    h = L // 2 + 1
    K = c.shape[-1]
    s = np.zeros_like(c)
    for i in range(h):
        lagged = np.zeros_like(c)
        lagged[..., i:] = c[..., :K - i]
        s += lagged * (4 ** (h - 1 - i))
    return s % (1 << L)


def _window_reversed(c, L):
    h = L // 2
    K = c.shape[-1]
    s = np.zeros_like(c)
    for i in range(h):
        lagged = np.zeros_like(c)
        lagged[..., i:] = c[..., :K - i]
        s += lagged * (4 ** i)
    return s


def _run_seed_off_by_one(c, L, run_start, run_len):
    out = orig["run_states"](c, L, run_start, run_len).copy()
    seed = orig["states_window"](c[..., :max(run_start, 1)], L)[..., max(run_start - 1, 0)]
    s = seed
    out[..., 0] = s
    for m in range(1, run_len):
        s = (s >> 2) | (c[..., run_start + m] << (L - 2))
        out[..., m] = s
    return out


def _run_shift_by_one(c, L, run_start, run_len):
    out = orig["run_states"](c, L, run_start, run_len).copy()
    s = out[..., 0]
    for m in range(1, run_len):
        s = ((s >> 1) | (c[..., run_start + m] << (L - 2))) & ((1 << L) - 1)
        out[..., m] = s
    return out


def _forward_no_router_weight(x_bits, topk_ids, topk_w, packed, lut_bits, L, rows=None):
    return orig["moe_forward"](x_bits, topk_ids, np.ones_like(topk_w), packed, lut_bits, L, rows)


def _forward_wrong_token(x_bits, topk_ids, topk_w, packed, lut_bits, L, rows=None):
    return orig["moe_forward"](np.roll(x_bits, 1, axis=0), topk_ids, topk_w, packed,
                               lut_bits, L, rows)


def _forward_negated(*a, **kw):
    return -orig["moe_forward"](*a, **kw)


def _lut_as_bf16(lut_bits):
    return orig["bf16_bits_to_f64"](lut_bits)


def _route_unstable(topk_ids, E):
    counts, offsets, sp = orig["route"](topk_ids, E)
    sp = sp.copy()
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        sp[a:b] = sp[a:b][::-1]
    return counts, offsets, sp


def _tile_map_off_by_one(offsets, tile_m):
    tiles = orig["tile_map"](offsets, tile_m)
    if len(tiles):
        tiles = tiles.copy()
        tiles[-1, 2] += 1
    return tiles


def _amortize_strict(n, top_k, E, tile_m):
    return n > 0 and orig["pairs_per_woken_expert"](n, top_k, E) > tile_m


def _ppw_wrong_exponent(n, top_k, E):
    if n <= 0:
        return 0.0
    return n * top_k / (E * (1 - (1 - top_k / E) ** (n - 1)))


def _bf16_ties_away(y32):
    u = np.ascontiguousarray(y32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x8000) >> 16).astype(np.uint16)


def _topk_ties_high(logits, top_k):
    lg = np.asarray(logits, dtype=np.float32).astype(np.float64)
    n, E = lg.shape
    order = np.lexsort((-np.broadcast_to(np.arange(E), (n, E)), -lg), axis=1)[:, :top_k]
    sel = np.take_along_axis(lg, order, axis=1)
    z = np.exp(sel - sel[:, :1])
    return order.astype(np.int32), z / z.sum(axis=1, keepdims=True)


def _topk_softmax_all(logits, top_k):
    ids, _ = orig["router_topk"](logits, top_k)
    lg = np.asarray(logits, dtype=np.float64)
    z = np.exp(lg - lg.max(axis=1, keepdims=True))
    full = z / z.sum(axis=1, keepdims=True)
    return ids, np.take_along_axis(full, ids.astype(np.int64), axis=1)


def _mlp_sigmoid_only(*a, **kw):
    saved = T.silu
    T.silu = lambda v: 1.0 / (1.0 + np.exp(-v))
    try:
        return orig["moe_mlp"](*a, **kw)
    finally:
        T.silu = saved


def _mlp_swapped_halves(x_bits, topk_ids, topk_w, packed_gu, lut_gu, packed_down, lut_down, L, tokens=None):
    I = packed_gu.shape[1] // 2
    swapped = np.concatenate([packed_gu[:, I:], packed_gu[:, :I]], axis=1)
    return orig["moe_mlp"](x_bits, topk_ids, topk_w, swapped, lut_gu, packed_down, lut_down, L, tokens)


def _capacity_too_small(n, top_k, E, tile_m):
    return max(orig["tile_map_capacity"](n, top_k, E, tile_m) - 1, 0)


def _flip_late(top_k, E, tile_m, limit=1 << 26):
    f = orig["grouped_min_tokens"](top_k, E, tile_m, limit)
    return f + 1 if f > 0 else f


def _dispatch_floor_strict(n, top_k, E, tile_m, pin="auto"):
    if pin in ("gemv", "grouped"):
        return pin
    if n < T.DECODE_REGIME_MAX_TOKENS or not T.tiles_amortize(n, top_k, E, tile_m):
        return "gemv"
    return "grouped"


def _ppw_with_replacement(n, top_k, E):
    if n <= 0:
        return 0.0
    return n * top_k / (E * (1 - (1 - 1 / E) ** (n * top_k)))


def _decode_symbols_reversed(packed_rows, lut_bits, L):
    lut = orig["lut_values"](lut_bits)
    c = np.ascontiguousarray(orig["symbols"](packed_rows)[..., ::-1])
    return lut[orig["states_window"](c, L)]


def _mlp_down_unweighted(x_bits, topk_ids, topk_w, *rest, **kw):
    return orig["moe_mlp"](x_bits, topk_ids, np.ones_like(topk_w), *rest, **kw)


def _activations_as_fp16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _forward_expert_off_by_one(x_bits, topk_ids, topk_w, packed, lut_bits, L, rows=None):
    E = packed.shape[0]
    return orig["moe_forward"](x_bits, (np.asarray(topk_ids) + 1) % E, topk_w, packed, lut_bits, L, rows)


def _forward_rows_reversed(x_bits, topk_ids, topk_w, packed, lut_bits, L, rows=None):
    return orig["moe_forward"](x_bits, topk_ids, topk_w, np.ascontiguousarray(packed[:, ::-1]), lut_bits, L, rows)


MUTATIONS = {
    "capacity_too_small": ("tile_map_capacity", _capacity_too_small),
    "flip_one_late": ("grouped_min_tokens", _flip_late),
    "decode_floor_strict": ("dispatch_arm", _dispatch_floor_strict),
    "woken_with_replacement": ("pairs_per_woken_expert", _ppw_with_replacement),
    "symbols_reversed_in_row": ("decode_rows", _decode_symbols_reversed),
    "mlp_down_unweighted": ("moe_mlp", _mlp_down_unweighted),
    "activations_as_fp16": ("bf16_bits_to_f64", _activations_as_fp16),
    "expert_off_by_one": ("moe_forward", _forward_expert_off_by_one),
    "output_rows_reversed": ("moe_forward", _forward_rows_reversed),
    "mlp_sigmoid_for_silu": ("moe_mlp", _mlp_sigmoid_only),
    "mlp_gate_up_swapped": ("moe_mlp", _mlp_swapped_halves),
    "topk_ties_high": ("router_topk", _topk_ties_high),
    "topk_softmax_over_all": ("router_topk", _topk_softmax_all),
    "symbol_off_by_one": ("symbols", _symbols_off_by_one),
    "state_mask": ("states_window", _window_wrong_mask),
    "window_too_wide": ("states_window", _window_too_wide),
    "window_reversed": ("states_window", _window_reversed),
    "seed_off_by_one": ("run_states", _run_seed_off_by_one),
    "shift_by_one": ("run_states", _run_shift_by_one),
    "no_router_weight": ("moe_forward", _forward_no_router_weight),
    "wrong_token": ("moe_forward", _forward_wrong_token),
    "wrong_sign": ("moe_forward", _forward_negated),
    "lut_as_bf16": ("lut_values", _lut_as_bf16),
    "route_unstable": ("route", _route_unstable),
    "tile_map_off_by_one": ("tile_map", _tile_map_off_by_one),
    "gate_strict": ("tiles_amortize", _amortize_strict),
    "fill_exponent": ("pairs_per_woken_expert", _ppw_wrong_exponent),
    "bf16_ties_away": ("bf16_rne_bits", _bf16_ties_away),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(T, attr, fn)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
        except Exception as exc:          # a crash under the mutation also counts
            caught.append(f"{pin.__name__}:{type(exc).__name__}")
    assert caught, f"mutation {name} escaped every pin"
