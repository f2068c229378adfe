"""Grouped GEMM and per-pair GEMV arms on the GPU against the CPU oracle.

Small problems (several tiles, ragged tails, every L, K of 1..many k-steps
and super-stages with a ragged last one, several 128-row blocks) are compared on every output; the five workloads at
full size on sampled rows.  Tolerance: max|y - ref| / max|ref| <= 1e-2 on the
fp32 accumulator (bf16 weights on the tensor cores; the GEMV widens fp16
weights exactly and is held to 1e-4)."""
import zlib

import numpy as np
import pytest
import torch

import moe_inputs
import oracle.trellis_moe as O
import trellis_quantized_moe_sort_gb300 as tq
from gpu_util import to_device, grouped_y32, gemv_y32, normwise, sample_rows, check_no_device_error

pytestmark = pytest.mark.gpu
TOL = 1e-2
TOL_GEMV = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_quantized_moe_sort_gb300 import build
    build.build()
    tq.tq_init(0)


# (E, top_k, n, K, N, L, tile_m, routing)
SMALL = {
    "tiny_e8_k2_n16_T16": (8, 2, 16, 256, 128, 12, 16, "uniform"),
    "tiny_T64": (8, 2, 16, 256, 128, 12, 64, "uniform"),
    "tiny_T1": (8, 2, 16, 256, 128, 12, 1, "uniform"),
    "ragged_n37_K192_N256": (4, 4, 37, 192, 256, 16, 16, "uniform"),
    "one_kstep_K64": (16, 3, 50, 64, 128, 8, 32, "uniform"),
    "big_tiles_T256": (8, 2, 300, 128, 384, 16, 256, "uniform"),
    "T48_L10": (6, 2, 40, 512, 128, 10, 48, "uniform"),
    "L2": (3, 3, 20, 320, 128, 2, 16, "uniform"),
    "L4_L6_mix": (5, 2, 24, 128, 128, 6, 16, "uniform"),
    "zipf_T128": (32, 4, 200, 256, 256, 14, 128, "zipf"),
    "zipf_perm_T256": (32, 4, 400, 320, 256, 16, 256, "zipf_perm"),
    # fp32 output > 24 MB and thousands of units: blocked row order, whole
    # units round-robin over the CTAs
    "interleaved_n6000_N1024": (64, 2, 6000, 64, 1024, 8, 16, "uniform"),
    # K past one super-stage (8 k-steps) with a ragged last one: the 4 stream
    # bytes carried across each boundary, and a final super-stage of 1 or 3
    # k-steps.  The first three hold fewer super-stage positions than there are
    # CTAs, so the walk splits every unit at every boundary; in the fourth each
    # CTA walks ~6 positions, crossing boundaries inside its own range.
    "ragged_ss_K576_L16": (4, 2, 24, 576, 128, 16, 16, "uniform"),
    "ragged_ss_K1216_T128": (6, 3, 60, 1216, 256, 14, 128, "zipf"),
    "ragged_ss_K2112_T256": (3, 2, 400, 2112, 1024, 12, 256, "uniform"),
    "ragged_ss_K1088_T64_zipf": (16, 4, 500, 1088, 1024, 16, 64, "zipf"),
    # the GEMV arm's largest K (one row = 16 super-stages)
    "kmax_K8192": (2, 1, 4, 8192, 128, 16, 16, "uniform"),
    # one expert holding every pair (128 + 128 + 44); the most experts the
    # routing sort takes, 393 of them woken by one or two pairs; one token
    "one_expert_E1": (1, 1, 300, 256, 128, 16, 128, "uniform"),
    "E1024_k8_n64": (1024, 8, 64, 256, 128, 12, 16, "uniform"),
    "one_token_n1": (16, 4, 1, 256, 256, 16, 16, "uniform"),
    "single_pair_k1": (4, 1, 1, 128, 128, 12, 16, "uniform"),
}


def _small(name):
    E, k, n, K, N, L, T, routing = SMALL[name]
    return moe_inputs.make_custom(E, k, n, K, N, L, seed=zlib.crc32(name.encode()) % 1000, routing=routing), T


@pytest.mark.parametrize("lay", [tq.X_TOKENS, tq.X_PAIR_SORTED])
@pytest.mark.parametrize("name", sorted(SMALL))
def test_grouped_small_all_outputs(name, lay):
    prob, T = _small(name)
    d = to_device(prob)
    y = grouped_y32(prob, d, T, lay).cpu().numpy()
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, prob.shape.L)
    err = normwise(y, ref)
    assert err <= TOL, err


# The GEMV arm's largest K with activations too large to stage beside the
# LUT (read from global memory, four 64-symbol chunks per lane), with one
# and with several pairs per token.
GEMV_EXTRA = {
    "gemv_K8192_n8_global_x": (2, 1, 8, 8192, 128, 16, 16, "uniform"),
    "gemv_K8192_n20_k3_global_x": (6, 3, 20, 8192, 256, 14, 16, "uniform"),
}


@pytest.mark.parametrize("name", sorted(SMALL) + sorted(GEMV_EXTRA))
def test_moe_forward_gemv_arm_small_all_outputs(name):
    """The whole product pinned to the GEMV arm (one launch: each warp sums a
    token's top_k pairs in registers and rounds once to bf16) on every small
    problem, all outputs: each within half a bf16 ulp of the oracle's value
    (round to nearest) plus the fp32 accumulation's slack."""
    if name in GEMV_EXTRA:
        E, k, n, K, N, L, _, routing = GEMV_EXTRA[name]
        prob = moe_inputs.make_custom(E, k, n, K, N, L, seed=zlib.crc32(name.encode()) % 1000, routing=routing)
    else:
        prob, _ = _small(name)
    d = to_device(prob)
    before = tq.tq_launch_counts()
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=16, pin=tq.ARM_GEMV)
    check_no_device_error()
    after = tq.tq_launch_counts()
    assert arm == tq.ARM_GEMV
    assert after["gemv"] == before["gemv"] + 1
    assert {k: after[k] - before[k] for k in after if k != "gemv"} == {k: 0 for k in after if k != "gemv"}
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, prob.shape.L)
    got = y.float().cpu().numpy().astype(np.float64)
    bound = np.abs(ref) * 2.0 ** -8 + 1e-5 * np.abs(ref).max()
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:4].tolist())


@pytest.mark.parametrize("N", [1, 3, 200])
def test_moe_forward_gemv_arm_any_output_width(N):
    """The GEMV arm of the whole product takes any N >= 1 (one (token, row)
    item per output element; a warp's range may wrap from a token's last row
    to the next token's first): all outputs within half a bf16 ulp of the
    oracle plus the fp32 slack; the grouped pin at such an N is refused."""
    prob = moe_inputs.make_custom(8, 2, 7, 256, N, 12, seed=900 + N)
    d = to_device(prob)
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=16, pin=tq.ARM_GEMV)
    check_no_device_error()
    assert arm == tq.ARM_GEMV and tuple(y.shape) == (7, N)
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, 12)
    got = y.float().cpu().numpy().astype(np.float64)
    assert not (np.abs(got - ref) > np.abs(ref) * 2.0 ** -8 + 1e-5 * np.abs(ref).max()).any()
    if N % 128:
        with pytest.raises(tq.TQError):
            tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=16, pin=tq.ARM_GROUPED)


@pytest.mark.parametrize("name", ["v4_fill_n1024", "v4_n128_down"])
def test_moe_forward_gemv_arm_full_size_sampled_rows(name):
    """The forward's GEMV arm at full V4 sizes (1024 tokens: 2 M (token, row)
    items with the activations read from global memory; the down projection
    at 128 tokens, K = 2048 -> N = 4096): sampled output columns within half a
    bf16 ulp of the oracle plus the fp32 slack."""
    prob = moe_inputs.make_problem(name)
    d = to_device(prob)
    s = prob.shape
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=16, pin=tq.ARM_GEMV)
    check_no_device_error()
    assert arm == tq.ARM_GEMV
    rows = sample_rows(s.N, 24, seed=77)
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, s.L, rows=rows)
    got = y.float().cpu().numpy()[:, rows].astype(np.float64)
    assert not (np.abs(got - ref) > np.abs(ref) * 2.0 ** -8 + 1e-5 * np.abs(ref).max()).any()


def test_moe_forward_gemv_arm_is_bit_reproducible():
    """The GEMV arm sums each token's pairs in a fixed order and writes each
    output once, so repeated calls (and a call on another stream) give the
    same bits (V4 up shape, 8 tokens)."""
    prob = moe_inputs.make_problem("v4_decode_n32", n=8)
    d = to_device(prob)
    outs = []
    for stream in (None, None, torch.cuda.Stream()):
        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
            y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=16, pin=tq.ARM_GEMV)
        torch.cuda.synchronize()
        assert arm == tq.ARM_GEMV
        outs.append(y.view(torch.int16).clone())
    check_no_device_error()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


# Expert sizes whose m-tiles at TILE_M 256 run through every transition of the
# accumulator slots (m-tiles above 128 pairs take both 128-column slots, the
# others one, alternating): 296 -> 256 + 40 (big -> small), 40 -> 200 (small ->
# big), 200 -> 130 (big -> big), 130 -> 128, 128 -> 1 (small -> small),
# 1 -> 129, 512 -> 256 + 256, 17, 255, 257 -> 256 + 1.
SLOT_PATTERN = [296, 200, 130, 128, 1, 129, 512, 17, 255, 257]


def _slot_problem(reps, N, seed, K=64):
    """top-1 routing with the expert sizes of SLOT_PATTERN repeated `reps`
    times (token order shuffled), router weights drawn in [0.5, 1.5)."""
    counts = np.array(SLOT_PATTERN * reps)
    E, n, L = len(counts), int(counts.sum()), 12
    rx, rr, rp, rl = moe_inputs._streams((moe_inputs.BASE_SEED, 4242, seed, reps, N, K))
    ids = np.repeat(np.arange(E, dtype=np.int32), counts)
    rr.shuffle(ids)
    w = rr.uniform(0.5, 1.5, size=(n, 1)).astype(np.float32)
    shp = moe_inputs.Shape(f"slots_{reps}_{N}", E, 1, n, K, N, L)
    return moe_inputs.Problem(shp, moe_inputs.draw_x(rx, n, K), ids.reshape(n, 1), w,
                              moe_inputs.draw_packed(rp, E, N, K), moe_inputs.draw_lut(rl, L, K))


@pytest.mark.parametrize("reps,N,T,K", [(60, 128, 256, 64), (60, 128, 192, 64), (30, 1024, 256, 64),
                                         (20, 128, 256, 1024)])
def test_grouped_accumulator_slots_all_outputs(reps, N, T, K):
    """m-tiles above 128 pairs with small and big tiles interleaved on every
    CTA: 780 one-row-block units (each CTA walks ~5 units in a row), 3120
    units over eight row blocks (whole units dealt round-robin), and 260 units
    of two super-stages each (K = 1024), which the contiguous walk splits
    between CTAs at super-stage boundaries.  Every output against the oracle,
    and the tile sizes the map holds are the pattern's."""
    prob = _slot_problem(reps, N, seed=T, K=K)
    counts, offsets, _ = O.route(prob.topk_ids, prob.shape.E)
    rows = O.tile_map(offsets, T)[:, 2]
    assert (rows > 128).any() and (rows <= 128).any() and (rows == 1).any()
    d = to_device(prob)
    y = grouped_y32(prob, d, T, tq.X_PAIR_SORTED).cpu().numpy()
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, prob.shape.L)
    assert normwise(y, ref) <= TOL


def _random_configs(count=24, seed=2026):
    """Seeded shapes anywhere inside the documented limits (K % 64 == 0,
    N % 128 == 0, L even in [2, 16], 1 <= tile_m <= 256, top_k <= E), small
    enough for the oracle on every output: (E, top_k, n, K, N, L, tile_m)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    while len(out) < count:
        E = int(rng.integers(1, 65))
        k = int(rng.integers(1, min(E, 8) + 1))
        n = int(rng.integers(1, 301))
        K = 64 * int(rng.integers(1, 41))
        N = 128 * int(rng.integers(1, 5))
        L = 2 * int(rng.integers(1, 9))
        T = int(rng.choice([1, 2, 5, 16, 24, 48, 64, 100, 128, 160, 192, 256]))
        if n * k * K * N <= 6e7:
            out.append((E, k, n, K, N, L, T))
    return out


@pytest.mark.parametrize("cfg", _random_configs(count=160), ids=lambda c: "E{}_k{}_n{}_K{}_N{}_L{}_T{}".format(*c))
def test_random_shapes_all_outputs(cfg):
    """Both arms, and the grouped arm on both activation layouts, on seeded
    random shapes: every output against the oracle; then the whole product
    on each arm at the shape's m-tile (the GEMV arm's bf16 outputs each within
    half a bf16 ulp of the oracle plus the fp32 slack)."""
    E, k, n, K, N, L, T = cfg
    prob = moe_inputs.make_custom(E, k, n, K, N, L, seed=zlib.crc32(repr(cfg).encode()) % 1000)
    d = to_device(prob)
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, L)
    for lay in (tq.X_TOKENS, tq.X_PAIR_SORTED):
        y = grouped_y32(prob, d, T, lay).cpu().numpy()
        assert normwise(y, ref) <= TOL, (lay, normwise(y, ref))
    y = gemv_y32(prob, d).cpu().numpy()
    assert normwise(y, ref) <= TOL_GEMV
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=T, pin=tq.ARM_GROUPED)
    check_no_device_error()
    assert arm == tq.ARM_GROUPED and normwise(y.float().cpu().numpy(), ref) <= TOL
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=T, pin=tq.ARM_GEMV)
    check_no_device_error()
    got = y.float().cpu().numpy().astype(np.float64)
    bad = np.abs(got - ref) > np.abs(ref) * 2.0 ** -8 + 1e-5 * np.abs(ref).max()
    assert arm == tq.ARM_GEMV and not bad.any(), (int(bad.sum()), np.argwhere(bad)[:4].tolist())


@pytest.mark.parametrize("name", sorted(SMALL))
def test_gemv_small_all_outputs(name):
    prob, _ = _small(name)
    d = to_device(prob)
    y = gemv_y32(prob, d).cpu().numpy()
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, prob.shape.L)
    assert normwise(y, ref) <= TOL_GEMV


def test_grouped_accumulates_into_y32():
    prob, T = _small("tiny_e8_k2_n16_T16")
    d = to_device(prob)
    s = prob.shape
    _, offsets, sp = tq.tq_route(d["ids"], s.E)
    cap = tq.tq_tile_map_capacity(s.n, s.top_k, s.E, T)
    tiles, nt = tq.tq_build_tile_map(offsets, T, cap)
    y32 = torch.ones((s.n, s.N), dtype=torch.float32, device="cuda")
    for _ in range(2):
        tq.tq_grouped_gemm(d["x"], d["packed"], d["lut"], sp, d["w"], tiles, nt, s.top_k, T, y32)
    check_no_device_error()
    ref = 1.0 + 2.0 * O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed,
                                    prob.lut_bits, s.L)
    assert normwise(y32.cpu().numpy(), ref) <= TOL


def test_grouped_onehot_x_reads_single_weight_column():
    """x[t] = e_i: y[t, r] = sum_j w W_e[r, i] -> checks the k ordering inside
    the decoded tile (a transposed or shifted A layout fails here)."""
    prob = moe_inputs.make_custom(4, 2, 8, 256, 128, 16, seed=77)
    x = np.zeros_like(prob.x_bits)
    cols = [0, 1, 15, 16, 63, 64, 130, 255]
    for t, i in enumerate(cols):
        x[t, i] = 0x3F80
    prob.x_bits = x
    d = to_device(prob)
    y = grouped_y32(prob, d, 16).cpu().numpy()
    ref = O.moe_forward(x, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, 16)
    assert normwise(y, ref) <= TOL


FULL = ["v4_decode_n32", "v4_n128_up", "v4_n128_down", "v4_fill_n512", "v4_fill_n683",
        "v4_fill_n1024", "v4_prefill_n8192_up", "v4_prefill_n8192_down"]


@pytest.fixture(scope="module")
def full_problems():
    cache = {}

    def get(name):
        if name not in cache:
            cache.clear()
            prob = moe_inputs.make_problem(name)
            cache[name] = (prob, to_device(prob))
        return cache[name]
    return get


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(name, full_problems):
    prob, d = full_problems(name)
    s = prob.shape
    rows = sample_rows(s.N, 48, seed=len(name))
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, s.L, rows=rows)
    # token rows gathered by the kernel and the pair-sorted copy (each at the
    # m-tile the whole-product calls use it with, and token rows at 128 too)
    for T, lay in ((16, tq.X_TOKENS), (128, tq.X_PAIR_SORTED), (128, tq.X_TOKENS)):
        y = grouped_y32(prob, d, T, lay)[:, torch.from_numpy(rows).cuda()].cpu().numpy()
        assert normwise(y, ref) <= TOL, (T, lay, normwise(y, ref))
    if s.n <= 1024:
        y = gemv_y32(prob, d)[:, torch.from_numpy(rows).cuda()].cpu().numpy()
        assert normwise(y, ref) <= TOL_GEMV


def test_moe_forward_gate_and_arms():
    """(top-2 of 8, TILE_M=16) flips at n = 64: below it the GEMV runs, at it
    the grouped GEMM; n <= 8 always GEMV; the pin forces either arm; the
    launch counters prove which kernel ran; y is bf16 of the product."""
    assert tq.tq_grouped_min_tokens(2, 8, 16) == 64
    for n, pin, want_arm in ((63, 0, 1), (64, 0, 2), (8, 0, 1), (5, 2, 2), (200, 1, 1)):
        prob = moe_inputs.make_custom(8, 2, n, 256, 128, 12, seed=n + 10 * pin)
        d = to_device(prob)
        before = tq.tq_launch_counts()
        y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=16, pin=pin)
        check_no_device_error()
        after = tq.tq_launch_counts()
        assert arm == want_arm
        ran = "grouped" if arm == 2 else "gemv"
        other = "gemv" if arm == 2 else "grouped"
        assert after[ran] == before[ran] + 1 and after[other] == before[other]
        # the grouped arm: one routing launch (clearing y32), the kernel gathers
        # activations itself, one combine; the GEMV arm: the GEMV alone (it
        # sums each token's pairs and writes bf16 y, so nothing to clear or
        # combine)
        assert after["gather"] == before["gather"] and after["clear"] == before["clear"]
        if arm == 2:
            assert after["route_tile_map"] == before["route_tile_map"] + 1
            assert after["combine"] == before["combine"] + 1
        else:
            assert after["route_tile_map"] == before["route_tile_map"]
            assert after["combine"] == before["combine"]
        ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, 12)
        got = y.float().cpu().numpy()
        assert normwise(got, ref) <= TOL


@pytest.mark.parametrize("pin", [tq.ARM_GROUPED, tq.ARM_GEMV])
@pytest.mark.parametrize("tile_m", [16, 64])
def test_moe_forward_dirty_workspace(pin, tile_m):
    """A workspace full of NaN bit patterns: every call clears what must start
    at zero itself (the grouped arm's accumulator, in the routing launch; the
    GEMV arm reads no workspace), so the result matches the oracle on every
    call."""
    prob = moe_inputs.make_custom(8, 2, 40, 256, 256, 12, seed=55)
    d = to_device(prob)
    s = prob.shape
    ws = torch.empty(tq.tq_moe_workspace_size(s.n, s.top_k, s.E, s.K, s.N, tile_m), dtype=torch.uint8,
                     device="cuda")
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, s.L)
    for _ in range(2):
        ws.fill_(0xFF)
        y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=tile_m, pin=pin,
                                   workspace=ws)
        check_no_device_error()
        assert arm == pin
        assert normwise(y.float().cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("tile_m,pin", [(16, tq.ARM_GROUPED), (64, tq.ARM_GROUPED), (16, tq.ARM_GEMV)])
def test_moe_forward_out_of_range_expert(tile_m, pin):
    """One pair routed to expert E (out of range): the call reports
    TQ_ERR_INVALID_ARG in the device error word and drops that pair (at m-tile
    64 its slot in the sort's inverse is -1 and the token-order copy skips it);
    every output equals the product over the remaining pairs.  The dropped
    pair's router weight is NaN: dropping means it is never multiplied in."""
    prob = moe_inputs.make_custom(8, 2, 40, 256, 128, 12, seed=4040)
    ids = prob.topk_ids.copy()
    ids[5, 1] = 8
    d = to_device(prob)
    d["ids"] = torch.from_numpy(ids).cuda()
    d["w"] = d["w"].clone()
    d["w"][5, 1] = float("nan")
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=tile_m, pin=pin)
    torch.cuda.synchronize()
    assert arm == pin
    code, _ = tq.tq_device_error()
    assert code == -1
    w = prob.topk_w.copy()
    w[5, 1] = 0.0
    keep = ids.copy()
    keep[5, 1] = 0
    ref = O.moe_forward(prob.x_bits, keep, w, prob.packed, prob.lut_bits, prob.shape.L)
    assert normwise(y.float().cpu().numpy(), ref) <= TOL


def test_moe_forward_gemv_ragged_output():
    """The GEMV arm of the whole product takes any N: 7 tokens x 130 rows (an
    odd output length, so the warps' ranges of (token, row) items start and
    end at odd rows), with a NaN-filled workspace that the arm never reads."""
    prob = moe_inputs.make_custom(8, 2, 7, 256, 130, 12, seed=61)
    d = to_device(prob)
    s = prob.shape
    ws = torch.empty(tq.tq_moe_workspace_size(s.n, s.top_k, s.E, s.K, s.N, 16) + 256, dtype=torch.uint8,
                     device="cuda")
    ws.fill_(0xFF)
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=16, pin=tq.ARM_GEMV,
                               workspace=ws)
    check_no_device_error()
    assert arm == tq.ARM_GEMV
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, s.L)
    assert normwise(y.float().cpu().numpy(), ref) <= TOL


def test_moe_forward_empty_batch():
    prob = moe_inputs.make_custom(8, 2, 4, 256, 128, 12, seed=3)
    d = to_device(prob)
    x0 = d["x"][:0]
    y, arm = tq.tq_moe_forward(x0, d["packed"], d["lut"], d["ids"][:0], d["w"][:0])
    check_no_device_error()
    assert tuple(y.shape) == (0, 128)


def test_moe_forward_measured_policy():
    """pin = ARM_MEASURED: the GEMV for a lone token (1 pair per woken expert),
    the grouped GEMM once experts are shared (3 tokens of top-2 of 8: 1.30),
    with the launch counters proving the arm and the output within tolerance."""
    for n, want_arm in ((1, 1), (3, 2), (40, 2)):
        prob = moe_inputs.make_custom(8, 2, n, 256, 128, 12, seed=70 + n)
        d = to_device(prob)
        before = tq.tq_launch_counts()
        y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=16,
                                   pin=tq.ARM_MEASURED)
        check_no_device_error()
        after = tq.tq_launch_counts()
        assert arm == want_arm
        ran = "grouped" if arm == 2 else "gemv"
        assert after[ran] == before[ran] + 1
        ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, 12)
        assert normwise(y.float().cpu().numpy(), ref) <= TOL


def test_binding_refuses_wrong_dtype_and_strides():
    """A tensor of the wrong dtype or a non-contiguous view is refused by the
    binding (TypeError / ValueError naming the argument), never read with the
    wrong layout."""
    prob, T = _small("tiny_e8_k2_n16_T16")
    d = to_device(prob)
    with pytest.raises(ValueError, match="topk_ids must be a CUDA tensor"):
        tq.tq_route(d["ids"].cpu(), prob.shape.E)
    with pytest.raises(TypeError, match="topk_ids"):
        tq.tq_route(d["ids"].long(), prob.shape.E)
    wide = torch.zeros((prob.shape.n, 2 * prob.shape.K), dtype=torch.int16, device="cuda")
    with pytest.raises(ValueError, match="must be contiguous"):
        tq.tq_gemv(wide[:, ::2], d["packed"], d["lut"], d["ids"], d["w"],
                   torch.zeros((prob.shape.n, prob.shape.N), dtype=torch.float32, device="cuda"))
    check_no_device_error()

