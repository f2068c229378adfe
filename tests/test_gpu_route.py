"""Routing sort, tile map and bf16 combine on the GPU: bit-exact against the
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle.trellis_moe as O
import trellis_quantized_moe_sort_gb300 as tq
from gpu_util import check_no_device_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_quantized_moe_sort_gb300 import build
    build.build()
    tq.tq_init(0)


def test_arch_witness_is_sm103():
    assert tq.tq_arch_witness(0) == 1030


def _ids_cases():
    rng = np.random.Generator(np.random.PCG64(5))
    cases = {
        "tiny": (moe_inputs.draw_routing(rng, 16, 8, 2)[0], 8),
        "v4_n32": (moe_inputs.draw_routing(rng, 32, 256, 6)[0], 256),
        "v4_n128": (moe_inputs.draw_routing(rng, 128, 256, 6)[0], 256),
        "v4_zipf_n8192": (moe_inputs.draw_routing(rng, 8192, 256, 6, "zipf")[0], 256),
        "one_expert_all": (np.full((1000, 1), 3, np.int32), 8),
        "E1024": (moe_inputs.draw_routing(rng, 300, 1024, 8)[0], 1024),
        "E1_k1": (np.zeros((5, 1), np.int32), 1),
        "ragged_P_37x3": (moe_inputs.draw_routing(rng, 37, 5, 3)[0], 5),
        "empty": (np.zeros((0, 6), np.int32), 256),
        # more than 8192 pairs: the sort is shared by several blocks (ragged
        # chunks, one expert spanning every chunk, many experts)
        "multi_one_expert_20000": (np.full((20000, 1), 3, np.int32), 8),
        "multi_E1024_n3000_k8": (moe_inputs.draw_routing(rng, 3000, 1024, 8)[0], 1024),
        "multi_ragged_9001x3": (moe_inputs.draw_routing(rng, 9001, 5, 3)[0], 5),
    }
    return cases


CASES = _ids_cases()


@pytest.mark.parametrize("name", sorted(CASES))
def test_route_bitexact(name):
    ids, E = CASES[name]
    d_ids = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    counts, offsets, sp = tq.tq_route(d_ids, E)
    check_no_device_error()
    c, o, s = O.route(ids, E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(sp.cpu().numpy(), s)


@pytest.mark.parametrize("name", ["tiny", "v4_n32", "v4_zipf_n8192", "one_expert_all", "E1024", "ragged_P_37x3",
                                  "multi_E1024_n3000_k8"])
@pytest.mark.parametrize("tile_m", [1, 7, 16, 64, 256])
def test_tile_map_bitexact(name, tile_m):
    ids, E = CASES[name]
    n, k = ids.shape
    d_ids = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    _, offsets, _ = tq.tq_route(d_ids, E)
    cap = tq.tq_tile_map_capacity(n, k, E, tile_m)
    tiles, nt = tq.tq_build_tile_map(offsets, tile_m, cap)
    check_no_device_error()
    want = O.tile_map(O.route(ids, E)[1], tile_m)
    got_n = int(nt.item())
    assert got_n == len(want)
    assert np.array_equal(tiles[:got_n].cpu().numpy(), want)


def test_tile_map_over_capacity_is_flagged():
    ids, E = CASES["v4_n32"]
    d_ids = torch.from_numpy(ids).cuda()
    _, offsets, _ = tq.tq_route(d_ids, E)
    want = O.tile_map(O.route(ids, E)[1], 16)
    cap = len(want) - 5
    tiles, nt = tq.tq_build_tile_map(offsets, 16, cap)
    torch.cuda.synchronize()
    assert int(nt.item()) == cap
    assert np.array_equal(tiles.cpu().numpy(), want[:cap])
    code, where = tq.tq_device_error()
    assert code == -3 and where == 2          # TQ_ERR_CAPACITY at the tile map
    check_no_device_error()


def test_route_flags_out_of_range_expert():
    ids = np.array([[0, 1], [2, 8], [3, 1]], np.int32)    # 8 is out of range for E=8
    counts, offsets, sp = tq.tq_route(torch.from_numpy(ids).cuda(), 8)
    torch.cuda.synchronize()
    code, where = tq.tq_device_error()
    assert code == -1 and where == 1
    c = counts.cpu().numpy()
    assert c.sum() == 5 and c[8 - 1] == 0
    check_no_device_error()


def test_route_multi_block_flags_out_of_range_expert():
    """More than 8192 pairs with a few ids out of range: they are reported,
    left out of the counts, and the rest sort exactly as the oracle sorts the
    valid pairs."""
    rng = np.random.Generator(np.random.PCG64(21))
    ids = moe_inputs.draw_routing(rng, 4000, 16, 4)[0].copy()
    ids[17, 2] = 16
    ids[3999, 0] = -2
    counts, offsets, sp = tq.tq_route(torch.from_numpy(ids).cuda(), 16)
    torch.cuda.synchronize()
    code, where = tq.tq_device_error()
    assert code == -1 and where == 1
    flat = ids.reshape(-1)
    valid = np.flatnonzero((flat >= 0) & (flat < 16))
    want = valid[np.argsort(flat[valid], kind="stable")]
    c = counts.cpu().numpy()
    assert c.sum() == len(valid)
    assert np.array_equal(sp[:len(valid)].cpu().numpy(), want)
    check_no_device_error()


def test_combine_bitexact():
    rng = np.random.Generator(np.random.PCG64(9))
    u = rng.integers(0, 1 << 16, 4096, dtype=np.uint32)
    ties = ((u << 16) | 0x8000).astype(np.uint32).view(np.float32)
    vals = np.concatenate([rng.standard_normal(100003).astype(np.float32),
                           ties[np.isfinite(ties)],
                           np.array([3.3895e38, -3.4e38, 0.0, -0.0, 1e-40], np.float32)])
    for arr in (vals, vals[:-1], vals[: (len(vals) // 4) * 4]):      # ragged and vector paths
        y32 = torch.from_numpy(arr.copy()).cuda()
        y = tq.tq_combine(y32)
        check_no_device_error()
        got = y.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, O.bf16_rne_bits(arr))


def test_prepare_equals_separate_calls():
    """tq_prepare (route + tile map in one launch whose other blocks clear
    y32, then the gather when x_sorted is given) gives bit for bit what
    tq_route, tq_build_tile_map and tq_gather_rows give, and leaves y32 zero
    (64 MiB of it at the prefill size)."""
    import moe_inputs
    for name, T in (("v4_decode_n32", 16), ("v4_prefill_n8192_up", 256)):
        prob = moe_inputs.make_problem(name, with_packed=False)
        s = prob.shape
        ids = torch.from_numpy(np.ascontiguousarray(prob.topk_ids)).cuda()
        x = torch.from_numpy(prob.x_bits.view(np.int16)).cuda()
        cap = tq.tq_tile_map_capacity(s.n, s.top_k, s.E, T)
        c1, o1, sp1 = tq.tq_route(ids, s.E)
        t1, nt1 = tq.tq_build_tile_map(o1, T, cap)
        xs1 = tq.tq_gather_rows(x, sp1, s.top_k)
        c2 = torch.empty_like(c1); o2 = torch.empty_like(o1); sp2 = torch.empty_like(sp1)
        t2 = torch.full_like(t1, -7); nt2 = torch.empty_like(nt1); xs2 = torch.empty_like(xs1)
        y32 = torch.full((s.n, s.N), 3.0, dtype=torch.float32, device="cuda")
        before = tq.tq_launch_counts()
        tq.tq_prepare(ids, x, s.E, T, cap, c2, o2, sp2, t2, nt2, xs2, y32)
        torch.cuda.synchronize()
        after = tq.tq_launch_counts()
        assert after["route_tile_map"] == before["route_tile_map"] + 1
        assert after["gather"] == before["gather"] + 1
        assert tq.tq_device_error() == (0, 0)
        for a, b in ((c1, c2), (o1, o2), (sp1, sp2), (nt1, nt2), (xs1, xs2)):
            assert torch.equal(a, b)
        ntiles = int(nt1.item())
        assert torch.equal(t1[:ntiles], t2[:ntiles])
        assert torch.count_nonzero(y32).item() == 0
        # without x_sorted: one launch, the same routing, y32 cleared
        y32.fill_(5.0)
        sp2.fill_(-1)
        before = tq.tq_launch_counts()
        tq.tq_prepare(ids, x, s.E, T, cap, c2, o2, sp2, t2, nt2, None, y32)
        torch.cuda.synchronize()
        after = tq.tq_launch_counts()
        assert after["route_tile_map"] == before["route_tile_map"] + 1
        assert after["gather"] == before["gather"]
        assert tq.tq_device_error() == (0, 0)
        assert torch.equal(sp1, sp2) and torch.equal(t1[:ntiles], t2[:ntiles])
        assert torch.count_nonzero(y32).item() == 0


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("tile_m", [1, 16, 256])
def test_prepare_bitexact_against_oracle(name, tile_m):
    """The fused route + tile map launch and the gather of tq_prepare against
    the oracle's route and tile map, bit for bit, on every routing case."""
    ids, E = CASES[name]
    n, k = ids.shape
    K = 64
    rng = np.random.Generator(np.random.PCG64(17))
    x_bits = moe_inputs.fp32_to_bf16_bits(rng.standard_normal((n, K), dtype=np.float32))
    d_ids = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    cap = tq.tq_tile_map_capacity(n, k, E, tile_m)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    sp = torch.empty(max(n * k, 1), dtype=torch.int32, device="cuda")
    tiles = torch.empty((max(cap, 1), 3), dtype=torch.int32, device="cuda")
    nt = torch.empty(1, dtype=torch.int32, device="cuda")
    xs = torch.empty((max(n * k, 1), K), dtype=torch.int16, device="cuda")
    tq.tq_prepare(d_ids, x, E, tile_m, max(cap, 1), counts, offsets, sp[:n * k], tiles, nt, xs[:n * k])
    check_no_device_error()
    c, o, s = O.route(ids, E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(sp[:n * k].cpu().numpy(), s)
    want = O.tile_map(o, tile_m)
    got_n = int(nt.item())
    assert got_n == len(want)
    assert np.array_equal(tiles[:got_n].cpu().numpy(), np.asarray(want, dtype=np.int32).reshape(-1, 3))
    if n * k:
        np.testing.assert_array_equal(xs[:n * k].cpu().numpy().view(np.uint16), x_bits[s // k])


def _random_routing(i, seed=404):
    """Seeded routing number i: E up to 1024, top_k up to 16, up to 40,000
    tokens (up to 640,000 pairs: the sort's largest grid), uniform, Zipf and
    shuffled-rank Zipf popularity, a random m-tile: (ids, E, tile_m).  Drawn
    when the test runs, so collecting the tests costs nothing."""
    rng = np.random.Generator(np.random.PCG64([seed, i]))
    E = int(rng.integers(1, 1025))
    k = int(rng.integers(1, min(E, 16) + 1))
    n = int(rng.choice([0, 1, int(rng.integers(2, 600)), int(rng.integers(600, 40001))],
                       p=[0.06, 0.06, 0.44, 0.44]))
    routing = str(rng.choice(["uniform", "zipf", "zipf_perm"]))
    ids, _ = moe_inputs.draw_routing(rng, n, E, k, routing)
    return ids.reshape(n, k), E, int(rng.integers(1, 257))


@pytest.mark.parametrize("i", range(64))
def test_prepare_random_routings_bitexact(i):
    """The fused route + tile map launch and the gather against the oracle's
    route and tile map, bit for bit, on seeded random routings."""
    ids, E, tile_m = _random_routing(i)
    n, k = ids.shape
    K = 64
    rng = np.random.Generator(np.random.PCG64(1000 + i))
    x_bits = moe_inputs.fp32_to_bf16_bits(rng.standard_normal((n, K), dtype=np.float32))
    d_ids = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    cap = tq.tq_tile_map_capacity(n, k, E, tile_m)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    sp = torch.empty(max(n * k, 1), dtype=torch.int32, device="cuda")
    tiles = torch.empty((max(cap, 1), 3), dtype=torch.int32, device="cuda")
    nt = torch.empty(1, dtype=torch.int32, device="cuda")
    xs = torch.empty((max(n * k, 1), K), dtype=torch.int16, device="cuda")
    tq.tq_prepare(d_ids, x, E, tile_m, max(cap, 1), counts, offsets, sp[:n * k], tiles, nt, xs[:n * k])
    check_no_device_error()
    c, o, s = O.route(ids, E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(sp[:n * k].cpu().numpy(), s)
    want = O.tile_map(o, tile_m)
    got_n = int(nt.item())
    assert got_n == len(want)
    assert np.array_equal(tiles[:got_n].cpu().numpy(), np.asarray(want, dtype=np.int32).reshape(-1, 3))
    if n * k:
        np.testing.assert_array_equal(xs[:n * k].cpu().numpy().view(np.uint16), x_bits[s // k])

