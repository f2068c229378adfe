"""Dequantize-materialize comparator on the GPU against the CPU oracle.

tq_dequantize must reproduce, bit for bit, the bf16 weights the oracle's
trellis decode gives (the fp16 table value rounded to bf16, nearest-even); the
dense grouped GEMM and the whole comparator path are held to the output
tolerance of the fused arms (max|y - ref| / max|ref| <= 1e-2), and the dense
GEMM fed the materialized weights must agree with the fused kernel to fp32
summation-order noise (both multiply the same bf16 weights and activations)."""
import zlib

import numpy as np
import pytest
import torch

import moe_inputs
import oracle.trellis_moe as O
import trellis_quantized_moe_sort_gb300 as tq
from gpu_util import to_device, grouped_y32, normwise, sample_rows, check_no_device_error

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_quantized_moe_sort_gb300 import build
    build.build()
    tq.tq_init(0)


def _expected_bits(packed_rows, lut_bits, L):
    """The oracle's decoded weights (exact fp16 values) rounded to bf16."""
    return O.bf16_rne_bits(O.decode_rows(packed_rows, lut_bits, L).astype(np.float32))


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


# (E, N, K, L)
DEQ = {
    "tiny_L12": (8, 128, 256, 12),
    "K72_one_partial_pass": (3, 5, 72, 16),
    "K264_ragged_pass": (2, 7, 264, 8),
    "K4104_two_chunks": (2, 3, 4104, 16),
    "L2": (4, 9, 512, 2),
    "L4": (2, 3, 128, 4),
    "L10": (2, 4, 1024, 10),
    "L14": (2, 6, 2048, 14),
}


@pytest.mark.parametrize("name", sorted(DEQ))
def test_dequantize_bit_exact(name):
    E, N, K, L = DEQ[name]
    prob = moe_inputs.make_custom(E, 1, 1, K, N, L, seed=zlib.crc32(name.encode()) % 1000)
    d = to_device(prob)
    w = tq.tq_dequantize(d["packed"], d["lut"])
    check_no_device_error()
    got = _bits(w)
    for e in range(E):
        np.testing.assert_array_equal(got[e], _expected_bits(prob.packed[e], prob.lut_bits, L), err_msg=f"e={e}")


def test_dequantize_v4_listed_experts_sampled_rows():
    """L = 16, 4096-symbol rows: experts listed out of order land in their
    slots; a negative id leaves its slot untouched."""
    prob = moe_inputs.make_problem("v4_decode_n32")
    s = prob.shape
    packed = torch.from_numpy(prob.packed).cuda()
    lut = torch.from_numpy(prob.lut_bits.view(np.int16)).cuda()
    ids = torch.tensor([255, 0, -1, 17], dtype=torch.int32, device="cuda")
    w = torch.full((4, s.N, s.K), 7.0, dtype=torch.bfloat16, device="cuda")
    tq.tq_dequantize(packed, lut, expert_ids=ids, w_out=w)
    check_no_device_error()
    rows = sample_rows(s.N, 24, seed=5)
    got = _bits(w[:, torch.from_numpy(rows).cuda()])
    for slot, e in enumerate([255, 0, None, 17]):
        if e is None:
            assert np.all(got[slot] == np.uint16(0x40E0)), "slot with id -1 was written"
            continue
        np.testing.assert_array_equal(got[slot], _expected_bits(prob.packed[e][rows], prob.lut_bits, s.L))


def test_dequantize_out_of_range_id_reports():
    prob = moe_inputs.make_custom(4, 1, 1, 128, 8, 8, seed=3)
    d = to_device(prob)
    ids = torch.tensor([1, 4], dtype=torch.int32, device="cuda")
    w = torch.zeros((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    tq.tq_dequantize(d["packed"], d["lut"], expert_ids=ids, w_out=w)
    torch.cuda.synchronize()
    code, _ = tq.tq_device_error()
    assert code == -1          # TQ_ERR_INVALID_ARG
    assert torch.count_nonzero(w[1]).item() == 0
    np.testing.assert_array_equal(_bits(w[0]), _expected_bits(prob.packed[1], prob.lut_bits, 8))


def _random_deq(count=12, seed=31):
    """Seeded (E, N, K, L): K a multiple of 8 up to 4600 (partial passes and
    several chunks), any N, every even L."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [(int(rng.integers(1, 5)), int(rng.integers(1, 40)), 8 * int(rng.integers(1, 576)),
             2 * int(rng.integers(1, 9))) for _ in range(count)]


@pytest.mark.parametrize("cfg", _random_deq(count=40), ids=lambda c: "E{}_N{}_K{}_L{}".format(*c))
def test_dequantize_random_shapes_bit_exact(cfg):
    E, N, K, L = cfg
    prob = moe_inputs.make_custom(E, 1, 1, K, N, L, seed=zlib.crc32(repr(cfg).encode()) % 1000)
    d = to_device(prob)
    w = tq.tq_dequantize(d["packed"], d["lut"])
    check_no_device_error()
    got = _bits(w)
    for e in range(E):
        np.testing.assert_array_equal(got[e], _expected_bits(prob.packed[e], prob.lut_bits, L), err_msg=f"e={e}")


# (E, top_k, n, K, N, L, tile_m, routing)
FWD = {
    "tiny_T16": (8, 2, 16, 256, 128, 12, 16, "uniform"),
    "ragged_n37_K192_N256_T7": (4, 4, 37, 192, 256, 16, 7, "uniform"),
    "zipf_T128": (32, 4, 200, 256, 256, 14, 128, "zipf"),
    "T256": (8, 2, 300, 128, 384, 16, 256, "uniform"),
    # 19 k-steps of materialized weights: two full super-stages and 3
    "ragged_ss_K1216_T128": (6, 3, 60, 1216, 256, 14, 128, "zipf"),
}


@pytest.mark.parametrize("name", sorted(FWD))
def test_forward_dequant_all_outputs(name):
    E, k, n, K, N, L, T, routing = FWD[name]
    prob = moe_inputs.make_custom(E, k, n, K, N, L, seed=zlib.crc32(name.encode()) % 1000, routing=routing)
    d = to_device(prob)
    before = tq.tq_launch_counts()
    y = tq.tq_moe_forward_dequant(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=T)
    check_no_device_error()
    after = tq.tq_launch_counts()
    assert after["dequant"] == before["dequant"] + 1 and after["grouped"] == before["grouped"] + 1
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, L)
    assert normwise(y.float().cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("workload,T", [("v4_decode_n32", 16), ("v4_n128_up", 128)])
def test_forward_dequant_v4_sampled_rows(workload, T):
    prob = moe_inputs.make_problem(workload)
    s = prob.shape
    d = to_device(prob)
    y = tq.tq_moe_forward_dequant(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=T)
    check_no_device_error()
    rows = sample_rows(s.N, 48, seed=11)
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, s.L, rows=rows)
    got = y.float().cpu().numpy()[:, rows]
    assert normwise(got, ref) <= TOL


def test_dense_gemm_equals_fused_on_materialized_weights():
    """Same bf16 weights, same activations, fp32 accumulation: the dense and
    the fused grouped kernels differ only in summation order."""
    prob = moe_inputs.make_problem("v4_n128_up")
    s = prob.shape
    d = to_device(prob)
    T = 128
    fused = grouped_y32(prob, d, T)
    counts, offsets, sp = tq.tq_route(d["ids"], s.E)
    cap = tq.tq_tile_map_capacity(s.n, s.top_k, s.E, T)
    tiles, nt = tq.tq_build_tile_map(offsets, T, cap)
    w_dense = tq.tq_dequantize(d["packed"], d["lut"])
    y32 = torch.zeros((s.n, s.N), dtype=torch.float32, device="cuda")
    tq.tq_grouped_gemm_dense(d["x"], w_dense, sp, d["w"], tiles, nt, s.top_k, T, y32)
    check_no_device_error()
    assert normwise(y32.cpu().numpy(), fused.cpu().numpy()) <= 1e-5


def test_forward_dequant_empty_and_bad_workspace():
    prob = moe_inputs.make_custom(8, 2, 4, 256, 128, 12, seed=3)
    d = to_device(prob)
    y = tq.tq_moe_forward_dequant(d["x"][:0], d["packed"], d["lut"], d["ids"][:0], d["w"][:0])
    assert tuple(y.shape) == (0, 128)
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(tq.TQError) as ei:
        tq.tq_moe_forward_dequant(d["x"], d["packed"], d["lut"], d["ids"], d["w"], workspace=small)
    assert ei.value.status == -8       # TQ_ERR_WORKSPACE
    check_no_device_error()
