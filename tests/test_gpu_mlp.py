"""The whole SwiGLU expert MLP (gate|up grouped GEMM per pair, SwiGLU, down
grouped GEMM combined per token) against the oracle, and its two new pieces
on their own: the per-pair grouped GEMM and the SwiGLU kernel.  Tolerance
max|y - ref| / max|ref| <= 1e-2 (bf16 weights and bf16 h on the GPU)."""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle.trellis_moe as O
import trellis_quantized_moe_sort_gb300 as tq
from gpu_util import to_device, normwise, check_no_device_error

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_quantized_moe_sort_gb300 import build
    build.build()
    tq.tq_init(0)


def _mlp_dev(prob):
    import warnings
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        return dict(x=c(prob.x_bits.view(np.int16)), ids=c(prob.topk_ids), w=c(prob.topk_w),
                    pgu=c(prob.packed_gu), lgu=c(prob.lut_gu.view(np.int16)),
                    pd=c(prob.packed_down), ld=c(prob.lut_down.view(np.int16)))


@pytest.mark.parametrize("tile_m,pin", [(16, tq.ARM_GROUPED), (64, tq.ARM_GROUPED), (16, tq.ARM_GEMV)])
def test_mlp_tiny_all_outputs(tile_m, pin):
    prob = moe_inputs.make_mlp_problem("tiny_mlp_e8_k2_n16")
    d = _mlp_dev(prob)
    before = tq.tq_launch_counts()
    y, arm = tq.tq_moe_mlp_forward(d["x"], d["pgu"], d["lgu"], d["pd"], d["ld"], d["ids"], d["w"], tile_m=tile_m,
                                   pin=pin)
    check_no_device_error()
    after = tq.tq_launch_counts()
    assert arm == pin
    ran = "grouped" if pin == tq.ARM_GROUPED else "gemv"
    assert after[ran] == before[ran] + 2     # gate|up and down
    # the gate|up input: token rows gathered in the kernel, or a pair-sorted
    # copy (one gather launch) above the in-kernel gather's m-tile
    gathers = 1 if pin == tq.ARM_GROUPED and tile_m > tq.GATHER_MAX_TILE_M else 0
    assert after["gather"] == before["gather"] + gathers
    # SwiGLU: one launch between the projections on either arm
    assert after["swiglu"] == before["swiglu"] + 1
    ref = O.moe_mlp(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed_gu, prob.lut_gu, prob.packed_down,
                    prob.lut_down, prob.L)
    assert normwise(y.float().cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("tile_m,pin", [(16, tq.ARM_GROUPED), (64, tq.ARM_GROUPED), (256, tq.ARM_GROUPED),
                                        (16, tq.ARM_GEMV)])
def test_mlp_ragged_superstages_all_outputs(tile_m, pin):
    """H = 640, I = 576: the gate|up projection takes 10 k-steps (one full
    super-stage of 8, then 2) and the down projection 9 (8, then 1), so both
    carry the stream history across a super-stage boundary into a ragged last
    one; every output of both arms against the oracle."""
    prob = moe_inputs.make_mlp_custom(6, 2, 40, 640, 576, 14, seed=5, routing="zipf")
    d = _mlp_dev(prob)
    y, arm = tq.tq_moe_mlp_forward(d["x"], d["pgu"], d["lgu"], d["pd"], d["ld"], d["ids"], d["w"], tile_m=tile_m,
                                   pin=pin)
    check_no_device_error()
    assert arm == pin
    ref = O.moe_mlp(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed_gu, prob.lut_gu, prob.packed_down,
                    prob.lut_down, prob.L)
    assert normwise(y.float().cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("tile_m,pin", [(16, tq.ARM_GROUPED), (64, tq.ARM_GROUPED), (16, tq.ARM_GEMV)])
def test_mlp_dirty_workspace(tile_m, pin):
    """A workspace of NaN bit patterns, twice: the gate|up rows are written
    once each and the accumulator is cleared by the call itself."""
    prob = moe_inputs.make_mlp_problem("tiny_mlp_e8_k2_n16")
    d = _mlp_dev(prob)
    n, k = prob.topk_ids.shape
    E, I2, _ = prob.packed_gu.shape
    H = prob.x_bits.shape[1]
    ws = torch.empty(tq.tq_moe_mlp_workspace_size(n, k, E, H, I2 // 2, tile_m), dtype=torch.uint8, device="cuda")
    ref = O.moe_mlp(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed_gu, prob.lut_gu, prob.packed_down,
                    prob.lut_down, prob.L)
    for _ in range(2):
        ws.fill_(0xFF)
        y, arm = tq.tq_moe_mlp_forward(d["x"], d["pgu"], d["lgu"], d["pd"], d["ld"], d["ids"], d["w"],
                                       tile_m=tile_m, pin=pin, workspace=ws)
        check_no_device_error()
        assert arm == pin
        assert normwise(y.float().cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("pin", [tq.ARM_GROUPED, tq.ARM_GEMV])
def test_mlp_v4_n32_sampled_tokens(pin):
    prob = moe_inputs.make_mlp_problem("v4_mlp_n32")
    d = _mlp_dev(prob)
    y, arm = tq.tq_moe_mlp_forward(d["x"], d["pgu"], d["lgu"], d["pd"], d["ld"], d["ids"], d["w"], tile_m=16,
                                   pin=pin)
    check_no_device_error()
    assert arm == pin
    tokens = [0, 17, 31]
    ref = O.moe_mlp(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed_gu, prob.lut_gu, prob.packed_down,
                    prob.lut_down, prob.L, tokens=tokens)
    assert normwise(y[tokens].float().cpu().numpy(), ref) <= TOL


def test_mlp_prefill_native_tile_sampled_tokens():
    """8192 tokens, Zipf routing, the native m-tile (256): the per-pair gate|up
    output is large enough for the blocked row order and the round-robin unit
    walk; three tokens against the oracle."""
    prob = moe_inputs.make_mlp_problem("v4_mlp_prefill_n8192")
    d = _mlp_dev(prob)
    y, arm = tq.tq_moe_mlp_forward(d["x"], d["pgu"], d["lgu"], d["pd"], d["ld"], d["ids"], d["w"],
                                   tile_m=tq.TILE_NATIVE)
    assert arm == tq.ARM_GROUPED     # 8192 tokens: the first page's predicate picks the grouped arm
    check_no_device_error()
    tokens = [370, 1221, 2109]    # three tokens sharing most of their 9 experts (keeps the oracle short)
    ref = O.moe_mlp(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed_gu, prob.lut_gu, prob.packed_down,
                    prob.lut_down, prob.L, tokens=tokens)
    assert normwise(y[tokens].float().cpu().numpy(), ref) <= TOL


def test_grouped_gemm_pairs_all_outputs():
    prob = moe_inputs.make_custom(8, 2, 24, 256, 256, 12, seed=91)
    d = to_device(prob)
    s = prob.shape
    _, offsets, sp = tq.tq_route(d["ids"], s.E)
    cap = tq.tq_tile_map_capacity(s.n, s.top_k, s.E, 16)
    tiles, nt = tq.tq_build_tile_map(offsets, 16, cap)
    xs = tq.tq_gather_rows(d["x"], sp, s.top_k)
    out = torch.zeros((s.pairs, s.N), dtype=torch.float32, device="cuda")
    p = lambda t: __import__("ctypes").c_void_p(t.data_ptr())
    rc = tq.lib().tq_grouped_gemm_pairs(p(xs), p(d["packed"]), p(d["lut"]), s.L, p(sp), p(tiles), p(nt), cap,
                                        s.n, s.top_k, s.E, s.K, s.N, 16, p(out),
                                        __import__("ctypes").c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    check_no_device_error()
    x = O.bf16_bits_to_f64(prob.x_bits)
    spn = sp.cpu().numpy()
    ref = np.zeros((s.pairs, s.N))
    for slot, pair in enumerate(spn):
        t, e = pair // s.top_k, int(prob.topk_ids.reshape(-1)[pair])
        ref[slot] = O.decode_rows(prob.packed[e], prob.lut_bits, s.L) @ x[t]
    assert normwise(out.cpu().numpy(), ref) <= TOL


def test_swiglu_kernel():
    rng = np.random.Generator(np.random.PCG64(3))
    gu = (rng.standard_normal((37, 2 * 96)) * 3).astype(np.float32)
    h = tq.tq_swiglu(torch.from_numpy(gu).cuda())
    check_no_device_error()
    g, u = gu[:, :96].astype(np.float64), gu[:, 96:].astype(np.float64)
    ref = O.silu(g) * u
    got = h.float().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)


def test_mlp_offsets_past_2_gib():
    """70,000 tokens x top-4 of 16 experts, H = I = 1024, native m-tile 256: the
    per-pair gate|up accumulator is 280,000 x 2048 fp32 = 2.29 GB, so its rows
    past 262,144 sit beyond 2^31 bytes (as do the SwiGLU's reads of them).
    Sampled tokens against the oracle's whole MLP."""
    E, k, n, H, I, L = 16, 4, 70000, 1024, 1024, 16
    prob = moe_inputs.make_mlp_custom(E, k, n, H, I, L, seed=70000)
    d = _mlp_dev(prob)
    y, arm = tq.tq_moe_mlp_forward(d["x"], d["pgu"], d["lgu"], d["pd"], d["ld"], d["ids"], d["w"],
                                   tile_m=tq.TILE_NATIVE, pin=tq.ARM_AUTO)
    check_no_device_error()
    assert arm == tq.ARM_GROUPED
    rng = np.random.Generator(np.random.PCG64(12))
    toks = np.unique(np.concatenate([[0, n - 1], rng.choice(n, 62, replace=False)]))
    ref = O.moe_mlp(prob.x_bits[toks], prob.topk_ids[toks], prob.topk_w[toks], prob.packed_gu, prob.lut_gu,
                    prob.packed_down, prob.lut_down, prob.L)
    got = y[torch.from_numpy(toks).cuda()].float().cpu().numpy()
    assert normwise(got, ref) <= TOL


@pytest.mark.parametrize("tile_m,pin", [(16, tq.ARM_GROUPED), (tq.TILE_NATIVE, tq.ARM_GROUPED), (16, tq.ARM_GEMV)])
def test_mlp_in_cuda_graph(tile_m, pin):
    """The whole expert MLP captured in a CUDA graph (every launch a
    programmatic dependent of the one before) and replayed on new inputs
    copied into the captured buffers, on both arms and at the native m-tile
    (256 here: 150 pairs per expert); every replay against the oracle."""
    probs = [moe_inputs.make_mlp_custom(8, 2, 600, 256, 256, 12, seed=sd) for sd in (901, 902)]
    p0 = probs[0]
    n, k, E, H, I = p0.n, p0.top_k, p0.E, p0.H, p0.I
    if tile_m == tq.TILE_NATIVE:
        assert tq.tq_native_tile_m(n, k, E) == 256
    devs = [_mlp_dev(p) for p in probs]
    d = {key: v.clone() for key, v in devs[0].items()}
    ws = torch.empty(tq.tq_moe_mlp_workspace_size(n, k, E, H, I, tile_m), dtype=torch.uint8, device="cuda")
    y = torch.empty((n, H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    call = lambda: tq.tq_moe_mlp_forward(d["x"], d["pgu"], d["lgu"], d["pd"], d["ld"], d["ids"], d["w"],
                                         tile_m=tile_m, pin=pin, workspace=ws, y=y)
    with torch.cuda.stream(stream):
        call()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    for prob, src in zip(probs + probs[:1], devs + devs[:1]):
        for key in d:
            d[key].copy_(src[key])
        g.replay()
        torch.cuda.synchronize()
        check_no_device_error()
        ref = O.moe_mlp(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed_gu, prob.lut_gu, prob.packed_down,
                        prob.lut_down, prob.L)
        assert normwise(y.float().cpu().numpy(), ref) <= TOL


def _random_mlp_configs(count=8, seed=77):
    """Seeded expert-MLP shapes inside the documented limits (H % 128 == 0,
    I % 64 == 0, L even): (E, top_k, n, H, I, L, tile_m, pin)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    while len(out) < count:
        E = int(rng.integers(1, 17))
        k = int(rng.integers(1, min(E, 4) + 1))
        n = int(rng.integers(1, 121))
        H = 128 * int(rng.integers(1, 5))
        I = 64 * int(rng.integers(1, 9))
        L = 2 * int(rng.integers(2, 9))
        T = int(rng.choice([16, 64, 256, tq.TILE_NATIVE]))
        pin = int(rng.choice([tq.ARM_GROUPED, tq.ARM_GEMV]))
        out.append((E, k, n, H, I, L, T, pin))
    return out


@pytest.mark.parametrize("cfg", _random_mlp_configs(count=32),
                         ids=lambda c: "E{}_k{}_n{}_H{}_I{}_L{}_T{}_arm{}".format(*c))
def test_mlp_random_shapes_all_outputs(cfg):
    """The whole expert MLP on seeded random shapes, every output against the oracle."""
    E, k, n, H, I, L, T, pin = cfg
    prob = moe_inputs.make_mlp_custom(E, k, n, H, I, L, seed=sum(cfg) % 997)
    d = _mlp_dev(prob)
    y, arm = tq.tq_moe_mlp_forward(d["x"], d["pgu"], d["lgu"], d["pd"], d["ld"], d["ids"], d["w"], tile_m=T,
                                   pin=pin)
    check_no_device_error()
    assert arm == pin
    ref = O.moe_mlp(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed_gu, prob.lut_gu, prob.packed_down,
                    prob.lut_down, prob.L)
    assert normwise(y.float().cpu().numpy(), ref) <= TOL

