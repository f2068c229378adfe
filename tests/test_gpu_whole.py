"""The whole routed-expert product through tq_moe_forward at full size
(sampled output rows against the oracle), and the decode-ceiling probe."""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle.trellis_moe as O
import trellis_quantized_moe_sort_gb300 as tq
from gpu_util import to_device, normwise, sample_rows, check_no_device_error

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_quantized_moe_sort_gb300 import build
    build.build()
    tq.tq_init(0)


@pytest.mark.parametrize("name,tile_m,pin", [("v4_decode_n32", 16, tq.ARM_GROUPED),
                                              ("v4_decode_n32", 16, tq.ARM_GEMV),
                                              ("v4_n128_down", 128, tq.ARM_AUTO),
                                              ("v4_fill_n683", 16, tq.ARM_AUTO)])
def test_moe_forward_full_size(name, tile_m, pin):
    prob = moe_inputs.make_problem(name)
    d = to_device(prob)
    s = prob.shape
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=tile_m, pin=pin)
    check_no_device_error()
    want_arm = pin if pin else tq.tq_select_arm(s.n, s.top_k, s.E, tile_m)
    assert arm == want_arm
    rows = sample_rows(s.N, 32, seed=7)
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, s.L, rows=rows)
    got = y[:, torch.from_numpy(rows).cuda()].float().cpu().numpy()
    assert normwise(got, ref) <= TOL


@pytest.mark.parametrize("n", [1, 2, 8])
def test_moe_forward_small_batch_decode_steps(n):
    """The decode steps at 1, 2 and 8 tokens at the V4 up shape through
    tq_moe_forward with the default selection: the n <= 8 floor sends them to
    the per-pair GEMV (launch counters), and sampled output rows match the
    oracle."""
    prob = moe_inputs.make_problem("v4_decode_n32", n=n)
    d = to_device(prob)
    s = prob.shape
    assert tq.tq_select_arm(n, s.top_k, s.E, 16) == tq.ARM_GEMV
    before = tq.tq_launch_counts()
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=tq.TILE_NATIVE)
    check_no_device_error()
    after = tq.tq_launch_counts()
    assert arm == tq.ARM_GEMV
    assert after["gemv"] == before["gemv"] + 1 and after["grouped"] == before["grouped"]
    rows = sample_rows(s.N, 32, seed=11 + n)
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, s.L, rows=rows)
    assert normwise(y.float().cpu().numpy()[:, rows], ref) <= TOL


@pytest.mark.parametrize("n", [13, 14])
def test_moe_forward_measured_policy_at_its_crossover(n):
    """pin = ARM_MEASURED at the V4 up shape on either side of the library's
    crossover (13 tokens: 1.148 pairs per woken expert -> GEMV; 14: 1.161 ->
    grouped, the threshold being TQ_MEASURED_CROSSOVER_PPW = 1.16): the arm the
    closed form predicts runs (launch counters) and sampled rows match the
    oracle."""
    prob = moe_inputs.make_problem("v4_decode_n32", n=n)
    d = to_device(prob)
    s = prob.shape
    want = tq.tq_select_arm(n, s.top_k, s.E, 16, tq.ARM_MEASURED)
    assert want == (tq.ARM_GROUPED if n == 14 else tq.ARM_GEMV)
    before = tq.tq_launch_counts()
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=tq.TILE_NATIVE,
                               pin=tq.ARM_MEASURED)
    check_no_device_error()
    after = tq.tq_launch_counts()
    assert arm == want
    ran = "grouped" if arm == tq.ARM_GROUPED else "gemv"
    assert after[ran] == before[ran] + 1
    rows = sample_rows(s.N, 32, seed=21 + n)
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, s.L, rows=rows)
    assert normwise(y.float().cpu().numpy()[:, rows], ref) <= TOL


def test_lut_probe_rate_is_sane():
    rate = tq.tq_probe_lut_rate(8, 128)
    # between random-address bank conflicts at their worst and 32 banks per clock
    assert 2.0 < rate <= 32.0, rate


@pytest.mark.parametrize("pin", [tq.ARM_GROUPED, tq.ARM_GEMV])
def test_moe_forward_in_cuda_graph(pin):
    """tq_moe_forward captured in a CUDA graph (its grouped kernel is a
    programmatic dependent of the routing launch) replays to the eager result, on new
    inputs copied into the captured buffers, within the fp32 summation-order
    noise of the atomics."""
    s = moe_inputs.shape("v4_decode_n32")
    probs = [moe_inputs.make_problem("v4_decode_n32", layer=i) for i in range(2)]
    devs = [to_device(p) for p in probs]
    d = {k: v.clone() for k, v in devs[0].items()}
    ws = torch.empty(tq.tq_moe_workspace_size(s.n, s.top_k, s.E, s.K, s.N, 16), dtype=torch.uint8, device="cuda")
    y = torch.empty((s.n, s.N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=16, pin=pin, workspace=ws, y=y)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=16, pin=pin, workspace=ws, y=y)
    for src in devs + devs[:1]:
        for k in d:
            d[k].copy_(src[k])
        g.replay()
        torch.cuda.synchronize()
        check_no_device_error()
        eager, _ = tq.tq_moe_forward(src["x"], src["packed"], src["lut"], src["ids"], src["w"], tile_m=16, pin=pin)
        torch.cuda.synchronize()
        assert normwise(y.float().cpu().numpy(), eager.float().cpu().numpy()) <= 1e-2


@pytest.mark.parametrize("name,pin,want_arm,want_tile", [
    ("tiny_e8_k2_n16", tq.ARM_GROUPED, tq.ARM_GROUPED, 128),
    ("tiny_e8_k2_n16", tq.ARM_AUTO, tq.ARM_GEMV, 128),
    ("v4_decode_n32", tq.ARM_GROUPED, tq.ARM_GROUPED, 16),
    ("v4_prefill_n8192_up", tq.ARM_AUTO, tq.ARM_GROUPED, 256),
    ("v4_prefill_n8192_down", tq.ARM_AUTO, tq.ARM_GROUPED, 256),
    ("v4_prefill_n8192_up_zipf_perm", tq.ARM_AUTO, tq.ARM_GROUPED, 256)])
def test_moe_forward_native_tile(name, pin, want_arm, want_tile):
    """tile_m = TQ_TILE_NATIVE: the pages' TILE_M gates the arm, the kernel runs
    its native tile (256 at the prefill sizes: the down projection's K = 2048
    and 128 MiB accumulator take the blocked row order and the round-robin
    unit walk); the launch counters show the arm and, through the gather
    launch that only m-tiles above 16 use, the tile; output rows match the
    oracle."""
    prob = moe_inputs.make_problem(name)
    d = to_device(prob)
    s = prob.shape
    assert tq.tq_native_tile_m(s.n, s.top_k, s.E) == want_tile
    before = tq.tq_launch_counts()
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=tq.TILE_NATIVE, pin=pin)
    check_no_device_error()
    after = tq.tq_launch_counts()
    assert arm == want_arm
    if want_arm == tq.ARM_GROUPED:
        assert after["grouped"] == before["grouped"] + 1 and after["gemv"] == before["gemv"]
        assert after["gather"] - before["gather"] == (1 if want_tile > tq.GATHER_MAX_TILE_M else 0)
    else:
        assert after["gemv"] == before["gemv"] + 1 and after["grouped"] == before["grouped"]
    rows = sample_rows(s.N, 24, seed=3) if s.N > 256 else np.arange(s.N)
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, s.L, rows=rows)
    assert normwise(y.float().cpu().numpy()[:, rows], ref) <= TOL


def test_moe_forward_offsets_past_2_gib():
    """65,536 tokens x top-6 of 256 experts at K = 4096, N = 2048 through the
    whole product at its native m-tile (256): the pair-sorted activations are
    393,216 rows x 8 KiB = 3.2 GB, so every address past row 262,144 is beyond
    2^31 bytes, and the route runs its largest grid (64 blocks of 6,144 pairs).
    Sampled tokens (their pairs land anywhere in the sorted order) and rows
    against the oracle."""
    E, k, n, K, N, L = 256, 6, 65536, 4096, 2048, 16
    prob = moe_inputs.make_custom(E, k, n, K, N, L, seed=65536)
    d = to_device(prob)
    y, arm = tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=tq.TILE_NATIVE,
                               pin=tq.ARM_AUTO)
    check_no_device_error()
    assert arm == tq.ARM_GROUPED and tq.tq_native_tile_m(n, k, E) == 256
    rng = np.random.Generator(np.random.PCG64(11))
    toks = np.unique(np.concatenate([[0, n - 1], rng.choice(n, 254, replace=False)]))
    rows = sample_rows(N, 32, seed=5)
    ref = O.moe_forward(prob.x_bits[toks], prob.topk_ids[toks], prob.topk_w[toks], prob.packed, prob.lut_bits, L,
                        rows=rows)
    got = y[torch.from_numpy(toks).cuda()][:, torch.from_numpy(rows).cuda()].float().cpu().numpy()
    assert normwise(got, ref) <= TOL


def test_moe_forward_in_cuda_graph_native_tile():
    """The whole product at its native m-tile 256 (the pair-sorted gather
    launch, then the grouped kernel with eight epilogue warps) captured in a
    CUDA graph and replayed on new inputs copied into the captured buffers;
    every replay against the oracle on all outputs."""
    probs = [moe_inputs.make_custom(16, 4, 2048, 512, 256, 12, seed=sd) for sd in (801, 802)]
    s = probs[0].shape
    assert tq.tq_native_tile_m(s.n, s.top_k, s.E) == 256
    devs = [to_device(p) for p in probs]
    d = {k: v.clone() for k, v in devs[0].items()}
    ws = torch.empty(tq.tq_moe_workspace_size(s.n, s.top_k, s.E, s.K, s.N, tq.TILE_NATIVE), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty((s.n, s.N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    call = lambda: tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=tq.TILE_NATIVE,
                                     pin=tq.ARM_GROUPED, workspace=ws, y=y)
    with torch.cuda.stream(stream):
        call()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    for prob, src in zip(probs + probs[:1], devs + devs[:1]):
        for k in d:
            d[k].copy_(src[k])
        g.replay()
        torch.cuda.synchronize()
        check_no_device_error()
        ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, s.L)
        assert normwise(y.float().cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("tile_m", [16, tq.TILE_NATIVE])
def test_moe_forward_concurrent_streams(tile_m):
    """Two whole-product calls enqueued on two streams at once, each with its
    own workspace and output: the library keeps no per-call state of its own
    (the workspace holds it all), so each result matches its oracle."""
    probs = [moe_inputs.make_custom(16, 4, 2048, 512, 256, 12, seed=sd) for sd in (811, 812)]
    s = probs[0].shape
    devs = [to_device(p) for p in probs]
    wss = [torch.empty(tq.tq_moe_workspace_size(s.n, s.top_k, s.E, s.K, s.N, tile_m), dtype=torch.uint8,
                       device="cuda") for _ in probs]
    ys = [torch.empty((s.n, s.N), dtype=torch.bfloat16, device="cuda") for _ in probs]
    streams = [torch.cuda.Stream() for _ in probs]
    torch.cuda.synchronize()
    for _ in range(3):
        for d, ws, y, st in zip(devs, wss, ys, streams):
            tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=tile_m, pin=tq.ARM_GROUPED,
                              workspace=ws, y=y, stream=st)
    torch.cuda.synchronize()
    check_no_device_error()
    for prob, y in zip(probs, ys):
        ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, s.L)
        assert normwise(y.float().cpu().numpy(), ref) <= TOL

