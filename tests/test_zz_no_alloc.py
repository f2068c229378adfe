"""tq_moe_forward_static — the allocation-free entry point — against
tq_moe_forward on the same inputs, called through the C ABI.

It serves callers that cannot allocate device memory (a plugin handed only its
input and output buffers by a host framework, a serving loop that forbids
cudaMalloc after start-up); its scratch is one fixed device array inside the
library, shared by every call.  This file is collected last; it must pass both
alone in a fresh process and after the other GPU tests (the array then holds
the previous calls' contents)."""
import ctypes

import numpy as np
import pytest
import torch

import moe_inputs
import trellis_quantized_moe_sort_gb300 as tq

pytestmark = pytest.mark.gpu
TOL = 1e-2          # max|y - ref| / max|ref|, as in the other parity tests


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_quantized_moe_sort_gb300 import build
    build.build()
    tq.tq_init(0)


def _dev(prob):
    import warnings
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        return (c(prob.x_bits.view(np.int16)), c(prob.packed), c(prob.lut_bits.view(np.int16)),
                c(prob.topk_ids), c(prob.topk_w))


def _call_static(x, packed, lut, ids, w, tile_m, pin, y):
    """Direct C-ABI call of tq_moe_forward_static."""
    n, K = x.shape
    E, N, _ = packed.shape
    L = lut.numel().bit_length() - 1
    arm = ctypes.c_int(-1)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = tq.lib().tq_moe_forward_static(p(x), p(packed), p(lut), L, p(ids), p(w), n, ids.shape[1], E, K, N,
                                        tile_m, pin, p(y), ctypes.byref(arm),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, arm.value


def _normwise(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def _oracle_rows(prob, rows):
    import oracle.trellis_moe as O
    return O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, prob.shape.L,
                         rows=rows)


def _sample_rows(N, count, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    fixed = [0, 1, 127, 128, N - 1] if N >= 256 else [0, N - 1]
    return np.unique(np.concatenate([fixed, rng.choice(N, size=min(count, N), replace=False)]))


# tile_m 16: the kernel gathers its token rows itself; tile_m 128: the call
# also carves the pair-sorted activation copy out of the array (v4_n128_up at
# 128 needs about 7.3 MB of it)
@pytest.mark.parametrize("name,tile_m,pin", [("v4_decode_n32", 16, tq.ARM_GROUPED),
                                              ("v4_n128_up", 128, tq.ARM_GROUPED),
                                              ("tiny_e8_k2_n16", 16, tq.ARM_AUTO)])
def test_static_matches_workspace_entry_point_two_calls(name, tile_m, pin):
    s = moe_inputs.shape(name)
    need = tq.tq_moe_workspace_size(s.n, s.top_k, s.E, s.K, s.N, tile_m)
    assert need <= tq.STATIC_SCRATCH_BYTES
    probs = [moe_inputs.make_problem(name, layer=0), moe_inputs.make_problem(name, layer=1)]
    for prob in probs:                                     # two calls in a row
        x, packed, lut, ids, w = _dev(prob)
        want, want_arm = tq.tq_moe_forward(x, packed, lut, ids, w, tile_m=tile_m, pin=pin)
        y = torch.empty_like(want)
        before = tq.tq_launch_counts()
        rc, arm = _call_static(x, packed, lut, ids, w, tile_m, pin, y)
        assert rc == 0, tq.tq_status_string(rc)
        torch.cuda.synchronize()
        after = tq.tq_launch_counts()
        assert tq.tq_device_error() == (0, 0)
        assert arm == want_arm
        if arm == tq.ARM_GROUPED:
            assert after["gather"] - before["gather"] == (1 if tile_m > tq.GATHER_MAX_TILE_M else 0)
        else:   # the GEMV arm is one launch: nothing else runs
            assert {k: after[k] - before[k] for k in after} == {k: int(k == "gemv") for k in after}
        assert _normwise(y, want) <= TOL
        rows = _sample_rows(s.N, 24, seed=11)
        got = y[:, torch.from_numpy(rows).cuda()]
        ref = torch.from_numpy(_oracle_rows(prob, rows))
        assert _normwise(got, ref) <= TOL


def test_static_rejects_shapes_beyond_its_array():
    # 8192 tokens x 2048 outputs need a 64 MiB fp32 accumulator: over the 16 MiB array
    assert tq.tq_moe_workspace_size(8192, 6, 256, 256, 2048, 16) > tq.STATIC_SCRATCH_BYTES
    prob = moe_inputs.make_custom(8, 2, 4, 256, 128, 12, seed=1)
    x, packed, lut, ids, w = _dev(prob)
    y = torch.empty((4, 128), dtype=torch.bfloat16, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    before = tq.tq_launch_counts()
    rc = tq.lib().tq_moe_forward_static(p(x), p(packed), p(lut), 12, p(ids), p(w), 8192, 6, 256, 256, 2048,
                                        16, 0, p(y), None, None)
    assert rc == -8                                        # TQ_ERR_WORKSPACE
    assert tq.tq_launch_counts() == before                 # nothing was launched
