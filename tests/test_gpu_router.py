"""Device router (top-k + softmax from fp32 logits) against the oracle:
expert ids bit-exact (the selection compares the same fp32 values), weights
within 1e-6 relative (fp32 exp vs fp64), and the fused route on its ids."""
import numpy as np
import pytest
import torch

import oracle.trellis_moe as O
import trellis_quantized_moe_sort_gb300 as tq
from gpu_util import check_no_device_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_quantized_moe_sort_gb300 import build
    build.build()
    tq.tq_init(0)


def _cases():
    rng = np.random.Generator(np.random.PCG64(55))
    ties = np.round(rng.standard_normal((300, 64)) * 2).astype(np.float32)      # many exact ties
    bad = rng.standard_normal((40, 256)).astype(np.float32)
    bad[::3, ::7] = np.nan
    bad[1::3, :200] = -np.inf
    bad[2] = np.nan                                                            # no finite logit
    return {
        "v4_n8192_E256_k6": (rng.standard_normal((8192, 256)).astype(np.float32), 6),
        "E8_k8_all": (rng.standard_normal((100, 8)).astype(np.float32), 8),
        "E1024_k8": (rng.standard_normal((257, 1024)).astype(np.float32), 8),
        "E300_k32": (rng.standard_normal((33, 300)).astype(np.float32), 32),
        "ties": (ties, 5),
        "non_finite": (bad, 6),
        "one_token_E1_k1": (np.zeros((1, 1), np.float32), 1),
    }


CASES = _cases()


@pytest.mark.parametrize("name", sorted(CASES))
def test_router_topk_matches_oracle(name):
    logits, k = CASES[name]
    ids, w = tq.tq_router_topk(torch.from_numpy(logits).cuda(), k)
    check_no_device_error()
    want_ids, want_w = O.router_topk(logits, k)
    assert np.array_equal(ids.cpu().numpy(), want_ids)
    got = w.cpu().numpy().astype(np.float64)
    assert np.allclose(got, want_w, rtol=1e-6, atol=1e-7)


def test_route_logits_equals_route_of_oracle_ids():
    logits, k = CASES["v4_n8192_E256_k6"]
    ids, w, counts, offsets, sp = tq.tq_route_logits(torch.from_numpy(logits).cuda(), k)
    check_no_device_error()
    want_ids, _ = O.router_topk(logits, k)
    c, o, s = O.route(want_ids, 256)
    assert np.array_equal(ids.cpu().numpy(), want_ids)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(sp.cpu().numpy(), s)


def _random_router_case(i, seed=909):
    """Seeded logits number i: E up to 1024, top_k up to min(E, 32), up to
    3000 tokens; every second case rounded to a few values so that exact ties
    are common.  Drawn when the test runs."""
    rng = np.random.Generator(np.random.PCG64([seed, i]))
    E = int(rng.integers(1, 1025))
    k = int(rng.integers(1, min(E, 32) + 1))
    n = int(rng.integers(1, 3001))
    logits = rng.standard_normal((n, E)).astype(np.float32)
    if i % 2:
        logits = np.round(logits * 2).astype(np.float32)
    return logits, k


@pytest.mark.parametrize("i", range(40))
def test_router_topk_random_matches_oracle(i):
    logits, k = _random_router_case(i)
    ids, w = tq.tq_router_topk(torch.from_numpy(logits).cuda(), k)
    check_no_device_error()
    want_ids, want_w = O.router_topk(logits, k)
    assert np.array_equal(ids.cpu().numpy(), want_ids)
    assert np.allclose(w.cpu().numpy().astype(np.float64), want_w, rtol=1e-6, atol=1e-7)

