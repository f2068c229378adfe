"""The seeded input recipe (CPU): the workloads have the stated shapes, the
draws are reproducible and independent per layer, and each input follows its
stated distribution and structure.  These inputs feed both the oracle and the
CUDA path, so a drifted recipe would move every parity case at once."""
import numpy as np
import pytest

import moe_inputs
import oracle.trellis_moe as O

# name -> (E, top_k, n, K, N, L, routing)
STATED = {
    "tiny_e8_k2_n16": (8, 2, 16, 256, 128, 12, "uniform"),
    "v4_decode_n32": (256, 6, 32, 4096, 2048, 16, "uniform"),
    "v4_n128_up": (256, 6, 128, 4096, 2048, 16, "uniform"),
    "v4_n128_down": (256, 6, 128, 2048, 4096, 16, "uniform"),
    "v4_fill_n512": (256, 6, 512, 4096, 2048, 16, "uniform"),
    "v4_fill_n683": (256, 6, 683, 4096, 2048, 16, "uniform"),
    "v4_fill_n1024": (256, 6, 1024, 4096, 2048, 16, "uniform"),
    "v4_prefill_n8192_up": (256, 6, 8192, 4096, 2048, 16, "zipf"),
    "v4_prefill_n8192_down": (256, 6, 8192, 2048, 4096, 16, "zipf"),
    "v4_prefill_n8192_up_zipf_perm": (256, 6, 8192, 4096, 2048, 16, "zipf_perm"),
}


def test_workload_shapes_are_the_stated_ones():
    assert set(moe_inputs.WORKLOADS) == set(STATED)
    for name, (E, k, n, K, N, L, routing) in STATED.items():
        s = moe_inputs.shape(name)
        assert (s.E, s.top_k, s.n, s.K, s.N, s.L, s.routing) == (E, k, n, K, N, L, routing), name


def test_draws_are_reproducible_and_layers_independent():
    a = moe_inputs.make_problem("tiny_e8_k2_n16")
    b = moe_inputs.make_problem("tiny_e8_k2_n16")
    c = moe_inputs.make_problem("tiny_e8_k2_n16", layer=1)
    for f in ("x_bits", "topk_ids", "topk_w", "packed", "lut_bits"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    assert not np.array_equal(a.packed, c.packed)
    assert not np.array_equal(a.lut_bits, c.lut_bits)
    assert not np.array_equal(a.x_bits, c.x_bits)


def test_value_distributions():
    p = moe_inputs.make_problem("v4_decode_n32", with_packed=False)
    s = p.shape
    x = O.bf16_bits_to_f64(p.x_bits)
    assert x.shape == (s.n, s.K)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02          # N(0, 1)
    lut = p.lut_bits.view(np.float16).astype(np.float64)
    assert lut.shape == (1 << s.L,)
    assert abs(lut.std() * np.sqrt(s.K) - 1.0) < 0.02                   # N(0, 1/K)
    # bf16 and fp16 values are the round-to-nearest images of their draws
    assert np.array_equal(moe_inputs.fp32_to_bf16_bits(x.astype(np.float32)), p.x_bits)


def test_packed_bytes_are_uniform():
    p = moe_inputs.make_problem("tiny_e8_k2_n16")
    s = p.shape
    assert p.packed.shape == (s.E, s.N, s.K // 4) and p.packed.dtype == np.uint8
    counts = np.bincount(p.packed.reshape(-1), minlength=256)
    expected = p.packed.size / 256
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 400   # 255 degrees of freedom: mean 255, sd ~23


@pytest.mark.parametrize("name", ["v4_decode_n32", "v4_prefill_n8192_up", "v4_prefill_n8192_up_zipf_perm"])
def test_routing_structure(name):
    p = moe_inputs.make_problem(name, with_packed=False)
    s = p.shape
    ids, w = p.topk_ids, p.topk_w
    assert ids.shape == (s.n, s.top_k) and ids.dtype == np.int32 and w.dtype == np.float32
    assert ids.min() >= 0 and ids.max() < s.E
    # k distinct experts per token, weights a softmax (positive, sum 1, in
    # descending order because the experts come in descending score order)
    assert all(len(set(row)) == s.top_k for row in ids)
    assert np.all(w > 0) and np.allclose(w.sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 1e-7)
    counts = np.bincount(ids.reshape(-1), minlength=s.E)
    if s.routing == "zipf":
        # popularity falls with the expert index: the first 16 experts take far
        # more than their 1/16 share of pairs, and the most popular is expert 0
        assert counts[:16].sum() > 0.25 * counts.sum()
        assert int(np.argmax(counts)) == 0
    elif s.routing == "zipf_perm":
        # the same skew with the ranks shuffled over the ids: the 16 most
        # popular experts still take far more than their share, but they are
        # not the lowest ids
        top = np.argsort(-counts, kind="stable")[:16]
        assert counts[top].sum() > 0.25 * counts.sum()
        assert top.max() >= 64 and int(np.argmax(counts)) != 0
    else:
        # uniform: no expert far above its share n*k/E
        assert counts.max() < 5 * s.n * s.top_k / s.E + 5
