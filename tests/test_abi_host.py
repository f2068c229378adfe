"""C ABI without a GPU: the library loads, exports every function the header
declares, and its host-only gate arithmetic (tile fill, amortization predicate,
flip point, tile-map capacity, arm selection) equals the oracle bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle.trellis_moe as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tqmoe.h")


@pytest.fixture(scope="module")
def tq():
    from trellis_quantized_moe_sort_gb300 import build
    build.build()
    import trellis_quantized_moe_sort_gb300 as tq
    return tq


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(tq):
    declared = _declared_functions()
    assert len(declared) >= 17
    h = ctypes.CDLL(tq.lib_path)
    missing = [name for name in declared if not hasattr(h, name)]
    assert not missing, missing
    assert sorted(tq.EXPORTED_SYMBOLS) == declared


def test_status_strings(tq):
    for code in range(0, -9, -1):
        s = tq.tq_status_string(code)
        assert s and "unknown" not in s
    assert "unknown" in tq.tq_status_string(-99)


SHAPES = [(k, E) for (k, E) in ((1, 1), (1, 8), (2, 8), (6, 8), (8, 8), (2, 16), (4, 32),
                                 (6, 64), (8, 128), (6, 256), (8, 256), (2, 256), (7, 1000))]


def test_pairs_per_woken_bitexact(tq):
    for k, E in SHAPES:
        for n in list(range(0, 50)) + [127, 128, 512, 682, 683, 1024, 1572, 2000, 8192, 10**6]:
            a = tq.tq_pairs_per_woken_expert(n, k, E)
            b = O.pairs_per_woken_expert(n, k, E)
            assert a == b, (n, k, E, a, b)


def test_gate_and_flip_bitexact(tq):
    for k, E in SHAPES:
        for T in (1, 4, 16, 64, 128, 256):
            flip = tq.tq_grouped_min_tokens(k, E, T)
            assert flip == O.grouped_min_tokens(k, E, T), (k, E, T)
            for n in sorted({0, 1, 8, 9, flip - 1, flip, flip + 1, 2 * flip}):
                if n < 0:
                    continue
                assert tq.tq_tiles_amortize(n, k, E, T) == O.tiles_amortize(n, k, E, T)
                assert tq.tq_tile_map_capacity(n, k, E, T) == O.tile_map_capacity(n, k, E, T)
                for pin, name in ((0, "auto"), (1, "gemv"), (2, "grouped")):
                    arm = tq.tq_select_arm(n, k, E, T, pin)
                    assert {1: "gemv", 2: "grouped"}[arm] == O.dispatch_arm(n, k, E, T, name)
    assert tq.tq_grouped_min_tokens(6, 256, 16) == 683


def test_gate_random_shapes_bitexact(tq):
    """2000 seeded random routing shapes (E up to 1024, k up to min(E, 16),
    TILE_M 1..256, n log-uniform up to 50,000 and around each shape's flip):
    the amortization predicate, the flip, the tile-map capacity, the pairs
    per woken expert and the arm under each pin agree with the oracle."""
    rng = np.random.default_rng(20261203)
    for _ in range(2000):
        E = int(rng.integers(1, 1025))
        k = int(rng.integers(1, min(E, 16) + 1))
        T = int(rng.integers(1, 257))
        flip = tq.tq_grouped_min_tokens(k, E, T)
        assert flip == O.grouped_min_tokens(k, E, T), (k, E, T)
        ns = {int(np.exp(rng.uniform(0.0, np.log(50_000)))), int(rng.integers(0, 10)), flip - 1, flip}
        for n in sorted(v for v in ns if v >= 0):
            assert tq.tq_tiles_amortize(n, k, E, T) == O.tiles_amortize(n, k, E, T), (n, k, E, T)
            assert tq.tq_tile_map_capacity(n, k, E, T) == O.tile_map_capacity(n, k, E, T), (n, k, E, T)
            got, want = tq.tq_pairs_per_woken_expert(n, k, E), O.pairs_per_woken_expert(n, k, E)
            assert got == want or (np.isnan(got) and np.isnan(want)), (n, k, E, got, want)
            for pin, name in ((0, "auto"), (1, "gemv"), (2, "grouped")):
                arm = tq.tq_select_arm(n, k, E, T, pin)
                assert {1: "gemv", 2: "grouped"}[arm] == O.dispatch_arm(n, k, E, T, name), (n, k, E, T, name)


def _header_crossover():
    """The measured policy's threshold as the header defines it (a library
    tuning value, read from the header rather than restated here)."""
    m = re.search(r"#define\s+TQ_MEASURED_CROSSOVER_PPW\s+([0-9.eE+-]+)", open(HEADER).read())
    assert m, "TQ_MEASURED_CROSSOVER_PPW not found in the header"
    return float(m.group(1))


def test_measured_policy_follows_closed_form(tq):
    """pin = TQ_ARM_MEASURED: the grouped arm iff n > 0 and the oracle's
    pairs-per-woken-expert closed form reaches the header's threshold, with
    no token floor and no tile-fill term (TILE_M does not matter)."""
    thr = _header_crossover()
    assert 1.0 < thr < 16.0
    for k, E in SHAPES:
        for n in list(range(0, 64)) + [127, 128, 512, 682, 683, 1024, 8192]:
            want = "grouped" if n > 0 and O.pairs_per_woken_expert(n, k, E) >= thr else "gemv"
            for T in (1, 16, 256):
                arm = tq.tq_select_arm(n, k, E, T, 3)
                assert {1: "gemv", 2: "grouped"}[arm] == want, (n, k, E, T)
    # k == E puts exactly n pairs on every expert: one token never selects,
    # two tokens always do (the threshold lies strictly between 1 and 2)
    if thr <= 2.0:
        for E in (1, 4, 64):
            assert tq.tq_select_arm(1, E, E, 16, 3) == 1
            assert tq.tq_select_arm(2, E, E, 16, 3) == 2


def test_host_functions_reject_invalid_arguments(tq):
    for args in ((5, 0, 8, 16), (5, 9, 8, 16), (5, 2, 8, 0), (-1, 2, 8, 16)):
        with pytest.raises(tq.TQError):
            tq.tq_tiles_amortize(*args)
        with pytest.raises(tq.TQError):
            tq.tq_tile_map_capacity(*args)
    with pytest.raises(tq.TQError):
        tq.tq_select_arm(10, 2, 8, 16, pin=7)
    assert np.isnan(tq.tq_pairs_per_woken_expert(4, 9, 8))
    # counts, offsets, sorted pairs, tile map, tile count, fp32 accumulator
    # (each region 256-byte aligned); no copy of the activations
    a256 = lambda b: (b + 255) // 256 * 256
    cap = tq.tq_tile_map_capacity(16, 2, 8, 16)
    assert tq.tq_moe_workspace_size(16, 2, 8, 256, 128, 16) == (
        a256(8 * 4) + a256(9 * 4) + a256(32 * 4) + a256(3 * cap * 4) + a256(4) + a256(16 * 128 * 4))
    # above the in-kernel gather's m-tile, the pair-sorted activations and the
    # sort's inverse (one slot per pair) too
    T = tq.GATHER_MAX_TILE_M + 1
    cap = tq.tq_tile_map_capacity(16, 2, 8, T)
    assert tq.tq_moe_workspace_size(16, 2, 8, 256, 128, T) == (
        a256(8 * 4) + a256(9 * 4) + a256(32 * 4) + a256(3 * cap * 4) + a256(4) + a256(16 * 128 * 4)
        + a256(32 * 256 * 2) + a256(32 * 4))


def test_device_calls_reject_bad_arguments_before_any_device_work(tq):
    """Argument checks come first: with no GPU present, a bad layout, size,
    window width, m-tile or workspace is reported as such (the addresses
    below are never dereferenced)."""
    lib = tq.lib()
    A = 0x10000            # 16-byte aligned stand-in address

    def gg(x_layout=0, L=16, K=256, N=128, tile_m=16):
        return lib.tq_grouped_gemm(A, x_layout, A, A, L, A, A, A, A, 16, 4, 2, 8, K, N, tile_m, A, None)

    INVALID, WORKSPACE = -1, -8
    assert gg(x_layout=7) == INVALID
    assert gg(N=100) == INVALID           # the grouped arm needs N % 128 == 0
    assert gg(K=100) == INVALID           # K % 64 != 0
    assert gg(L=15) == INVALID            # odd window
    assert gg(L=18) == INVALID            # window wider than 16 bits
    assert gg(tile_m=0) == INVALID and gg(tile_m=257) == INVALID
    assert lib.tq_grouped_gemm_dense(A, 5, A, A, A, A, A, 16, 4, 2, 8, 256, 128, 16, A, None) == INVALID
    arm = ctypes.c_int(-1)
    # grouped pin with a workspace one byte short
    need = tq.tq_moe_workspace_size(4, 2, 8, 256, 128, 16)
    rc = lib.tq_moe_forward(A, A, A, 12, A, A, 4, 2, 8, 256, 128, 16, 2, A, need - 1, A, ctypes.byref(arm), None)
    assert rc == WORKSPACE
    rc = lib.tq_moe_forward(A, A, A, 12, A, A, 4, 2, 8, 256, 128, 16, 9, A, need, A, ctypes.byref(arm), None)
    assert rc == INVALID                  # unknown pin


def test_env_tile_m_overrides_native_tile(tq, monkeypatch):
    """TQ_TILE_M sets the kernel m-tile of TILE_NATIVE calls (seen in the
    workspace they need); 0, out-of-range and non-numeric values leave the
    native tile."""
    n, k, E, K, N = 512, 6, 256, 4096, 2048
    native = tq.tq_moe_workspace_size(n, k, E, K, N, 0)
    assert native == tq.tq_moe_workspace_size(n, k, E, K, N, tq.tq_native_tile_m(n, k, E))
    monkeypatch.setenv("TQ_TILE_M", "16")
    assert tq.tq_moe_workspace_size(n, k, E, K, N, 0) == tq.tq_moe_workspace_size(n, k, E, K, N, 16)
    assert tq.tq_moe_workspace_size(n, k, E, K, N, 0) != native
    assert tq.tq_moe_mlp_workspace_size(n, k, E, K, N, 0) == tq.tq_moe_mlp_workspace_size(n, k, E, K, N, 16)
    for bad in ("0", "257", "-3", "x16", ""):
        monkeypatch.setenv("TQ_TILE_M", bad)
        assert tq.tq_moe_workspace_size(n, k, E, K, N, 0) == native, bad


def test_native_tile(tq):
    """TQ_TILE_NATIVE: 16 while the expected pairs per woken expert stay at
    most 4, 128 above, 256 once they reach 128 (the oracle's closed form
    decides which); the workspace of tile_m = 0 is that of the native tile."""
    assert tq.TILE_NATIVE == 0
    for n, k, E in ((1, 6, 256), (32, 6, 256), (128, 6, 256), (512, 6, 256), (1024, 6, 256), (8192, 6, 256),
                    (5000, 2, 8), (0, 2, 8)):
        ppw = O.pairs_per_woken_expert(n, k, E) if n > 0 else 0.0
        want = 256 if ppw >= 128 else (128 if ppw > 4 else 16)
        assert tq.tq_native_tile_m(n, k, E) == want, (n, k, E)
        assert tq.tq_moe_workspace_size(n, k, E, 4096, 2048, 0) == tq.tq_moe_workspace_size(n, k, E, 4096, 2048, want)
        assert (tq.tq_moe_mlp_workspace_size(n, k, E, 4096, 2048, 0)
                == tq.tq_moe_mlp_workspace_size(n, k, E, 4096, 2048, want))
    assert tq.tq_native_tile_m(32, 6, 256) == 16 and tq.tq_native_tile_m(512, 6, 256) == 128
    assert tq.tq_native_tile_m(8192, 6, 256) == 256
    with pytest.raises(tq.TQError):
        tq.tq_native_tile_m(4, 9, 8)
    assert tq.tq_moe_workspace_size(16, 2, 8, 256, 128, 257) == 0


def test_device_calls_fail_loudly_without_a_gpu(tq):
    """No CPU fallback: without a CUDA device every device call raises before
    the library is asked to do anything (with one, a host tensor is refused
    as not a CUDA tensor)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    with pytest.raises(RuntimeError, match="needs a CUDA device"):
        tq.tq_route(torch.zeros((4, 2), dtype=torch.int32), 8)
    with pytest.raises(RuntimeError, match="needs a CUDA device"):
        tq.tq_combine(torch.zeros(8, dtype=torch.float32))

