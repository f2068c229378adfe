"""Helpers for the GPU tests: move a seeded problem to the device and run the
library's path through its Python binding (which calls the C ABI)."""
import warnings

import numpy as np
import torch

import trellis_quantized_moe_sort_gb300 as tq


def to_device(prob):
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")            # read-only numpy buffers are copied anyway
        return {
            "x": torch.from_numpy(prob.x_bits.view(np.int16)).cuda(),
            "ids": torch.from_numpy(np.ascontiguousarray(prob.topk_ids)).cuda(),
            "w": torch.from_numpy(np.ascontiguousarray(prob.topk_w)).cuda(),
            "packed": torch.from_numpy(prob.packed).cuda(),
            "lut": torch.from_numpy(prob.lut_bits.view(np.int16)).cuda(),
        }


def check_no_device_error():
    torch.cuda.synchronize()
    code, where = tq.tq_device_error()
    assert (code, where) == (0, 0), f"device error word: code={code} where={where}"


def grouped_y32(prob, d, tile_m, x_layout=tq.X_TOKENS):
    """The grouped GEMM's fp32 output; x_layout picks token rows (gathered in
    the kernel) or the pair-sorted copy from tq_gather_rows."""
    s = prob.shape
    counts, offsets, sp = tq.tq_route(d["ids"], s.E)
    cap = tq.tq_tile_map_capacity(s.n, s.top_k, s.E, tile_m)
    tiles, nt = tq.tq_build_tile_map(offsets, tile_m, cap)
    y32 = torch.zeros((s.n, s.N), dtype=torch.float32, device="cuda")
    x = d["x"] if x_layout == tq.X_TOKENS else tq.tq_gather_rows(d["x"], sp, s.top_k)
    tq.tq_grouped_gemm(x, d["packed"], d["lut"], sp, d["w"], tiles, nt, s.top_k, tile_m, y32, x_layout=x_layout)
    check_no_device_error()
    return y32


def gemv_y32(prob, d):
    s = prob.shape
    y32 = torch.zeros((s.n, s.N), dtype=torch.float32, device="cuda")
    tq.tq_gemv(d["x"], d["packed"], d["lut"], d["ids"], d["w"], y32)
    check_no_device_error()
    return y32


def normwise(y, ref):
    """max |y - ref| / max |ref| (the output tolerance metric)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(y - ref).max() / max(np.abs(ref).max(), 1e-30))


def sample_rows(N, count=64, seed=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    fixed = [0, 1, 127, 128, N - 1, N - 128] if N >= 256 else [0, 1, N - 1]
    extra = rng.choice(N, size=min(count, N), replace=False)
    return np.unique(np.concatenate([fixed, extra]))
