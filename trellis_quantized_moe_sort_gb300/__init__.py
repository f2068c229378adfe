"""Python binding of libtqmoe.so (C ABI: include/tqmoe.h).

Argument marshalling only: every step of the MoE path runs in the library's
CUDA kernels.  PyTorch provides device memory and the current stream.  There
is no CPU fallback: if the library is missing or no sm_103a device is present,
calls raise.

Tensor conventions: bf16 activations (torch.bfloat16 or 16-bit integer views),
packed bitstreams torch.uint8 [E, N, K/4], LUT fp16 (torch.float16 or 16-bit
integer view) [2^L], router ids torch.int32 [n, top_k], router weights
torch.float32 [n, top_k].
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "TQError", "lib", "lib_path", "tq_init", "tq_arch_witness", "tq_pairs_per_woken_expert",
    "tq_tiles_amortize", "tq_grouped_min_tokens", "tq_tile_map_capacity", "tq_native_tile_m", "TILE_NATIVE", "tq_select_arm",
    "tq_route", "tq_router_topk", "tq_route_logits", "tq_build_tile_map", "tq_gather_rows", "tq_prepare", "tq_grouped_gemm", "tq_gemv", "tq_combine",
    "tq_moe_workspace_size", "tq_moe_forward", "tq_moe_forward_static", "tq_device_error", "tq_launch_counts",
    "tq_status_string", "tq_probe_lut_rate", "tq_probe_wait_timeout", "tq_grouped_gemm_pairs", "tq_swiglu",
    "tq_moe_mlp_workspace_size", "tq_moe_mlp_forward", "tq_dequantize", "tq_grouped_gemm_dense",
    "tq_moe_dequant_workspace_size", "tq_moe_forward_dequant", "ARM_AUTO", "ARM_GEMV", "ARM_GROUPED", "ARM_MEASURED", "EXPORTED_SYMBOLS",
    "X_TOKENS", "X_PAIR_SORTED", "GATHER_MAX_TILE_M",
]

ARM_AUTO, ARM_GEMV, ARM_GROUPED, ARM_MEASURED = 0, 1, 2, 3
TILE_NATIVE = 0          # tile_m of the whole-product calls: the kernel's native m-tile
X_TOKENS, X_PAIR_SORTED = 0, 1   # activation layouts of tq_grouped_gemm / tq_grouped_gemm_dense
GATHER_MAX_TILE_M = 16   # the whole-product calls gather rows in the kernel up to this m-tile
_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libtqmoe.so")

_c_i64, _c_int, _c_dbl, _c_p, _c_sz = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_size_t

# name -> (restype, argtypes); the same set include/tqmoe.h declares
_SIGS = {
    "tq_status_string": (ctypes.c_char_p, [_c_int]),
    "tq_init": (_c_int, [_c_int]),
    "tq_arch_witness": (_c_int, [_c_int, ctypes.POINTER(_c_int)]),
    "tq_pairs_per_woken_expert": (_c_dbl, [_c_i64, _c_int, _c_int]),
    "tq_tiles_amortize": (_c_int, [_c_i64, _c_int, _c_int, _c_int]),
    "tq_grouped_min_tokens": (_c_i64, [_c_int, _c_int, _c_int]),
    "tq_tile_map_capacity": (_c_i64, [_c_i64, _c_int, _c_int, _c_int]),
    "tq_native_tile_m": (_c_int, [_c_i64, _c_int, _c_int]),
    "tq_select_arm": (_c_int, [_c_i64, _c_int, _c_int, _c_int, _c_int]),
    "tq_route": (_c_int, [_c_p, _c_i64, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p]),
    "tq_build_tile_map": (_c_int, [_c_p, _c_int, _c_int, _c_p, _c_p, _c_i64, _c_p]),
    "tq_router_topk": (_c_int, [_c_p, _c_i64, _c_int, _c_int, _c_p, _c_p, _c_p]),
    "tq_route_logits": (_c_int, [_c_p, _c_i64, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]),
    "tq_grouped_gemm": (_c_int, [_c_p, _c_int, _c_p, _c_p, _c_int, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64,
                                 _c_int, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p]),
    "tq_gemv": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_i64, _c_int, _c_int, _c_int,
                         _c_int, _c_p, _c_p]),
    "tq_combine": (_c_int, [_c_p, _c_p, _c_i64, _c_p]),
    "tq_gather_rows": (_c_int, [_c_p, _c_p, _c_i64, _c_int, _c_int, _c_p, _c_p]),
    "tq_prepare": (_c_int, [_c_p, _c_p, _c_i64, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p,
                            _c_i64, _c_p, _c_p, _c_i64, _c_p]),
    "tq_moe_workspace_size": (_c_sz, [_c_i64, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "tq_moe_forward": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_i64, _c_int, _c_int,
                                _c_int, _c_int, _c_int, _c_int, _c_p, _c_sz, _c_p,
                                ctypes.POINTER(_c_int), _c_p]),
    "tq_moe_forward_static": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_i64, _c_int, _c_int,
                                       _c_int, _c_int, _c_int, _c_int, _c_p, ctypes.POINTER(_c_int), _c_p]),
    "tq_probe_lut_rate": (_c_int, [_c_p, _c_int, _c_int, _c_p, _c_p, _c_p]),
    "tq_probe_wait_timeout": (_c_int, [_c_i64, _c_p, _c_p]),
    "tq_grouped_gemm_pairs": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_int, _c_int,
                                       _c_int, _c_int, _c_int, _c_p, _c_p]),
    "tq_swiglu": (_c_int, [_c_p, _c_i64, _c_int, _c_p, _c_p]),
    "tq_moe_mlp_workspace_size": (_c_sz, [_c_i64, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "tq_moe_mlp_forward": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_i64, _c_int, _c_int, _c_int,
                                    _c_int, _c_int, _c_int, _c_p, _c_sz, _c_p, ctypes.POINTER(_c_int), _c_p]),
    "tq_dequantize": (_c_int, [_c_p, _c_p, _c_int, _c_p, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p]),
    "tq_grouped_gemm_dense": (_c_int, [_c_p, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_int, _c_int,
                                       _c_int,
                                       _c_int, _c_int, _c_p, _c_p]),
    "tq_moe_dequant_workspace_size": (_c_sz, [_c_i64, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "tq_moe_forward_dequant": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_i64, _c_int, _c_int, _c_int,
                                        _c_int, _c_int, _c_p, _c_sz, _c_p, _c_p]),
    "tq_device_error": (_c_int, [ctypes.POINTER(_c_int), ctypes.POINTER(_c_int)]),
    "tq_launch_counts": (None, [ctypes.POINTER(_c_i64)]),
}
EXPORTED_SYMBOLS = tuple(_SIGS)

_lib = None


class TQError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {tq_status_string(status)} ({status})" if what else
                         f"{tq_status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load libtqmoe.so (built by __graft_entry__.build()); raise if missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(lib_path):
            raise RuntimeError(f"{lib_path} is not built; run `python -c 'import __graft_entry__ as g; "
                               f"g.build()'` (nvcc, sm_103a)")
        h = ctypes.CDLL(lib_path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def tq_status_string(status: int) -> str:
    return lib().tq_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise TQError(rc, what)


# ------------------------------------------------------------------ torch glue

_torch_mod = None


def _torch():
    """torch, once a CUDA device has been seen (checked on the first call only)."""
    global _torch_mod
    if _torch_mod is None:
        import torch
        if not torch.cuda.is_available():
            raise RuntimeError("trellis_quantized_moe_sort_gb300 needs a CUDA device (sm_103a); none found")
        _torch_mod = torch
    return _torch_mod


def _dev_ptr(t, dtypes, name):
    """Device address of a contiguous CUDA tensor of one of `dtypes`."""
    try:
        ok = t.is_cuda and (not dtypes or t.dtype in dtypes) and t.is_contiguous()
    except AttributeError:
        raise TypeError(f"{name} must be a torch.Tensor") from None
    if not ok:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if dtypes and t.dtype not in dtypes:
            raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _current_stream_fast():
    """Raw handle of torch's current stream on the current device."""
    torch = _torch()
    return torch.cuda.current_stream().cuda_stream


_raw_stream_fn = None


def _stream(stream):
    global _raw_stream_fn
    if stream is not None:
        return stream.cuda_stream
    torch = _torch()
    if _raw_stream_fn is None:
        # the C-level getter of torch's current stream (a plain integer), when
        # this torch build has it; else the public (slower) route
        getter = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _raw_stream_fn = ((lambda: getter(torch.cuda.current_device())) if getter is not None
                          else _current_stream_fast)
    return _raw_stream_fn()


_bits16_types = None


def _bits16():
    global _bits16_types
    if _bits16_types is None:
        torch = _torch()
        _bits16_types = (torch.bfloat16, torch.float16, torch.int16, torch.uint16)
    return _bits16_types


# ------------------------------------------------------------------ API

def tq_init(device: int = 0) -> None:
    _check(lib().tq_init(device), "tq_init")


def tq_arch_witness(device: int = 0) -> int:
    arch = ctypes.c_int(0)
    _check(lib().tq_arch_witness(device, ctypes.byref(arch)), "tq_arch_witness")
    return arch.value


def tq_pairs_per_woken_expert(n: int, top_k: int, E: int) -> float:
    return lib().tq_pairs_per_woken_expert(n, top_k, E)


def tq_tiles_amortize(n: int, top_k: int, E: int, tile_m: int) -> bool:
    rc = lib().tq_tiles_amortize(n, top_k, E, tile_m)
    if rc < 0:
        raise TQError(rc, "tq_tiles_amortize")
    return bool(rc)


def tq_grouped_min_tokens(top_k: int, E: int, tile_m: int) -> int:
    rc = lib().tq_grouped_min_tokens(top_k, E, tile_m)
    if rc < 0:
        raise TQError(int(rc), "tq_grouped_min_tokens")
    return int(rc)


def tq_native_tile_m(n: int, top_k: int, E: int) -> int:
    v = lib().tq_native_tile_m(n, top_k, E)
    if v < 0:
        raise TQError(v, "tq_native_tile_m")
    return int(v)


def tq_tile_map_capacity(n: int, top_k: int, E: int, tile_m: int) -> int:
    rc = lib().tq_tile_map_capacity(n, top_k, E, tile_m)
    if rc < 0:
        raise TQError(int(rc), "tq_tile_map_capacity")
    return int(rc)


def tq_select_arm(n: int, top_k: int, E: int, tile_m: int, pin: int = ARM_AUTO) -> int:
    rc = lib().tq_select_arm(n, top_k, E, tile_m, pin)
    if rc < 0:
        raise TQError(rc, "tq_select_arm")
    return rc


def tq_route(topk_ids, E: int, counts=None, offsets=None, sorted_pairs=None, stream=None):
    """Stable sort of pairs by expert -> (counts[E], offsets[E+1], sorted_pairs[P])."""
    torch = _torch()
    n, k = topk_ids.shape
    dev = topk_ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev) if counts is None else counts
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if offsets is None else offsets
    if sorted_pairs is None:
        sorted_pairs = torch.empty(max(n * k, 1), dtype=torch.int32, device=dev)
    _check(lib().tq_route(_dev_ptr(topk_ids, (torch.int32,), "topk_ids"), n, k, E,
                          _dev_ptr(counts, (torch.int32,), "counts"),
                          _dev_ptr(offsets, (torch.int32,), "offsets"),
                          _dev_ptr(sorted_pairs, (torch.int32,), "sorted_pairs"), _stream(stream)),
           "tq_route")
    return counts, offsets, sorted_pairs[: n * k]


def tq_router_topk(logits, top_k: int, topk_ids=None, topk_w=None, stream=None):
    """Per-token top_k experts and softmax weights from fp32 logits [n, E]."""
    torch = _torch()
    n, E = logits.shape
    topk_ids = torch.empty((n, top_k), dtype=torch.int32, device=logits.device) if topk_ids is None else topk_ids
    topk_w = torch.empty((n, top_k), dtype=torch.float32, device=logits.device) if topk_w is None else topk_w
    _check(lib().tq_router_topk(_dev_ptr(logits, (torch.float32,), "logits"), n, E, top_k,
                                _dev_ptr(topk_ids, (torch.int32,), "topk_ids"),
                                _dev_ptr(topk_w, (torch.float32,), "topk_w"), _stream(stream)), "tq_router_topk")
    return topk_ids, topk_w


def tq_route_logits(logits, top_k: int, stream=None):
    """Router top-k then the routing sort -> (ids, w, counts, offsets, sorted_pairs)."""
    torch = _torch()
    n, E = logits.shape
    dev = logits.device
    ids = torch.empty((n, top_k), dtype=torch.int32, device=dev)
    w = torch.empty((n, top_k), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(max(n * top_k, 1), dtype=torch.int32, device=dev)
    _check(lib().tq_route_logits(_dev_ptr(logits, (torch.float32,), "logits"), n, E, top_k,
                                 _dev_ptr(ids, (torch.int32,), "topk_ids"), _dev_ptr(w, (torch.float32,), "topk_w"),
                                 _dev_ptr(counts, (torch.int32,), "counts"), _dev_ptr(offsets, (torch.int32,), "offsets"),
                                 _dev_ptr(sp, (torch.int32,), "sorted_pairs"), _stream(stream)), "tq_route_logits")
    return ids, w, counts, offsets, sp[: n * top_k]


def tq_build_tile_map(offsets, tile_m: int, cap: int, tiles=None, num_tiles=None, stream=None):
    """m-tile map -> (tiles[cap, 3], num_tiles[1]) (device)."""
    torch = _torch()
    E = offsets.numel() - 1
    dev = offsets.device
    tiles = torch.empty((cap, 3), dtype=torch.int32, device=dev) if tiles is None else tiles
    num_tiles = torch.empty(1, dtype=torch.int32, device=dev) if num_tiles is None else num_tiles
    _check(lib().tq_build_tile_map(_dev_ptr(offsets, (torch.int32,), "offsets"), E, tile_m,
                                   _dev_ptr(tiles, (torch.int32,), "tiles"),
                                   _dev_ptr(num_tiles, (torch.int32,), "num_tiles"), cap, _stream(stream)),
           "tq_build_tile_map")
    return tiles, num_tiles


def _shapes(x, packed, lut):
    n, K = x.shape
    E, N, kb = packed.shape
    if kb * 4 != K:
        raise ValueError(f"packed has {kb} bytes per row, expected K/4 = {K // 4}")
    L = lut.numel().bit_length() - 1
    if lut.numel() != (1 << L):
        raise ValueError("lut must have 2^L entries")
    return n, K, E, N, L


def tq_gather_rows(x, sorted_pairs, top_k: int, x_sorted=None, stream=None):
    """Pair-sorted copy of the activations: x_sorted[s] = x[sorted_pairs[s] // top_k]."""
    torch = _torch()
    n, K = x.shape
    P = n * top_k
    x_sorted = torch.empty((max(P, 1), K), dtype=x.dtype, device=x.device) if x_sorted is None else x_sorted
    _check(lib().tq_gather_rows(_dev_ptr(x, _bits16(), "x"), _dev_ptr(sorted_pairs, (torch.int32,), "sorted_pairs"),
                                n, top_k, K, _dev_ptr(x_sorted, _bits16(), "x_sorted"), _stream(stream)),
           "tq_gather_rows")
    return x_sorted[:P]


def tq_prepare(topk_ids, x, E: int, tile_m: int, cap: int, counts, offsets, sorted_pairs, tiles, num_tiles,
               x_sorted=None, y32=None, stream=None) -> None:
    """Route + tile map in one launch, clearing y32 (fp32) in the same launch
    when it is given; with x_sorted, also the pair-sorted copy of x (what
    tq_grouped_gemm_pairs reads; tq_grouped_gemm gathers the rows itself)."""
    torch = _torch()
    n, top_k = topk_ids.shape
    K = x.shape[1]
    y32_ptr = None if y32 is None else _dev_ptr(y32, (torch.float32,), "y32")
    xs_ptr = None if x_sorted is None else _dev_ptr(x_sorted, _bits16(), "x_sorted")
    _check(lib().tq_prepare(_dev_ptr(topk_ids, (torch.int32,), "topk_ids"), _dev_ptr(x, _bits16(), "x"), n, top_k,
                            E, K, tile_m, _dev_ptr(counts, (torch.int32,), "counts"),
                            _dev_ptr(offsets, (torch.int32,), "offsets"),
                            _dev_ptr(sorted_pairs, (torch.int32,), "sorted_pairs"),
                            _dev_ptr(tiles, (torch.int32,), "tiles"), _dev_ptr(num_tiles, (torch.int32,), "num_tiles"),
                            cap, xs_ptr, y32_ptr, 0 if y32 is None else y32.numel(), _stream(stream)), "tq_prepare")


def _x_rows(x, x_layout: int, top_k: int) -> int:
    """Tokens n of an activation tensor in either layout."""
    if x_layout == X_TOKENS:
        return x.shape[0]
    if x_layout != X_PAIR_SORTED:
        raise ValueError(f"x_layout must be X_TOKENS or X_PAIR_SORTED, not {x_layout}")
    if x.shape[0] % top_k:
        raise ValueError("pair-sorted x must have n*top_k rows")
    return x.shape[0] // top_k


def tq_grouped_gemm(x, packed, lut, sorted_pairs, topk_w, tiles, num_tiles, top_k: int, tile_m: int,
                    y32, x_layout: int = X_TOKENS, stream=None) -> None:
    """y32 += grouped product (y32 fp32 [n, N], zero it for a plain product).
    x: the token activations [n, K] (X_TOKENS: the kernel gathers each m-tile's
    rows through sorted_pairs) or their pair-sorted copy [n*top_k, K] from
    tq_gather_rows (X_PAIR_SORTED)."""
    torch = _torch()
    n = _x_rows(x, x_layout, top_k)
    K = x.shape[1]
    E, N, kb = packed.shape
    if kb * 4 != K:
        raise ValueError(f"packed has {kb} bytes per row, expected K/4 = {K // 4}")
    L = lut.numel().bit_length() - 1
    cap = tiles.shape[0]
    _check(lib().tq_grouped_gemm(_dev_ptr(x, _bits16(), "x"), x_layout, _dev_ptr(packed, (torch.uint8,), "packed"),
                                 _dev_ptr(lut, _bits16(), "lut"), L,
                                 _dev_ptr(sorted_pairs, (torch.int32,), "sorted_pairs"),
                                 _dev_ptr(topk_w, (torch.float32,), "topk_w"),
                                 _dev_ptr(tiles, (torch.int32,), "tiles"),
                                 _dev_ptr(num_tiles, (torch.int32,), "num_tiles"), cap, n, top_k, E, K, N,
                                 tile_m, _dev_ptr(y32, (torch.float32,), "y32"), _stream(stream)),
           "tq_grouped_gemm")


def tq_gemv(x, packed, lut, topk_ids, topk_w, y32, stream=None) -> None:
    """y32 += per-pair GEMV product."""
    torch = _torch()
    n, K, E, N, L = _shapes(x, packed, lut)
    top_k = topk_ids.shape[1]
    _check(lib().tq_gemv(_dev_ptr(x, _bits16(), "x"), _dev_ptr(packed, (torch.uint8,), "packed"),
                         _dev_ptr(lut, _bits16(), "lut"), L, _dev_ptr(topk_ids, (torch.int32,), "topk_ids"),
                         _dev_ptr(topk_w, (torch.float32,), "topk_w"), n, top_k, E, K, N,
                         _dev_ptr(y32, (torch.float32,), "y32"), _stream(stream)), "tq_gemv")


def tq_combine(y32, y=None, stream=None):
    """bf16 (round to nearest even) copy of y32."""
    torch = _torch()
    y = torch.empty(y32.shape, dtype=torch.bfloat16, device=y32.device) if y is None else y
    _check(lib().tq_combine(_dev_ptr(y32, (torch.float32,), "y32"), _dev_ptr(y, _bits16(), "y"),
                            y32.numel(), _stream(stream)), "tq_combine")
    return y


def tq_moe_workspace_size(n: int, top_k: int, E: int, K: int, N: int, tile_m: int) -> int:
    return int(lib().tq_moe_workspace_size(n, top_k, E, K, N, tile_m))


def tq_moe_forward(x, packed, lut, topk_ids, topk_w, tile_m: int = 16, pin: int = ARM_AUTO,
                   workspace=None, y=None, stream=None):
    """Whole routed-expert product -> (y bf16 [n, N], arm used)."""
    torch = _torch()
    n, K, E, N, L = _shapes(x, packed, lut)
    top_k = topk_ids.shape[1]
    need = tq_moe_workspace_size(n, top_k, E, K, N, tile_m)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    y = torch.empty((n, N), dtype=torch.bfloat16, device=x.device) if y is None else y
    arm = ctypes.c_int(-1)
    _check(lib().tq_moe_forward(_dev_ptr(x, _bits16(), "x"), _dev_ptr(packed, (torch.uint8,), "packed"),
                                _dev_ptr(lut, _bits16(), "lut"), L,
                                _dev_ptr(topk_ids, (torch.int32,), "topk_ids"),
                                _dev_ptr(topk_w, (torch.float32,), "topk_w"), n, top_k, E, K, N, tile_m, pin,
                                _dev_ptr(workspace, (torch.uint8,), "workspace"), workspace.numel(),
                                _dev_ptr(y, _bits16(), "y"), ctypes.byref(arm), _stream(stream)),
           "tq_moe_forward")
    return y, arm.value


STATIC_SCRATCH_BYTES = 16 * 1024 * 1024   # TQ_STATIC_SCRATCH_BYTES in include/tqmoe.h


def tq_moe_forward_static(x, packed, lut, topk_ids, topk_w, tile_m: int = 16, pin: int = ARM_AUTO,
                          y=None, stream=None):
    """Whole routed-expert product with the library's fixed scratch array
    instead of a workspace (for callers that cannot allocate device memory;
    here only `y` is allocated, and only when not given) -> (y, arm used).
    Calls sharing a device must not overlap on the GPU."""
    torch = _torch()
    n, K, E, N, L = _shapes(x, packed, lut)
    top_k = topk_ids.shape[1]
    y = torch.empty((n, N), dtype=torch.bfloat16, device=x.device) if y is None else y
    arm = ctypes.c_int(-1)
    _check(lib().tq_moe_forward_static(_dev_ptr(x, _bits16(), "x"), _dev_ptr(packed, (torch.uint8,), "packed"),
                                       _dev_ptr(lut, _bits16(), "lut"), L,
                                       _dev_ptr(topk_ids, (torch.int32,), "topk_ids"),
                                       _dev_ptr(topk_w, (torch.float32,), "topk_w"), n, top_k, E, K, N, tile_m,
                                       pin, _dev_ptr(y, _bits16(), "y"), ctypes.byref(arm), _stream(stream)),
           "tq_moe_forward_static")
    return y, arm.value


def tq_probe_wait_timeout(timeout_ns: int, stream=None) -> tuple[bool, int]:
    """Run the bounded-wait probe: (whether the wait completed, microseconds
    waited).  The give-up is recorded in the device error word."""
    torch = _torch()
    out = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    _check(lib().tq_probe_wait_timeout(int(timeout_ns), _dev_ptr(out, (torch.int32,), "out"), _stream(stream)),
           "tq_probe_wait_timeout")
    torch.cuda.synchronize()
    done, us = out.tolist()
    return bool(done), int(us)


def tq_probe_lut_rate(warps_per_sm: int = 8, iters: int = 512, stream=None) -> float:
    """Measured random 16-bit shared-memory lookups per clock per SM (the
    resource that bounds the trellis decode)."""
    torch = _torch()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    table = torch.zeros(65536, dtype=torch.int16, device="cuda")
    sink = torch.empty(sms * warps_per_sm * 32, dtype=torch.int32, device="cuda")
    cycles = torch.zeros(sms, dtype=torch.int64, device="cuda")
    _check(lib().tq_probe_lut_rate(_dev_ptr(table, _bits16(), "table"), warps_per_sm, iters,
                                   _dev_ptr(sink, (torch.int32,), "sink"), _dev_ptr(cycles, (torch.int64,), "cycles"),
                                   _stream(stream)), "tq_probe_lut_rate")
    torch.cuda.synchronize()
    c = float(cycles.double().mean())
    return warps_per_sm * 32 * iters * 16 / c


def tq_moe_mlp_workspace_size(n: int, top_k: int, E: int, H: int, I: int, tile_m: int) -> int:
    return int(lib().tq_moe_mlp_workspace_size(n, top_k, E, H, I, tile_m))


def tq_moe_mlp_forward(x, packed_gu, lut_gu, packed_down, lut_down, topk_ids, topk_w, tile_m: int = 16,
                       pin: int = ARM_AUTO, workspace=None, y=None, stream=None):
    """Whole SwiGLU expert MLP -> (y bf16 [n, H], arm used)."""
    torch = _torch()
    n, H = x.shape
    E, I2, hb = packed_gu.shape
    I = I2 // 2
    if hb * 4 != H or tuple(packed_down.shape) != (E, H, I // 4):
        raise ValueError("packed_gu must be [E, 2I, H/4] and packed_down [E, H, I/4]")
    L = lut_gu.numel().bit_length() - 1
    if lut_down.numel() != lut_gu.numel():
        raise ValueError("both LUTs need 2^L entries")
    top_k = topk_ids.shape[1]
    need = tq_moe_mlp_workspace_size(n, top_k, E, H, I, tile_m)
    workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device) if workspace is None else workspace
    y = torch.empty((n, H), dtype=torch.bfloat16, device=x.device) if y is None else y
    arm = ctypes.c_int(-1)
    _check(lib().tq_moe_mlp_forward(_dev_ptr(x, _bits16(), "x"), _dev_ptr(packed_gu, (torch.uint8,), "packed_gu"),
                                    _dev_ptr(lut_gu, _bits16(), "lut_gu"),
                                    _dev_ptr(packed_down, (torch.uint8,), "packed_down"),
                                    _dev_ptr(lut_down, _bits16(), "lut_down"), L,
                                    _dev_ptr(topk_ids, (torch.int32,), "topk_ids"),
                                    _dev_ptr(topk_w, (torch.float32,), "topk_w"), n, top_k, E, H, I, tile_m,
                                    pin, _dev_ptr(workspace, (torch.uint8,), "workspace"), workspace.numel(),
                                    _dev_ptr(y, _bits16(), "y"), ctypes.byref(arm), _stream(stream)),
           "tq_moe_mlp_forward")
    return y, arm.value


def tq_swiglu(gate_up, h=None, stream=None):
    """h = bf16(silu(gate) * up) for gate_up fp32 [P, 2I]."""
    torch = _torch()
    P, I2 = gate_up.shape
    h = torch.empty((P, I2 // 2), dtype=torch.bfloat16, device=gate_up.device) if h is None else h
    _check(lib().tq_swiglu(_dev_ptr(gate_up, (torch.float32,), "gate_up"), P, I2 // 2, _dev_ptr(h, _bits16(), "h"),
                           _stream(stream)), "tq_swiglu")
    return h


def tq_dequantize(packed, lut, expert_ids=None, w_out=None, stream=None):
    """Materialized bf16 weights [m, N, K] of the listed experts (all E when
    expert_ids is None) -- the dequantize-materialize comparator's first step."""
    torch = _torch()
    E, N, kb = packed.shape
    K = kb * 4
    L = lut.numel().bit_length() - 1
    if lut.numel() != (1 << L):
        raise ValueError("lut must have 2^L entries")
    m = E if expert_ids is None else expert_ids.numel()
    w_out = torch.empty((m, N, K), dtype=torch.bfloat16, device=packed.device) if w_out is None else w_out
    ids = None if expert_ids is None else _dev_ptr(expert_ids, (torch.int32,), "expert_ids")
    _check(lib().tq_dequantize(_dev_ptr(packed, (torch.uint8,), "packed"), _dev_ptr(lut, _bits16(), "lut"), L, ids,
                               m, E, N, K, _dev_ptr(w_out, _bits16(), "w_out"), _stream(stream)), "tq_dequantize")
    return w_out


def tq_grouped_gemm_dense(x, w_dense, sorted_pairs, topk_w, tiles, num_tiles, top_k: int, tile_m: int,
                          y32, x_layout: int = X_TOKENS, stream=None) -> None:
    """y32 += grouped product with dense bf16 weights w_dense [E, N, K];
    x and x_layout as in tq_grouped_gemm."""
    torch = _torch()
    n = _x_rows(x, x_layout, top_k)
    K = x.shape[1]
    E, N, K2 = w_dense.shape
    if K2 != K:
        raise ValueError(f"w_dense has K = {K2}, x has {K}")
    _check(lib().tq_grouped_gemm_dense(_dev_ptr(x, _bits16(), "x"), x_layout,
                                       _dev_ptr(w_dense, _bits16(), "w_dense"),
                                       _dev_ptr(sorted_pairs, (torch.int32,), "sorted_pairs"),
                                       _dev_ptr(topk_w, (torch.float32,), "topk_w"),
                                       _dev_ptr(tiles, (torch.int32,), "tiles"),
                                       _dev_ptr(num_tiles, (torch.int32,), "num_tiles"), tiles.shape[0], n,
                                       top_k, E, K, N, tile_m, _dev_ptr(y32, (torch.float32,), "y32"),
                                       _stream(stream)), "tq_grouped_gemm_dense")


def tq_moe_dequant_workspace_size(n: int, top_k: int, E: int, K: int, N: int, tile_m: int) -> int:
    return int(lib().tq_moe_dequant_workspace_size(n, top_k, E, K, N, tile_m))


def tq_moe_forward_dequant(x, packed, lut, topk_ids, topk_w, tile_m: int = 16, workspace=None, y=None,
                           stream=None):
    """Dequantize-materialize comparator: the routed-expert product through
    dense bf16 copies of the woken experts -> y bf16 [n, N]."""
    torch = _torch()
    n, K, E, N, L = _shapes(x, packed, lut)
    top_k = topk_ids.shape[1]
    need = tq_moe_dequant_workspace_size(n, top_k, E, K, N, tile_m)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    y = torch.empty((n, N), dtype=torch.bfloat16, device=x.device) if y is None else y
    _check(lib().tq_moe_forward_dequant(_dev_ptr(x, _bits16(), "x"), _dev_ptr(packed, (torch.uint8,), "packed"),
                                        _dev_ptr(lut, _bits16(), "lut"), L,
                                        _dev_ptr(topk_ids, (torch.int32,), "topk_ids"),
                                        _dev_ptr(topk_w, (torch.float32,), "topk_w"), n, top_k, E, K, N, tile_m,
                                        _dev_ptr(workspace, (torch.uint8,), "workspace"), workspace.numel(),
                                        _dev_ptr(y, _bits16(), "y"), _stream(stream)), "tq_moe_forward_dequant")
    return y


def tq_device_error() -> tuple[int, int]:
    """(code, where) of the first device-side error since the last call; clears it."""
    code, where = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().tq_device_error(ctypes.byref(code), ctypes.byref(where)), "tq_device_error")
    return code.value, where.value


LAUNCH_COUNTERS = ("route", "tile_map", "grouped", "gemv", "combine", "gather", "router", "dequant",
                   "route_tile_map", "clear", "swiglu")


def tq_launch_counts() -> dict:
    arr = (ctypes.c_int64 * len(LAUNCH_COUNTERS))()
    lib().tq_launch_counts(arr)
    return dict(zip(LAUNCH_COUNTERS, list(arr)))
