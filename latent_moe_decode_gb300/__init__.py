"""GB300 (sm_103a) routing-and-combine path of a decode-step latent-MoE layer.

A thin ctypes binding over ``libmoe_decode.so`` (C ABI in ``include/moe_decode.h``):
it checks torch tensors (device, dtype, shape, contiguity), passes their device
pointers and the current CUDA stream, and turns status codes into exceptions. Every
step of the path runs in the library's CUDA kernels; there is no fallback.

BF16 tensors are ``torch.bfloat16``; E4M3 / E8M0 outputs are ``torch.uint8``.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "MoeError", "load", "router_logits", "router_logits_workspace", "front_projection",
    "front_projection_workspace", "topk_route",
    "build_routing_lists", "build_routing_lists_workspace", "unit_windows", "unit_windows_capacity",
    "mxfp8_quantize_rows", "mxfp8_quantize_rows_tcgen05", "mxfp8_tcgen05_scales_bytes",
    "finalize", "finalize_rmsnorm", "route_finalize", "route_finalize_workspace", "device_error", "RouteFinalize",
    "ROUTER_AUTO", "ROUTER_SIMT", "ROUTER_TCGEN05", "MXFP8_SCALE_FLOOR", "MXFP8_SCALE_CEIL",
    "DEVERR_ROW_INDEX", "DEVERR_EXPERT_ID", "DEVERR_TIMEOUT", "DEVERR_CAPACITY",
]

OK, ERR_INVALID_ARGUMENT, ERR_ALIGNMENT, ERR_CAPACITY, ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_CUDA = range(7)
DEVERR_ROW_INDEX, DEVERR_EXPERT_ID, DEVERR_TIMEOUT, DEVERR_CAPACITY = 0x1, 0x2, 0x4, 0x8
ROUTER_AUTO, ROUTER_SIMT, ROUTER_TCGEN05 = 0, 1, 2
MXFP8_SCALE_FLOOR, MXFP8_SCALE_CEIL = 0, 1
DTYPE_F32, DTYPE_BF16 = 0, 1

# Every symbol the header declares, with its ctypes signature.
_P, _I, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_version": (_I, []),
    "moe_device_error": (_I, [ctypes.POINTER(ctypes.c_uint32), _I]),
    "moe_router_logits_workspace": (_SZ, [_I, _I, _I]),
    "moe_router_logits": (_I, [_P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "moe_router_logits_ex": (_I, [_P, _P, _P, _I, _I, _I, _P, _SZ, _I, _P]),
    "moe_router_logits_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _P]),
    "moe_front_projection_workspace": (_SZ, [_I, _I, _I, _I]),
    "moe_front_projection": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _SZ, _P]),
    "moe_topk_route": (_I, [_P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
    "moe_topk_route_quantize": (_I, [_P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P, _I, _I, _P, _P, _P]),
    "moe_build_routing_lists_workspace": (_SZ, [_I, _I, _I]),
    "moe_build_routing_lists": (_I, [_P, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "moe_unit_windows_capacity": (_I, [_I, _I, _I, _I]),
    "moe_build_unit_windows": (_I, [_P, _I, _I, _P, _P, _P, _P, _I, _P]),
    "mxfp8_quantize_rows": (_I, [_P, _I, _I, _P, _P, _P]),
    "mxfp8_quantize_rows_ex": (_I, [_P, _I, _I, _P, _P, _I, _P]),
    "mxfp8_tcgen05_scales_bytes": (_SZ, [_I, _I]),
    "mxfp8_quantize_rows_tcgen05": (_I, [_P, _I, _I, _P, _P, _I, _P]),
    "moe_finalize": (_I, [_P, ctypes.c_int64, _P, _P, _I, _P, _F, _I, _I, _I, _P, _P]),
    "moe_finalize_rmsnorm": (_I, [_P, ctypes.c_int64, _P, _P, _I, _F, _P, _F, _I, _I, _I, _P, _P, _P]),
    "moe_route_finalize_workspace": (_SZ, [_I, _I, _I, _I]),
    "moe_route_finalize": (_I, [_P] * 5 + [_I] * 6 + [_F] + [_P] * 9 + [_P, _SZ, _P]),
}

_lib = None


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = load().moe_status_string(status).decode()
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


def load(path: str | None = None):
    """Load the CUDA library (built in-tree by ``build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build the CUDA library first (latent_moe_decode_gb300.build.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != OK:
        raise MoeError(fn, status)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, shape=None, name="tensor"):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


# ---------------------------------------------------------------------------
def router_logits_workspace(T: int, H: int, E: int) -> int:
    return int(load().moe_router_logits_workspace(T, H, E))


def router_logits(x, w, out=None, workspace=None, algo: int = ROUTER_AUTO, stream=None):
    """FP32 logits [T, E] = x [T, H] (BF16) @ w [E, H]^T (BF16)."""
    T, H = x.shape
    E = w.shape[0]
    _need(x, torch.bfloat16, (T, H), "x")
    _need(w, torch.bfloat16, (E, H), "w")
    out = _empty((T, E), torch.float32, x) if out is None else _need(out, torch.float32, (T, E), "out")
    need = router_logits_workspace(T, H, E)
    if need and workspace is None:
        workspace = _empty((need,), torch.uint8, x)
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("moe_router_logits_ex", load().moe_router_logits_ex(
        _ptr(x), _ptr(w), _ptr(out), T, H, E, _ptr(workspace), wb, algo, _stream(stream)))
    return out


def front_projection_workspace(T: int, H: int, E: int, L: int) -> int:
    return int(load().moe_front_projection_workspace(T, H, E, L))


def front_projection(x, w_router, w_down, logits=None, latent=None, workspace=None, stream=None):
    """(FP32 logits [T, E] = x @ w_router^T, BF16 latent [T, L] = bf16(x @ w_down^T)), one launch."""
    T, H = x.shape
    E, L = w_router.shape[0], w_down.shape[0]
    _need(x, torch.bfloat16, (T, H), "x")
    _need(w_router, torch.bfloat16, (E, H), "w_router")
    _need(w_down, torch.bfloat16, (L, H), "w_down")
    logits = _empty((T, E), torch.float32, x) if logits is None else _need(logits, torch.float32, (T, E), "logits")
    latent = _empty((T, L), torch.bfloat16, x) if latent is None else _need(latent, torch.bfloat16, (T, L), "latent")
    need = front_projection_workspace(T, H, E, L)
    if need and workspace is None:
        workspace = _empty((need,), torch.uint8, x)
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("moe_front_projection", load().moe_front_projection(
        _ptr(x), _ptr(w_router), _ptr(w_down), _ptr(logits), _ptr(latent), T, H, E, L, _ptr(workspace), wb,
        _stream(stream)))
    return logits, latent


def topk_route(logits, bias, K: int, renormalize: bool = True, scale: float = 1.0,
               ids=None, weights=None, weights_bf16=None, want_bf16: bool = True, stream=None):
    """(ids int32 [T,K], weights FP32 [T,K], weights BF16 [T,K] or None)."""
    T, E = logits.shape
    _need(logits, torch.float32, (T, E), "logits")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    ids = _empty((T, K), torch.int32, logits) if ids is None else _need(ids, torch.int32, (T, K), "ids")
    weights = _empty((T, K), torch.float32, logits) if weights is None else _need(weights, torch.float32, (T, K), "weights")
    if weights_bf16 is None and want_bf16:
        weights_bf16 = _empty((T, K), torch.bfloat16, logits)
    elif weights_bf16 is not None:
        _need(weights_bf16, torch.bfloat16, (T, K), "weights_bf16")
    _check("moe_topk_route", load().moe_topk_route(
        _ptr(logits), _ptr(bias), T, E, K, int(bool(renormalize)), float(scale),
        _ptr(ids), _ptr(weights), _ptr(weights_bf16), _stream(stream)))
    return ids, weights, weights_bf16


def topk_route_quantize(logits, bias, K: int, latent, renormalize: bool = True, scale: float = 1.0, ids=None,
                        weights=None, weights_bf16=None, q=None, scales=None, stream=None):
    """topk_route and mxfp8_quantize_rows(latent) in one launch:
    (ids, weights, weights_bf16, q, scales)."""
    T, E = logits.shape
    _need(logits, torch.float32, (T, E), "logits")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    rows, cols = latent.shape
    _need(latent, torch.bfloat16, (rows, cols), "latent")
    ids = _empty((T, K), torch.int32, logits) if ids is None else _need(ids, torch.int32, (T, K), "ids")
    weights = _empty((T, K), torch.float32, logits) if weights is None else _need(weights, torch.float32, (T, K), "weights")
    weights_bf16 = _empty((T, K), torch.bfloat16, logits) if weights_bf16 is None else _need(weights_bf16, torch.bfloat16, (T, K), "weights_bf16")
    q = _empty((rows, cols), torch.uint8, latent) if q is None else _need(q, torch.uint8, (rows, cols), "q")
    scales = _empty((rows, cols // 32), torch.uint8, latent) if scales is None else _need(scales, torch.uint8, (rows, cols // 32), "scales")
    _check("moe_topk_route_quantize", load().moe_topk_route_quantize(
        _ptr(logits), _ptr(bias), T, E, K, int(bool(renormalize)), float(scale), _ptr(ids), _ptr(weights),
        _ptr(weights_bf16), _ptr(latent), rows, cols, _ptr(q), _ptr(scales), _stream(stream)))
    return ids, weights, weights_bf16, q, scales


def build_routing_lists_workspace(T: int, K: int, E: int) -> int:
    return int(load().moe_build_routing_lists_workspace(T, K, E))


def build_routing_lists(ids, E: int, offsets=None, pairs=None, workspace=None, stream=None):
    """CSR lists: offsets int32 [E+1], pairs int32 [T*K] (pair code t*K + k)."""
    T, K = ids.shape
    _need(ids, torch.int32, (T, K), "ids")
    offsets = _empty((E + 1,), torch.int32, ids) if offsets is None else _need(offsets, torch.int32, (E + 1,), "offsets")
    pairs = _empty((T * K,), torch.int32, ids) if pairs is None else _need(pairs, torch.int32, (T * K,), "pairs")
    need = build_routing_lists_workspace(T, K, E)
    if need and workspace is None:
        workspace = _empty((need,), torch.uint8, ids)
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("moe_build_routing_lists", load().moe_build_routing_lists(
        _ptr(ids), T, K, E, _ptr(offsets), _ptr(pairs), _ptr(workspace), wb, _stream(stream)))
    return offsets, pairs


def unit_windows_capacity(T: int, K: int, E: int, window: int = 8) -> int:
    n = int(load().moe_unit_windows_capacity(T, K, E, window))
    if n < 0:
        raise MoeError("moe_unit_windows_capacity", ERR_INVALID_ARGUMENT)
    return n


def unit_windows(offsets, window: int = 8, max_units: int | None = None, unit_offsets=None, unit_expert=None,
                 unit_start=None, unit_len=None, stream=None):
    """Units of `window` listed pairs per expert from CSR offsets int32 [E+1]:
    (unit_offsets [E+1], unit_expert, unit_start, unit_len [max_units]); the first
    unit_offsets[E] entries are the units."""
    E = offsets.shape[0] - 1
    _need(offsets, torch.int32, (E + 1,), "offsets")
    if max_units is None:
        max_units = unit_expert.shape[0] if unit_expert is not None else None
    if max_units is None:
        raise ValueError("max_units (or preallocated unit arrays) required: see unit_windows_capacity()")
    unit_offsets = _empty((E + 1,), torch.int32, offsets) if unit_offsets is None else _need(unit_offsets, torch.int32, (E + 1,), "unit_offsets")
    outs = []
    for t, name in ((unit_expert, "unit_expert"), (unit_start, "unit_start"), (unit_len, "unit_len")):
        if t is None:
            t = _empty((max_units,), torch.int32, offsets)
        elif _need(t, torch.int32, None, name).dim() != 1 or t.shape[0] < max_units:
            raise ValueError(f"{name}: expected a 1-D tensor of at least {max_units} entries")
        outs.append(t)
    _check("moe_build_unit_windows", load().moe_build_unit_windows(
        _ptr(offsets), E, int(window), _ptr(unit_offsets), _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), int(max_units),
        _stream(stream)))
    return (unit_offsets, *outs)


def mxfp8_quantize_rows(x, q=None, scales=None, stream=None, scale_rule: int = MXFP8_SCALE_FLOOR):
    """(E4M3 bytes uint8 [rows, cols], E8M0 scale bytes uint8 [rows, cols/32]);
    scale_rule MXFP8_SCALE_FLOOR (OCP) or MXFP8_SCALE_CEIL (no saturation)."""
    rows, cols = x.shape
    _need(x, torch.bfloat16, (rows, cols), "x")
    q = _empty((rows, cols), torch.uint8, x) if q is None else _need(q, torch.uint8, (rows, cols), "q")
    nb = cols // 32
    scales = _empty((rows, nb), torch.uint8, x) if scales is None else _need(scales, torch.uint8, (rows, nb), "scales")
    _check("mxfp8_quantize_rows_ex", load().mxfp8_quantize_rows_ex(_ptr(x), rows, cols, _ptr(q), _ptr(scales),
                                                                   int(scale_rule), _stream(stream)))
    return q, scales


def mxfp8_tcgen05_scales_bytes(rows: int, cols: int) -> int:
    """Bytes of the tcgen05 block-scaling scale layout of a [rows, cols] MXFP8 tensor."""
    return int(load().mxfp8_tcgen05_scales_bytes(rows, cols))


def mxfp8_quantize_rows_tcgen05(x, q=None, scales=None, stream=None, scale_rule: int = MXFP8_SCALE_FLOOR):
    """(E4M3 bytes uint8 [rows, cols], E8M0 scales uint8 [mxfp8_tcgen05_scales_bytes]
    in the tcgen05 block-scaling tile layout)."""
    rows, cols = x.shape
    _need(x, torch.bfloat16, (rows, cols), "x")
    q = _empty((rows, cols), torch.uint8, x) if q is None else _need(q, torch.uint8, (rows, cols), "q")
    n = mxfp8_tcgen05_scales_bytes(rows, cols)
    scales = _empty((n,), torch.uint8, x) if scales is None else _need(scales, torch.uint8, (n,), "scales")
    _check("mxfp8_quantize_rows_tcgen05", load().mxfp8_quantize_rows_tcgen05(
        _ptr(x), rows, cols, _ptr(q), _ptr(scales), int(scale_rule), _stream(stream)))
    return q, scales


def finalize(rows, weights, T: int, K: int, row_index=None, shared=None, scale: float = 1.0, out=None, stream=None):
    """BF16 out [T, H] = sum_k w[t,k] * rows[r(t,k)] (+ shared[t])."""
    n_rows, H = rows.shape
    _need(rows, torch.bfloat16, (n_rows, H), "rows")
    if weights.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif weights.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise TypeError("weights: expected float32 or bfloat16")
    _need(weights, weights.dtype, (T, K), "weights")
    if row_index is not None:
        _need(row_index, torch.int32, (T, K), "row_index")
    if shared is not None:
        _need(shared, torch.bfloat16, (T, H), "shared")
    out = _empty((T, H), torch.bfloat16, rows) if out is None else _need(out, torch.bfloat16, (T, H), "out")
    _check("moe_finalize", load().moe_finalize(
        _ptr(rows), n_rows, _ptr(row_index), _ptr(weights), dt, _ptr(shared), float(scale), T, K, H, _ptr(out),
        _stream(stream)))
    return out


def finalize_rmsnorm(rows, weights, T: int, K: int, norm_weight, eps: float = 1e-5, row_index=None,
                     scale: float = 1.0, routed=None, out=None, want_routed: bool = True, stream=None):
    """(routed BF16 [T, H] or None, RMSNorm(routed) * norm_weight BF16 [T, H])."""
    n_rows, H = rows.shape
    _need(rows, torch.bfloat16, (n_rows, H), "rows")
    if weights.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif weights.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise TypeError("weights: expected float32 or bfloat16")
    _need(weights, weights.dtype, (T, K), "weights")
    _need(norm_weight, torch.bfloat16, (H,), "norm_weight")
    if row_index is not None:
        _need(row_index, torch.int32, (T, K), "row_index")
    if routed is None and want_routed:
        routed = _empty((T, H), torch.bfloat16, rows)
    elif routed is not None:
        _need(routed, torch.bfloat16, (T, H), "routed")
    out = _empty((T, H), torch.bfloat16, rows) if out is None else _need(out, torch.bfloat16, (T, H), "out")
    _check("moe_finalize_rmsnorm", load().moe_finalize_rmsnorm(
        _ptr(rows), n_rows, _ptr(row_index), _ptr(weights), dt, float(scale), _ptr(norm_weight), float(eps), T, K, H,
        _ptr(routed), _ptr(out), _stream(stream)))
    return routed, out


def device_error(clear: bool = True) -> int:
    """The library's device error word (DEVERR_* bits); synchronises the device."""
    v = ctypes.c_uint32(0)
    _check("moe_device_error", load().moe_device_error(ctypes.byref(v), int(bool(clear))))
    return int(v.value)


def route_finalize_workspace(T: int, H: int, E: int, K: int) -> int:
    return int(load().moe_route_finalize_workspace(T, H, E, K))


def route_finalize(x, w, bias, latent, rows, K: int, renormalize: bool, scale: float, logits, ids, weights,
                   weights_bf16, offsets, pairs, q, scales, out, workspace=None, stream=None):
    """The whole step in one library call (all outputs preallocated): router logits ->
    top-K + MXFP8 -> routing lists -> Finalize of rows [T*K, L] with the BF16 weights."""
    T, H = x.shape
    E = w.shape[0]
    L = latent.shape[1]
    _need(x, torch.bfloat16, (T, H), "x")
    _need(w, torch.bfloat16, (E, H), "w")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    _need(latent, torch.bfloat16, (T, L), "latent")
    _need(rows, torch.bfloat16, (T * K, L), "rows")
    for t, dt, shape, name in ((logits, torch.float32, (T, E), "logits"), (ids, torch.int32, (T, K), "ids"),
                               (weights_bf16, torch.bfloat16, (T, K), "weights_bf16"),
                               (offsets, torch.int32, (E + 1,), "offsets"), (pairs, torch.int32, (T * K,), "pairs"),
                               (q, torch.uint8, (T, L), "q"), (scales, torch.uint8, (T, L // 32), "scales"),
                               (out, torch.bfloat16, (T, L), "out")):
        _need(t, dt, shape, name)
    if weights is not None:
        _need(weights, torch.float32, (T, K), "weights")
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("moe_route_finalize", load().moe_route_finalize(
        _ptr(x), _ptr(w), _ptr(bias), _ptr(latent), _ptr(rows), T, H, L, E, K, int(bool(renormalize)), float(scale),
        _ptr(logits), _ptr(ids), _ptr(weights), _ptr(weights_bf16), _ptr(offsets), _ptr(pairs), _ptr(q), _ptr(scales),
        _ptr(out), _ptr(workspace), ws, _stream(stream)))
    return out


class RouteFinalize:
    """The whole routing-and-combine step, with its buffers preallocated:
    router logits -> sigmoid+bias top-K with the MXFP8 latent in the same launch ->
    Finalize, whose launch also builds the routing lists (Finalize does not read them),
    on one stream.

    ``run()`` launches the library's kernels (programmatic dependent launch between
    consecutive kernels of a stream) and allocates nothing, so it can be captured in a
    CUDA graph. With the automatic router choice it is one library call
    (``moe_route_finalize``); with a forced router family, the four calls.
    """

    def __init__(self, T: int, H: int, L: int, E: int, K: int, device="cuda", renormalize=True, scale=1.0,
                 router_algo: int = ROUTER_AUTO):
        self.T, self.H, self.L, self.E, self.K = T, H, L, E, K
        self.renormalize, self.scale, self.router_algo = renormalize, scale, router_algo
        dev = torch.device(device)
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
        self.logits = e((T, E), torch.float32)
        self.ids = e((T, K), torch.int32)
        self.weights = e((T, K), torch.float32)
        self.weights_bf16 = e((T, K), torch.bfloat16)
        self.offsets = e((E + 1,), torch.int32)
        self.pairs = e((T * K,), torch.int32)
        self.q = e((T, L), torch.uint8)
        self.scales = e((T, L // 32), torch.uint8)
        self.out = e((T, L), torch.bfloat16)
        self.router_ws = e((max(1, router_logits_workspace(T, H, E)),), torch.uint8)
        self.lists_ws = e((max(1, build_routing_lists_workspace(T, K, E)),), torch.uint8)
        self.chain_ws = e((max(1, route_finalize_workspace(T, H, E, K)),), torch.uint8)
        self.launches = self._count_launches()

    def _count_launches(self) -> int:
        """Kernels one run() launches."""
        if self.router_algo == ROUTER_AUTO:
            # the one-call step: router (its split-K partials summed by the top-K launch),
            # top-k + MXFP8, Finalize with the routing lists
            return 3
        # the four calls; a forced router family may add its split-K reduce kernel
        return 4 + (1 if router_logits_workspace(self.T, self.H, self.E) > 0 else 0)

    def run(self, x, w, bias, latent, rows, stream=None):
        main = stream if stream is not None else torch.cuda.current_stream()
        if self.router_algo == ROUTER_AUTO:
            return route_finalize(x, w, bias, latent, rows, self.K, self.renormalize, self.scale, self.logits, self.ids,
                                  self.weights, self.weights_bf16, self.offsets, self.pairs, self.q, self.scales,
                                  self.out, workspace=self.chain_ws, stream=main)
        router_logits(x, w, out=self.logits, workspace=self.router_ws, algo=self.router_algo, stream=main)
        topk_route_quantize(self.logits, bias, self.K, latent, self.renormalize, self.scale, ids=self.ids,
                            weights=self.weights, weights_bf16=self.weights_bf16, q=self.q, scales=self.scales,
                            stream=main)
        build_routing_lists(self.ids, self.E, offsets=self.offsets, pairs=self.pairs, workspace=self.lists_ws,
                            stream=main)
        finalize(rows, self.weights_bf16, self.T, self.K, out=self.out, stream=main)
        return self.out
