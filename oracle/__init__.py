"""CPU oracle for the latent-MoE decode routing-and-combine path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg are the only users. The product library
(``latent_moe_decode_gb300``) neither imports this package nor shares code with it.

The arithmetic lives in ``oracle.c`` (plain C, built with ``-ffp-contract=off``);
this module only builds it and marshals numpy arrays. BF16 tensors are numpy
``uint16`` arrays of raw bits, E4M3/E8M0 tensors ``uint8`` arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
# A prebuilt library to load instead (the mutation tests point this at oracle
# copies with planted mistakes, to show that the pins catch them).
_LIB_OVERRIDE = os.environ.get("MOE_ORACLE_LIB")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, no CUDA)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(_LIB_OVERRIDE or build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_router_logits.argtypes = [P, P, I, I, I, P, P]
        lib.oracle_router_logits_sampled.argtypes = [P, P, I, I, P, P, P, P]
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f64_to_bf16_array.argtypes = [P, P, ctypes.c_long]
        lib.oracle_exp_spec.argtypes = [ctypes.c_float]
        lib.oracle_exp_spec.restype = ctypes.c_float
        lib.oracle_sigmoid.argtypes = [ctypes.c_float]
        lib.oracle_sigmoid.restype = ctypes.c_float
        lib.oracle_sigmoid_array.argtypes = [P, P, ctypes.c_long]
        lib.oracle_topk_route.argtypes = [P, P, I, I, I, I, ctypes.c_float, P, P, P]
        lib.oracle_topk_route.restype = I
        lib.oracle_routing_lists.argtypes = [P, I, I, I, P, P]
        lib.oracle_routing_lists.restype = I
        lib.oracle_rmsnorm.argtypes = [P, P, I, I, ctypes.c_double, P]
        lib.oracle_unit_windows.argtypes = [P, I, I, P, P, P, P, I]
        lib.oracle_unit_windows.restype = I
        lib.oracle_mxfp8_quantize.argtypes = [P, I, I, P, P]
        lib.oracle_mxfp8_quantize_rule.argtypes = [P, I, I, I, P, P]
        lib.oracle_mxfp8_tcgen05_scales_bytes.argtypes = [I, I]
        lib.oracle_mxfp8_tcgen05_scales_bytes.restype = ctypes.c_size_t
        lib.oracle_mxfp8_scales_tcgen05.argtypes = [P, I, I, P]
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_finalize.argtypes = [P, ctypes.c_long, P, P, I, P, ctypes.c_float, I, I, I, P]
        lib.oracle_finalize.restype = I
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


# ---------------------------------------------------------------------------
_PARALLEL_MACS = 1 << 26  # inputs larger than this many multiply-adds use every host core


def router_logits(x: np.ndarray, w: np.ndarray, threads: int | None = None):
    """FP64 logits [T,E] and sum_j |x*w| [T,E] of BF16 x [T,H], W [E,H].

    Every token's row is independent, so large inputs are cut into contiguous token
    ranges, each computed by the same C function on its own host thread (ctypes
    releases the GIL during the call); the per-element arithmetic is unchanged."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    T, H = x.shape
    E = w.shape[0]
    assert w.shape[1] == H
    out = np.empty((T, E), np.float64)
    ab = np.empty((T, E), np.float64)
    lib = _load()
    if threads is None:
        threads = (os.cpu_count() or 1) if T * E * H > _PARALLEL_MACS else 1
    threads = max(1, min(int(threads), T))
    if threads == 1:
        lib.oracle_router_logits(_ptr(x), _ptr(w), T, H, E, _ptr(out), _ptr(ab))
        return out, ab
    from concurrent.futures import ThreadPoolExecutor

    bounds = np.linspace(0, T, threads + 1).astype(int)

    def part(i):
        t0, t1 = int(bounds[i]), int(bounds[i + 1])
        if t1 > t0:
            lib.oracle_router_logits(_ptr(x[t0:t1]), _ptr(w), t1 - t0, H, E, _ptr(out[t0:t1]), _ptr(ab[t0:t1]))

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(part, range(threads)))
    return out, ab


def router_logits_sampled(x, w, tok, exp_):
    """FP64 logits and |x*w| sums at the (tok[i], exp_[i]) pairs only."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    tok = _c(np.asarray(tok, np.int32), np.int32)
    exp_ = _c(np.asarray(exp_, np.int32), np.int32)
    n = tok.size
    out = np.empty(n, np.float64)
    ab = np.empty(n, np.float64)
    _load().oracle_router_logits_sampled(_ptr(x), _ptr(w), x.shape[1], n, _ptr(tok), _ptr(exp_), _ptr(out), _ptr(ab))
    return out, ab


def f64_to_bf16(v) -> np.ndarray:
    """BF16 bits of FP64 values, rounded once (nearest, ties to even)."""
    v = _c(np.asarray(v, np.float64), np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_f64_to_bf16_array(_ptr(v), _ptr(out), v.size)
    return out


def latent_down(x, w_down, rel_tol=1e-5):
    """Exact FP64 latent [T, L] = x @ w_down^T, its BF16 rounding, and the BF16 bounds
    (lo, hi) that any FP32 sum within rel_tol * sum|x w| of exact rounds into."""
    ref, ab = router_logits(x, w_down)
    return ref, f64_to_bf16(ref), f64_to_bf16(ref - rel_tol * ab), f64_to_bf16(ref + rel_tol * ab)


def exp_spec(y: float) -> float:
    return _load().oracle_exp_spec(float(y))


def sigmoid(x: np.ndarray) -> np.ndarray:
    x = _c(np.asarray(x, np.float32), np.float32)
    out = np.empty_like(x)
    _load().oracle_sigmoid_array(_ptr(x), _ptr(out), x.size)
    return out


def topk_route(logits, bias, K, renormalize=True, scale=1.0):
    """ids int32 [T,K], weights FP32 [T,K], weights BF16 bits [T,K]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    b = None if bias is None else _c(bias, np.float32)
    ids = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    wb = np.empty((T, K), np.uint16)
    rc = _load().oracle_topk_route(_ptr(logits), _ptr(b), T, E, K, int(bool(renormalize)), float(scale), _ptr(ids), _ptr(w), _ptr(wb))
    if rc != 0:
        raise ValueError(f"oracle_topk_route failed ({rc})")
    return ids, w, wb


def routing_lists(ids, E):
    """CSR lists: offsets int32 [E+1], pairs int32 [T*K] (pair code t*K + k)."""
    ids = _c(ids, np.int32)
    T, K = ids.shape
    off = np.empty(E + 1, np.int32)
    pairs = np.empty(T * K, np.int32)
    rc = _load().oracle_routing_lists(_ptr(ids), T, K, E, _ptr(off), _ptr(pairs))
    if rc != 0:
        raise ValueError(f"oracle_routing_lists failed ({rc})")
    return off, pairs


def unit_windows(offsets, window=8):
    """(unit_offsets int32 [E+1], unit_expert, unit_start, unit_len int32 [units])."""
    offsets = _c(offsets, np.int32)
    E = offsets.size - 1
    cap = max(1, int(offsets[-1]))
    uo = np.empty(E + 1, np.int32)
    ue, us, ul = (np.empty(cap, np.int32) for _ in range(3))
    rc = _load().oracle_unit_windows(_ptr(offsets), E, int(window), _ptr(uo), _ptr(ue), _ptr(us), _ptr(ul), cap)
    if rc != 0:
        raise ValueError(f"oracle_unit_windows failed ({rc})")
    n = int(uo[-1])
    return uo, ue[:n], us[:n], ul[:n]


def mxfp8_quantize(x, rule=0):
    """E4M3 bytes [rows, cols] and E8M0 scale bytes [rows, cols/32]; rule 0 = the OCP
    floor scale, 1 = the round-up scale (no saturation)."""
    x = _c(x, np.uint16)
    rows, cols = x.shape
    assert cols % 32 == 0
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 32), np.uint8)
    if rule == 0:
        _load().oracle_mxfp8_quantize(_ptr(x), rows, cols, _ptr(q), _ptr(s))
    else:
        _load().oracle_mxfp8_quantize_rule(_ptr(x), rows, cols, int(rule), _ptr(q), _ptr(s))
    return q, s


def mxfp8_scales_tcgen05(scales):
    """Row-major E8M0 scales [rows, nsc] in the tcgen05 block-scaling tile layout
    (128 x 4 tiles of 512 bytes, padding 0): a flat uint8 array."""
    scales = _c(scales, np.uint8)
    rows, nsc = scales.shape
    lib = _load()
    out = np.empty(lib.oracle_mxfp8_tcgen05_scales_bytes(rows, nsc), np.uint8)
    lib.oracle_mxfp8_scales_tcgen05(_ptr(scales), rows, nsc, _ptr(out))
    return out


def e4m3_encode(y: float) -> int:
    return int(_load().oracle_e4m3_encode(float(y)))


def e4m3_decode(c: int) -> float:
    return float(_load().oracle_e4m3_decode(int(c)))


def finalize(rows, weights, T, K, row_index=None, shared=None, scale=1.0):
    """BF16 bits out [T,H]. ``weights`` is float32 or BF16 bits (uint16) [T,K]."""
    rows = _c(rows, np.uint16)
    n_rows, H = rows.shape
    if weights.dtype == np.uint16:
        wb, is_bf16 = _c(weights, np.uint16), 1
    else:
        wb, is_bf16 = _c(weights, np.float32), 0
    ri = None if row_index is None else _c(row_index, np.int32)
    sh = None if shared is None else _c(shared, np.uint16)
    out = np.empty((T, H), np.uint16)
    rc = _load().oracle_finalize(_ptr(rows), n_rows, _ptr(ri), _ptr(wb), is_bf16, _ptr(sh), float(scale), T, K, H, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_finalize failed ({rc})")
    return out


def rmsnorm(x, g, eps=1e-5):
    """FP64 RMSNorm of BF16 rows x [T, H] with BF16 weight g [H]."""
    x = _c(x, np.uint16)
    g = _c(g, np.uint16)
    T, H = x.shape
    assert g.shape == (H,)
    y = np.empty((T, H), np.float64)
    _load().oracle_rmsnorm(_ptr(x), _ptr(g), T, H, float(eps), _ptr(y))
    return y


def rmsnorm_bounds(y, rel_tol=2.0 ** -16):
    """BF16 bits (lo, hi): every value within rel_tol * |y| of y rounds into [lo, hi]."""
    return f64_to_bf16(y - rel_tol * np.abs(y)), f64_to_bf16(y + rel_tol * np.abs(y))


def bf16_to_f32(b: int) -> float:
    return float(_load().oracle_bf16_to_f32(int(b)))


def f32_to_bf16(f: float) -> int:
    return int(_load().oracle_f32_to_bf16(float(f)))
