"""The C-ABI library builds, loads and exports every function that include/*.h
declares; argument validation runs on the host before any CUDA call (no GPU needed)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"#[^\n]*", "", text)
        for m in re.finditer(r"\b([A-Za-z_]\w*)\s*\(([^;{}]*)\)\s*;", text):
            if m.group(1) not in ("sizeof",):
                names.append(m.group(1))
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from latent_moe_decode_gb300 import build, load

    build.build()
    return load()


def test_header_declares_the_five_calls():
    names = declared_functions()
    for fn in ["moe_router_logits", "moe_topk_route", "moe_build_routing_lists", "mxfp8_quantize_rows", "moe_finalize"]:
        assert fn in names


def test_every_declared_symbol_is_exported(lib):
    import latent_moe_decode_gb300 as m

    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in m.SIGNATURES, f"binding lacks a signature for {name}"


def test_status_strings(lib):
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(4) == b"workspace missing or too small"
    assert lib.moe_status_string(99) == b"unknown status"
    assert lib.moe_version() >= 100


P = ctypes.c_void_p
A16 = P(256)  # a 16-byte aligned stand-in address; never dereferenced (validation fails first)


def test_validation_before_any_cuda_call(lib):
    # bad sizes / flags are rejected on the host, whether or not a GPU exists
    assert lib.moe_finalize(A16, 64, None, A16, 0, None, 1.0, -1, 16, 3584, A16, None) == 1
    assert lib.moe_finalize(A16, 64, None, A16, 0, None, 1.0, 4, 0, 3584, A16, None) == 1
    assert lib.moe_finalize(A16, 64, None, A16, 0, None, 1.0, 4, 33, 3584, A16, None) == 1
    assert lib.moe_finalize(A16, 64, None, A16, 0, None, 1.0, 4, 16, 3583, A16, None) == 1
    assert lib.moe_finalize(A16, 64, None, A16, 2, None, 1.0, 4, 16, 3584, A16, None) == 1
    assert lib.moe_finalize(A16, 63, None, A16, 0, None, 1.0, 4, 16, 3584, A16, None) == 1  # n_rows < T*K
    assert lib.moe_finalize(P(258), 64, None, A16, 0, None, 1.0, 4, 16, 3584, A16, None) == 2
    assert lib.moe_finalize(A16, 64, None, A16, 0, None, 1.0, 0, 16, 3584, A16, None) == 0  # T = 0: no-op
    assert lib.moe_topk_route(A16, None, 4, 896, 0, 1, 1.0, A16, None, None, None) == 1
    assert lib.moe_topk_route(A16, None, 4, 16, 17, 1, 1.0, A16, None, None, None) == 1
    assert lib.moe_topk_route(A16, None, 4, 4097, 16, 1, 1.0, A16, None, None, None) == 3
    assert lib.moe_topk_route(A16, None, 4, 896, 33, 1, 1.0, A16, None, None, None) == 3
    assert lib.mxfp8_quantize_rows(A16, 4, 33, A16, A16, None) == 1
    assert lib.mxfp8_quantize_rows(A16, 4, 0, A16, A16, None) == 1
    assert lib.mxfp8_quantize_rows(P(264), 4, 64, A16, A16, None) == 2
    assert lib.mxfp8_quantize_rows_ex(A16, 4, 64, A16, A16, 2, None) == 1
    assert lib.mxfp8_quantize_rows_ex(A16, 4, 33, A16, A16, 1, None) == 1
    assert lib.moe_build_routing_lists(A16, 4, 0, 896, A16, A16, None, 0, None) == 1
    assert lib.moe_build_routing_lists(A16, 4, 16, 4097, A16, A16, None, 0, None) == 3
    assert lib.moe_router_logits_ex(A16, A16, A16, 0, 7168, 896, None, 0, 0, None) == 1
    assert lib.moe_router_logits_ex(A16, A16, A16, 8, 7167, 896, None, 0, 0, None) == 1
    assert lib.moe_router_logits_ex(A16, A16, A16, 8, 7168, 896, None, 0, 7, None) == 1
    # the whole step: T >= 1, K >= 1, BF16 weights required
    chain = lambda T, K, wb: lib.moe_route_finalize(A16, A16, None, A16, A16, T, 7168, 3584, 896, K, 1, 1.0, A16, A16,
                                                    None, wb, A16, A16, A16, A16, A16, None, 0, None)
    assert chain(0, 16, A16) == 1
    assert chain(8, 0, A16) == 1
    assert chain(8, 16, None) == 1
    bad_x = lambda: lib.moe_route_finalize(P(264), A16, None, A16, A16, 8, 7168, 3584, 896, 16, 1, 1.0, A16, A16,
                                           None, A16, A16, A16, A16, A16, A16, None, 0, None)
    assert bad_x() == 2  # the step checks x itself (its router is launched directly)
    assert lib.moe_router_logits_ex(P(264), A16, A16, 8, 7168, 896, None, 0, 0, None) == 2
    assert lib.moe_build_unit_windows(A16, 0, 8, A16, A16, A16, A16, 4, None) == 1
    assert lib.moe_build_unit_windows(A16, 896, 0, A16, A16, A16, A16, 4, None) == 1
    assert lib.moe_build_unit_windows(A16, 4097, 8, A16, A16, A16, A16, 4, None) == 3
    assert lib.moe_build_unit_windows(A16, 896, 8, A16, None, A16, A16, 4, None) == 1
    assert lib.moe_build_unit_windows(P(258), 896, 8, A16, A16, A16, A16, 4, None) == 2
    assert lib.moe_unit_windows_capacity(1020, 16, 896, 8) == 2040 + 896
    assert lib.moe_unit_windows_capacity(10, 16, 896, 8) == 160  # at most one unit per pair
    assert lib.moe_unit_windows_capacity(10, 16, 896, 0) == -1
    fn = lambda T, K, H, eps=1e-5, g=A16, wdt=1: lib.moe_finalize_rmsnorm(A16, 1 << 20, None, A16, wdt, 1.0, g, eps, T,
                                                                           K, H, None, A16, None)
    assert fn(-1, 16, 3584) == 1
    assert fn(4, 0, 3584) == 1
    assert fn(4, 16, 3500) == 1  # H % 256
    assert fn(4, 16, 3584, eps=-1.0) == 1
    assert fn(4, 16, 3584, wdt=2) == 1
    assert fn(4, 16, 8448) == 3  # H > 8192
    assert fn(4, 16, 3584, g=None) == 1
    assert fn(4, 16, 3584, g=P(264)) == 2
    assert fn(0, 16, 3584) == 0  # T = 0: no-op
    front = lambda T, H, E, L, x=A16, wd=A16, lat=A16: lib.moe_front_projection(x, A16, wd, A16, lat, T, H, E, L, None,
                                                                               0, None)
    assert front(0, 7168, 896, 3584) == 1
    assert front(8, 7167, 896, 3584) == 1
    assert front(8, 7168, 0, 3584) == 1
    assert front(8, 7168, 896, 0) == 1
    assert front(8, 7168, 896, 3584, wd=None) == 1
    assert front(8, 7168, 1 << 23, 1 << 23) == 3
    assert front(8, 7168, 896, 3584, x=P(264)) == 2
    assert front(8, 7168, 896, 3584, lat=P(257)) == 2


def test_lists_workspace_query(lib):
    # the expert-parallel filter needs no scratch at any size
    for T in (0, 1, 1024, 1025, 4096, 65536):
        assert lib.moe_build_routing_lists_workspace(T, 16, 896) == 0


def test_python_binding_fails_loudly_without_library(tmp_path):
    import latent_moe_decode_gb300 as m

    saved = m._lib
    try:
        m._lib = None
        with pytest.raises(ImportError):
            m.load(str(tmp_path / "missing.so"))
    finally:
        m._lib = saved
