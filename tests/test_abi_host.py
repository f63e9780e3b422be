"""The C-ABI library loads and exports what include/moe.h declares, and its
host-side argument checks reject bad calls before any CUDA work.  Runs
without a GPU: no call here launches a kernel."""
import ctypes
import os
import re

import pytest
import torch

from mixture_experts_transformer_sigmoid_b300 import binding as B
from mixture_experts_transformer_sigmoid_b300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text, re.M)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(B.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_config_struct_matches_header():
    text = open(HEADER).read()
    body = re.search(r"typedef struct \{(.*?)\} moe_config;", text, re.S).group(1)
    fields = re.findall(r"(?:int32_t|float)\s+(\w+);", body)
    assert fields == [f for f, _ in B.MoeConfig._fields_]


def test_status_strings(lib):
    for s in range(6):
        assert len(B.status_string(s)) > 0
    assert B.status_string(0) == "ok"
    assert B.status_string(99) == "unknown status"


def good_cfg(**kw):
    c = dict(max_tokens=64, hidden=256, n_experts=8, inter=128, shared_inter=128, max_top_k=2,
             dtype=B.DTYPE_BF16, eps=1e-6, device=0, gemm_path=0, dense_inter=0)
    c.update(kw)
    return B.MoeConfig(**c)


@pytest.mark.parametrize("kw,status", [
    (dict(max_tokens=0), B.MOE_ERR_INVALID_ARG),
    (dict(hidden=0), B.MOE_ERR_INVALID_ARG),
    (dict(n_experts=0), B.MOE_ERR_INVALID_ARG),
    (dict(n_experts=2000), B.MOE_ERR_INVALID_ARG),
    (dict(max_top_k=0), B.MOE_ERR_INVALID_ARG),
    (dict(max_top_k=9), B.MOE_ERR_INVALID_ARG),      # > n_experts
    (dict(dtype=7), B.MOE_ERR_INVALID_ARG),
    (dict(eps=float("nan")), B.MOE_ERR_INVALID_ARG),
    (dict(eps=-1.0), B.MOE_ERR_INVALID_ARG),
    (dict(device=-1), B.MOE_ERR_INVALID_ARG),
    (dict(gemm_path=5), B.MOE_ERR_INVALID_ARG),
    (dict(shared_inter=-1), B.MOE_ERR_INVALID_ARG),
    (dict(hidden=200), B.MOE_ERR_UNSUPPORTED),       # tensor-core path needs multiples of 64
    (dict(inter=100), B.MOE_ERR_UNSUPPORTED),
    (dict(hidden=36, dtype=B.DTYPE_FP32), B.MOE_OK),                # valid fp32 shape
    (dict(dense_inter=-1), B.MOE_ERR_INVALID_ARG),
    (dict(dense_inter=100), B.MOE_ERR_UNSUPPORTED),  # tensor-core path needs multiples of 64
    (dict(dense_inter=512), B.MOE_OK),               # MoE handle with dense workspace
    # a handle for the dense block only: no experts, no routed sizes
    (dict(n_experts=0, inter=0, shared_inter=0, max_top_k=0, dense_inter=512), B.MOE_OK),
    (dict(n_experts=0, inter=0, shared_inter=0, max_top_k=0, dense_inter=0), B.MOE_ERR_INVALID_ARG),
    (dict(n_experts=0, inter=128, shared_inter=0, max_top_k=0, dense_inter=512), B.MOE_ERR_INVALID_ARG),
    (dict(n_experts=0, inter=0, shared_inter=0, max_top_k=1, dense_inter=512), B.MOE_ERR_INVALID_ARG),
    # the CUDA-core path stages one fp32 input row in 48 KB of shared memory
    (dict(dtype=B.DTYPE_FP32, dense_inter=12288), B.MOE_OK),
    (dict(dtype=B.DTYPE_FP32, dense_inter=12292), B.MOE_ERR_UNSUPPORTED),
    (dict(dtype=B.DTYPE_FP32, hidden=12800), B.MOE_ERR_UNSUPPORTED),
])
def test_init_rejects_bad_config(lib, kw, status):
    c = good_cfg(**kw)
    h = ctypes.c_void_p()
    rc = lib.moe_init(ctypes.byref(c), ctypes.byref(h))
    if status == B.MOE_OK:
        # a valid config: on a machine without a GPU the device query fails
        if torch.cuda.is_available():
            assert rc == B.MOE_OK
            lib.moe_destroy(h)
        else:
            assert rc == B.MOE_ERR_CUDA
        return
    assert rc == status
    assert not h.value


def test_init_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.moe_init(None, ctypes.byref(h)) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_init(ctypes.byref(good_cfg()), None) == B.MOE_ERR_INVALID_ARG


def test_calls_on_null_handle(lib):
    p = ctypes.c_void_p(16)
    assert lib.moe_forward(None, 1, p, p, p, p, p, p, p, p, p, 1, 1.0, p, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_host(None, 1, p, p, p, p, p, p, p, p, p, 1, 1.0, p, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_get_routing(None, None, None, None, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_get_intermediate(None, 0, p, 16, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_sync_status(None, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_dense_forward(None, 1, p, p, p, p, p, 64, p, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_wait_timeout(None, 1000, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_destroy(None) == B.MOE_OK


def test_binding_fails_loudly_without_library(tmp_path):
    B2 = B
    saved = B2._lib
    try:
        B2._lib = None
        with pytest.raises(RuntimeError):
            B2.load_library(str(tmp_path / "missing.so"))
    finally:
        B2._lib = saved


@pytest.mark.parametrize("T,E,k,status", [
    (-1, 8, 2, B.MOE_ERR_INVALID_ARG), (64, 0, 1, B.MOE_ERR_INVALID_ARG),
    (64, 8, 0, B.MOE_ERR_INVALID_ARG), (64, 8, 9, B.MOE_ERR_INVALID_ARG),
    (64, 2000, 2, B.MOE_ERR_INVALID_ARG), (128 * 513, 256, 8, B.MOE_ERR_UNSUPPORTED),
    (64, 8, 2, B.MOE_ERR_INVALID_ARG),   # valid sizes, null pointers
    (0, 8, 2, B.MOE_OK),                 # nothing to do, no pointer read
])
def test_route_static_host_checks(lib, T, E, k, status):
    nulls = [None] * 9
    assert lib.moe_route_static(T, E, k, 1.0, *nulls, None) == status


def test_route_static_rejects_overlap_before_touching_the_device(lib):
    """Outputs overlapping an input or each other are rejected by the host
    checks, before any CUDA call (fake, aligned addresses: nothing is read)."""
    T, E, k = 256, 16, 2                        # logits 16 KB, each [T, k] array 2 KB
    base = [ctypes.c_void_p((i + 1) << 20) for i in range(9)]
    logits, bias, idx, w, counts, offsets, pos, row_tok, row_w = base
    over_logits = ctypes.c_void_p((1 << 20) + 4096)
    assert lib.moe_route_static(T, E, k, 1.0, logits, bias, idx, over_logits, counts, offsets, pos,
                                row_tok, row_w, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_route_static(T, E, k, 1.0, logits, bias, idx, w, counts, offsets, pos,
                                ctypes.c_void_p((7 << 20) + 1024), row_w, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_route_static(T, E, k, 1.0, logits, bias, idx, w, bias, offsets, pos,
                                row_tok, row_w, None) == B.MOE_ERR_INVALID_ARG


def test_host_io_entry_points_reject_a_null_handle(lib):
    nulls = [None] * 11
    assert lib.moe_forward_host_async(None, 4, *nulls[:9], 2, 1.0, None, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_host_wait(None) == B.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("E,d,I,eb,status", [
    (-1, 64, 64, 2, B.MOE_ERR_INVALID_ARG), (2, 0, 64, 2, B.MOE_ERR_INVALID_ARG),
    (2, 64, 0, 2, B.MOE_ERR_INVALID_ARG), (2, 64, 64, 3, B.MOE_ERR_INVALID_ARG),
    (70000, 64, 64, 2, B.MOE_ERR_UNSUPPORTED),           # grid z limit
    (2, 63, 64, 2, B.MOE_ERR_UNSUPPORTED),               # bf16 moves whole 4-byte words
    (2, 64, 65, 2, B.MOE_ERR_UNSUPPORTED),
    (0, 64, 64, 2, B.MOE_OK),                            # nothing to do, no pointer read
])
def test_pack_experts_host_checks(lib, E, d, I, eb, status):
    p = [ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20), ctypes.c_void_p(3 << 20)]
    out = [ctypes.c_void_p(8 << 20), ctypes.c_void_p(16 << 20)]
    assert lib.moe_pack_experts(E, d, I, eb, *p, *out, None) == status


def test_pack_experts_pointer_checks(lib):
    g, u, dn = ctypes.c_void_p(1 << 24), ctypes.c_void_p(2 << 24), ctypes.c_void_p(3 << 24)
    gu, do = ctypes.c_void_p(4 << 24), ctypes.c_void_p(6 << 24)
    E, d, I = 2, 64, 64       # each HF stack is 16 KB, gate_up 32 KB
    assert lib.moe_pack_experts(E, d, I, 2, g, u, dn, None, None, None) == B.MOE_OK  # no outputs
    assert lib.moe_pack_experts(E, d, I, 2, None, u, dn, gu, None, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_pack_experts(E, d, I, 2, g, u, None, None, do, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_pack_experts(E, d, I, 2, ctypes.c_void_p((1 << 24) + 2), u, dn, gu, None,
                                None) == B.MOE_ERR_INVALID_ARG                   # misaligned
    assert lib.moe_pack_experts(E, d, I, 2, g, u, dn, ctypes.c_void_p((2 << 24) + 64), None,
                                None) == B.MOE_ERR_INVALID_ARG                   # output over `up`
    assert lib.moe_pack_experts(E, d, I, 2, g, u, dn, gu, ctypes.c_void_p((4 << 24) + 1024),
                                None) == B.MOE_ERR_INVALID_ARG                   # outputs overlap
