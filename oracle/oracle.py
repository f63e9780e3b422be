"""ctypes front end of the CPU oracle (moe_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg.  The product path never imports it.

``build()`` compiles moe_oracle.c with gcc/OpenMP into liboracle.so next to
this file; ``load()`` builds on first use when the library is missing or
older than its source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
HDR = os.path.join(HERE, "moe_oracle.h")
LIB = os.path.join(HERE, "liboracle.so")


class OracleCfg(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("E", ctypes.c_int32), ("I", ctypes.c_int32),
                ("Is", ctypes.c_int32), ("k", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("eps", ctypes.c_float), ("routed_scale", ctypes.c_float)]


def build(force: bool = False) -> str:
    stale = (not os.path.exists(LIB)
             or os.path.getmtime(LIB) < max(os.path.getmtime(SRC), os.path.getmtime(HDR)))
    if force or stale:
        # -ffp-contract=off: no fused multiply-adds, so every fp32 step of the
        # RMSNorm rounds exactly where the definition rounds.
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-std=c11", "-o", LIB + ".tmp", SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(LIB + ".tmp", LIB)
    return LIB


_lib = None


def load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.oracle_rmsnorm.argtypes = [ctypes.POINTER(OracleCfg), ctypes.c_int64, P, P, P]
        lib.oracle_route.argtypes = [ctypes.POINTER(OracleCfg), ctypes.c_int64, P, P, P,
                                     P, P, P, P]
        lib.oracle_select.argtypes = [ctypes.POINTER(OracleCfg), ctypes.c_int64, P, P, P, P, P]
        lib.oracle_forward.argtypes = [ctypes.POINTER(OracleCfg), ctypes.c_int64, P,
                                       P, P, P, P, P, P, P, P, P, P,
                                       P, P, P, P, P, P]
        lib.oracle_dense_forward.argtypes = [ctypes.POINTER(OracleCfg), ctypes.c_int64, P,
                                             P, P, P, P, P, P, P]
        lib.oracle_q_latent.argtypes = [ctypes.POINTER(OracleCfg), ctypes.c_int32, ctypes.c_int64,
                                        P, P, P, P, P, P]
        lib.oracle_param_count.argtypes = [ctypes.POINTER(OracleCfg)]
        lib.oracle_param_count.restype = ctypes.c_int64
        lib.oracle_num_threads.restype = ctypes.c_int
        for f in (lib.oracle_rmsnorm, lib.oracle_route, lib.oracle_select, lib.oracle_forward,
                  lib.oracle_dense_forward, lib.oracle_q_latent):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def cfg(d, E, I, Is, k, dtype, eps=1e-6, routed_scale=1.0) -> OracleCfg:
    dt = {"fp32": 0, "bf16": 1, 0: 0, 1: 1}[dtype]
    return OracleCfg(d, E, I, Is, k, dt, eps, routed_scale)


def cfg_from_workload(w) -> OracleCfg:
    return cfg(w.d, w.E, w.I, w.Is, w.k, w.dtype, w.eps, w.routed_scale)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check_storage(c: OracleCfg, *arrs):
    want = np.float32 if c.dtype == 0 else np.uint16
    for a in arrs:
        if a is not None:
            assert a.dtype == want and a.flags.c_contiguous, (a.dtype, want)


def rmsnorm(c: OracleCfg, x: np.ndarray, gain: np.ndarray) -> np.ndarray:
    _check_storage(c, x, gain)
    n = x.shape[0]
    xn = np.empty((n, c.d), np.float32)
    rc = load().oracle_rmsnorm(ctypes.byref(c), n, _ptr(x), _ptr(gain), _ptr(xn))
    assert rc == 0, rc
    return xn


def route(c: OracleCfg, xn: np.ndarray, router_w: np.ndarray, bias: np.ndarray):
    """Steps B-D on given xn (fp32 values).  Returns logits, idx, w, margin."""
    _check_storage(c, router_w)
    xn = np.ascontiguousarray(xn, np.float32)
    bias = np.ascontiguousarray(bias, np.float32)
    n = xn.shape[0]
    logits = np.empty((n, c.E), np.float32)
    idx = np.empty((n, c.k), np.int32)
    w = np.empty((n, c.k), np.float32)
    margin = np.empty((n,), np.float32)
    rc = load().oracle_route(ctypes.byref(c), n, _ptr(xn), _ptr(router_w), _ptr(bias),
                             _ptr(logits), _ptr(idx), _ptr(w), _ptr(margin))
    assert rc == 0, rc
    return logits, idx, w, margin


def select(c: OracleCfg, logits: np.ndarray, bias: np.ndarray):
    """Steps C-D on given fp32 logits [n, E].  Returns idx, w, margin."""
    logits = np.ascontiguousarray(logits, np.float32)
    bias = np.ascontiguousarray(bias, np.float32)
    n = logits.shape[0]
    idx = np.empty((n, c.k), np.int32)
    w = np.empty((n, c.k), np.float32)
    margin = np.empty((n,), np.float32)
    rc = load().oracle_select(ctypes.byref(c), n, _ptr(logits), _ptr(bias), _ptr(idx), _ptr(w),
                              _ptr(margin))
    assert rc == 0, rc
    return idx, w, margin


def forward(c: OracleCfg, a: dict, rows: Optional[np.ndarray] = None,
            forced_idx: Optional[np.ndarray] = None):
    """The whole sublayer.  ``a`` holds host arrays as stored (see
    workloads.host_arrays).  Returns a dict of out, idx, w, margin, xn, logits
    for the selected rows (all rows when ``rows`` is None)."""
    _check_storage(c, a["x"], a["norm_w"], a["router_w"], a["gate_up"], a["down"])
    n = a["x"].shape[0] if rows is None else len(rows)
    rows_arr = None if rows is None else np.ascontiguousarray(rows, np.int64)
    forced = None if forced_idx is None else np.ascontiguousarray(forced_idx, np.int32)
    res = {
        "out": np.empty((n, c.d), np.float32),
        "idx": np.empty((n, c.k), np.int32),
        "w": np.empty((n, c.k), np.float32),
        "margin": np.empty((n,), np.float32),
        "xn": np.empty((n, c.d), np.float32),
        "logits": np.empty((n, c.E), np.float32),
    }
    bias = np.ascontiguousarray(a["corr_bias"], np.float32)
    rc = load().oracle_forward(
        ctypes.byref(c), n, _ptr(rows_arr), _ptr(a["x"]), _ptr(a["norm_w"]),
        _ptr(a["router_w"]), _ptr(bias), _ptr(a["gate_up"]), _ptr(a["down"]),
        _ptr(a.get("shared_gate")), _ptr(a.get("shared_up")), _ptr(a.get("shared_down")),
        _ptr(forced), _ptr(res["out"]), _ptr(res["idx"]), _ptr(res["w"]),
        _ptr(res["margin"]), _ptr(res["xn"]), _ptr(res["logits"]))
    assert rc == 0, rc
    return res


def dense_cfg(d: int, inter: int, dtype, eps: float = 1e-6) -> OracleCfg:
    """Configuration of the dense block: ``inter`` travels in the Is field."""
    return cfg(d, 1, 1, inter, 1, dtype, eps)


def dense_forward(c: OracleCfg, a: dict, rows: Optional[np.ndarray] = None):
    """The dense feed-forward block x + GlmMoeDsaMLP(RMSNorm(x)).  ``a``
    holds host arrays as stored: x, norm_w, dense_gate, dense_up, dense_down.
    Returns out and xn (fp32) for the selected rows."""
    _check_storage(c, a["x"], a["norm_w"], a["dense_gate"], a["dense_up"], a["dense_down"])
    n = a["x"].shape[0] if rows is None else len(rows)
    rows_arr = None if rows is None else np.ascontiguousarray(rows, np.int64)
    res = {"out": np.empty((n, c.d), np.float32), "xn": np.empty((n, c.d), np.float32)}
    rc = load().oracle_dense_forward(
        ctypes.byref(c), n, _ptr(rows_arr), _ptr(a["x"]), _ptr(a["norm_w"]),
        _ptr(a["dense_gate"]), _ptr(a["dense_up"]), _ptr(a["dense_down"]),
        _ptr(res["out"]), _ptr(res["xn"]))
    assert rc == 0, rc
    return res


def q_latent(d: int, rank: int, dtype, hidden: np.ndarray, w_qa: np.ndarray, gain: np.ndarray,
             eps: float = 1e-6, rows: Optional[np.ndarray] = None):
    """The query compression of GLM-5's sparse latent attention (GLM-5 "Query
    latent" page: q_resid = q_a_layernorm(q_a_proj(hidden_states)), q_a_proj
    an nn.Linear(d -> rank) without bias, q_a_layernorm a GlmMoeDsaRMSNorm(rank)).
    hidden [n, d], w_qa [rank, d] and gain [rank] as stored.  Returns (c, q):
    the query latent before and after the norm, [n, rank] fp32 values."""
    c = cfg(d, 1, 1, 0, 1, dtype, eps)
    _check_storage(c, hidden, w_qa, gain)
    n = hidden.shape[0] if rows is None else len(rows)
    rows_arr = None if rows is None else np.ascontiguousarray(rows, np.int64)
    c_out = np.empty((n, rank), np.float32)
    q_out = np.empty((n, rank), np.float32)
    rc = load().oracle_q_latent(ctypes.byref(c), rank, n, _ptr(rows_arr), _ptr(hidden), _ptr(w_qa),
                                _ptr(gain), _ptr(c_out), _ptr(q_out))
    assert rc == 0, rc
    return c_out, q_out


def pack_experts(gate: np.ndarray, up: np.ndarray, down: np.ndarray):
    """HF per-expert nn.Linear weights -> the grouped native layout (NeMo
    AutoModel GLM4-MoE state dict adapter page, Glm4MoeStateDictAdapter:
    experts.{E}.gate_proj / up_proj / down_proj are grouped into
    gate_and_up_projs [n_experts, dim, 2*moe_inter_dim] and down_projs
    [n_experts, moe_inter_dim, dim]).  gate, up [E, I, d] and down [E, d, I]
    are the experts' HF tensors stacked; gate_and_up[e] = [gate[e]^T | up[e]^T]
    (gate columns first), down_projs[e] = down[e]^T.  Pure data movement: any
    dtype, bit for bit."""
    gate_up = np.ascontiguousarray(np.concatenate([gate.transpose(0, 2, 1), up.transpose(0, 2, 1)],
                                                  axis=2))
    down_projs = np.ascontiguousarray(down.transpose(0, 2, 1))
    return gate_up, down_projs


def param_count(c: OracleCfg) -> int:
    return int(load().oracle_param_count(ctypes.byref(c)))


def num_threads() -> int:
    return int(load().oracle_num_threads())
