"""Thin Python binding of the C ABI in include/moe.h (ctypes).

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of libmoe_b300.so.  PyTorch is used for device memory and streams.
Loading fails loudly when the library has not been built; there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_b300.so")

(MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_OOM, MOE_ERR_TIMEOUT,
 MOE_ERR_RANGE) = range(7)
DTYPE_FP32, DTYPE_BF16 = 0, 1
T_XN, T_LOGITS, T_OFFSETS, T_POS, T_ROW_TOK, T_H, T_YP = range(7)

# Functions the header declares (kept in sync by the ABI test).
EXPORTS = ("moe_init", "moe_forward", "moe_forward_host", "moe_forward_host_async",
           "moe_forward_host_wait", "moe_dense_forward", "moe_q_latent", "moe_get_routing",
           "moe_get_intermediate", "moe_sync_status", "moe_selftest_wait_timeout",
           "moe_set_profiling", "moe_read_stats",
           "moe_destroy", "moe_route_static", "moe_pack_experts", "moe_status_string")
# Stages of one forward (the gate_up and down launches carry the routed
# experts and the shared expert).
STAGES = ("rmsnorm", "router", "topk", "scan", "scatter", "gather", "gate_up_swiglu",
          "down_weighted", "combine")


class MoeConfig(ctypes.Structure):
    _fields_ = [("max_tokens", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("max_top_k", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("eps", ctypes.c_float),
                ("device", ctypes.c_int32), ("gemm_path", ctypes.c_int32),
                ("dense_inter", ctypes.c_int32)]


class MoeStats(ctypes.Structure):
    _fields_ = [("forwards", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("n_stages", ctypes.c_int32), ("stage_ms", ctypes.c_float * 16)]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libmoe_b300.so and declares the signatures.  Raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m mixture_experts_transformer_sigmoid_b300.build`")
    lib = ctypes.CDLL(path)
    P, I32, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    lib.moe_init.argtypes = [ctypes.POINTER(MoeConfig), ctypes.POINTER(ctypes.c_void_p)]
    fwd = [P, I32, P, P, P, P, P, P, P, P, P, I32, F32, P, P]
    lib.moe_forward.argtypes = fwd
    lib.moe_forward_host.argtypes = fwd
    lib.moe_forward_host_async.argtypes = fwd
    lib.moe_forward_host_wait.argtypes = [P]
    lib.moe_dense_forward.argtypes = [P, I32, P, P, P, P, P, I32, P, P]
    lib.moe_q_latent.argtypes = [P, I32, I32, P, P, P, P, P, P]
    lib.moe_get_routing.argtypes = [P, P, P, P, P]
    lib.moe_get_intermediate.argtypes = [P, ctypes.c_int, P, ctypes.c_size_t, P]
    lib.moe_sync_status.argtypes = [P, P]
    lib.moe_selftest_wait_timeout.argtypes = [P, ctypes.c_uint32, P]
    lib.moe_set_profiling.argtypes = [P, I32]
    lib.moe_read_stats.argtypes = [P, ctypes.POINTER(MoeStats)]
    lib.moe_destroy.argtypes = [P]
    lib.moe_route_static.argtypes = [I32, I32, I32, F32, P, P, P, P, P, P, P, P, P, P]
    lib.moe_pack_experts.argtypes = [I32, I32, I32, I32, P, P, P, P, P, P]
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_status_string.restype = ctypes.c_char_p
    for name in EXPORTS[:-1]:
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class MoeSublayer:
    """One handle of the C ABI: workspace for up to ``max_tokens`` tokens."""

    def __init__(self, *, max_tokens: int, hidden: int, n_experts: int, inter: int,
                 shared_inter: int, max_top_k: int, dtype: str = "bf16", eps: float = 1e-6,
                 device: int = 0, gemm_path: int = 0, dense_inter: int = 0):
        self.lib = load_library()
        self.cfg = MoeConfig(max_tokens, hidden, n_experts, inter, shared_inter, max_top_k,
                             DTYPE_BF16 if dtype == "bf16" else DTYPE_FP32, eps, device, gemm_path,
                             dense_inter)
        self.dtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.tensor_cores = dtype == "bf16" and gemm_path == 0   # the library's tcgen05 path
        self.device = torch.device("cuda", device)
        h = ctypes.c_void_p()
        _check(self.lib.moe_init(ctypes.byref(self.cfg), ctypes.byref(h)), "moe_init")
        self.handle = h
        self.last_T = 0
        self.last_k = 0

    def close(self):
        if self.handle is not None and self.handle.value:
            self.lib.moe_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _stream(stream):
        if stream is None:
            stream = torch.cuda.current_stream()
        return ctypes.c_void_p(stream.cuda_stream)

    def forward(self, x, w: dict, top_k: int, routed_scale: float, out=None, stream=None):
        """x [T, d] on the device; w holds norm_w, router_w, corr_bias,
        gate_up, down, shared_gate, shared_up, shared_down (device tensors)."""
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        st = self._stream(stream)
        _check(self.lib.moe_forward(
            self.handle, T, _ptr(x), _ptr(w["norm_w"]), _ptr(w["router_w"]), _ptr(w["corr_bias"]),
            _ptr(w["gate_up"]), _ptr(w["down"]), _ptr(w.get("shared_gate")),
            _ptr(w.get("shared_up")), _ptr(w.get("shared_down")), top_k, routed_scale,
            _ptr(out), st), "moe_forward")
        self.last_T, self.last_k = T, top_k
        return out

    def dense_forward(self, x, w: dict, out=None, stream=None):
        """moe_dense_forward: x + GlmMoeDsaMLP(RMSNorm(x)); w holds norm_w,
        dense_gate, dense_up [I, d] and dense_down [d, I] (device tensors)."""
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        _check(self.lib.moe_dense_forward(
            self.handle, T, _ptr(x), _ptr(w["norm_w"]), _ptr(w["dense_gate"]), _ptr(w["dense_up"]),
            _ptr(w["dense_down"]), w["dense_gate"].shape[0], _ptr(out), self._stream(stream)),
            "moe_dense_forward")
        return out

    def q_latent(self, hidden, w_qa, q_norm_w, c_out=None, q_out=None, stream=None):
        """moe_q_latent: the query compression of the sparse latent attention,
        (c, q) = (q_a_proj(hidden), q_a_layernorm(c)); hidden [T, d], w_qa
        [q_rank, d], q_norm_w [q_rank] (device tensors)."""
        T, rank = hidden.shape[0], w_qa.shape[0]
        if c_out is None:
            c_out = torch.empty((T, rank), dtype=hidden.dtype, device=hidden.device)
        if q_out is None:
            q_out = torch.empty((T, rank), dtype=hidden.dtype, device=hidden.device)
        _check(self.lib.moe_q_latent(self.handle, T, rank, _ptr(hidden), _ptr(w_qa), _ptr(q_norm_w),
                                     _ptr(c_out), _ptr(q_out), self._stream(stream)), "moe_q_latent")
        return c_out, q_out

    def forward_host(self, x_host, w: dict, top_k: int, routed_scale: float, out_host,
                     stream=None):
        """x_host / out_host: CPU tensors (pinned for asynchronous copies)."""
        T = x_host.shape[0]
        _check(self.lib.moe_forward_host(
            self.handle, T, _ptr(x_host), _ptr(w["norm_w"]), _ptr(w["router_w"]),
            _ptr(w["corr_bias"]), _ptr(w["gate_up"]), _ptr(w["down"]),
            _ptr(w.get("shared_gate")), _ptr(w.get("shared_up")), _ptr(w.get("shared_down")),
            top_k, routed_scale, _ptr(out_host), self._stream(stream)), "moe_forward_host")
        self.last_T, self.last_k = T, top_k
        return out_host

    def forward_host_async(self, x_host, w: dict, top_k: int, routed_scale: float, out_host,
                           stream=None):
        """Queues one host-buffer forward without waiting (pipelined copies);
        out_host is filled once forward_host_wait returns."""
        T = x_host.shape[0]
        _check(self.lib.moe_forward_host_async(
            self.handle, T, _ptr(x_host), _ptr(w["norm_w"]), _ptr(w["router_w"]),
            _ptr(w["corr_bias"]), _ptr(w["gate_up"]), _ptr(w["down"]),
            _ptr(w.get("shared_gate")), _ptr(w.get("shared_up")), _ptr(w.get("shared_down")),
            top_k, routed_scale, _ptr(out_host), self._stream(stream)), "moe_forward_host_async")
        self.last_T, self.last_k = T, top_k
        return out_host

    def forward_host_wait(self):
        _check(self.lib.moe_forward_host_wait(self.handle), "moe_forward_host_wait")

    def routing(self, stream=None):
        T, k, E = self.last_T, self.last_k, self.cfg.n_experts
        idx = torch.empty((T, k), dtype=torch.int32, device=self.device)
        wt = torch.empty((T, k), dtype=torch.float32, device=self.device)
        counts = torch.empty((E,), dtype=torch.int32, device=self.device)
        _check(self.lib.moe_get_routing(self.handle, _ptr(idx), _ptr(wt), _ptr(counts),
                                        self._stream(stream)), "moe_get_routing")
        return idx, wt, counts

    def intermediate(self, which: int, stream=None):
        T, k, c = self.last_T, self.last_k, self.cfg
        shapes = {T_XN: ((T, c.hidden), self.dtype), T_LOGITS: ((T, c.n_experts), torch.float32),
                  T_OFFSETS: ((c.n_experts + 1,), torch.int32), T_POS: ((T, k), torch.int32),
                  T_ROW_TOK: ((T * k,), torch.int32), T_H: ((T * k, c.inter), self.dtype),
                  T_YP: ((T * k, c.hidden), torch.float16 if self.tensor_cores else self.dtype)}
        shape, dt = shapes[which]
        dst = torch.empty(shape, dtype=dt, device=self.device)
        _check(self.lib.moe_get_intermediate(self.handle, which, _ptr(dst),
                                             dst.numel() * dst.element_size(),
                                             self._stream(stream)), "moe_get_intermediate")
        return dst

    def sync_status(self, stream=None) -> int:
        return self.lib.moe_sync_status(self.handle, self._stream(stream))

    def selftest_wait_timeout(self, timeout_us: int, stream=None):
        """Queues a bounded wait that nothing completes; the next
        sync_status reports MOE_ERR_TIMEOUT."""
        _check(self.lib.moe_selftest_wait_timeout(self.handle, timeout_us, self._stream(stream)),
               "moe_selftest_wait_timeout")

    def set_profiling(self, enable: bool):
        _check(self.lib.moe_set_profiling(self.handle, 1 if enable else 0), "moe_set_profiling")

    def read_stats(self) -> dict:
        """Counters since the last call: forwards, kernel launches, and the
        summed GPU milliseconds of each stage (profiling on)."""
        st = MoeStats()
        _check(self.lib.moe_read_stats(self.handle, ctypes.byref(st)), "moe_read_stats")
        return {"forwards": st.forwards, "launches": st.launches,
                "stage_ms": {STAGES[i]: float(st.stage_ms[i]) for i in range(st.n_stages)}}


# Scratch limit of moe_route_static: ceil(T / 128) * E histogram cells.
ROUTE_STATIC_MAX_CELLS = 131072


def route_static(logits: torch.Tensor, corr_bias: torch.Tensor, top_k: int,
                 routed_scale: float, out: Optional[dict] = None, stream=None) -> dict:
    """moe_route_static: routing of a batch from fp32 router logits [T, E]
    on the current device, with no allocation inside the library (for
    callers that cannot allocate device memory).  ``out`` may hold the
    caller's output tensors (idx, w, counts, offsets, pos, row_tok, row_w);
    missing ones are created here with torch.  Calls that overlap on the GPU
    share one static scratch array and race."""
    if logits.dim() != 2 or logits.dtype != torch.float32 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous fp32 [T, E] tensor")
    T, E = logits.shape
    dev = logits.device
    if dev.type != "cuda":
        raise ValueError("logits must be on a CUDA device")
    if (corr_bias.dtype != torch.float32 or not corr_bias.is_contiguous()
            or corr_bias.numel() != E or corr_bias.device != dev):
        raise ValueError("corr_bias must be a contiguous fp32 [E] tensor on the logits' device")
    shapes = {"idx": ((T, top_k), torch.int32), "w": ((T, top_k), torch.float32),
              "counts": ((E,), torch.int32), "offsets": ((E + 1,), torch.int32),
              "pos": ((T, top_k), torch.int32), "row_tok": ((T * top_k,), torch.int32),
              "row_w": ((T * top_k,), torch.float32)}
    res = dict(out or {})
    for name, (shape, dt) in shapes.items():
        if name not in res:
            res[name] = torch.empty(shape, dtype=dt, device=dev)
        else:
            t = res[name]
            if (t.dtype != dt or not t.is_contiguous() or t.numel() != int(torch.Size(shape).numel())
                    or t.device != dev):
                raise ValueError(f"out[{name!r}] must be a contiguous {dt} tensor of {shape} "
                                 f"elements on {dev}")
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):   # the library takes its scratch address from the current device
        st = load_library().moe_route_static(
            T, E, top_k, routed_scale, _ptr(logits), _ptr(corr_bias), _ptr(res["idx"]),
            _ptr(res["w"]), _ptr(res["counts"]), _ptr(res["offsets"]), _ptr(res["pos"]),
            _ptr(res["row_tok"]), _ptr(res["row_w"]), ctypes.c_void_p(stream.cuda_stream))
    if st == MOE_ERR_UNSUPPORTED:
        raise MoeError(st, f"moe_route_static: ceil(T/128)*E = {-(-T // 128) * E} exceeds the "
                           f"static scratch limit of {ROUTE_STATIC_MAX_CELLS} cells")
    _check(st, "moe_route_static")
    return res


def pack_experts(gate: torch.Tensor, up: torch.Tensor, down: torch.Tensor,
                 gate_up: Optional[torch.Tensor] = None, down_projs: Optional[torch.Tensor] = None,
                 stream=None):
    """moe_pack_experts: HF per-expert weights (gate, up [E, I, d], down
    [E, d, I], stacked) -> the grouped layout gate_up [E, d, 2I] and
    down_projs [E, I, d] that MoeSublayer.forward reads."""
    E, I, d = gate.shape
    if gate_up is None:
        gate_up = torch.empty((E, d, 2 * I), dtype=gate.dtype, device=gate.device)
    if down_projs is None:
        down_projs = torch.empty((E, I, d), dtype=down.dtype, device=down.device)
    if stream is None:
        stream = torch.cuda.current_stream(gate.device)
    _check(load_library().moe_pack_experts(E, d, I, gate.element_size(), _ptr(gate), _ptr(up), _ptr(down),
                                           _ptr(gate_up), _ptr(down_projs),
                                           ctypes.c_void_p(stream.cuda_stream)), "moe_pack_experts")
    return gate_up, down_projs
