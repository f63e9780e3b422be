"""Seeded synthetic workloads for the GLM MoE feed-forward sublayer.

This module only draws random numbers and casts them to the storage dtype.
It holds none of the sublayer's arithmetic, so both the CUDA path and the
CPU oracle can be fed from it without sharing any computation.

Shapes follow the grouped native layout of the NeMo AutoModel GLM4-MoE state
dict adapter page ("Our native format groups them into"):
``gate_and_up_projs [E, d, 2I]`` and ``down_projs [E, I, d]``; the shared
expert keeps ``nn.Linear`` weights ``[out, in]`` (GlmMoeDsaMLP on the GLM-5
shared-expert page).

Recipe (every tensor has its own generator so that two workloads with the
same weight shapes share the same weights, e.g. GLM-5 prefill and decode):

  tensor index:  x=0, norm_w=1, router_w=2, corr_bias=3, gate_up=4, down=5,
                 shared_gate=6, shared_up=7, shared_down=8, hot_experts=9,
                 dense_gate=10, dense_up=11, dense_down=12, w_qa=13, q_norm_w=14
  generator seed: seed * 16 + tensor index

  x ~ N(0, 1); norm_w ~ U(0.5, 1.5); all projection weights ~ N(0, 0.02);
  corr_bias ~ U(-b, b) (b = 0.1 for the tiny fp32 case, 0.05 otherwise),
  plus +0.5 on ``n_hot`` experts taken from randperm(E)[:n_hot] when the
  workload is skewed.  gate_up / down are drawn one expert at a time.
  Values are drawn in fp32 and rounded (RNE) to the storage dtype.

The dense feed-forward block of the first decoder layers (GlmMoeDsaMLP with
its RMSNorm and residual) has workloads of its own (``DENSE_WORKLOADS``):
the same x and norm_w recipe, and nn.Linear gate, up [I, d] and down [d, I]
weights ~ N(0, 0.02).  The pages do not print GLM-5's dense intermediate
size; the GLM-5-sized dense workloads take I = 2 d = 12288.

The query compression of the sparse latent attention (``QLATENT_WORKLOADS``)
draws hidden ~ N(0, 1) (from the x generator), w_qa ~ N(0, 0.02) [rank, d]
and q_norm_w ~ U(0.5, 1.5).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

TENSOR_INDEX = {
    "x": 0, "norm_w": 1, "router_w": 2, "corr_bias": 3, "gate_up": 4,
    "down": 5, "shared_gate": 6, "shared_up": 7, "shared_down": 8,
    "hot_experts": 9, "dense_gate": 10, "dense_up": 11, "dense_down": 12,
    "w_qa": 13, "q_norm_w": 14,
}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int                  # tokens (B * S)
    d: int                  # hidden size
    E: int                  # routed experts
    I: int                  # routed expert intermediate size (moe_inter_dim)
    Is: int                 # shared expert intermediate size (0 = none)
    k: int                  # top_k
    routed_scale: float
    dtype: str              # "fp32" or "bf16": storage of x, weights, out
    bias_range: float = 0.05
    n_hot: int = 0          # experts given +hot_bias (skewed routing)
    hot_bias: float = 0.5
    eps: float = 1e-6
    description: str = ""

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five synthetic workloads: a tiny fp32 case, a small bf16 case, a
# GLM-4.5-Air-like prefill, the GLM-5-shaped prefill and GLM-5-shaped decode
# (the GLM-5 shapes: d = 6144 from the block in/out shape on the GLM-5 MoE
# block page; 256 routed experts with I = 2048 and one shared expert, which
# that page's parameter count 9,702,998,272 fixes).
WORKLOADS: Dict[str, Workload] = {
    "tiny_fp32": Workload("tiny_fp32", T=64, d=256, E=8, I=128, Is=128, k=2,
                          routed_scale=1.0, dtype="fp32", bias_range=0.1,
                          description="T64 d256 E8 I128 Is128 k2 fp32"),
    "small_bf16": Workload("small_bf16", T=2048, d=2048, E=64, I=768, Is=768,
                           k=4, routed_scale=1.0, dtype="bf16",
                           description="T2048 d2048 E64 I768 k4 bf16"),
    "air_prefill": Workload("air_prefill", T=4096, d=4096, E=128, I=1408,
                            Is=1408, k=8, routed_scale=2.5, dtype="bf16",
                            description="T4096 d4096 E128 I1408 k8 bf16"),
    "glm5_prefill": Workload("glm5_prefill", T=8192, d=6144, E=256, I=2048,
                             Is=2048, k=8, routed_scale=2.5, dtype="bf16",
                             description="T8192 d6144 E256 I2048 k8 bf16"),
    "glm5_decode": Workload("glm5_decode", T=64, d=6144, E=256, I=2048,
                            Is=2048, k=8, routed_scale=2.5, dtype="bf16",
                            n_hot=16,
                            description="T64 d6144 E256 I2048 k8 bf16, 16 hot experts"),
    # GLM-5 expert shapes with 32 experts and the same tokens per expert as
    # the prefill workload (2.5 GB of weights): the profiling case.
    "glm5_slice": Workload("glm5_slice", T=1024, d=6144, E=32, I=2048,
                           Is=2048, k=8, routed_scale=2.5, dtype="bf16",
                           description="T1024 d6144 E32 I2048 k8 bf16"),
    # GLM-5 routing shapes (tokens, hidden, experts, top-k) with narrow
    # experts (0.6 GB of weights): the profiling case of the routing kernels.
    "glm5_routing": Workload("glm5_routing", T=8192, d=6144, E=256, I=64,
                             Is=64, k=8, routed_scale=2.5, dtype="bf16",
                             description="T8192 d6144 E256 I64 k8 bf16"),
}


@dataclasses.dataclass(frozen=True)
class DenseWorkload:
    name: str
    T: int                  # tokens
    d: int                  # hidden size
    I: int                  # intermediate size of the dense MLP
    dtype: str              # "fp32" or "bf16"
    eps: float = 1e-6
    description: str = ""

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def with_(self, **kw) -> "DenseWorkload":
        return dataclasses.replace(self, **kw)


DENSE_WORKLOADS: Dict[str, DenseWorkload] = {
    "dense_tiny_fp32": DenseWorkload("dense_tiny_fp32", T=40, d=256, I=384, dtype="fp32",
                                     description="T40 d256 I384 fp32"),
    "dense_small_bf16": DenseWorkload("dense_small_bf16", T=700, d=1024, I=1536, dtype="bf16",
                                      description="T700 d1024 I1536 bf16"),
    "glm5_dense_prefill": DenseWorkload("glm5_dense_prefill", T=8192, d=6144, I=12288,
                                        dtype="bf16",
                                        description="T8192 d6144 I12288 bf16"),
    "glm5_dense_decode": DenseWorkload("glm5_dense_decode", T=64, d=6144, I=12288,
                                       dtype="bf16", description="T64 d6144 I12288 bf16"),
}


@dataclasses.dataclass(frozen=True)
class QLatentWorkload:
    """The query compression of the sparse latent attention: hidden [T, d]
    (the attention input) -> q_a_proj (w_qa [rank, d]) -> q_a_layernorm."""
    name: str
    T: int
    d: int
    rank: int               # q_lora_rank
    dtype: str
    eps: float = 1e-6
    description: str = ""

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def with_(self, **kw) -> "QLatentWorkload":
        return dataclasses.replace(self, **kw)


# GLM-5: d = 6144 and q_lora_rank = 2048 (the query latent's shape on the GLM-5
# "Query latent" page); the small cases cover both GEMM paths and ragged sizes.
QLATENT_WORKLOADS: Dict[str, QLatentWorkload] = {
    "q_tiny_fp32": QLatentWorkload("q_tiny_fp32", T=40, d=256, rank=64, dtype="fp32"),
    "q_small_bf16": QLatentWorkload("q_small_bf16", T=300, d=512, rank=192, dtype="bf16"),
    "q_pair_bf16": QLatentWorkload("q_pair_bf16", T=4800, d=1024, rank=1024, dtype="bf16"),
    "glm5_q_prefill": QLatentWorkload("glm5_q_prefill", T=8192, d=6144, rank=2048, dtype="bf16",
                                      description="T8192 d6144 q_lora_rank 2048 bf16"),
    "glm5_q_decode": QLatentWorkload("glm5_q_decode", T=64, d=6144, rank=2048, dtype="bf16",
                                     description="T64 d6144 q_lora_rank 2048 bf16"),
}


def make_q_inputs(w: QLatentWorkload, seed: int = 0, device: str = "cpu", T: Optional[int] = None,
                  weights_from: Optional[Dict[str, torch.Tensor]] = None) -> Dict[str, torch.Tensor]:
    """hidden ~ N(0, 1) (the attention input, an RMSNorm output), w_qa ~ N(0,
    0.02) as nn.Linear [rank, d], q_norm_w ~ U(0.5, 1.5); the x, w_qa and
    q_norm_w generators of the recipe above."""
    T = w.T if T is None else T
    dt = w.torch_dtype
    out: Dict[str, torch.Tensor] = {}
    out["hidden"] = _normal((T, w.d), 1.0, _gen(seed, "x", device), device, dt)
    if weights_from is not None:
        out["w_qa"], out["q_norm_w"] = weights_from["w_qa"], weights_from["q_norm_w"]
        return out
    out["w_qa"] = _normal((w.rank, w.d), 0.02, _gen(seed, "w_qa", device), device, dt)
    g = _gen(seed, "q_norm_w", device)
    out["q_norm_w"] = (torch.rand(w.rank, generator=g, device=device) + 0.5).to(dt)
    return out


def _gen(seed: int, name: str, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + TENSOR_INDEX[name])
    return g


def _normal(shape, std, gen, device, dtype):
    return (torch.randn(*shape, generator=gen, device=device,
                        dtype=torch.float32) * std).to(dtype)


def make_inputs(w: Workload, seed: int = 0, device: str = "cpu",
                T: Optional[int] = None,
                weights_from: Optional[Dict[str, torch.Tensor]] = None
                ) -> Dict[str, torch.Tensor]:
    """Draw every input of one forward.

    ``device`` selects where the generator runs ("cpu" or "cuda"); the two
    give different (each reproducible) values.  ``weights_from`` reuses the
    weight tensors of another workload with the same weight shapes (only x
    and corr_bias are drawn again).  Returns contiguous tensors on
    ``device``; corr_bias is always fp32.
    """
    T = w.T if T is None else T
    dt = w.torch_dtype
    out: Dict[str, torch.Tensor] = {}
    out["x"] = _normal((T, w.d), 1.0, _gen(seed, "x", device), device, dt)
    names = ("norm_w", "router_w", "gate_up", "down", "shared_gate",
             "shared_up", "shared_down")
    if weights_from is not None:
        for n in names:
            out[n] = weights_from[n]
    else:
        g = _gen(seed, "norm_w", device)
        out["norm_w"] = (torch.rand(w.d, generator=g, device=device) + 0.5).to(dt)
        out["router_w"] = _normal((w.E, w.d), 0.02,
                                  _gen(seed, "router_w", device), device, dt)
        gu = torch.empty((w.E, w.d, 2 * w.I), dtype=dt, device=device)
        g = _gen(seed, "gate_up", device)
        for e in range(w.E):
            gu[e] = _normal((w.d, 2 * w.I), 0.02, g, device, dt)
        out["gate_up"] = gu
        dn = torch.empty((w.E, w.I, w.d), dtype=dt, device=device)
        g = _gen(seed, "down", device)
        for e in range(w.E):
            dn[e] = _normal((w.I, w.d), 0.02, g, device, dt)
        out["down"] = dn
        Is = max(w.Is, 0)
        out["shared_gate"] = _normal((Is, w.d), 0.02,
                                     _gen(seed, "shared_gate", device), device, dt)
        out["shared_up"] = _normal((Is, w.d), 0.02,
                                   _gen(seed, "shared_up", device), device, dt)
        out["shared_down"] = _normal((w.d, Is), 0.02,
                                     _gen(seed, "shared_down", device), device, dt)
    g = _gen(seed, "corr_bias", device)
    bias = (torch.rand(w.E, generator=g, device=device) * 2.0 - 1.0) * w.bias_range
    if w.n_hot > 0:
        gh = _gen(seed, "hot_experts", device)
        hot = torch.randperm(w.E, generator=gh, device=device)[: w.n_hot]
        bias[hot] += w.hot_bias
    out["corr_bias"] = bias.to(torch.float32).contiguous()
    return out


def make_dense_inputs(w: DenseWorkload, seed: int = 0, device: str = "cpu",
                      T: Optional[int] = None,
                      weights_from: Optional[Dict[str, torch.Tensor]] = None
                      ) -> Dict[str, torch.Tensor]:
    """Draw every input of one dense-block forward: x, norm_w, dense_gate,
    dense_up [I, d] and dense_down [d, I] (the same conventions as
    ``make_inputs``)."""
    T = w.T if T is None else T
    dt = w.torch_dtype
    out: Dict[str, torch.Tensor] = {}
    out["x"] = _normal((T, w.d), 1.0, _gen(seed, "x", device), device, dt)
    if weights_from is not None:
        for n in ("norm_w", "dense_gate", "dense_up", "dense_down"):
            out[n] = weights_from[n]
        return out
    g = _gen(seed, "norm_w", device)
    out["norm_w"] = (torch.rand(w.d, generator=g, device=device) + 0.5).to(dt)
    out["dense_gate"] = _normal((w.I, w.d), 0.02, _gen(seed, "dense_gate", device), device, dt)
    out["dense_up"] = _normal((w.I, w.d), 0.02, _gen(seed, "dense_up", device), device, dt)
    out["dense_down"] = _normal((w.d, w.I), 0.02, _gen(seed, "dense_down", device), device, dt)
    return out


def host_arrays(inputs: Dict[str, torch.Tensor]):
    """numpy views of the inputs as stored: bf16 tensors become uint16 bit
    patterns, fp32 stays fp32.  Copies to host memory when needed."""
    res = {}
    for k, v in inputs.items():
        v = v.detach().contiguous().cpu()
        if v.dtype == torch.bfloat16:
            res[k] = v.view(torch.int16).numpy().view("uint16")
        else:
            res[k] = v.numpy()
    return res
