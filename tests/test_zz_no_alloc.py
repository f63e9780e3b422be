"""moe_route_static, the routing entry point that allocates nothing.

Some callers cannot call cudaMalloc: a serving engine that reserved all
device memory for its own pool up front, or code that must not let an
allocation synchronise the device mid-step.  moe_route_static serves them
with scratch in a static device array.  Its outputs must equal, bit for bit,
the routing moe_forward computed from the same logits (integer and index
work is compared exactly, like every routing test here; the weights come
from the same fp32 operations, so they are exact too).

Two calls run back to back, the second on a smaller, ragged batch, so the
second reads the shared scratch right after the first left its own
contents there.  This file sorts last so that a run stopping at the first
failure has run every other test before it.
"""
import numpy as np
import pytest
import torch

import parity
from mixture_experts_transformer_sigmoid_b300 import binding as B
from mixture_experts_transformer_sigmoid_b300 import build as build_mod
from mixture_experts_transformer_sigmoid_b300 import workloads as wl
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def forward_routing(layer, inp, w, T):
    """Routing tensors of one moe_forward over the first T tokens."""
    layer.forward(inp["x"][:T].contiguous(), inp, w.k, w.routed_scale)
    idx, wt, counts = layer.routing()
    ref = {"idx": idx, "w": wt, "counts": counts,
           "logits": layer.intermediate(B.T_LOGITS),
           "offsets": layer.intermediate(B.T_OFFSETS),
           "pos": layer.intermediate(B.T_POS),
           "row_tok": layer.intermediate(B.T_ROW_TOK)}
    assert layer.sync_status() == B.MOE_OK
    return ref


def check_same(got, ref, T, k):
    for name in ("idx", "counts", "offsets", "pos", "row_tok"):
        assert torch.equal(got[name], ref[name]), name
    assert torch.equal(got["w"], ref["w"])
    # row_w is the weight of each permuted row: w scattered through pos
    expect_row_w = torch.empty(T * k, dtype=torch.float32, device=ref["w"].device)
    expect_row_w[ref["pos"].reshape(-1).long()] = ref["w"].reshape(-1)
    assert torch.equal(got["row_w"], expect_row_w)


def test_route_static_matches_forward_on_two_calls_in_a_row():
    build_mod.build()
    w = wl.Workload("route_static", T=2048, d=512, E=64, I=128, Is=128, k=6,
                    routed_scale=2.5, dtype="bf16")
    inp = {k: v.cuda() for k, v in wl.make_inputs(w, seed=3).items()}
    layer = B.MoeSublayer(max_tokens=w.T, hidden=w.d, n_experts=w.E, inter=w.I,
                          shared_inter=w.Is, max_top_k=w.k, dtype=w.dtype, eps=w.eps)
    try:
        sizes = (w.T, 777)  # a full batch, then a ragged one (not a multiple of 128)
        refs = [forward_routing(layer, inp, w, T) for T in sizes]
        torch.cuda.synchronize()
        outs = [B.route_static(r["logits"], inp["corr_bias"], w.k, w.routed_scale)
                for r in refs]
        torch.cuda.synchronize()
        for T, got, ref in zip(sizes, outs, refs):
            check_same(got, ref, T, w.k)
            assert int(got["counts"].sum()) == T * w.k
    finally:
        layer.close()


def test_route_static_rejects_sizes_beyond_its_scratch():
    logits = torch.zeros((128 * 513, 256), dtype=torch.float32, device="cuda")
    bias = torch.zeros(256, dtype=torch.float32, device="cuda")
    with pytest.raises(B.MoeError) as ei:
        B.route_static(logits, bias, 8, 1.0)
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED


def test_route_static_matches_oracle_selection():
    """The selection and weights against the oracle's steps C-D run on the
    same fp32 logits: the same set of experts per token (a k-th / (k+1)-th
    margin below 1e-5 excepted), an order the scores allow, and weights
    within 2e-6 relative."""
    T, E, k, scale = 1000, 96, 6, 2.5
    g = torch.Generator().manual_seed(11)
    logits = torch.randn((T, E), generator=g) * 1.5
    bias = (torch.rand(E, generator=g) * 2 - 1) * 0.05
    got = B.route_static(logits.cuda(), bias.cuda(), k, scale)
    torch.cuda.synchronize()
    c = orc.cfg(d=64, E=E, I=64, Is=0, k=k, dtype="fp32", routed_scale=scale)
    oidx, ow, margin = orc.select(c, logits.numpy(), bias.numpy())
    gi, gw = got["idx"].cpu().numpy(), got["w"].cpu().numpy()
    set_diff, order_bad = parity.selection_diff(gi, oidx, parity.biased_scores(logits.numpy(), bias.numpy()))
    assert not (set_diff & (margin >= parity.NEAR_TIE)).any()
    assert not order_bad.any()
    ok = ~set_diff
    np.testing.assert_allclose(parity.by_expert(gi[ok], gw[ok]), parity.by_expert(oidx[ok], ow[ok]),
                               rtol=2e-6, atol=1e-7)


def test_route_static_rejects_overlapping_buffers():
    T, E, k = 300, 16, 2
    logits = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    bias = torch.zeros(E, dtype=torch.float32, device="cuda")
    # w written over the logits it reads
    with pytest.raises(B.MoeError) as ei:
        B.route_static(logits, bias, k, 1.0, out={"w": logits.view(-1)[: T * k]})
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
    # two outputs sharing memory
    buf = torch.empty(T * k, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoeError) as ei:
        B.route_static(logits, bias, k, 1.0, out={"pos": buf.view(T, k), "row_tok": buf})
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
