"""Parity of the dense feed-forward block (moe_dense_forward, through the C
ABI) with the CPU oracle: out = x + GlmMoeDsaMLP(RMSNorm(x)), the block the
first first_k_dense_replace decoder layers use instead of the MoE (decoder
layer excerpt on the GLM-5 shared-expert page).

Small cases compare every token on both GEMM paths (single-CTA tiles below
128 tokens, with both projections split over k-ranges; CTA pairs from 128
up) and the CUDA-core path; the GLM-5-sized
cases compare a seeded sample of tokens.  The output is held to the
sublayer's tolerances (tests/parity.py).  The MLP's own contribution
out - x is checked too: in fp32 to 1e-4 of its rms; in bf16 elementwise to
2^-8 |out| (the worst case of the one rounding of out to bf16, which is
relative to |out|, not to the contribution) plus 2e-2 of its rms.  With the
workloads' N(0, 0.02) weights a small block's contribution is a few percent
of x, so the small cases scale the three weights by 4 (exact in bf16 and
fp32): the contribution is then as large as x and the second check has
teeth.
"""
import numpy as np
import pytest
import torch

import parity
from mixture_experts_transformer_sigmoid_b300 import binding as B
from mixture_experts_transformer_sigmoid_b300 import workloads as wl
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

DW = wl.DenseWorkload
SMALL = {
    "dense_tiny_fp32": wl.DENSE_WORKLOADS["dense_tiny_fp32"],
    "dense_small_bf16": wl.DENSE_WORKLOADS["dense_small_bf16"],
    # partial feature tiles in both GEMMs: I = 192 (1.5 pair tiles), d = 320 (1.25 pair tiles)
    "dense_pair_odd_bf16": DW("dense_pair_odd_bf16", T=333, d=320, I=192, dtype="bf16"),
    "dense_single_odd_bf16": DW("dense_single_odd_bf16", T=77, d=320, I=192, dtype="bf16"),
    "dense_one_token_bf16": DW("dense_one_token_bf16", T=1, d=512, I=256, dtype="bf16"),
    "dense_ragged_fp32": DW("dense_ragged_fp32", T=53, d=128, I=96, dtype="fp32"),
    # prefill-sized batches (at least 8 tokens per SM): the RMSNorm with rows staged in
    # shared memory, 40 vectors per row (lanes hold one or two), in bf16 and in fp32
    "dense_prefill_odd_bf16": DW("dense_prefill_odd_bf16", T=1250, d=320, I=192, dtype="bf16"),
    "dense_prefill_fp32": DW("dense_prefill_fp32", T=1250, d=160, I=96, dtype="fp32"),
}


def dense_layer(w, gemm_path=0, T=None):
    return B.MoeSublayer(max_tokens=max(w.T if T is None else T, 1), hidden=w.d, n_experts=0,
                         inter=0, shared_inter=0, max_top_k=0, dtype=w.dtype, eps=w.eps,
                         gemm_path=gemm_path, dense_inter=w.I)


def run_dense(w, dev, gemm_path=0):
    layer = dense_layer(w, gemm_path)
    try:
        # NaN first: an output element no tile writes stays NaN
        out = torch.full_like(dev["x"], float("nan"))
        layer.dense_forward(dev["x"], dev, out=out)
        st = layer.sync_status()
        assert st == B.MOE_OK, B.status_string(st)
        return parity.to_np_f32(out)
    finally:
        layer.close()


WEIGHT_SCALE = 4.0   # exact in bf16 and fp32


def scaled(inp):
    """The small cases' inputs with the three dense weights times 4."""
    out = dict(inp)
    for n in ("dense_gate", "dense_up", "dense_down"):
        out[n] = (inp[n] * WEIGHT_SCALE).contiguous()
    return out


def compare(w, gout, host, rows):
    c = orc.dense_cfg(w.d, w.I, w.dtype, w.eps)
    r = orc.dense_forward(c, host, rows=rows)
    x = host["x"][rows]
    x = (x.astype(np.uint32) << 16).view(np.float32) if x.dtype == np.uint16 else x
    g, ref = gout[rows].astype(np.float64), r["out"].astype(np.float64)
    st = parity.output_errors(g, ref)
    sd = parity.output_errors(g - x, ref - x)
    tol = parity.TOL[w.dtype]
    if w.dtype == "bf16":
        parity.check_bf16_max(g, ref, tol["max_rms"])
        assert st["mean_rel"] <= tol["mean_rel"], (st, sd)
        # the MLP's contribution: the one rounding of out (relative to |out|) plus 2e-2 of its rms
        rms_delta = float(np.sqrt(np.mean((ref - x) ** 2)))
        excess = np.abs(g - ref) - (2.0 ** -8 * np.abs(ref) + 2e-2 * rms_delta)
        assert excess.max() <= 0.0, (st, sd, float(excess.max()))
    else:
        assert st["max_over_rms"] <= tol["max_rms"], (st, sd)
        assert sd["max_over_rms"] <= tol["max_rms"], (st, sd)
    return st, sd


@pytest.mark.parametrize("name", list(SMALL))
def test_small_dense_case_matches_oracle(name):
    w = SMALL[name]
    inp = scaled(wl.make_dense_inputs(w))
    host = wl.host_arrays(inp)
    gout = run_dense(w, {k: v.cuda() for k, v in inp.items()})
    print(name, compare(w, gout, host, np.arange(w.T)))


def test_dense_cuda_core_path_on_bf16_storage():
    w = SMALL["dense_single_odd_bf16"]
    inp = scaled(wl.make_dense_inputs(w))
    gout = run_dense(w, {k: v.cuda() for k, v in inp.items()}, gemm_path=1)
    print(compare(w, gout, wl.host_arrays(inp), np.arange(w.T)))


@pytest.mark.parametrize("name", ["glm5_dense_prefill", "glm5_dense_decode"])
def test_glm5_sized_dense_block_sampled_tokens(name):
    w = wl.DENSE_WORKLOADS[name]
    dev = wl.make_dense_inputs(w, device="cuda")
    gout = run_dense(w, dev)
    host = wl.host_arrays(dev)
    n = min(w.T, 48)
    rows = np.sort(np.random.default_rng(7).choice(w.T, size=n, replace=False))
    assert np.isfinite(gout).all(), "output elements no tile wrote"
    print(name, compare(w, gout, host, rows))


def test_dense_empty_input_queues_nothing():
    w = SMALL["dense_small_bf16"]
    layer = dense_layer(w)
    try:
        out = torch.empty((0, w.d), dtype=torch.bfloat16, device="cuda")
        assert layer.lib.moe_dense_forward(layer.handle, 0, None, None, None, None, None, w.I, None,
                                           None) == B.MOE_OK
        assert layer.sync_status() == B.MOE_OK
        assert out.shape == (0, w.d)
    finally:
        layer.close()


def test_dense_argument_checks_on_a_live_handle():
    w = SMALL["dense_small_bf16"]
    dev = {k: v.cuda() for k, v in wl.make_dense_inputs(w).items()}
    layer = dense_layer(w)
    try:
        out = torch.empty_like(dev["x"])
        args = [B._ptr(dev["x"]), B._ptr(dev["norm_w"]), B._ptr(dev["dense_gate"]),
                B._ptr(dev["dense_up"]), B._ptr(dev["dense_down"])]
        call = lambda T, inter, o: layer.lib.moe_dense_forward(layer.handle, T, *args, inter, o, None)
        assert call(w.T + 1, w.I, B._ptr(out)) == B.MOE_ERR_INVALID_ARG     # T > max_tokens
        assert call(w.T, w.I + 64, B._ptr(out)) == B.MOE_ERR_INVALID_ARG    # inter > dense_inter
        assert call(w.T, w.I - 32, B._ptr(out)) == B.MOE_ERR_UNSUPPORTED    # not a multiple of 64
        assert call(w.T, w.I, args[0]) == B.MOE_ERR_INVALID_ARG             # out aliases x
        assert call(w.T, w.I, None) == B.MOE_ERR_INVALID_ARG
        # the MoE entry points reject a handle without experts
        p = B._ptr(out)
        assert layer.lib.moe_forward(layer.handle, 4, p, p, p, p, p, p, p, p, p, 1, 1.0, p,
                                     None) == B.MOE_ERR_INVALID_ARG
        assert layer.sync_status() == B.MOE_OK
    finally:
        layer.close()


def test_dense_on_a_moe_handle_leaves_the_moe_results_alone():
    """One handle serves both blocks: a dense call between two MoE forwards
    changes neither the MoE output nor its own (same bytes as on a handle
    for the dense block only)."""
    wm = wl.Workload("moe_for_dense", T=300, d=512, E=16, I=192, Is=128, k=4, routed_scale=1.0,
                     dtype="bf16")
    wd = DW("dense_for_moe", T=300, d=512, I=384, dtype="bf16")
    mi = {k: v.cuda() for k, v in wl.make_inputs(wm).items()}
    di = {k: v.cuda() for k, v in wl.make_dense_inputs(wd, seed=3).items()}
    layer = B.MoeSublayer(max_tokens=300, hidden=512, n_experts=16, inter=192, shared_inter=128,
                          max_top_k=4, dtype="bf16", dense_inter=384)
    try:
        a = layer.forward(mi["x"], mi, 4, 1.0).clone()
        d1 = layer.dense_forward(di["x"], di).clone()
        b = layer.forward(mi["x"], mi, 4, 1.0).clone()
        assert layer.sync_status() == B.MOE_OK
    finally:
        layer.close()
    assert torch.equal(a, b)
    np.testing.assert_array_equal(parity.to_np_f32(d1), run_dense(wd, di))


@pytest.mark.parametrize("name", ["dense_pair_odd_bf16", "dense_single_odd_bf16"])  # CTA pairs / split-K
def test_dense_graph_replay_matches_direct_call(name):
    w = SMALL[name]
    dev = {k: v.cuda() for k, v in wl.make_dense_inputs(w).items()}
    layer = dense_layer(w)
    try:
        direct = layer.dense_forward(dev["x"], dev).clone()
        out = torch.zeros_like(direct)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            layer.dense_forward(dev["x"], dev, out=out, stream=s)   # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        out.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer.dense_forward(dev["x"], dev, out=out)
        g.replay()
        torch.cuda.synchronize()
        assert layer.sync_status() == B.MOE_OK
    finally:
        layer.close()
    assert torch.equal(out, direct)
