"""Parity of moe_q_latent (the query compression of GLM-5's sparse latent
attention, q_a_layernorm(q_a_proj(hidden)), GLM-5 "Query latent" page) with
the CPU oracle.

The query latent c is the Linear's output rounded to bf16.  Its rounding is a
decision that floating point takes: the GPU accumulates in fp32 on the tensor
cores and the oracle rounds the exact sum, so an element whose exact value
lies within the GPU's accumulation error of a rounding boundary may
legitimately round to another bf16 value.  The checks therefore are:
  1. c: every element is the bf16 rounding of a value within
     ACC_TOL * sum_j |h_j w_j| of the exact sum; elements that differ from
     the oracle's (which rounds the exact sum) are counted and reported;
  2. q on the GPU's own c: the oracle's RMSNorm of the GPU's c equals the
     GPU's q on >= 99.9 % of the elements, the rest within one bf16 ulp;
  3. q end to end: max|gpu - oracle| <= 2e-2 * rms(oracle) on the rows whose
     c rounded exactly as the oracle's (elsewhere a c element that took the
     other rounding moves its own q by up to a few bf16 ulps, and the row's
     mean of squares, whose reciprocal root then rounds some neighbours'
     c * r the other way: checks 1 and 2 cover those rows), and mean relative
     error <= 5e-3 over all elements.
fp32 storage: max|gpu - oracle| <= 1e-4 * rms(oracle) for c and q.
"""
import numpy as np
import pytest
import torch

from mixture_experts_transformer_sigmoid_b300 import binding as B
from mixture_experts_transformer_sigmoid_b300 import workloads as wl
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

# Bound of the tensor cores' fp32 accumulation error over the contraction,
# relative to sum_j |h_j w_j| (it grows with the chain of MMAs into one
# accumulator: about 1e-6 of that sum at d = 6144).
ACC_TOL = 4e-6
QW = wl.QLATENT_WORKLOADS


def bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 \
        else t.contiguous().cpu().numpy()


def as_f64(a):
    return ((a.astype(np.uint32) << 16).view(np.float32) if a.dtype == np.uint16 else a).astype(np.float64)


def ulp_bf16(v):
    a = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def run_case(w, inp, rows=None):
    layer = B.MoeSublayer(max_tokens=max(w.T, 1), hidden=w.d, n_experts=0, inter=0, shared_inter=0,
                          max_top_k=0, dtype=w.dtype, eps=w.eps, dense_inter=64)
    try:
        dev = {k: v.cuda() for k, v in inp.items()}
        c, q = layer.q_latent(dev["hidden"], dev["w_qa"], dev["q_norm_w"])
        assert layer.sync_status() == B.MOE_OK
        c_g, q_g = c.float().cpu().numpy(), q.float().cpu().numpy()
    finally:
        layer.close()
    hid, wq, g = bits(inp["hidden"]), bits(inp["w_qa"]), bits(inp["q_norm_w"])
    rows = np.arange(w.T) if rows is None else rows
    c_o, q_o = orc.q_latent(w.d, w.rank, w.dtype, hid, wq, g, eps=w.eps, rows=rows)
    c_g, q_g = c_g[rows], q_g[rows]
    h64, w64 = as_f64(hid[rows]), as_f64(wq)
    exact = h64 @ w64.T
    scale = np.abs(h64) @ np.abs(w64).T
    return c_g, q_g, c_o, q_o, exact, scale, g


def check(w, c_g, q_g, c_o, q_o, exact, scale, g):
    rms = float(np.sqrt(np.mean(q_o.astype(np.float64) ** 2)))
    if w.dtype == "fp32":
        assert np.abs(c_g - c_o).max() <= 1e-4 * float(np.sqrt(np.mean(c_o.astype(np.float64) ** 2)))
        assert np.abs(q_g - q_o).max() <= 1e-4 * rms
        return {"max_over_rms": float(np.abs(q_g - q_o).max() / rms)}
    # 1. c is the rounding of a value within the accumulation tolerance of the exact sum
    eps = ACC_TOL * scale
    lo = torch.from_numpy(exact - eps).to(torch.bfloat16).double().numpy()
    hi = torch.from_numpy(exact + eps).to(torch.bfloat16).double().numpy()
    assert np.all((lo <= c_g) & (c_g <= hi)), "c is not a rounding of the sum within the tolerance"
    flip = c_g != c_o
    # 2. the norm on the GPU's own c
    c_bits = torch.from_numpy(c_g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q_own = orc.rmsnorm(orc.cfg(w.rank, 1, 1, 0, 1, "bf16", eps=w.eps), np.ascontiguousarray(c_bits), g)
    same = q_own == q_g
    assert same.mean() >= 0.999
    assert (np.abs(q_own - q_g) / np.maximum(np.abs(q_own), 1e-30))[~same].max(initial=0) <= 2.0 ** -7 + 1e-9
    # 3. end to end
    err = np.abs(q_g.astype(np.float64) - q_o.astype(np.float64))
    clean = ~flip.any(axis=1)
    assert err[clean].max(initial=0.0) <= 2e-2 * rms
    mean_rel = float(err.sum() / np.abs(q_o).sum())
    assert mean_rel <= 5e-3
    return {"max_over_rms": float(err.max() / rms), "max_over_rms_clean_rows": float(err[clean].max(initial=0) / rms),
            "clean_rows": int(clean.sum()), "rows": int(clean.size), "c_flips": int(flip.sum()),
            "c_elements": int(flip.size), "q_own_bit_exact": float(same.mean()), "mean_rel": mean_rel}


@pytest.mark.parametrize("name", ["q_tiny_fp32", "q_small_bf16", "q_pair_bf16", "glm5_q_decode"])
def test_q_latent_matches_oracle(name):
    w = QW[name]
    inp = wl.make_q_inputs(w, seed=0)
    st = check(w, *run_case(w, inp))
    print(name, st)


@pytest.mark.parametrize("T", [1, 100, 128, 129, 777])   # split-K ranges, single-CTA tails, ragged
def test_q_latent_token_range(T):
    w = QW["glm5_q_decode"].with_(T=T)
    inp = wl.make_q_inputs(w, seed=T)
    st = check(w, *run_case(w, inp))
    print(T, st)


def test_q_latent_glm5_prefill_sampled_rows():
    w = QW["glm5_q_prefill"]
    inp = wl.make_q_inputs(w, seed=0, device="cuda")
    rows = np.sort(np.random.default_rng(0).choice(w.T, size=1024, replace=False))
    st = check(w, *run_case(w, inp, rows=rows))
    print(st)


def test_q_latent_rejects_bad_arguments():
    w = QW["q_small_bf16"]
    inp = {k: v.cuda() for k, v in wl.make_q_inputs(w).items()}
    layer = B.MoeSublayer(max_tokens=w.T, hidden=w.d, n_experts=0, inter=0, shared_inter=0,
                          max_top_k=0, dtype=w.dtype, dense_inter=64)
    try:
        with pytest.raises(B.MoeError) as e:      # q written over the input
            layer.q_latent(inp["hidden"], inp["w_qa"], inp["q_norm_w"],
                           q_out=inp["hidden"].view(-1)[: w.T * w.rank].view(w.T, w.rank))
        assert e.value.status == B.MOE_ERR_INVALID_ARG
        with pytest.raises(B.MoeError) as e:      # rank not a multiple of 64
            layer.q_latent(inp["hidden"], inp["w_qa"][:100], inp["q_norm_w"][:100])
        assert e.value.status == B.MOE_ERR_UNSUPPORTED
    finally:
        layer.close()
