"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks one oracle function against something the pages or plain
mathematics fix: the GLM-5 parameter count printed on the GLM-5 MoE block
page, closed forms of RMSNorm, brute-force enumeration of the top-k,
the reduction of the sublayer to a dense SwiGLU MLP (GlmMoeDsaMLP.forward),
and invariants of the routed combine.  Expected values are computed here with
numpy/math, never with the oracle or the CUDA path.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(v):
    """Round fp32 values to bf16 (RNE) and return them as fp32 (numpy)."""
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).float().numpy()


def bf16_bits(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def silu(z):
    return z / (1.0 + np.exp(-z))


def rand_inputs(rng, T, d, E, I, Is, dtype="fp32", bias_range=0.1, wstd=0.3):
    """Small random inputs; wstd is large so that routing margins are wide."""
    f = {
        "x": rng.standard_normal((T, d)).astype(np.float32),
        "norm_w": rng.uniform(0.5, 1.5, d).astype(np.float32),
        "router_w": (rng.standard_normal((E, d)) * wstd).astype(np.float32),
        "corr_bias": rng.uniform(-bias_range, bias_range, E).astype(np.float32),
        "gate_up": (rng.standard_normal((E, d, 2 * I)) * 0.05).astype(np.float32),
        "down": (rng.standard_normal((E, I, d)) * 0.05).astype(np.float32),
        "shared_gate": (rng.standard_normal((Is, d)) * 0.05).astype(np.float32),
        "shared_up": (rng.standard_normal((Is, d)) * 0.05).astype(np.float32),
        "shared_down": (rng.standard_normal((d, Is)) * 0.05).astype(np.float32),
    }
    if dtype == "bf16":
        f = {k: (v if k == "corr_bias" else bf16_bits(v)) for k, v in f.items()}
    return f


def as_f64(a, dtype):
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# ---------------------------------------------------------------------------
# Parameter accounting: the GLM-5 MoE block page prints the exact counts.
# ---------------------------------------------------------------------------
def test_param_count_matches_glm5_page():
    g = json.load(open(os.path.join(GOLDEN, "glm5_moe_counts.json")))
    c = orc.cfg(d=g["hidden"], E=256, I=2048, Is=2048, k=8, dtype="bf16")
    moe = orc.param_count(c)
    assert moe == g["moe_sublayer_params"]
    block = g["attention_rmsnorm_params"] + g["mla_params"] + g["moe_rmsnorm_params"] + moe
    assert block == g["block_params"]
    assert block * g["moe_blocks"] == g["all_blocks_params"]
    assert c.E * g["moe_blocks"] == g["correction_bias_values_all_blocks"]
    gib = 2 * (moe - c.E) / 2**30 + 4 * c.E / 2**30   # bf16 weights, fp32 bias
    assert round(gib, 1) == g["moe_weights_gib_bf16_rounded"]
    assert round(2 * block / 2**30, 1) == g["block_weights_gib_bf16_rounded"]


def test_param_count_catches_wrong_shapes():
    base = orc.param_count(orc.cfg(6144, 256, 2048, 2048, 8, "bf16"))
    assert orc.param_count(orc.cfg(6144, 256, 2048, 0, 8, "bf16")) != base
    assert orc.param_count(orc.cfg(6144, 255, 2048, 2048, 8, "bf16")) != base


# ---------------------------------------------------------------------------
# RMSNorm (GlmMoeDsaRMSNorm.forward): closed forms.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cval,eps", [(0.5, 0.25), (3.0, 1e-6), (0.01, 1e-4), (1.75, 2.0)])
def test_rmsnorm_constant_row_closed_form(cval, eps):
    d = 64
    c = orc.cfg(d, 4, 64, 0, 1, "fp32", eps=eps)
    x = np.full((1, d), cval, np.float32)
    g = np.linspace(0.5, 1.5, d).astype(np.float32)
    xn = orc.rmsnorm(c, x, g)
    # mean(x^2) = c^2 exactly for a constant row; n = c / sqrt(c^2 + eps)
    n = np.float32(cval) / np.float32(math.sqrt(np.float32(np.float32(cval) ** 2 + np.float32(eps))))
    np.testing.assert_allclose(xn[0], g * n, rtol=2e-7)


def test_rmsnorm_rms_of_output_closed_form():
    rng = np.random.default_rng(1)
    d, eps = 512, 0.05
    c = orc.cfg(d, 4, 64, 0, 1, "fp32", eps=eps)
    x = (rng.standard_normal((16, d)) * 0.3).astype(np.float32)
    xn = orc.rmsnorm(c, x, np.ones(d, np.float32))
    ms = (x.astype(np.float64) ** 2).mean(1)
    want = np.sqrt(ms / (ms + eps))
    got = np.sqrt((xn.astype(np.float64) ** 2).mean(1))
    np.testing.assert_allclose(got, want, rtol=1e-6)


def test_rmsnorm_gain_is_per_feature_and_scale_invariant():
    rng = np.random.default_rng(2)
    d = 256
    c = orc.cfg(d, 4, 64, 0, 1, "fp32", eps=1e-6)
    x = rng.standard_normal((4, d)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    xn = orc.rmsnorm(c, x, g)
    # xn / (g * x) is the same reciprocal rms for every feature of a row
    ratio = xn.astype(np.float64) / (g.astype(np.float64) * x)
    np.testing.assert_allclose(ratio, ratio[:, :1].repeat(d, 1), rtol=3e-7)
    # scaling the row by a power of two leaves the output unchanged (eps << ms)
    xn8 = orc.rmsnorm(c, (x * 8).astype(np.float32), g)
    np.testing.assert_allclose(xn8, xn, rtol=1e-6)


def test_rmsnorm_bf16_casts_before_gain():
    """The page casts the normalised fp32 values to the input dtype and only
    then multiplies by the gain.  Find inputs where that order differs from
    multiplying first, and check the oracle follows the page."""
    d, eps = 8, 0.25
    c = orc.cfg(d, 4, 64, 0, 1, "bf16", eps=eps)
    found = 0
    for cval, gval in itertools.product(np.linspace(0.3, 2.0, 40), np.linspace(0.55, 1.45, 40)):
        cv = float(bf16(cval))
        gv = float(bf16(gval))
        n = np.float32(cv) / np.float32(math.sqrt(np.float32(np.float32(cv) ** 2 + np.float32(eps))))
        cast_first = bf16(np.float32(gv) * bf16(n))
        mult_first = bf16(np.float32(gv) * n)
        if cast_first != mult_first:
            x = bf16_bits(np.full((1, d), cv, np.float32))
            gw = bf16_bits(np.full(d, gv, np.float32))
            xn = orc.rmsnorm(c, x, gw)
            assert np.all(xn == cast_first)
            found += 1
    assert found >= 3


def test_rmsnorm_bf16_agrees_with_torch_cpu_formula():
    """The page's formula executed by torch on the CPU.  Sum order differs
    (torch reduces pairwise in fp32), so allow rare one-ulp flips."""
    rng = np.random.default_rng(3)
    T, d = 256, 1024
    c = orc.cfg(d, 4, 64, 0, 1, "bf16", eps=1e-6)
    x = bf16_bits(rng.standard_normal((T, d)))
    g = bf16_bits(rng.uniform(0.5, 1.5, d))
    xn = orc.rmsnorm(c, x, g)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    gt = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16)
    h = xt.to(torch.float32)
    var = h.pow(2).mean(-1, keepdim=True)
    h = h * torch.rsqrt(var + 1e-6)
    ref = (gt * h.to(torch.bfloat16)).float().numpy()
    same = xn == ref
    assert same.mean() > 0.999
    ulp = np.abs(xn - ref) / np.maximum(np.abs(ref), 1e-30)
    assert ulp[~same].max(initial=0) <= 2 ** -7 + 1e-9


# ---------------------------------------------------------------------------
# Router: brute-force selection, exact ties, weights.
# ---------------------------------------------------------------------------
def numpy_scores(xn, Wr, bias):
    l = (xn.astype(np.float64) @ Wr.astype(np.float64).T).astype(np.float32)
    s = (1.0 / (1.0 + np.exp(-l.astype(np.float64)))).astype(np.float32)
    b = (s + bias).astype(np.float32)
    return l, s, b


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (8, 2), (10, 3)])
def test_routing_matches_bruteforce(E, k):
    rng = np.random.default_rng(100 + E * 10 + k)
    d, T = 32, 200
    c = orc.cfg(d, E, 16, 0, k, "fp32", routed_scale=1.0)
    xn = rng.standard_normal((T, d)).astype(np.float32)
    Wr = (rng.standard_normal((E, d)) * 0.3).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    logits, idx, w, margin = orc.route(c, xn, Wr, bias)
    l, s, b = numpy_scores(xn, Wr, bias)
    np.testing.assert_allclose(logits, l, rtol=1e-6, atol=1e-6)
    for t in range(T):
        best, best_sum = None, None
        for sub in itertools.combinations(range(E), k):     # lexicographic order
            tot = math.fsum(sorted(float(b[t, e]) for e in sub))
            if best_sum is None or tot > best_sum:
                best, best_sum = sub, tot
        assert sorted(idx[t].tolist()) == list(best)
        # slot order: biased score descending, lower index first on ties
        order = sorted(best, key=lambda e: (-float(b[t, e]), e))
        assert idx[t].tolist() == order
        rest = [float(b[t, e]) for e in range(E) if e not in best]
        want_margin = float(b[t, order[-1]]) - max(rest) if rest else math.inf
        assert margin[t] == pytest.approx(want_margin, abs=1e-7)


def test_exact_ties_go_to_lower_index():
    d, E = 16, 6
    rng = np.random.default_rng(7)
    row = rng.standard_normal(d).astype(np.float32)
    Wr = np.stack([row * 0.1, row, row * 0.2, row, row * 0.3, row]).astype(np.float32)
    bias = np.zeros(E, np.float32)
    xn = row[None, :].copy()
    for k, want in [(1, [1]), (2, [1, 3]), (3, [1, 3, 5])]:
        c = orc.cfg(d, E, 16, 0, k, "fp32")
        _, idx, _, margin = orc.route(c, xn, Wr, bias)
        assert idx[0].tolist() == want
    # all experts identical: the first k indices
    c = orc.cfg(d, E, 16, 0, 4, "fp32")
    _, idx, w, margin = orc.route(c, xn, np.tile(row, (E, 1)), bias)
    assert idx[0].tolist() == [0, 1, 2, 3]
    assert margin[0] == 0.0
    np.testing.assert_allclose(w[0], 0.25, rtol=1e-7)


def test_bias_selects_but_does_not_weight():
    rng = np.random.default_rng(8)
    d, E, k, T = 32, 8, 2, 64
    xn = rng.standard_normal((T, d)).astype(np.float32)
    Wr = (rng.standard_normal((E, d)) * 0.3).astype(np.float32)
    bias = np.zeros(E, np.float32)
    bias[[2, 5]] = 10.0                        # experts 2 and 5 always selected
    for scale in (1.0, 2.5):
        c = orc.cfg(d, E, 16, 0, k, "fp32", routed_scale=scale)
        logits, idx, w, _ = orc.route(c, xn, Wr, bias)
        l, s, b = numpy_scores(xn, Wr, bias)
        assert np.all(np.sort(idx, 1) == np.array([2, 5]))
        sel = np.take_along_axis(s, idx, 1).astype(np.float64)
        want = scale * sel / sel.sum(1, keepdims=True)
        np.testing.assert_allclose(w, want, rtol=2e-7)
        np.testing.assert_allclose(w.astype(np.float64).sum(1), scale, rtol=1e-6)


# ---------------------------------------------------------------------------
# The whole sublayer: reductions to dense SwiGLU and combine invariants.
# ---------------------------------------------------------------------------
def dense_swiglu(xn, G, U, Dlin):
    """GlmMoeDsaMLP.forward with nn.Linear weights G, U [I, d], Dlin [d, I]."""
    return (silu(xn @ G.T) * (xn @ U.T)) @ Dlin.T


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_one_expert_top1_reduces_to_dense_swiglu(dtype):
    rng = np.random.default_rng(11)
    T, d, I = 24, 64, 48
    G = (rng.standard_normal((I, d)) * 0.1).astype(np.float32)
    U = (rng.standard_normal((I, d)) * 0.1).astype(np.float32)
    Dlin = (rng.standard_normal((d, I)) * 0.1).astype(np.float32)
    gate_up = np.concatenate([G.T, U.T], axis=1)[None]      # [1, d, 2I]
    down = Dlin.T[None]                                     # [1, I, d]
    a = {
        "x": rng.standard_normal((T, d)).astype(np.float32),
        "norm_w": rng.uniform(0.5, 1.5, d).astype(np.float32),
        "router_w": (rng.standard_normal((1, d)) * 0.1).astype(np.float32),
        "corr_bias": np.array([0.03], np.float32),
        "gate_up": np.ascontiguousarray(gate_up), "down": np.ascontiguousarray(down),
    }
    if dtype == "bf16":
        a = {k: (v if k == "corr_bias" else bf16_bits(v)) for k, v in a.items()}
    c = orc.cfg(d, 1, I, 0, 1, dtype, routed_scale=1.0)
    r = orc.forward(c, a)
    assert np.all(r["idx"] == 0)
    np.testing.assert_array_equal(r["w"], 1.0)
    xn = r["xn"].astype(np.float64)
    Gd = as_f64(a["gate_up"], dtype)[0][:, :I].T
    Ud = as_f64(a["gate_up"], dtype)[0][:, I:].T
    Dd = as_f64(a["down"], dtype)[0].T
    y = dense_swiglu(xn, Gd, Ud, Dd)
    x64 = as_f64(a["x"], dtype)
    np.testing.assert_allclose(r["out"], (x64 + y).astype(np.float32), rtol=1e-6, atol=1e-6)
    # the result must depend on which half is the gate: swapping fails
    y_swapped = dense_swiglu(xn, Ud, Gd, Dd)
    assert np.abs(y_swapped - y).max() > 100 * np.abs(r["out"] - (x64 + y)).max() + 1e-6


def test_shared_expert_alone():
    rng = np.random.default_rng(12)
    T, d, E, I, Is, k = 16, 64, 4, 32, 40, 2
    a = rand_inputs(rng, T, d, E, I, Is)
    a["gate_up"][:] = 0.0          # routed experts output silu(0) * 0 = 0
    c = orc.cfg(d, E, I, Is, k, "fp32", routed_scale=1.7)
    r = orc.forward(c, a)
    xn = r["xn"].astype(np.float64)
    sh = dense_swiglu(xn, a["shared_gate"].astype(np.float64),
                      a["shared_up"].astype(np.float64), a["shared_down"].astype(np.float64))
    np.testing.assert_allclose(r["out"], (a["x"] + sh).astype(np.float32), rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("scale", [1.0, 2.5])
def test_identical_experts_give_scaled_dense_mlp(scale):
    rng = np.random.default_rng(13)
    T, d, E, I, Is, k = 32, 64, 6, 32, 24, 3
    a = rand_inputs(rng, T, d, E, I, Is)
    a["gate_up"][:] = a["gate_up"][0]
    a["down"][:] = a["down"][0]
    c = orc.cfg(d, E, I, Is, k, "fp32", routed_scale=scale)
    r = orc.forward(c, a)
    xn = r["xn"].astype(np.float64)
    f64 = {k2: v.astype(np.float64) for k2, v in a.items()}
    G, U = f64["gate_up"][0][:, :I].T, f64["gate_up"][0][:, I:].T
    y = dense_swiglu(xn, G, U, f64["down"][0].T)
    sh = dense_swiglu(xn, f64["shared_gate"], f64["shared_up"], f64["shared_down"])
    np.testing.assert_allclose(r["out"], (f64["x"] + sh + scale * y).astype(np.float32),
                               rtol=1e-5, atol=1e-6)


def test_routed_sum_matches_explicit_weighted_experts():
    """out - x - shared equals sum_j w_j * expert_{idx_j}(xn) with each expert
    evaluated densely from its grouped weights."""
    rng = np.random.default_rng(14)
    T, d, E, I, Is, k = 20, 64, 8, 32, 16, 3
    a = rand_inputs(rng, T, d, E, I, Is)
    c = orc.cfg(d, E, I, Is, k, "fp32", routed_scale=2.5)
    r = orc.forward(c, a)
    xn = r["xn"].astype(np.float64)
    f64 = {k2: v.astype(np.float64) for k2, v in a.items()}
    sh = dense_swiglu(xn, f64["shared_gate"], f64["shared_up"], f64["shared_down"])
    want = f64["x"] + sh
    for t in range(T):
        for j in range(k):
            e = r["idx"][t, j]
            G, U = f64["gate_up"][e][:, :I].T, f64["gate_up"][e][:, I:].T
            want[t] += r["w"][t, j] * dense_swiglu(xn[t:t + 1], G, U, f64["down"][e].T)[0]
    np.testing.assert_allclose(r["out"], want.astype(np.float32), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(r["w"].astype(np.float64).sum(1), 2.5, rtol=1e-6)


def test_linear_in_routed_scale():
    rng = np.random.default_rng(15)
    T, d, E, I, Is, k = 16, 64, 8, 32, 16, 2
    a = rand_inputs(rng, T, d, E, I, Is)
    outs = {}
    for s in (0.0, 1.0, 2.0):
        outs[s] = orc.forward(orc.cfg(d, E, I, Is, k, "fp32", routed_scale=s), a)["out"]
    np.testing.assert_allclose(outs[2.0] - outs[1.0], outs[1.0] - outs[0.0], atol=3e-6)


def test_tokens_are_independent():
    rng = np.random.default_rng(16)
    T, d, E, I, Is, k = 40, 64, 8, 32, 16, 2
    a = rand_inputs(rng, T, d, E, I, Is, dtype="bf16")
    c = orc.cfg(d, E, I, Is, k, "bf16", routed_scale=1.0)
    full = orc.forward(c, a)
    perm = rng.permutation(T)
    sub = orc.forward(c, a, rows=perm)
    for key in ("out", "idx", "w", "xn"):
        np.testing.assert_array_equal(sub[key], full[key][perm])
    one = orc.forward(c, a, rows=np.array([7]))
    np.testing.assert_array_equal(one["out"][0], full["out"][7])


def test_forced_selection():
    rng = np.random.default_rng(17)
    T, d, E, I, Is, k = 12, 64, 8, 32, 16, 2
    a = rand_inputs(rng, T, d, E, I, Is)
    c = orc.cfg(d, E, I, Is, k, "fp32", routed_scale=1.0)
    r = orc.forward(c, a)
    same = orc.forward(c, a, forced_idx=r["idx"])
    np.testing.assert_array_equal(same["out"], r["out"])
    other = (r["idx"] + 1) % E
    f = orc.forward(c, a, forced_idx=other)
    np.testing.assert_array_equal(f["idx"], other)
    _, s, _ = numpy_scores(r["xn"], a["router_w"], a["corr_bias"])
    sel = np.take_along_axis(s, other, 1).astype(np.float64)
    np.testing.assert_allclose(f["w"], sel / sel.sum(1, keepdims=True), rtol=2e-7)


@pytest.mark.parametrize("E,k", [(5, 2), (9, 3)])
def test_select_from_logits_matches_bruteforce(E, k):
    """Steps C-D alone, on given logits: the brute-force k-subset with the
    largest biased sum, slot order by biased score, weights from the
    unbiased sigmoids."""
    rng = np.random.default_rng(200 + E)
    T = 150
    c = orc.cfg(32, E, 16, 0, k, "fp32", routed_scale=2.5)
    logits = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    idx, w, margin = orc.select(c, logits, bias)
    s = (1.0 / (1.0 + np.exp(-logits.astype(np.float64)))).astype(np.float32)
    b = (s + bias).astype(np.float32)
    for t in range(T):
        best = max(itertools.combinations(range(E), k),
                   key=lambda sub: (math.fsum(sorted(float(b[t, e]) for e in sub)),
                                    [-e for e in sub]))
        assert idx[t].tolist() == sorted(best, key=lambda e: (-float(b[t, e]), e))
        sel = s[t, idx[t]].astype(np.float64)
        np.testing.assert_allclose(w[t], 2.5 * sel / sel.sum(), rtol=2e-7)
    # route() = step B followed by select() on its own logits
    xn = rng.standard_normal((T, 32)).astype(np.float32)
    Wr = (rng.standard_normal((E, 32)) * 0.3).astype(np.float32)
    lg, idx2, w2, m2 = orc.route(c, xn, Wr, bias)
    idx3, w3, m3 = orc.select(c, lg, bias)
    np.testing.assert_array_equal(idx2, idx3)
    np.testing.assert_array_equal(w2, w3)
    np.testing.assert_array_equal(m2, m3)


# ---------------------------------------------------------------------------
# The dense feed-forward block of the first decoder layers: the decoder-layer
# excerpt on the GLM-5 shared-expert page applies post_attention_layernorm,
# then GlmMoeDsaMLP, then the residual add.  Pinned against the MLP formula
# written out in numpy (fp64) on the oracle's pinned RMSNorm output.
# ---------------------------------------------------------------------------
def dense_inputs(rng, T, d, I, dtype):
    a = {
        "x": rng.standard_normal((T, d)).astype(np.float32),
        "norm_w": rng.uniform(0.5, 1.5, d).astype(np.float32),
        "dense_gate": (rng.standard_normal((I, d)) * 0.1).astype(np.float32),
        "dense_up": (rng.standard_normal((I, d)) * 0.1).astype(np.float32),
        "dense_down": (rng.standard_normal((d, I)) * 0.1).astype(np.float32),
    }
    if dtype == "bf16":
        a = {k: bf16_bits(v) for k, v in a.items()}
    return a


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_dense_block_is_residual_plus_swiglu_mlp(dtype):
    rng = np.random.default_rng(31)
    T, d, I = 20, 64, 96          # I != d: a transposed weight reads the wrong values
    a = dense_inputs(rng, T, d, I, dtype)
    c = orc.dense_cfg(d, I, dtype)
    r = orc.dense_forward(c, a)
    np.testing.assert_array_equal(r["xn"], orc.rmsnorm(c, a["x"], a["norm_w"]))
    xn = r["xn"].astype(np.float64)
    G, U, Dl = (as_f64(a[n], dtype) for n in ("dense_gate", "dense_up", "dense_down"))
    y = dense_swiglu(xn, G, U, Dl)
    x64 = as_f64(a["x"], dtype)
    np.testing.assert_allclose(r["out"], (x64 + y).astype(np.float32), rtol=1e-6, atol=1e-6)
    # the gate is the projection inside silu: swapping gate and up changes the result
    y_swapped = dense_swiglu(xn, U, G, Dl)
    assert np.abs(y_swapped - y).max() > 100 * np.abs(r["out"] - (x64 + y)).max() + 1e-6


def test_dense_block_zero_down_returns_the_residual():
    rng = np.random.default_rng(32)
    T, d, I = 8, 32, 48
    a = dense_inputs(rng, T, d, I, "fp32")
    a["dense_down"][:] = 0.0
    r = orc.dense_forward(orc.dense_cfg(d, I, "fp32"), a)
    np.testing.assert_array_equal(r["out"], a["x"])


def test_dense_block_rows_are_independent():
    rng = np.random.default_rng(33)
    T, d, I = 12, 32, 40
    a = dense_inputs(rng, T, d, I, "bf16")
    c = orc.dense_cfg(d, I, "bf16")
    full = orc.dense_forward(c, a)["out"]
    rows = np.array([11, 0, 5, 5], np.int64)
    np.testing.assert_array_equal(orc.dense_forward(c, a, rows=rows)["out"], full[rows])


# ---------------------------------------------------------------------------
# HF -> grouped layout packing (state dict adapter page): the packed tensors,
# fed to the sublayer oracle, give the SwiGLU MLP of the HF nn.Linear weights
# (GlmMoeDsaMLP orientation, y = x W^T) for every expert.
# ---------------------------------------------------------------------------
def test_packed_layout_gives_the_hf_experts():
    rng = np.random.default_rng(41)
    T, d, E, I = 9, 32, 3, 24
    G = (rng.standard_normal((E, I, d)) * 0.2).astype(np.float32)
    U = (rng.standard_normal((E, I, d)) * 0.2).astype(np.float32)
    Dn = (rng.standard_normal((E, d, I)) * 0.2).astype(np.float32)
    gate_up, down = orc.pack_experts(G, U, Dn)
    assert gate_up.shape == (E, d, 2 * I) and down.shape == (E, I, d)
    x = rng.standard_normal((T, d)).astype(np.float32)
    for e in range(E):
        # one expert at a time: top-1 over a single expert routes every token to it
        a = {"x": x, "norm_w": np.ones(d, np.float32), "router_w": np.zeros((1, d), np.float32),
             "corr_bias": np.zeros(1, np.float32), "gate_up": np.ascontiguousarray(gate_up[e:e + 1]),
             "down": np.ascontiguousarray(down[e:e + 1])}
        r = orc.forward(orc.cfg(d, 1, I, 0, 1, "fp32", routed_scale=1.0), a)
        xn = r["xn"].astype(np.float64)
        y = dense_swiglu(xn, G[e].astype(np.float64), U[e].astype(np.float64), Dn[e].astype(np.float64))
        np.testing.assert_allclose(r["out"], (x + y).astype(np.float32), rtol=1e-6, atol=1e-6)


def test_packing_is_exact_data_movement():
    rng = np.random.default_rng(42)
    E, d, I = 2, 5, 3
    bits = rng.integers(0, 2 ** 16, size=(3, E, I, d), dtype=np.uint16)
    G, U, Dn = bits[0], bits[1], bits[2].transpose(0, 2, 1).copy()
    gate_up, down = orc.pack_experts(G, U, Dn)
    for e in range(E):
        for j in range(d):
            for i in range(I):
                assert gate_up[e, j, i] == G[e, i, j] and gate_up[e, j, I + i] == U[e, i, j]
                assert down[e, i, j] == Dn[e, j, i]


# ---------------------------------------------------------------------------
# Query compression of the sparse latent attention (GLM-5 "Query latent" page:
# q_resid = q_a_layernorm(q_a_proj(hidden_states)), q_a_proj = nn.Linear(d ->
# q_lora_rank, no bias), q_a_layernorm = GlmMoeDsaRMSNorm(q_lora_rank)).
# ---------------------------------------------------------------------------
def torch_rmsnorm_bf16(cq, gain, eps):
    """The RMSNorm excerpt's formula executed by torch on bf16 tensors."""
    h = cq.to(torch.float32)
    var = h.pow(2).mean(-1, keepdim=True)
    h = h * torch.rsqrt(var + eps)
    return (gain * h.to(torch.bfloat16)).float()


def test_q_latent_is_linear_then_rmsnorm():
    """Inputs on a coarse grid (integers times powers of two), so that every
    sum of the projection is exact in fp32: torch's fp32 matmul then gives the
    exact value, and its bf16 cast rounds it once, as the Linear's bf16 output
    does.  The norm is then the page's formula run by torch."""
    rng = np.random.default_rng(21)
    n, d, rank = 48, 256, 96
    hid = (rng.integers(-64, 65, (n, d)) * 2.0 ** -5).astype(np.float32)      # 7-bit values
    wq = (rng.integers(-32, 33, (rank, d)) * 2.0 ** -8).astype(np.float32)    # 6-bit values
    g = (rng.integers(64, 192, rank) * 2.0 ** -7).astype(np.float32)
    c_or, q_or = orc.q_latent(d, rank, "bf16", bf16_bits(hid), bf16_bits(wq), bf16_bits(g))
    c_t = (torch.from_numpy(hid) @ torch.from_numpy(wq).T).to(torch.bfloat16)
    np.testing.assert_array_equal(c_or, c_t.float().numpy())
    assert (c_t.float() != torch.from_numpy(hid) @ torch.from_numpy(wq).T).any()   # rounding happened
    q_t = torch_rmsnorm_bf16(c_t, torch.from_numpy(g).to(torch.bfloat16), 1e-6).numpy()
    same = q_or == q_t
    assert same.mean() > 0.995                   # sum order of the mean of squares may flip an ulp
    ulp = np.abs(q_or - q_t) / np.maximum(np.abs(q_t), 1e-30)
    assert ulp[~same].max(initial=0) <= 2 ** -7 + 1e-9


def test_q_latent_identity_projection_is_the_norm_of_the_leading_features():
    """W = [I | 0] ([rank, d], nn.Linear orientation): c is the first rank
    features of the row, and q their RMSNorm (step A, pinned above)."""
    rng = np.random.default_rng(22)
    n, d, rank = 20, 128, 48
    hid = bf16_bits(rng.standard_normal((n, d)))
    wq = np.zeros((rank, d), np.float32)
    wq[np.arange(rank), np.arange(rank)] = 1.0
    g = bf16_bits(rng.uniform(0.5, 1.5, rank))
    c_or, q_or = orc.q_latent(d, rank, "bf16", hid, bf16_bits(wq), g)
    lead = np.ascontiguousarray(hid[:, :rank])
    np.testing.assert_array_equal(c_or, as_f64(lead, "bf16").astype(np.float32))
    np.testing.assert_array_equal(q_or, orc.rmsnorm(orc.cfg(rank, 1, 1, 0, 1, "bf16"), lead, g))


def test_q_latent_fp32_and_selected_rows():
    rng = np.random.default_rng(23)
    n, d, rank = 16, 64, 32
    hid = rng.standard_normal((n, d)).astype(np.float32)
    wq = (rng.standard_normal((rank, d)) * 0.1).astype(np.float32)
    g = rng.uniform(0.5, 1.5, rank).astype(np.float32)
    c_or, q_or = orc.q_latent(d, rank, "fp32", hid, wq, g, eps=1e-6)
    np.testing.assert_allclose(c_or, hid.astype(np.float64) @ wq.astype(np.float64).T, rtol=1e-6, atol=1e-7)
    cd = c_or.astype(np.float64)
    np.testing.assert_allclose(q_or, g * cd / np.sqrt((cd ** 2).mean(1, keepdims=True) + 1e-6), rtol=2e-6)
    rows = np.array([7, 2, 11])
    c2, q2 = orc.q_latent(d, rank, "fp32", hid, wq, g, rows=rows)
    np.testing.assert_array_equal(q2, q_or[rows])
    np.testing.assert_array_equal(c2, c_or[rows])
