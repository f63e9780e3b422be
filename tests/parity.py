"""Helpers shared by the GPU parity tests, the smoke check and the benchmark:
run the CUDA path through the C ABI and compare it with the CPU oracle.

Tolerances (floating point), as stated for this sublayer:
  bf16 storage: max|gpu - oracle| <= 2e-2 * rms(oracle)  and
                sum|gpu - oracle| / sum|oracle| <= 5e-3
  fp32 storage: max|gpu - oracle| <= 1e-4 * rms(oracle)
The oracle's output is fp64 rounded to fp32; the GPU's is the stored dtype.
Routing: expert ids are compared exactly; a token may differ only when its
top-k margin b_(k) - b_(k+1) is below 1e-5 (several selections are then
correct), or when its RMSNorm output differs from the oracle's in a bf16
rounding whose effect on the biased scores can reach that token's margin
(bounded by the router weights; see check_end_to_end_routing).  Output
parity is judged against the oracle run on the GPU's own selection, so a
correct alternative selection is not counted as an error.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as orc

NEAR_TIE = 1e-5
# Slot order inside a selection follows each side's own fp32 scores; two
# selected experts whose biased scores differ by less than this may appear in
# either order (one rounding of the sigmoid can swap them).
ORDER_TOL = 1e-6
TOL = {"bf16": dict(max_rms=2e-2, mean_rel=5e-3), "fp32": dict(max_rms=1e-4, mean_rel=1e-5)}


def biased_scores(logits: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """b = fp32(sigmoid(l)) + bias, for checking the order of a selection."""
    s = (1.0 / (1.0 + np.exp(-logits.astype(np.float64)))).astype(np.float32)
    return (s + bias.astype(np.float32)).astype(np.float32)


def selection_diff(gi: np.ndarray, oi: np.ndarray, b: np.ndarray):
    """Per token: whether the selected sets differ, and whether the GPU's
    slot order contradicts the scores b by more than ORDER_TOL."""
    set_diff = np.any(np.sort(gi, axis=1) != np.sort(oi, axis=1), axis=1)
    bg = np.take_along_axis(b, gi.astype(np.int64), axis=1).astype(np.float64)
    order_bad = np.any(bg[:, :-1] < bg[:, 1:] - ORDER_TOL, axis=1)
    return set_diff, order_bad


def by_expert(idx: np.ndarray, vals: np.ndarray) -> np.ndarray:
    """Values of a selection reordered by ascending expert id."""
    order = np.argsort(idx, axis=1, kind="stable")
    return np.take_along_axis(vals, order, axis=1)


def to_np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def run_gpu(w, dev_inputs, top_k=None, routed_scale=None, gemm_path=0, T=None, keep=True):
    """Runs one forward through the C ABI; returns numpy copies of the output
    and of every intermediate the tests inspect."""
    from mixture_experts_transformer_sigmoid_b300 import binding as B
    T = dev_inputs["x"].shape[0] if T is None else T
    k = w.k if top_k is None else top_k
    scale = w.routed_scale if routed_scale is None else routed_scale
    layer = B.MoeSublayer(max_tokens=max(T, 1), hidden=w.d, n_experts=w.E, inter=w.I,
                          shared_inter=w.Is, max_top_k=k, dtype=w.dtype, eps=w.eps,
                          gemm_path=gemm_path)
    try:
        x = dev_inputs["x"][:T]
        out = layer.forward(x, dev_inputs, k, scale)
        st = layer.sync_status()
        assert st == B.MOE_OK, B.status_string(st)
        res = {"out": to_np_f32(out)}
        if T > 0:
            idx, wt, counts = layer.routing()
            res.update(idx=idx.cpu().numpy(), w=wt.cpu().numpy(), counts=counts.cpu().numpy())
            if keep:
                res["xn"] = to_np_f32(layer.intermediate(B.T_XN))
                res["logits"] = layer.intermediate(B.T_LOGITS).cpu().numpy()
                res["offsets"] = layer.intermediate(B.T_OFFSETS).cpu().numpy()
                res["pos"] = layer.intermediate(B.T_POS).cpu().numpy()
                res["row_tok"] = layer.intermediate(B.T_ROW_TOK).cpu().numpy()
        assert layer.sync_status() == B.MOE_OK
        return res
    finally:
        layer.close()


def check_permutation(g, T, E, k):
    """Histogram / scan / scatter invariants (bit-exact integer work)."""
    idx, counts, offsets, pos, row_tok = g["idx"], g["counts"], g["offsets"], g["pos"], g["row_tok"]
    P = T * k
    assert idx.shape == (T, k)
    assert idx.min() >= 0 and idx.max() < E
    for t in range(min(T, 4096)):
        assert len(set(idx[t].tolist())) == k, "an expert chosen twice"
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    flat = pos.ravel()
    assert np.array_equal(np.sort(flat), np.arange(P)), "pos is not a bijection onto the rows"
    tok = np.repeat(np.arange(T), k)
    np.testing.assert_array_equal(row_tok[flat], tok)
    # rows of each expert hold that expert's tokens in ascending order
    exp_of_row = np.searchsorted(offsets, np.arange(P), side="right") - 1
    np.testing.assert_array_equal(exp_of_row[flat], idx.ravel())
    for e in range(E):
        seg = row_tok[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)


def check_xn(g_xn, ref_xn, dtype):
    if dtype == "fp32":
        np.testing.assert_allclose(g_xn, ref_xn, rtol=2e-6, atol=1e-6)
        return 0
    same = g_xn == ref_xn
    n_diff = int((~same).sum())
    assert same.mean() >= 0.999, f"{n_diff} xn elements differ"
    rel = np.abs(g_xn - ref_xn) / np.maximum(np.abs(ref_xn), 1e-30)
    assert rel[~same].max(initial=0.0) <= 2.0 ** -7 + 1e-9, "xn differs by more than one bf16 ulp"
    return n_diff


LOGIT_ABS_TOL = 2e-5   # |dl| <= 2e-5 keeps |db| = |ds| <= 0.25 |dl| at half the near-tie margin


def check_routing_stage(g, host, c, rows=None):
    """Stage checks of the router on the GPU's own intermediates.
    (1) logits: oracle step B on the GPU's xn, |gpu - oracle| <= 2e-5;
    (2) top-k + weights: oracle steps C-D on the GPU's logits; ids equal
        except near-ties, weights within 2e-6 relative;
    (3) ids against oracle steps B-D on the GPU's xn: equal except where the
        oracle's margin is below 1e-5."""
    sel = slice(None) if rows is None else rows
    xn = g["xn"][sel]
    logits, idx, wts, margin = orc.route(c, xn, host["router_w"], host["corr_bias"])
    gl = g["logits"][sel]
    dl = float(np.abs(gl.astype(np.float64) - logits).max())
    assert dl <= LOGIT_ABS_TOL, f"router logits differ by {dl}"
    gi, gw = g["idx"][sel], g["w"][sel]
    # (2) selection and weights from identical logits: the same set of experts
    # (near-ties at the k-th place excepted), in an order the scores allow
    sidx, sw, smargin = orc.select(c, gl, host["corr_bias"])
    smis, order_bad = selection_diff(gi, sidx, biased_scores(gl, host["corr_bias"]))
    assert not (smis & (smargin >= NEAR_TIE)).any(), "top-k differs from the oracle on the same logits"
    assert not order_bad.any(), "slot order contradicts the scores"
    ok = ~smis
    np.testing.assert_allclose(by_expert(gi[ok], gw[ok]), by_expert(sidx[ok], sw[ok]), rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(gw.astype(np.float64).sum(1), c.routed_scale, rtol=2e-6)
    # (3) selection against the oracle's own logits
    mismatch, _ = selection_diff(gi, idx, biased_scores(logits, host["corr_bias"]))
    bad = mismatch & (margin >= NEAR_TIE)
    assert not bad.any(), f"{int(bad.sum())} tokens routed differently with margin >= {NEAR_TIE}"
    return {"max_logit_err": dl, "mismatch": int(mismatch.sum()),
            "near_tie": int((margin < NEAR_TIE).sum()), "select_mismatch": int(smis.sum()),
            "order_swaps": int(np.any(gi != sidx, axis=1).sum() - smis.sum())}


def output_errors(gpu, ref):
    diff = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    return {"max_over_rms": float(diff.max() / rms) if rms > 0 else float(diff.max()),
            "mean_rel": float(diff.sum() / max(np.abs(ref).sum(), 1e-30))}


def check_bf16_max(gpu, ref, max_rms):
    """max|gpu - ref| <= max_rms * rms(ref) over every compared element."""
    ref64 = ref.astype(np.float64)
    rms = float(np.sqrt(np.mean(ref64 ** 2)))
    err = float(np.abs(gpu.astype(np.float64) - ref64).max(initial=0.0))
    assert err <= max_rms * rms, f"bf16 output error {err / rms:.5f} * rms(oracle) > {max_rms}"


def check_output(g, host, c, dtype, rows=None):
    """Oracle on the GPU's selection for the given rows; returns error stats
    of the output and of the MoE delta (out - x)."""
    rows_arr = np.arange(g["out"].shape[0]) if rows is None else np.asarray(rows)
    r = orc.forward(c, host, rows=rows_arr, forced_idx=g["idx"][rows_arr])
    gout = g["out"][rows_arr]
    st = output_errors(gout, r["out"])
    x = host["x"][rows_arr]
    x = (x.astype(np.uint32) << 16).view(np.float32) if x.dtype == np.uint16 else x
    sd = output_errors(gout - x, r["out"] - x)
    tol = TOL[dtype]
    if dtype == "bf16":
        check_bf16_max(gout, r["out"], tol["max_rms"])
        assert st["mean_rel"] <= tol["mean_rel"], st
    else:
        assert st["max_over_rms"] <= tol["max_rms"], st
    return {"out": st, "delta": sd}


def flip_reach(g_xn, o_xn, router_w):
    """Per token: an upper bound of how far the GPU's and the oracle's
    biased-score gap between any two experts can move because their RMSNorm
    outputs differ.  |dl_e| <= sum_j |dxn_j| |Wr[e, j]|, the sigmoid's slope
    is at most 1/4, and two experts' scores can move towards each other, so
    the reach is 2 * (max_e |dl_e| / 4 + the router's own logit error / 4)."""
    wr = ((router_w.astype(np.uint32) << 16).view(np.float32) if router_w.dtype == np.uint16
          else router_w.astype(np.float32))
    dxn = np.abs(g_xn.astype(np.float64) - o_xn.astype(np.float64))
    dl = dxn @ np.abs(wr.astype(np.float64)).T
    return 2.0 * (dl.max(axis=1) / 4.0 + LOGIT_ABS_TOL / 4.0)


def check_end_to_end_routing(g, host, c, rows):
    """Oracle's own routing (its own xn) against the GPU's, for the sampled
    rows.  A difference must be a near-tie (margin < 1e-5) or a token whose
    RMSNorm output differs from the oracle's by enough to reach its margin
    (flip_reach >= margin); both are counted and reported apart."""
    r = orc.forward(c, host, rows=np.asarray(rows))
    gi = g["idx"][rows]
    mismatch = np.any(np.sort(gi, axis=1) != np.sort(r["idx"], axis=1), axis=1)
    near_tie = r["margin"] < NEAR_TIE
    xn_diff = np.any(g["xn"][rows] != r["xn"], axis=1)
    reach = np.zeros(len(rows))
    cand = mismatch & ~near_tie & xn_diff
    if cand.any():
        reach[cand] = flip_reach(g["xn"][rows][cand], r["xn"][cand], host["router_w"])
    excused_flip = cand & (reach >= r["margin"])
    unexplained = mismatch & ~near_tie & ~excused_flip
    assert not unexplained.any(), f"{int(unexplained.sum())} unexplained routing differences"
    return {"mismatch": int(mismatch.sum()), "near_tie": int(near_tie.sum()),
            "near_tie_mismatch": int((mismatch & near_tie).sum()),
            "xn_flip_excused": int(excused_flip.sum()), "xn_rows_differ": int(xn_diff.sum())}
