"""CPU self-test of the parity harness: given the oracle's own results as the
'device' result, every check passes; given a planted error, the checks fail."""
import numpy as np
import pytest
import torch

import parity
from mixture_experts_transformer_sigmoid_b300 import workloads as wl
from oracle import oracle as orc


def fake_gpu(w, host, c):
    r = orc.forward(c, host)
    T, k, E = w.T, w.k, w.E
    idx = r["idx"]
    counts = np.bincount(idx.ravel(), minlength=E).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    order = sorted(range(T * k), key=lambda p: (idx.ravel()[p], p // k))
    pos = np.empty(T * k, np.int32)
    pos[np.array(order)] = np.arange(T * k)
    row_tok = np.empty(T * k, np.int32)
    row_tok[pos] = np.repeat(np.arange(T), k)
    return {"out": r["out"], "xn": r["xn"], "logits": r["logits"], "idx": idx, "w": r["w"],
            "counts": counts, "offsets": offsets, "pos": pos.reshape(T, k), "row_tok": row_tok}


@pytest.fixture(scope="module")
def case():
    w = wl.Workload("h", T=90, d=128, E=10, I=64, Is=32, k=3, routed_scale=2.5, dtype="bf16")
    inp = wl.make_inputs(w, seed=3)
    host = wl.host_arrays(inp)
    c = orc.cfg_from_workload(w)
    return w, host, c, fake_gpu(w, host, c)


def test_harness_accepts_the_oracle(case):
    w, host, c, g = case
    parity.check_permutation(g, w.T, w.E, w.k)
    parity.check_xn(g["xn"], g["xn"], w.dtype)
    parity.check_routing_stage(g, host, c)
    parity.check_output(g, host, c, w.dtype)
    parity.check_end_to_end_routing(g, host, c, np.arange(w.T))


def test_harness_catches_planted_errors(case):
    w, host, c, g = case
    bad = dict(g, out=g["out"] * 1.05)
    with pytest.raises(AssertionError):
        parity.check_output(bad, host, c, w.dtype)
    p2 = g["pos"].copy()
    p2[0, 0], p2[1, 0] = p2[1, 0], p2[0, 0]
    with pytest.raises(AssertionError):
        parity.check_permutation(dict(g, pos=p2), w.T, w.E, w.k)
    i2 = g["idx"].copy()
    i2[:, [0, 1]] = i2[:, [1, 0]]
    with pytest.raises(AssertionError):
        parity.check_routing_stage(dict(g, idx=i2), host, c)
    w2 = g["w"] * 1.001
    with pytest.raises(AssertionError):
        parity.check_routing_stage(dict(g, w=w2), host, c)


def test_slot_order_may_swap_only_near_tied_experts():
    b = np.array([[0.9, 0.5, 0.5 + 5e-7, 0.1]], np.float32)
    oracle_sel = np.array([[0, 2, 1]])
    set_diff, order_bad = parity.selection_diff(np.array([[0, 1, 2]]), oracle_sel, b)
    assert not set_diff.any() and not order_bad.any()      # 1 and 2 are 5e-7 apart
    set_diff, order_bad = parity.selection_diff(np.array([[1, 0, 2]]), oracle_sel, b)
    assert not set_diff.any() and order_bad.all()          # 0.5 placed before 0.9
    set_diff, _ = parity.selection_diff(np.array([[0, 1, 3]]), oracle_sel, b)
    assert set_diff.all()


def test_routing_difference_is_excused_only_when_an_xn_flip_can_reach_the_margin(case):
    w, host, c, g = case
    r = orc.forward(c, host)
    t = int(np.argmax(r["margin"]))                       # the clearest selection
    order = np.argsort(-parity.biased_scores(r["logits"][t:t + 1], host["corr_bias"])[0], kind="stable")
    i2 = g["idx"].copy()
    i2[t, -1] = order[w.k]                               # the (k+1)-th expert instead of the k-th
    # no xn difference: unexplained
    with pytest.raises(AssertionError):
        parity.check_end_to_end_routing(dict(g, idx=i2), host, c, np.arange(w.T))
    # one element one bf16 ulp off: its reach is far below this token's margin
    x1 = g["xn"].copy()
    x1[t, 0] = x1[t, 0] * (1 + 2.0 ** -7)
    assert parity.flip_reach(x1[t:t + 1], r["xn"][t:t + 1], host["router_w"])[0] < r["margin"][t]
    with pytest.raises(AssertionError):
        parity.check_end_to_end_routing(dict(g, idx=i2, xn=x1), host, c, np.arange(w.T))
    # a large RMSNorm difference can move the scores past the margin: excused and counted
    x2 = g["xn"].copy()
    x2[t] = -x2[t]
    rt = parity.check_end_to_end_routing(dict(g, idx=i2, xn=x2), host, c, np.arange(w.T))
    assert rt["xn_flip_excused"] == 1 and rt["mismatch"] == 1


def test_bf16_max_check_allows_rounding_and_catches_more():
    rng = np.random.default_rng(4)
    ref = (rng.standard_normal(200000) * 1.7).astype(np.float32)
    rounded = torch.from_numpy(ref).to(torch.bfloat16).float().numpy()
    parity.check_bf16_max(rounded, ref, 2e-2)            # the exact result, stored in bf16
    bad = rounded.copy()
    bad[123] += 0.05 * 1.7                               # 5e-2 rms off in one element
    with pytest.raises(AssertionError):
        parity.check_bf16_max(bad, ref, 2e-2)
