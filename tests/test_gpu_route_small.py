"""Small batches (at most 32 tokens, at most 256 experts) route in one fused
block (route_small_kernel): split-K logit sum, scores, top-k, histogram, scan,
stable scatter and, for a few rows, the row gather.

* Every shape below runs the fused block and is checked against the CPU oracle
  like the other small cases: the permutation invariants exactly, the routing
  and the output within the stated tolerances.
* The fused block must take the same decisions, bit for bit, as the separate
  kernels that route larger batches.  A batch of 48 tokens (separate kernels)
  and its first t tokens as a batch of their own (fused) share the router's
  split of K (the same 64-token router tile), so their logits, expert indices
  and weights must be identical.
"""
import numpy as np
import pytest

import parity
from mixture_experts_transformer_sigmoid_b300 import workloads as wl
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

W = wl.Workload
FUSED = {
    "t1_wide": W("t1_wide", T=1, d=2048, E=256, I=64, Is=64, k=8, routed_scale=2.5, dtype="bf16"),
    "t2_no_shared": W("t2_no_shared", T=2, d=256, E=8, I=64, Is=0, k=2, routed_scale=1.0, dtype="bf16"),
    "t3_k_equals_E": W("t3_k_equals_E", T=3, d=256, E=4, I=64, Is=64, k=4, routed_scale=1.0,
                       dtype="bf16"),
    # E not a multiple of 32
    "t5_odd_experts": W("t5_odd_experts", T=5, d=256, E=200, I=64, Is=64, k=6, routed_scale=1.0,
                        dtype="bf16"),
    # E above the fused block's 256: the separate kernels route it
    "t5_many_experts": W("t5_many_experts", T=5, d=256, E=300, I=64, Is=64, k=6, routed_scale=1.0,
                         dtype="bf16"),
    "t16_skewed": W("t16_skewed", T=16, d=512, E=32, I=128, Is=128, k=4, routed_scale=2.5,
                    dtype="bf16", n_hot=4),
    # the rows too many for the block's own gather
    "t24_wide": W("t24_wide", T=24, d=1024, E=256, I=64, Is=64, k=8, routed_scale=2.5, dtype="bf16"),
    # 32 tokens: the last bit of the per-expert token masks; top-1
    "t32_top1": W("t32_top1", T=32, d=256, E=12, I=128, Is=64, k=1, routed_scale=1.0, dtype="bf16"),
    # too many router partials for the block: router_reduce_kernel adds them first
    "t32_reduced_first": W("t32_reduced_first", T=32, d=2048, E=256, I=64, Is=64, k=8,
                           routed_scale=2.5, dtype="bf16"),
}


def device_inputs(inputs):
    return {k: v.cuda() for k, v in inputs.items()}


@pytest.mark.parametrize("name", list(FUSED))
def test_fused_routing_matches_oracle(name):
    w = FUSED[name]
    inp = wl.make_inputs(w, seed=3)
    host = wl.host_arrays(inp)
    g = parity.run_gpu(w, device_inputs(inp))
    c = orc.cfg_from_workload(w)
    parity.check_permutation(g, w.T, w.E, w.k)
    r = orc.forward(c, host)
    parity.check_xn(g["xn"], r["xn"], w.dtype)
    parity.check_routing_stage(g, host, c)
    stats = parity.check_output(g, host, c, w.dtype)
    rt = parity.check_end_to_end_routing(g, host, c, np.arange(w.T))
    print(name, stats, rt)


@pytest.mark.parametrize("d,E,k", [(1024, 64, 6), (2048, 256, 8)])
def test_fused_routing_is_bitwise_the_separate_kernels(d, E, k):
    big = W("big", T=48, d=d, E=E, I=64, Is=64, k=k, routed_scale=2.5, dtype="bf16")
    inp = device_inputs(wl.make_inputs(big, seed=11))
    ref = parity.run_gpu(big, inp)
    for t in (1, 7, 32):
        w = W(f"t{t}", T=t, d=d, E=E, I=64, Is=64, k=k, routed_scale=2.5, dtype="bf16")
        g = parity.run_gpu(w, inp, T=t)
        np.testing.assert_array_equal(g["logits"].view(np.uint32),
                                      ref["logits"][:t].view(np.uint32))
        np.testing.assert_array_equal(g["idx"], ref["idx"][:t])
        np.testing.assert_array_equal(g["w"].view(np.uint32), ref["w"][:t].view(np.uint32))
        parity.check_permutation(g, t, E, k)
