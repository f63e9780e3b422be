"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes (moe_selftest_wait_timeout, the same wait helper the tensor-core
kernels use) gives up, the host reads MOE_ERR_TIMEOUT from the device error
flag, the flag is cleared, and the same handle then runs a forward that
gives the same bytes as before."""
import time

import pytest
import torch

from mixture_experts_transformer_sigmoid_b300 import binding as B
from mixture_experts_transformer_sigmoid_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_stays_usable():
    w = wl.Workload("wait_bf16", T=300, d=512, E=16, I=192, Is=128, k=4, routed_scale=1.0,
                    dtype="bf16")
    inp = {k: v.cuda() for k, v in wl.make_inputs(w).items()}
    layer = B.MoeSublayer(max_tokens=w.T, hidden=w.d, n_experts=w.E, inter=w.I, shared_inter=w.Is,
                          max_top_k=w.k, dtype=w.dtype)
    try:
        before = layer.forward(inp["x"], inp, w.k, w.routed_scale).clone()
        assert layer.sync_status() == B.MOE_OK
        layer.selftest_wait_timeout(20000)            # 20 ms
        t0 = time.perf_counter()
        assert layer.sync_status() == B.MOE_ERR_TIMEOUT
        assert time.perf_counter() - t0 >= 0.01       # the wait ran until its limit
        assert layer.sync_status() == B.MOE_OK        # the flag was cleared
        after = layer.forward(inp["x"], inp, w.k, w.routed_scale)
        assert layer.sync_status() == B.MOE_OK
        assert torch.equal(before, after)
    finally:
        layer.close()
