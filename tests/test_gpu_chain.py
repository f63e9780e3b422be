"""The sublayer across the decode token range and chained over several
layers: the post-attention half of consecutive decoder layers, each layer's
output being the next layer's residual input (GlmMoeDsaDecoderLayer.forward
on the GLM-5 shared-expert page).

Decode: T in {1, 8, 16, 32, 128} on the GLM-5 weights with the skewed
routing of the decode workload (16 experts with +0.5 bias), every token
checked.  Chain: three layers with their own weights on one handle, each
layer's output checked against the oracle on that layer's input, and the
whole chain captured in one CUDA graph must give the same bytes."""
import numpy as np
import pytest
import torch

import parity
from mixture_experts_transformer_sigmoid_b300 import binding as B
from mixture_experts_transformer_sigmoid_b300 import workloads as wl
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

DECODE_T = [1, 8, 16, 32, 128]


@pytest.fixture(scope="module")
def glm5_decode_weights():
    w = wl.WORKLOADS["glm5_decode"]
    inp = wl.make_inputs(w, device="cuda")
    host = wl.host_arrays({k: v for k, v in inp.items() if k != "x"})
    return w, inp, host


@pytest.mark.parametrize("T", DECODE_T)
def test_glm5_decode_token_range(glm5_decode_weights, T):
    w0, inp, host_w = glm5_decode_weights
    w = w0.with_(T=T)
    x = wl.make_inputs(w, seed=T, device="cuda", weights_from=inp)["x"]
    dev = dict(inp)
    dev["x"] = x
    g = parity.run_gpu(w, dev)
    host = dict(host_w)
    host["x"] = wl.host_arrays({"x": x})["x"]
    c = orc.cfg_from_workload(w)
    parity.check_permutation(g, T, w.E, w.k)
    rs = parity.check_routing_stage(g, host, c)
    rows = np.arange(T)
    stats = parity.check_output(g, host, c, w.dtype, rows=rows)
    rt = parity.check_end_to_end_routing(g, host, c, rows)
    print("T", T, "active experts", int((g["counts"] > 0).sum()), rs, stats, rt)


def test_chained_layers_match_oracle_and_graph():
    w = wl.Workload("chain_bf16", T=200, d=256, E=16, I=128, Is=64, k=4, routed_scale=2.5,
                    dtype="bf16", n_hot=2)
    layers_w = [{k: v.cuda() for k, v in wl.make_inputs(w, seed=s).items()} for s in (11, 12, 13)]
    x0 = layers_w[0]["x"]
    layer = B.MoeSublayer(max_tokens=w.T, hidden=w.d, n_experts=w.E, inter=w.I, shared_inter=w.Is,
                          max_top_k=w.k, dtype=w.dtype)
    c = orc.cfg_from_workload(w)
    try:
        xs = [x0]
        for lw in layers_w:        # layer by layer, each checked on its own input
            out = layer.forward(xs[-1], lw, w.k, w.routed_scale)
            idx, wt, counts = layer.routing()
            assert layer.sync_status() == B.MOE_OK
            host = wl.host_arrays({k: v for k, v in lw.items() if k != "x"})
            host["x"] = wl.host_arrays({"x": xs[-1]})["x"]
            g = {"out": parity.to_np_f32(out), "idx": idx.cpu().numpy()}
            print(parity.check_output(g, host, c, w.dtype))
            xs.append(out)
        outs = [torch.empty_like(x0) for _ in layers_w]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            src = x0
            for lw, o in zip(layers_w, outs):
                layer.forward(src, lw, w.k, w.routed_scale, out=o)
                src = o
        graph.replay()
        torch.cuda.synchronize()
        assert layer.sync_status() == B.MOE_OK
    finally:
        layer.close()
    for direct, replayed in zip(xs[1:], outs):
        assert torch.equal(direct, replayed)
