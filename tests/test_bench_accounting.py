"""The benchmark's FLOP and byte accounting (the numerators of its roofline
fractions) against per-workload totals worked out from the shapes
(FLOPs = 2·T·d·E + 6·T·k·d·I + 6·T·d·Is for the sublayer, 6·T·d·I for the
dense block), and the GLM-5 weight bytes against the parameter count the
GLM-5 MoE block page prints (9,702,998,272 values per MoE sublayer).
Runs on the CPU: nothing here touches a GPU."""
import pytest

import bench
from mixture_experts_transformer_sigmoid_b300 import workloads as wl


@pytest.mark.parametrize("name,flops", [
    ("tiny_fp32", 3.80e7), ("small_bf16", 9.72e10), ("air_prefill", 1.28e12),
    ("glm5_prefill", 5.592e12), ("glm5_decode", 4.37e10),
])
def test_sublayer_flops(name, flops):
    w = wl.WORKLOADS[name]
    assert bench.total_flops(w, w.T) == pytest.approx(flops, rel=5e-3)
    assert bench.total_flops(w, w.T) == pytest.approx(
        2 * w.T * w.d * w.E + bench.gate_up_flops(w, w.T) + bench.down_flops(w, w.T))


def test_gate_up_is_two_thirds_of_the_expert_flops():
    w = wl.WORKLOADS["glm5_prefill"]
    assert bench.gate_up_flops(w, w.T) == pytest.approx(2 * bench.down_flops(w, w.T))
    assert bench.gate_up_flops(w, w.T) == pytest.approx(3.71e12, rel=2e-3)


def test_glm5_weight_bytes_match_the_printed_parameter_count():
    w = wl.WORKLOADS["glm5_prefill"]
    params = 9_702_998_272          # 257 SwiGLU experts of 3·6144·2048, router 256·6144, 256 biases
    # bf16 values, fp32 correction bias (256 values: 2 more bytes each), plus the RMSNorm gain
    assert bench.weight_bytes(w) == 2 * params + 2 * w.E + 2 * w.d
    assert bench.weight_bytes(w) == pytest.approx(19.41e9, rel=1e-3)


def test_decode_bytes_count_each_active_expert_once():
    w = wl.WORKLOADS["glm5_decode"]
    per_expert = 3 * w.d * w.I * 2
    b59 = bench.decode_bytes(w, w.T, 59)
    assert bench.decode_bytes(w, w.T, 60) - b59 == per_expert
    assert b59 == pytest.approx(4.53e9, rel=2e-3)         # 59 active experts + the shared one
    assert bench.gate_up_decode_bytes(w, 59) == 59 * w.d * 2 * w.I * 2 + 2 * w.d * w.Is * 2


def test_dense_block_flops():
    w = wl.DENSE_WORKLOADS["glm5_dense_prefill"]
    assert 6 * w.T * w.d * w.I == pytest.approx(3.7109e12, rel=1e-4)
