"""moe_pack_experts (HF per-expert weights -> the grouped layout moe_forward
reads, state dict adapter page) against the numpy definition in the oracle:
exact data movement, so every element is compared bit for bit."""
import numpy as np
import pytest
import torch

from mixture_experts_transformer_sigmoid_b300 import binding as B
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def hf_stacks(E, d, I, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *shape: torch.randn(*shape, generator=g).to(dtype)
    return mk(E, I, d), mk(E, I, d), mk(E, d, I)


def bits(t):
    t = t.cpu()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.view(torch.int32).numpy()


@pytest.mark.parametrize("E,d,I,dtype", [
    (3, 320, 192, torch.bfloat16),      # several 64-element tiles, partial in both directions
    (2, 200, 130, torch.bfloat16),      # sizes that are no multiple of the tile
    (1, 6, 2, torch.bfloat16),          # smaller than one tile
    (2, 72, 100, torch.float32),
    (3, 33, 17, torch.float32),         # odd sizes (4-byte elements)
])
def test_pack_matches_definition(E, d, I, dtype):
    G, U, Dn = hf_stacks(E, d, I, dtype, seed=E * 1000 + d)
    gu, dp = B.pack_experts(G.cuda(), U.cuda(), Dn.cuda())
    torch.cuda.synchronize()
    want_gu, want_dp = orc.pack_experts(bits(G), bits(U), bits(Dn))
    np.testing.assert_array_equal(bits(gu), want_gu)
    np.testing.assert_array_equal(bits(dp), want_dp)


def test_pack_one_expert_at_a_time_equals_the_stacked_call():
    E, d, I = 4, 128, 192
    G, U, Dn = (t.cuda() for t in hf_stacks(E, d, I, torch.bfloat16, seed=5))
    gu, dp = B.pack_experts(G, U, Dn)
    gu1 = torch.empty_like(gu)
    dp1 = torch.empty_like(dp)
    for e in range(E):
        B.pack_experts(G[e:e + 1], U[e:e + 1], Dn[e:e + 1], gate_up=gu1[e:e + 1], down_projs=dp1[e:e + 1])
    torch.cuda.synchronize()
    assert torch.equal(gu1, gu) and torch.equal(dp1, dp)


def test_pack_skips_a_null_output():
    E, d, I = 2, 64, 64
    G, U, Dn = (t.cuda() for t in hf_stacks(E, d, I, torch.bfloat16, seed=6))
    dp = torch.full((E, I, d), 7.0, dtype=torch.bfloat16, device="cuda")
    gu = torch.empty((E, d, 2 * I), dtype=torch.bfloat16, device="cuda")
    st = B.load_library().moe_pack_experts(E, d, I, 2, B._ptr(G), B._ptr(U), None, B._ptr(gu), None,
                                           B.ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == B.MOE_OK
    torch.cuda.synchronize()
    assert torch.all(dp == 7.0)
    want_gu, _ = orc.pack_experts(bits(G), bits(U), bits(Dn))
    np.testing.assert_array_equal(bits(gu), want_gu)


def test_pack_glm5_sized_experts_sampled():
    """The GLM-5 expert stacks (256 experts, d 6144, I 2048: 19.3 GB in, 19.3
    GB out); three experts compared with the definition on the host."""
    E, d, I = 256, 6144, 2048
    g = torch.Generator(device="cuda").manual_seed(9)
    G = torch.randn(E, I, d, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    U = torch.randn(E, I, d, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    Dn = torch.randn(E, d, I, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    gu, dp = B.pack_experts(G, U, Dn)
    torch.cuda.synchronize()
    for e in (0, 137, 255):
        want_gu, want_dp = orc.pack_experts(bits(G[e:e + 1]), bits(U[e:e + 1]), bits(Dn[e:e + 1]))
        np.testing.assert_array_equal(bits(gu[e:e + 1]), want_gu)
        np.testing.assert_array_equal(bits(dp[e:e + 1]), want_dp)
