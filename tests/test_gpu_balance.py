"""The two balance controls next to the layer -- router z-loss and one step
of auxiliary-loss-free bias balancing -- on the GPU through the C ABI, against
the CPU oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from sparse_mixture_experts_65_b300 import layer as L
from sparse_mixture_experts_65_b300 import workloads as W

from gpu_harness import run_gpu

pytestmark = pytest.mark.gpu

Z_RTOL = 1e-5   # float32 log-partition per token, double sum of squares

Z_CASES = [
    # T, E, scale, shift
    (0, 8, 1.0, 0.0),            # empty batch: 0
    (1, 1, 2.0, 0.5),            # E = 1: mean square of the logits
    (37, 5, 3.0, 0.0),           # scalar path (E not a multiple of 4), ragged
    (4096, 64, 1.0, 0.0),        # Switch-sized router
    (4096, 256, 2.0, 0.0),       # DeepSeek-V3-sized router
    (5000, 128, 8.0, 30.0),      # large logits, more tokens than cluster threads
    (9000, 512, 0.5, -3.0),      # the widest router, several tokens per thread
]


@pytest.mark.parametrize("T,E,scale,shift", Z_CASES)
def test_router_z_loss_matches_oracle(T, E, scale, shift):
    s = W.make_logits(T, E, seed=T + E, scale=scale, shift=shift)
    z = L.router_z_loss(s.cuda())
    z2 = L.router_z_loss(s.cuda())
    torch.cuda.synchronize()
    ref = O.router_z_loss(s.numpy())
    got = float(z.item())
    assert torch.equal(z, z2)                      # fixed summation order
    if T == 0:
        assert got == 0.0
    else:
        assert abs(got - ref) <= Z_RTOL * abs(ref), (got, ref)


@pytest.mark.parametrize("name", ["switch", "dsv3"])
def test_router_z_loss_of_full_size_router_logits(name):
    """The z-loss of the logits the layer routes with (moe_router_scores)."""
    shape = W.get(name)
    inp = W.make_inputs(shape, "cuda")
    cfg = L.config_for(shape)
    s = L.router_scores(cfg, inp.x, inp.W_r, inp.logit_offset)
    z = L.router_z_loss(s)
    torch.cuda.synchronize()
    ref = O.router_z_loss(s.cpu().numpy())
    assert abs(float(z.item()) - ref) <= Z_RTOL * abs(ref)
    del inp


BIAS_CASES = [
    # E, T, k, gamma, skew
    (1, 5, 1, 0.3, 1.0),
    (7, 5, 1, 1e-3, 1.0),          # mean load below one token
    (64, 4096, 1, 1e-3, 2.0),      # Switch-shaped, skewed
    (256, 4096, 8, 1e-3, 1.0),     # DeepSeek-V3-shaped, many at the mean
    (512, 1000, 3, 2.0 ** -10, 0.5),
    (128, 0, 4, 1e-3, 1.0),        # empty batch: every expert at the mean
]


@pytest.mark.parametrize("E,T,k,gamma,skew", BIAS_CASES)
def test_bias_update_bit_exact(E, T, k, gamma, skew):
    counts = W.make_routed_counts(E, T, k, seed=E + T, skew=skew)
    g = torch.Generator().manual_seed(E * 7 + k)
    b0 = (torch.rand(E, generator=g, dtype=torch.float32) * 2 - 1) * 0.05
    b = b0.cuda()
    L.bias_update(b, counts.cuda(), T, k, gamma)
    torch.cuda.synchronize()
    ref = O.bias_update(b0.numpy(), counts.numpy(), T, k, gamma)
    np.testing.assert_array_equal(b.cpu().numpy(), ref)


def test_bias_update_on_the_layers_routed_counts():
    """A DeepSeek-V3-style layer (sigmoid gates, selection bias): the routed
    counts moe_forward writes drive one balancing step; the updated bias then
    routes the next call."""
    from sparse_mixture_experts_65_b300.workloads import LayerShape
    shape = LayerShape("bias_step", 37, T=512, d=128, E=32, k=4, f=64, act=W.ACT_SWIGLU,
                       gate=W.GATE_SIGMOID_RENORM, dtype="bf16", alpha=1e-4,
                       sel_bias_halfwidth=0.05)
    inp = W.make_inputs(shape, "cuda")
    _, out = run_gpu(inp)
    before = inp.sel_bias.clone()
    L.bias_update(inp.sel_bias, out.routed_counts, shape.T, shape.k, 1e-3)
    torch.cuda.synchronize()
    ref = O.bias_update(before.cpu().numpy(), out.routed_counts.cpu().numpy(), shape.T,
                        shape.k, 1e-3)
    np.testing.assert_array_equal(inp.sel_bias.cpu().numpy(), ref)
    _, out2 = run_gpu(inp)           # the next call sees the new bias
    r2 = O.route(inp.x.float().cpu().numpy(), inp.W_r.float().cpu().numpy(), shape.k,
                 O.GATE_SIGMOID_RENORM, sel_bias=inp.sel_bias.cpu().numpy())
    agree = (out2.topk_idx.cpu().numpy() == r2[2]).all(axis=1).mean()
    assert agree > 0.99


def test_balance_controls_reject_bad_arguments():
    s = torch.zeros((4, 8), device="cuda")
    z = torch.zeros(1, device="cuda")
    lib = L.N.lib()
    assert lib.moe_router_z_loss(L._ptr(s), -1, 8, L._ptr(z), None) == L.N.MOE_ERR_ARG
    assert lib.moe_router_z_loss(L._ptr(s), 4, 513, L._ptr(z), None) == L.N.MOE_ERR_ARG
    assert lib.moe_router_z_loss(L._ptr(s), 4, 8, None, None) == L.N.MOE_ERR_ARG
    c = torch.zeros(8, dtype=torch.int32, device="cuda")
    b = torch.zeros(8, device="cuda")
    import ctypes
    for args in ((8, 4, 0, 1e-3), (8, 4, 9, 1e-3), (0, 4, 1, 1e-3), (8, 4, 1, -1.0),
                 (8, 4, 1, float("inf")), (8, -1, 1, 1e-3)):
        E, T, k, gm = args
        assert lib.moe_bias_update(L._ptr(c), E, T, k, ctypes.c_float(gm), L._ptr(b), None) \
            == L.N.MOE_ERR_ARG, args
    torch.cuda.synchronize()
    assert torch.equal(b, torch.zeros(8, device="cuda"))
