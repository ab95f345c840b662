"""moe_router_scores_noalloc: router logits for callers that cannot allocate
device memory per call (a host framework that owns all device memory, or a
latency path that must not enter the CUDA allocator).  Its scratch is an 8 MiB
array inside the library; its results must equal moe_router_scores, which uses
a caller workspace, and lie within the router tolerance of the float64
definition in the CPU oracle.  This file runs last so that a failure here
comes after every other test has run; it also passes alone in a fresh process
(the first call in the context does the array's set-up)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle.moe_oracle as O

from sparse_mixture_experts_65_b300 import _native as N
from sparse_mixture_experts_65_b300 import layer as L
from sparse_mixture_experts_65_b300 import workloads as W

pytestmark = pytest.mark.gpu

ROUTER_ATOL = 5e-6     # the router tolerance of the parity tests (half the near-tie band)


def _router_inputs(shape, seed):
    """x, W_r and the logit offset of a layer, without its expert weights."""
    g = torch.Generator(device="cuda")
    g.manual_seed(1000 * shape.cid + 17 + seed)
    dt = W.torch_dtype(shape)
    x = torch.randn((shape.T, shape.d), generator=g, device="cuda").to(dt)
    W_r = (torch.randn((shape.E, shape.d), generator=g, device="cuda") / shape.d ** 0.5).to(dt)
    off = None
    if shape.logit_offset_var > 0:
        off = torch.randn(shape.E, generator=g, device="cuda") * shape.logit_offset_var ** 0.5
    return x, W_r, off


def _noalloc(cfg, x, W_r, off, out):
    fn = N.lib().moe_router_scores_noalloc
    fn.argtypes = [ctypes.POINTER(N.MoeConfig)] + [ctypes.c_void_p] * 5
    fn.restype = ctypes.c_int
    return fn(ctypes.byref(cfg), x.data_ptr(), W_r.data_ptr(),
              None if off is None else off.data_ptr(), out.data_ptr(),
              torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("order", [("switch", "gptoss256"), ("gptoss256", "switch")])
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(order):
    for name in order:                     # the second call finds the first one's leftovers
        shape = W.get(name)
        x, W_r, off = _router_inputs(shape, seed=3)
        cfg = L.config_for(shape)
        ref = L.router_scores(cfg, x, W_r, off)
        out = torch.full((shape.T, shape.E), float("nan"), device="cuda")
        assert _noalloc(cfg, x, W_r, off, out) == N.MOE_OK
        torch.cuda.synchronize()
        diff = (out - ref).abs().max().item()
        assert np.isfinite(diff) and diff <= ROUTER_ATOL, (name, diff)
        # with moe_router_scores on the same float32 kernel the bits agree too
        with L.tuning(router="simt"):
            ref_same = L.router_scores(cfg, x, W_r, off)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_same), name
        # and the logits are the float64 definition's within the router tolerance
        def h(t):
            return None if t is None else t.float().cpu().numpy().astype(np.float64)
        exact = O.router_logits(h(x), h(W_r), h(off))
        err = np.abs(out.cpu().numpy().astype(np.float64) - exact).max()
        assert err <= ROUTER_ATOL, (name, err)


def test_noalloc_rejects_layers_beyond_its_scratch():
    shape = W.DSV3                                   # 4096 x 256 logits in 9 splits: 36 MiB
    x, W_r, _ = _router_inputs(shape, seed=0)
    out = torch.empty((shape.T, shape.E), device="cuda")
    assert _noalloc(L.config_for(shape), x, W_r, None, out) == N.MOE_ERR_UNSUPPORTED
