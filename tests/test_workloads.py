"""The seeded synthetic inputs follow the stated recipe (no GPU).

Recipe: tensor i of workload c is drawn from a generator seeded 1000*c + i
(plus 100003 times the caller's seed), in the fixed order x, W_r, W1, W2, W3,
logit offset, selection bias, Ws1, Ws3, Ws2; N(0, v) names a normal of
VARIANCE v; weights are N(0, 1/fan_in); bf16 values are float32 draws rounded
once; e4m3 weights are stored per output channel as a float32 scale amax/448
and codes rounded to nearest.
"""
import math

import pytest
import torch

from sparse_mixture_experts_65_b300 import workloads as W

MID = W.LayerShape("recipe_mid", 70, T=2048, d=256, E=4, k=2, f=512, act=W.ACT_SWIGLU,
                   gate=W.GATE_SIGMOID_RENORM, dtype="bf16", n_shared=1, f_shared=384,
                   sel_bias_halfwidth=0.05, logit_offset_var=1.5)
WIDE_E = W.LayerShape("recipe_wide_e", 71, T=4, d=8, E=8192, k=2, f=8, act=W.ACT_RELU,
                      gate=W.GATE_SOFTMAX_FULL, dtype="f32", logit_offset_var=1.5,
                      sel_bias_halfwidth=0.05)


def _std(t):
    return t.double().std().item()


def test_inputs_are_deterministic_per_seed():
    a, b = W.make_inputs(MID, "cpu"), W.make_inputs(MID, "cpu")
    for name in ("x", "W_r", "W1", "W2", "W3", "logit_offset", "sel_bias", "Ws1", "Ws3", "Ws2"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    c = W.make_inputs(MID, "cpu", seed=1)
    assert not torch.equal(a.x, c.x) and not torch.equal(a.W1, c.W1)
    assert torch.equal(W.make_x(MID, "cpu"), a.x)


def test_seeds_and_single_rounding_follow_the_recipe():
    """Re-draw three tensors by the recipe alone: the generator seed, the
    float32 draw, the scale, one rounding to bf16."""
    inp = W.make_inputs(MID, "cpu")
    base = 1000 * MID.cid

    def draw(i, shape, std):
        g = torch.Generator().manual_seed(base + i)
        return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)

    assert torch.equal(inp.x, draw(0, (MID.T, MID.d), 1.0))
    assert torch.equal(inp.W_r, draw(1, (MID.E, MID.d), 1.0 / math.sqrt(MID.d)))
    assert torch.equal(inp.W2, draw(3, (MID.E, MID.d, MID.f), 1.0 / math.sqrt(MID.f)))
    g = torch.Generator().manual_seed(base + 100003 + 0)
    x1 = (torch.randn((MID.T, MID.d), generator=g, dtype=torch.float32)).to(torch.bfloat16)
    assert torch.equal(W.make_x(MID, "cpu", seed=1), x1)


def test_weight_and_activation_scales():
    """Standard deviations 1 for x and 1/sqrt(fan_in) for every weight matrix,
    means near 0 (2 % on at least 2^17 draws, whose sampling error is ~0.2 %)."""
    inp = W.make_inputs(MID, "cpu")
    d, f, fs = MID.d, MID.f, MID.f_shared
    want = {"x": 1.0, "W_r": 1 / math.sqrt(d), "W1": 1 / math.sqrt(d), "W3": 1 / math.sqrt(d),
            "W2": 1 / math.sqrt(f), "Ws1": 1 / math.sqrt(d), "Ws3": 1 / math.sqrt(d),
            "Ws2": 1 / math.sqrt(fs)}
    for name, sd in want.items():
        t = getattr(inp, name)
        if t.numel() < (1 << 17):
            continue
        assert abs(_std(t) / sd - 1) < 0.02, (name, _std(t), sd)
        assert abs(t.double().mean().item()) < 0.02 * sd, name
    assert inp.W_r.numel() < (1 << 17)          # checked on the wide router below


def test_logit_skew_and_selection_bias_distributions():
    """The logit skew is N(0, 1.5): variance 1.5 (10 % on 8192 draws, sampling
    error ~1.6 %); the selection bias is U(-h, h): inside the interval, variance
    h^2 / 3; both float32.  The router weights of this layer: N(0, 1/d)."""
    inp = W.make_inputs(WIDE_E, "cpu")
    off, b = inp.logit_offset, inp.sel_bias
    assert off.dtype == torch.float32 and b.dtype == torch.float32
    assert abs(off.double().var().item() / 1.5 - 1) < 0.10
    assert abs(off.double().mean().item()) < 0.1
    h = WIDE_E.sel_bias_halfwidth
    assert b.abs().max().item() <= h
    assert abs(b.double().var().item() / (h * h / 3) - 1) < 0.10
    assert abs(_std(inp.W_r) * math.sqrt(WIDE_E.d) - 1) < 0.02
    none = W.make_inputs(W.LayerShape("recipe_plain", 72, T=2, d=8, E=4, k=1, f=8,
                                      act=W.ACT_RELU, gate=W.GATE_SOFTMAX_TOPK,
                                      dtype="f32"), "cpu")
    assert none.logit_offset is None and none.sel_bias is None and none.W3 is None


@pytest.mark.parametrize("w2", [False, True])
def test_e4m3_weights_are_channel_scaled_codes_of_the_bf16_draw(w2):
    """The e4m3 layer draws the same float32 weights (same seeds) and stores
    them per output channel: scale = amax / 448, so every channel's largest
    code is +-448; code * scale is the draw to within e4m3 rounding (relative
    2^-4 in the normal range, an absolute 2^-10 * scale below it)."""
    import dataclasses
    shape = dataclasses.replace(MID, name="recipe_fp8", w_fp8=True, w2_fp8=w2, n_shared=0,
                                f_shared=0)
    f8 = W.make_inputs(shape, "cpu")
    base = 1000 * shape.cid
    for q, s, i, std in ((f8.W1q, f8.W1s, 2, 1 / math.sqrt(shape.d)),
                         (f8.W3q, f8.W3s, 4, 1 / math.sqrt(shape.d)),
                         (f8.W2q, f8.W2s, 3, 1 / math.sqrt(shape.f))):
        if q is None:
            assert not w2 and f8.W2 is not None and f8.W2s is None
            continue
        assert q.dtype == torch.uint8 and s.dtype == torch.float32
        assert s.shape == q.shape[:2]
        g = torch.Generator().manual_seed(base + i)
        ref = torch.stack([torch.randn(q.shape[1:], generator=g, dtype=torch.float32) * std
                           for _ in range(q.shape[0])])
        val = q.view(torch.float8_e4m3fn).float()
        assert torch.all(val.abs().amax(dim=2) == 448.0)
        deq = val * s[:, :, None]
        err = (deq - ref).abs()
        tol = torch.maximum(ref.abs() * 2.0 ** -4, s[:, :, None] * 2.0 ** -10)
        assert torch.all(err <= tol * (1 + 1e-6))
