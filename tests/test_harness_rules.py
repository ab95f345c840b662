"""The GPU parity harness applies the parity rules it states (no GPU).

The harness (tests/gpu_harness.py) is what turns a GPU call into a pass or a
failure, so its rules are tested here on the CPU: outputs built from the
oracle itself stand in for a GPU call.  They must pass; a token that chose
differently inside the near-tie band must pass and be counted; a different
choice outside the band, or any integer, gate, loss or output off the rules,
must fail.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gpu_harness
import oracle.moe_oracle as O
from gpu_harness import check_layer, host64
from sparse_mixture_experts_65_b300 import layer as L
from sparse_mixture_experts_65_b300 import workloads as W


@pytest.fixture(autouse=True)
def _keep_routing_report_to_gpu_calls():
    """The end-of-run routing summary lists GPU calls only: these stand-in
    calls are taken back out of it."""
    saved = list(gpu_harness.ROUTING_REPORTS)
    yield
    gpu_harness.ROUTING_REPORTS[:] = saved


SHAPE = W.LayerShape("harness_bf16", 95, T=48, d=32, E=6, k=2, f=16, act=W.ACT_SWIGLU,
                     gate=W.GATE_SOFTMAX_TOPK, dtype="bf16", capacity_factor=1.0)


def _oracle(inp, forced_idx=None):
    s = inp.shape
    return O.moe_forward(host64(inp.x), host64(inp.W_r), host64(inp.W1), host64(inp.W2), s.k,
                         s.act, s.gate, W3=host64(inp.W3), logit_offset=host64(inp.logit_offset),
                         sel_bias=host64(inp.sel_bias), capacity_factor=s.capacity_factor,
                         alpha=s.alpha, forced_idx=forced_idx)


def _as_outputs(r):
    """The oracle's result in the layout of a GPU call's outputs (y rounded
    to bf16 once, float32 gates and statistics, int32 indices)."""
    i32 = lambda a: torch.tensor(np.asarray(a), dtype=torch.int32)   # noqa: E731
    f32 = lambda a: torch.tensor(np.asarray(a), dtype=torch.float32)  # noqa: E731
    return L.MoeOutputs(y=torch.tensor(r.y).to(torch.bfloat16), topk_idx=i32(r.topk_idx),
                        topk_w=f32(r.topk_w), expert_counts=i32(r.asg.kept),
                        aux_loss=f32([r.aux_loss]), routed_counts=i32(r.asg.routed),
                        offsets=i32(r.asg.offsets), slot_pos=i32(r.asg.slot_pos), f=f32(r.f),
                        P=f32(r.P))


def _far_token(inp, r):
    """A token whose top-k list is far from any tie (gap above 1e-2)."""
    far = np.nonzero(r.gap > 1e-2)[0]
    assert far.size
    return int(far[0])


def test_the_oracle_itself_passes():
    inp = W.make_inputs(SHAPE, "cpu")
    r = _oracle(inp)
    assert r.asg.kept.sum() < SHAPE.T * SHAPE.k          # capacity drops some slots
    rep = check_layer(inp, _as_outputs(r))
    assert rep["flipped_tokens"] == 0 and rep["rel_l2"] < 1e-2


def _mutations(inp, r):
    t = _far_token(inp, r)
    out = _as_outputs(r)

    def swapped_choice(o):
        idx = o.topk_idx.clone()
        other = [e for e in range(SHAPE.E) if e not in idx[t].tolist()][0]
        idx[t, 0] = other
        return dataclasses.replace(o, topk_idx=idx)

    def repeated(o):
        idx = o.topk_idx.clone()
        idx[t, 1] = idx[t, 0]
        return dataclasses.replace(o, topk_idx=idx)

    def slot(o):
        sp = o.slot_pos.clone()
        j = int(torch.nonzero(sp.flatten() >= 0)[0])
        sp.view(-1)[j] += 1
        return dataclasses.replace(o, slot_pos=sp)

    def count(o):
        c = o.expert_counts.clone()
        c[0] += 1
        return dataclasses.replace(o, expert_counts=c)

    def offsets(o):
        c = o.offsets.clone()
        c[-1] -= 1
        return dataclasses.replace(o, offsets=c)

    def gate(o):
        w = o.topk_w.clone()
        w[t, 0] += 1e-4
        return dataclasses.replace(o, topk_w=w)

    def loss(o):
        return dataclasses.replace(o, aux_loss=o.aux_loss * (1 + 1e-4))

    def y_element(o):
        y = o.y.float().clone()
        y[t, 3] += 0.05
        return dataclasses.replace(o, y=y.to(torch.bfloat16))

    def y_nan(o):
        y = o.y.clone()
        y[t, 0] = float("nan")
        return dataclasses.replace(o, y=y)

    def y_scaled(o):
        return dataclasses.replace(o, y=(o.y.float() * 1.05).to(torch.bfloat16))

    fns = (swapped_choice, repeated, slot, count, offsets, gate, loss, y_element, y_nan,
           y_scaled)
    return {fn.__name__: fn(out) for fn in fns}


@pytest.mark.parametrize("case", ["swapped_choice", "repeated", "slot", "count", "offsets",
                                  "gate", "loss", "y_element", "y_nan", "y_scaled"])
def test_outputs_off_the_rules_fail(case):
    inp = W.make_inputs(SHAPE, "cpu")
    r = _oracle(inp)
    bad = _mutations(inp, r)[case]
    with pytest.raises(AssertionError):
        check_layer(inp, bad)


def test_a_near_tie_flip_passes_and_is_counted():
    """Experts 0 and 1 get identical router rows, so every token that picks
    one of them ties exactly with the other: choosing the other one instead is
    inside the band.  The outputs are then the oracle's conditioned on that
    choice (the integers follow the changed choice), and they must pass with
    the flips counted; the same flip on a token far from a tie must not."""
    inp = W.make_inputs(SHAPE, "cpu")
    inp.W_r[1] = inp.W_r[0]
    r = _oracle(inp)
    idx = r.topk_idx.copy()
    tied = [t for t in range(SHAPE.T) if (0 in idx[t]) != (1 in idx[t])]
    assert len(tied) >= 3
    for t in tied[:3]:
        idx[t] = [1 if e == 0 else 0 if e == 1 else e for e in idx[t]]
    r2 = _oracle(inp, forced_idx=idx)
    rep = check_layer(inp, _as_outputs(r2))
    assert rep["flipped_tokens"] == 3 and rep["near_tie_tokens"] >= 3
    far = [t for t in range(SHAPE.T) if r.gap[t] > 1e-2]
    idx_far = r.topk_idx.copy()
    t = far[0]
    idx_far[t] = [e for e in range(SHAPE.E) if e not in idx_far[t]][:SHAPE.k]
    with pytest.raises(AssertionError, match="outside the near-tie band"):
        check_layer(inp, _as_outputs(_oracle(inp, forced_idx=idx_far)))
