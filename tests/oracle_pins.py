"""Checks that pin the CPU oracle to facts outside itself.

Each check raises AssertionError on failure.  ``test_oracle_pins.py`` runs
them against the oracle as written; ``test_oracle_mutations.py`` plants a
plausible mistake in the oracle (on the CPU) and shows that a check fails.

What each check leans on:
  brute force      -- enumeration of all k-subsets; dense evaluation of all E
                      experts with a gate vector that is zero off the chosen set
  closed forms     -- hand-derived gate and loss values for tiny inputs
  library cases    -- E = 1, k = 1 reduces the layer to one dense FFN, checked
                      against torch.nn.functional in float64
  page numbers     -- tests/golden/*.txt, each with its source
"""

import itertools
import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle.moe_oracle as O

from conftest import read_golden


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- stage 1
def check_router_onehot():
    """x_t = unit vector e_c picks out column c of W_r (catches a transposed
    or mis-indexed router product) and the offset adds per expert."""
    rng = _rng(1)
    E, d = 3, 5
    W_r = rng.normal(size=(E, d))
    x = np.eye(d)
    s = O.router_logits(x, W_r)
    assert s.shape == (d, E)
    for c in range(d):
        np.testing.assert_array_equal(s[c], W_r[:, c])
    off = np.array([0.5, -1.0, 2.0])
    s2 = O.router_logits(x, W_r, off)
    np.testing.assert_allclose(s2 - s, np.tile(off, (d, 1)), rtol=0, atol=1e-15)
    # linearity in x with a general vector
    xv = rng.normal(size=(1, d))
    ref = sum(xv[0, c] * W_r[:, c] for c in range(d))
    np.testing.assert_allclose(O.router_logits(xv, W_r)[0], ref, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------- stage 2
def check_topk_bruteforce():
    """For every E <= 7 and k <= E the chosen set maximises the summed selection
    score over all C(E, k) subsets and is listed in descending order."""
    rng = _rng(2)
    for E in range(1, 8):
        for k in range(1, E + 1):
            sel = rng.normal(size=(6, E))
            idx = O.topk_indices(sel, k)
            for t in range(sel.shape[0]):
                best = max(itertools.combinations(range(E), k),
                           key=lambda c: sum(sel[t, list(c)]))
                assert set(idx[t].tolist()) == set(best)
                vals = sel[t, idx[t]]
                assert np.all(np.diff(vals) <= 0)


def check_topk_ties():
    """Equal scores resolve to the lower expert index."""
    sel = np.array([[1.0, 3.0, 3.0, 2.0], [0.0, 0.0, 0.0, 0.0]])
    idx = O.topk_indices(sel, 2)
    assert idx[0].tolist() == [1, 2]
    assert idx[1].tolist() == [0, 1]
    assert O.topk_indices(sel, 4)[1].tolist() == [0, 1, 2, 3]


def check_topk_gap():
    """The near-tie gap: the smallest neighbouring difference among the k+1
    best scores.  Hand cases, then its meaning: moving every score by less than
    half the gap never changes the ordered top-k list, and moving the closest
    pair toward each other by a little more than half of it always does."""
    g = O.topk_gap(np.array([[3.0, 1.0, 2.0, 0.0]]), 2)
    assert g.tolist() == [1.0]                       # 3 | 2 | 1: both gaps are 1
    sel = np.array([[5.0, 4.5, 1.0, 0.9]])
    assert O.topk_gap(sel, 1).tolist() == [0.5]      # 5 vs 4.5 decides the set
    assert O.topk_gap(sel, 2).tolist() == [0.5]      # inside the set: the order
    np.testing.assert_allclose(O.topk_gap(sel, 3), [0.1], rtol=1e-12)   # 1 vs 0.9
    far = np.array([[10.0, 5.0, 1.0, 1.0]])          # a tie below the (k+1)-th is irrelevant
    assert O.topk_gap(far, 1).tolist() == [5.0]
    assert O.topk_gap(np.array([[1.0, 2.0, 2.0, 0.0]]), 1).tolist() == [0.0]   # exact tie
    assert O.topk_gap(np.array([[1.0, 3.0]]), 2).tolist() == [2.0]   # k = E: the order only
    assert O.topk_gap(np.array([[0.7]]), 1).tolist() == [math.inf]   # E = 1: nothing to swap
    assert O.near_tie_tokens(np.array([[1.0, 1.0 + 5e-6, 0.0], [3.0, 2.0, 1.0]]), 1).tolist() \
        == [True, False]
    rng = _rng(21)
    for E, k in ((6, 2), (9, 4), (5, 5), (12, 1)):
        sel = rng.normal(size=(40, E))
        gap = O.topk_gap(sel, k)
        base = O.topk_indices(sel, k)
        for t in range(sel.shape[0]):
            for _ in range(5):   # any perturbation below half the gap keeps the list
                d = rng.uniform(-1, 1, size=E) * 0.49 * gap[t]
                assert O.topk_indices(sel[t:t + 1] + d, k)[0].tolist() == base[t].tolist()
            srt = np.argsort(-sel[t], kind="stable")[:min(k + 1, E)]
            vals = sel[t, srt]
            i = int(np.argmin(vals[:-1] - vals[1:]))
            d = np.zeros(E)
            d[srt[i]] -= 0.51 * gap[t]
            d[srt[i + 1]] += 0.51 * gap[t]
            assert O.topk_indices(sel[t:t + 1] + d, k)[0].tolist() != base[t].tolist()


def check_gates_closed_form():
    """Hand-derived gates for logits [2, 1, 0, -1] with k = 2."""
    s = np.array([[2.0, 1.0, 0.0, -1.0]])
    idx = np.array([[0, 1]])
    e = math.e
    g = O.gate_values(s, idx, O.GATE_SOFTMAX_TOPK)
    np.testing.assert_allclose(g[0], [e / (e + 1), 1 / (e + 1)], rtol=1e-14)
    g = O.gate_values(s, idx, O.GATE_SOFTMAX_FULL)
    z = math.exp(2) + math.exp(1) + 1 + math.exp(-1)
    np.testing.assert_allclose(g[0], [math.exp(2) / z, math.exp(1) / z], rtol=1e-14)
    g = O.gate_values(s, idx, O.GATE_SIGMOID_RENORM)
    s2, s1 = 1 / (1 + math.exp(-2)), 1 / (1 + math.exp(-1))
    np.testing.assert_allclose(g[0], [s2 / (s1 + s2), s1 / (s1 + s2)], rtol=1e-14)


def check_gates_invariants():
    """Softmax over the chosen equals the full softmax renormalised over them;
    top-k and sigmoid gates sum to 1; top-1 softmax-over-chosen is exactly 1."""
    rng = _rng(3)
    s = rng.normal(size=(20, 9)) * 2
    for k in (1, 2, 3, 9):
        idx = O.topk_indices(s, k)
        g = O.gate_values(s, idx, O.GATE_SOFTMAX_TOPK)
        full = O.softmax_rows(s)
        ren = np.take_along_axis(full, idx, 1)
        ren = ren / ren.sum(1, keepdims=True)
        np.testing.assert_allclose(g, ren, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(g.sum(1), 1.0, rtol=1e-14)
        gs = O.gate_values(s, idx, O.GATE_SIGMOID_RENORM)
        np.testing.assert_allclose(gs.sum(1), 1.0, rtol=1e-14)
        assert np.all(gs > 0)
        if k == 1:
            np.testing.assert_array_equal(g, 1.0)
        gf = O.gate_values(s, idx, O.GATE_SOFTMAX_FULL)
        np.testing.assert_allclose(gf, np.take_along_axis(full, idx, 1), rtol=1e-13)


def check_router_probs():
    """Full distributions: softmax rows and normalised sigmoids sum to 1 and
    match hand values."""
    s = np.array([[2.0, 1.0, 0.0, -1.0]])
    p = O.router_probs(s, O.GATE_SOFTMAX_TOPK)
    z = math.exp(2) + math.exp(1) + 1 + math.exp(-1)
    np.testing.assert_allclose(p[0], [math.exp(v) / z for v in (2, 1, 0, -1)], rtol=1e-14)
    q = O.router_probs(s, O.GATE_SIGMOID_RENORM)
    sg = [1 / (1 + math.exp(-v)) for v in (2, 1, 0, -1)]
    np.testing.assert_allclose(q[0], [v / sum(sg) for v in sg], rtol=1e-14)


def check_selection_bias():
    """The bias changes which experts are chosen, never the gate values; a
    uniform shift of the bias changes nothing; a zero bias equals no bias."""
    s = np.array([[0.0, 0.1, 0.2]])
    b = np.array([0.5, 0.0, 0.0])
    sel = O.selection_scores(s, O.GATE_SIGMOID_RENORM, b)
    np.testing.assert_allclose(sel[0], [0.5 + 0.5, 1 / (1 + math.exp(-0.1)),
                                        1 / (1 + math.exp(-0.2))], rtol=1e-14)
    idx = O.topk_indices(sel, 2)
    assert idx[0].tolist() == [0, 2]
    g = O.gate_values(s, idx, O.GATE_SIGMOID_RENORM)
    a0, a2 = 0.5, 1 / (1 + math.exp(-0.2))
    np.testing.assert_allclose(g[0], [a0 / (a0 + a2), a2 / (a0 + a2)], rtol=1e-14)
    rng = _rng(4)
    s = rng.normal(size=(30, 8))
    b = rng.uniform(-0.05, 0.05, size=8)
    for mode in O.GATE_MODES:
        r0 = O.route(s[:, :8] @ np.eye(8), np.eye(8), 3, mode, sel_bias=b)
        r1 = O.route(s[:, :8] @ np.eye(8), np.eye(8), 3, mode, sel_bias=b + 0.37)
        np.testing.assert_array_equal(r0[2], r1[2])
        np.testing.assert_allclose(r0[3], r1[3], rtol=1e-14)
        rz = O.route(s, np.eye(8), 3, mode, sel_bias=np.zeros(8))
        rn = O.route(s, np.eye(8), 3, mode)
        np.testing.assert_array_equal(rz[2], rn[2])
        np.testing.assert_array_equal(rz[3], rn[3])
        # gates depend on the unbiased logits only
        np.testing.assert_allclose(r0[3], O.gate_values(s, r0[2], mode), rtol=1e-14)


# ---------------------------------------------------------------- stage 3
def check_capacity_formula():
    """C = ceil(k*T*rho/E): the Switch layer gives 80; ragged cases round up;
    no factor means no limit."""
    assert O.expert_capacity(4096, 1, 64, 1.25) == 80
    assert O.expert_capacity(10, 1, 3, 1.0) == 4
    assert O.expert_capacity(10, 2, 3, 1.0) == 7
    assert O.expert_capacity(7, 1, 8, 0.5) == 1
    assert O.expert_capacity(100, 1, 4, 0.0) is None
    assert O.expert_capacity(100, 1, 4, None) is None


def check_capacity_drops():
    """Top-1 drops equal sum_e max(0, routed_e - C) over a rho sweep 0.5..2.0
    (chapter 11, exercise 4); kept + drops = T*k; no drops once rho >= E/k;
    the kept assignments of each expert are its first C keys."""
    rng = _rng(5)
    T, E = 300, 6
    for k in (1, 2, 3):
        probs = rng.dirichlet([0.6] * E, size=T)
        idx = np.stack([rng.choice(E, size=k, replace=False, p=probs[t]) for t in range(T)])
        for rho in (0.5, 0.75, 1.0, 1.25, 1.5, 2.0, E / k):
            C = O.expert_capacity(T, k, E, rho)
            a = O.assign_slots(idx, E, C)
            counts = np.bincount(idx.ravel(), minlength=E)
            np.testing.assert_array_equal(a.routed, counts)
            drops = int(sum(max(0, int(c) - C) for c in counts))
            assert int(a.kept.sum()) == T * k - drops
            np.testing.assert_array_equal(a.kept, np.minimum(counts, C))
            if rho >= E / k:
                assert drops == 0
            # first come by token index: keys of expert e in key order
            for e in range(E):
                keys = [(t * k + j) for t in range(T) for j in range(k) if idx[t, j] == e]
                kept_keys = [(t * k + j) for t in range(T) for j in range(k)
                             if idx[t, j] == e and a.slot_pos[t, j] >= 0]
                assert kept_keys == keys[:C]


def check_offsets_and_permutation():
    """offsets are the exclusive scan of kept counts; every kept slot has a
    unique row inside its expert's segment; rows within a segment follow key
    order; the permutation round-trips."""
    rng = _rng(6)
    T, E, k = 97, 5, 2
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    for C in (None, 30, 7):
        a = O.assign_slots(idx, E, C)
        assert a.offsets[0] == 0
        np.testing.assert_array_equal(np.diff(a.offsets), a.kept)
        rows = O.permutation_rows(a, idx)
        assert np.all(rows >= 0)
        seen = set()
        for t in range(T):
            for j in range(k):
                r = a.slot_pos[t, j]
                if r < 0:
                    continue
                e = idx[t, j]
                assert a.offsets[e] <= r < a.offsets[e + 1]
                assert rows[r] == t
                seen.add(int(r))
        assert seen == set(range(int(a.offsets[-1])))
        for e in range(E):
            seg = rows[a.offsets[e]:a.offsets[e + 1]]
            assert np.all(np.diff(seg) > 0)   # one key per (token, expert); key order


# ---------------------------------------------------------------- stage 5/6
def _rand_layer(seed, T, d, E, f, swiglu):
    rng = _rng(seed)
    x = rng.normal(size=(T, d))
    W_r = rng.normal(size=(E, d)) / math.sqrt(d)
    W1 = rng.normal(size=(E, f, d)) / math.sqrt(d)
    W2 = rng.normal(size=(E, d, f)) / math.sqrt(f)
    W3 = rng.normal(size=(E, f, d)) / math.sqrt(d) if swiglu else None
    return x, W_r, W1, W2, W3


def _dense_reference(x, W_r, W1, W2, W3, k, act, mode, sel_bias=None, Ws=None):
    """Brute force: all E experts on every token, mixed by a dense gate vector
    that is zero outside the chosen set, written without the oracle's sparse
    loop; the expert itself is written out with torch.nn.functional."""
    s = x @ W_r.T
    sel = O.selection_scores(s, mode, sel_bias)
    idx = O.topk_indices(sel, k)
    g = O.gate_values(s, idx, mode)
    T, E = s.shape
    dense_g = np.zeros((T, E))
    for t in range(T):
        dense_g[t, idx[t]] = g[t]
    xt = torch.from_numpy(x)
    y = torch.zeros_like(xt)
    for e in range(E):
        a = F.linear(xt, torch.from_numpy(W1[e]))
        if act == O.ACT_GELU:
            h = F.gelu(a, approximate="none")
        elif act == O.ACT_RELU:
            h = F.relu(a)
        else:
            h = F.silu(a) * F.linear(xt, torch.from_numpy(W3[e]))
        y += torch.from_numpy(dense_g[:, e:e + 1]) * F.linear(h, torch.from_numpy(W2[e]))
    if Ws is not None:
        Ws1, Ws3, Ws2 = (torch.from_numpy(w) for w in Ws)
        y += F.linear(F.silu(F.linear(xt, Ws1)) * F.linear(xt, Ws3), Ws2)
    return y.numpy()


def check_sparse_equals_dense():
    """The sparse evaluation (only chosen experts run) equals the dense mixture
    with zero gates off the chosen set, for every activation and gate mode."""
    for n, (act, mode, k) in enumerate([
            (O.ACT_GELU, O.GATE_SOFTMAX_TOPK, 2),
            (O.ACT_RELU, O.GATE_SOFTMAX_FULL, 1),
            (O.ACT_SWIGLU, O.GATE_SIGMOID_RENORM, 3),
            (O.ACT_SWIGLU, O.GATE_SOFTMAX_TOPK, 6)]):
        T, d, E, f = 13, 8, 6, 12
        x, W_r, W1, W2, W3 = _rand_layer(10 + n, T, d, E, f, act == O.ACT_SWIGLU)
        b = _rng(20 + n).uniform(-0.05, 0.05, E) if mode == O.GATE_SIGMOID_RENORM else None
        r = O.moe_forward(x, W_r, W1, W2, k, act, mode, W3=W3, sel_bias=b)
        ref = _dense_reference(x, W_r, W1, W2, W3, k, act, mode, sel_bias=b)
        np.testing.assert_allclose(r.y, ref, rtol=1e-12, atol=1e-12)
    # with a shared SwiGLU expert added at weight 1
    T, d, E, f = 9, 8, 4, 10
    x, W_r, W1, W2, W3 = _rand_layer(40, T, d, E, f, True)
    rng = _rng(41)
    Ws = (rng.normal(size=(6, d)), rng.normal(size=(6, d)), rng.normal(size=(d, 6)))
    r = O.moe_forward(x, W_r, W1, W2, 2, O.ACT_SWIGLU, O.GATE_SOFTMAX_TOPK, W3=W3,
                      Ws1=Ws[0], Ws3=Ws[1], Ws2=Ws[2])
    ref = _dense_reference(x, W_r, W1, W2, W3, 2, O.ACT_SWIGLU, O.GATE_SOFTMAX_TOPK, Ws=Ws)
    np.testing.assert_allclose(r.y, ref, rtol=1e-12, atol=1e-12)



def check_shared_expert_outside_routing():
    """The shared expert is always on: it takes no part in routing (choices,
    gates, slots, f, P and L are those of the layer without it), it is
    outside capacity (a token whose every slot was dropped still gets its
    output) and it is added at weight 1 to every token, whatever its gates.
    Its output is written out with torch.nn.functional."""
    T, d, E, f, k = 12, 6, 3, 8, 2
    x, W_r, W1, W2, W3 = _rand_layer(42, T, d, E, f, True)
    rng = _rng(43)
    Ws = (rng.normal(size=(5, d)), rng.normal(size=(5, d)), rng.normal(size=(d, 5)))
    kw = dict(W3=W3, capacity_factor=0.3)            # C = ceil(24 * 0.3 / 3) = 3
    base = O.moe_forward(x, W_r, W1, W2, k, O.ACT_SWIGLU, O.GATE_SOFTMAX_TOPK, **kw)
    sh = O.moe_forward(x, W_r, W1, W2, k, O.ACT_SWIGLU, O.GATE_SOFTMAX_TOPK, **kw,
                       Ws1=Ws[0], Ws3=Ws[1], Ws2=Ws[2])
    assert sh.asg.capacity == 3
    np.testing.assert_array_equal(sh.topk_idx, base.topk_idx)
    np.testing.assert_array_equal(sh.topk_w, base.topk_w)
    np.testing.assert_array_equal(sh.asg.slot_pos, base.asg.slot_pos)
    np.testing.assert_array_equal(sh.asg.kept, base.asg.kept)
    np.testing.assert_array_equal(sh.f, base.f)
    np.testing.assert_array_equal(sh.P, base.P)
    assert sh.aux_loss == base.aux_loss
    xt = torch.from_numpy(x)
    Ws1, Ws3, Ws2 = (torch.from_numpy(w) for w in Ws)
    shared = F.linear(F.silu(F.linear(xt, Ws1)) * F.linear(xt, Ws3), Ws2).numpy()
    np.testing.assert_allclose(sh.y - base.y, shared, rtol=1e-12, atol=1e-12)
    all_dropped = np.all(sh.asg.slot_pos < 0, axis=1)
    partly = np.any(sh.asg.slot_pos < 0, axis=1) & ~all_dropped
    assert all_dropped.any() and partly.any()        # the case the reading is about
    np.testing.assert_allclose(sh.y[all_dropped], shared[all_dropped], rtol=1e-12, atol=1e-12)


def check_conditioning_and_token_sample():
    """Two evaluation modes the parity tests use.  (1) Conditioning on another
    implementation's choice: forcing the oracle's own choice changes nothing;
    forcing another choice gives that choice's gates, counts, slots and
    statistics.  (2) A token sample: y is evaluated for the sampled tokens
    only, but routing and capacity are those of the whole batch, so a sampled
    token that the batch drops stays dropped."""
    T, d, E, f, k = 16, 6, 3, 5, 2
    x, W_r, W1, W2, W3 = _rand_layer(44, T, d, E, f, True)
    kw = dict(W3=W3, capacity_factor=0.5)            # C = ceil(32 * 0.5 / 3) = 6
    full = O.moe_forward(x, W_r, W1, W2, k, O.ACT_SWIGLU, O.GATE_SOFTMAX_TOPK, **kw)
    same = O.moe_forward(x, W_r, W1, W2, k, O.ACT_SWIGLU, O.GATE_SOFTMAX_TOPK, **kw,
                         forced_idx=full.topk_idx)
    np.testing.assert_array_equal(same.y, full.y)
    np.testing.assert_array_equal(same.asg.slot_pos, full.asg.slot_pos)
    other = full.topk_idx.copy()
    other[1::2] = other[1::2, ::-1]                  # odd tokens: the two choices swapped
    other[0] = [(full.topk_idx[0, 0] + 1) % E, full.topk_idx[0, 0]]
    if other[0, 0] == other[0, 1]:
        raise AssertionError("test layer: need two distinct experts")
    forced = O.moe_forward(x, W_r, W1, W2, k, O.ACT_SWIGLU, O.GATE_SOFTMAX_TOPK, **kw,
                           forced_idx=other)
    np.testing.assert_array_equal(forced.topk_idx, other)
    np.testing.assert_array_equal(forced.asg.routed, np.bincount(other.ravel(), minlength=E))
    s = x @ W_r.T
    np.testing.assert_allclose(forced.topk_w, O.gate_values(s, other, O.GATE_SOFTMAX_TOPK),
                               rtol=1e-15)
    assert not np.array_equal(forced.asg.slot_pos, full.asg.slot_pos)
    dropped = np.nonzero(np.all(full.asg.slot_pos < 0, axis=1))[0]
    assert len(dropped) > 0
    sample = np.array([dropped[-1], 0, T - 1, 5])
    part = O.moe_forward(x, W_r, W1, W2, k, O.ACT_SWIGLU, O.GATE_SOFTMAX_TOPK, **kw,
                         tokens=sample)
    # the same sums over other groupings of the rows: equal to rounding
    np.testing.assert_allclose(part.y, full.y[sample], rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(part.y[0], 0.0)   # dropped by the batch, not by the sample
    np.testing.assert_array_equal(part.asg.slot_pos, full.asg.slot_pos)
    assert part.aux_loss == full.aux_loss

def check_drop_is_identity_branch():
    """A dropped slot contributes zero (the caller's residual carries the token);
    the surviving slot keeps its gate (no renormalisation)."""
    T, d, E, f, k = 8, 4, 2, 6, 2
    x, W_r, W1, W2, W3 = _rand_layer(50, T, d, E, f, False)
    full = O.moe_forward(x, W_r, W1, W2, k, O.ACT_RELU, O.GATE_SOFTMAX_TOPK)
    capped = O.moe_forward(x, W_r, W1, W2, k, O.ACT_RELU, O.GATE_SOFTMAX_TOPK,
                           capacity_factor=0.25)   # C = ceil(16*0.25/2) = 2
    assert capped.asg.capacity == 2
    for t in range(T):
        ref = np.zeros(d)
        for j in range(k):
            if capped.asg.slot_pos[t, j] >= 0:
                e = capped.topk_idx[t, j]
                ref += full.topk_w[t, j] * O.expert_ffn(x[t], W1[e], W2[e], O.ACT_RELU)
        np.testing.assert_allclose(capped.y[t], ref, rtol=1e-13, atol=1e-14)
    # tokens 0 and 1 fill both experts (k = E = 2): every later token is dropped
    assert np.all(capped.asg.slot_pos[2:] == -1)
    np.testing.assert_array_equal(capped.y[2:], 0.0)


def check_dense_ffn_special_case():
    """E = 1, k = 1, no capacity: the layer is one dense FFN (gate 1), checked
    against torch.nn.functional in float64 for GELU (erf), ReLU and SwiGLU."""
    rng = _rng(7)
    T, d, f = 11, 16, 24
    x = rng.normal(size=(T, d))
    W_r = rng.normal(size=(1, d))
    W1 = rng.normal(size=(1, f, d)) / 4
    W3 = rng.normal(size=(1, f, d)) / 4
    W2 = rng.normal(size=(1, d, f)) / 5
    xt = torch.from_numpy(x)
    for act in O.ACTS:
        r = O.moe_forward(x, W_r, W1, W2, 1, act, O.GATE_SOFTMAX_TOPK,
                          W3=W3 if act == O.ACT_SWIGLU else None)
        a = F.linear(xt, torch.from_numpy(W1[0]))
        if act == O.ACT_GELU:
            h = F.gelu(a, approximate="none")
        elif act == O.ACT_RELU:
            h = F.relu(a)
        else:
            h = F.silu(a) * F.linear(xt, torch.from_numpy(W3[0]))
        ref = F.linear(h, torch.from_numpy(W2[0])).numpy()
        np.testing.assert_allclose(r.y, ref, rtol=1e-12, atol=1e-13)


def check_elementwise_primitives():
    """The scalar maps of the stages against library routines in float64 and
    the identities they satisfy.  sigmoid: scipy's expit, sigma(z) + sigma(-z)
    = 1, sigma(0) = 1/2.  Row softmax: scipy's softmax, unchanged by a shift of
    its row, finite at |z| = 1000.  GELU (erf form) and SiLU: torch's, and
    both odd parts equal z, act(z) - act(-z) = z.  Affinity: the sigmoid of the
    logit in the sigmoid gate mode, the logit itself in the softmax modes."""
    from scipy import special
    z = np.linspace(-40.0, 40.0, 801)
    np.testing.assert_allclose(O.sigmoid(z), special.expit(z), rtol=1e-14, atol=0)
    np.testing.assert_allclose(O.sigmoid(z) + O.sigmoid(-z), 1.0, rtol=0, atol=4e-16)
    assert O.sigmoid(np.array([0.0]))[0] == 0.5
    rng = _rng(91)
    S = rng.normal(scale=4.0, size=(7, 13))
    np.testing.assert_allclose(O.softmax_rows(S), special.softmax(S, axis=-1), rtol=1e-13)
    shifted = S + 50.0 * rng.normal(size=(7, 1))
    np.testing.assert_allclose(O.softmax_rows(shifted), O.softmax_rows(S), rtol=1e-11)
    wide = np.array([[1000.0, 999.0, -1000.0]])
    got = O.softmax_rows(wide)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, special.softmax(wide, axis=-1), rtol=1e-14)
    u = np.linspace(-10.0, 10.0, 401)
    ut = torch.from_numpy(u)
    np.testing.assert_allclose(O.gelu_erf(u), F.gelu(ut, approximate="none").numpy(),
                               rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(O.silu(u), F.silu(ut).numpy(), rtol=1e-13, atol=1e-15)
    for act in (O.gelu_erf, O.silu):
        np.testing.assert_allclose(act(u) - act(-u), u, rtol=0, atol=1e-14)
        assert act(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(O.affinity(S, O.GATE_SIGMOID_RENORM), special.expit(S),
                               rtol=1e-14)
    for mode in (O.GATE_SOFTMAX_TOPK, O.GATE_SOFTMAX_FULL):
        assert np.array_equal(O.affinity(S, mode), S)
    try:
        O.affinity(S, "no such mode")
    except ValueError:
        pass
    else:
        raise AssertionError("an unknown gate mode must be refused")


def check_expert_ffn_rows_bruteforce():
    """One expert on n rows by explicit sums over every index, with torch's
    scalar activations (GELU erf form, ReLU, SiLU): f != d so a transposed
    operand cannot pass; each row is independent of the others; the multiply
    counter adds n*d*f per projection."""
    rng = _rng(92)
    n, d, f = 3, 4, 6
    X = rng.normal(size=(n, d))
    W1 = rng.normal(size=(f, d))
    W3 = rng.normal(size=(f, d))
    W2 = rng.normal(size=(d, f))
    scalar_act = {
        O.ACT_GELU: lambda a: float(F.gelu(torch.tensor(a, dtype=torch.float64),
                                           approximate="none")),
        O.ACT_RELU: lambda a: float(F.relu(torch.tensor(a, dtype=torch.float64))),
    }
    for act in O.ACTS:
        ref = np.zeros((n, d))
        for r in range(n):
            h = np.zeros(f)
            for i in range(f):
                a = sum(W1[i, c] * X[r, c] for c in range(d))
                if act == O.ACT_SWIGLU:
                    b = sum(W3[i, c] * X[r, c] for c in range(d))
                    h[i] = float(F.silu(torch.tensor(a, dtype=torch.float64))) * b
                else:
                    h[i] = scalar_act[act](a)
            for m in range(d):
                ref[r, m] = sum(W2[m, i] * h[i] for i in range(f))
        cnt = O.MultiplyCounter()
        got = O.expert_ffn_rows(X, W1, W2, act, W3=W3 if act == O.ACT_SWIGLU else None,
                                counter=cnt)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)
        assert cnt.count == n * d * f * (3 if act == O.ACT_SWIGLU else 2)
        for r in range(n):
            one = O.expert_ffn(X[r], W1, W2, act, W3=W3 if act == O.ACT_SWIGLU else None)
            np.testing.assert_allclose(one, ref[r], rtol=1e-12, atol=1e-13)


def check_multiply_counts():
    """Toy layer multiplies per token (page figure): 65,536 at top-2 and
    262,144 when all 8 experts fire; SwiGLU experts cost 3*d*f; the active
    fraction equals k/E (2/64 = 3.1%, 2/8 = 25%)."""
    g = read_golden("toy_multiplies.txt")
    acc = read_golden("expert_accounting.txt")
    E, d, f = g["experts"], g["d_model"], g["d_ffn"]
    assert 2 * d * f == g["weights_per_expert"]
    T = 4
    x, W_r, W1, W2, _ = _rand_layer(8, T, d, E, f, False)
    r2 = O.moe_forward(x, W_r, W1, W2, 2, O.ACT_GELU, O.GATE_SOFTMAX_TOPK, count_multiplies=True)
    assert r2.multiplies == T * g["multiplies_top2"]
    r8 = O.moe_forward(x, W_r, W1, W2, E, O.ACT_GELU, O.GATE_SOFTMAX_TOPK, count_multiplies=True)
    assert r8.multiplies == T * g["multiplies_all_fire"]
    assert g["multiplies_all_fire"] // g["multiplies_top2"] == 4
    # SwiGLU expert: 3*d*f multiplies per token; Mixtral shapes give ~5.6B per expert
    c = O.MultiplyCounter()
    dd, ff = 6, 10
    rng = _rng(9)
    O.expert_ffn(rng.normal(size=dd), rng.normal(size=(ff, dd)), rng.normal(size=(dd, ff)),
                 O.ACT_SWIGLU, rng.normal(size=(ff, dd)), c)
    assert c.count == 3 * dd * ff
    per_expert = 3 * acc["d_model"] * acc["d_ffn"] * acc["layers"]
    assert round(per_expert / 1e9, 1) == acc["per_expert_billions_rounded"]
    # active fraction k/E from the counter, E = 64 and E = 8 at k = 2
    for E_, pct in ((64, acc["active_fraction_percent_E64_k2"]), (8, acc["active_fraction_percent_E8_k2"])):
        x, W_r, W1, W2, _ = _rand_layer(11, 3, 4, E_, 4, False)
        rk = O.moe_forward(x, W_r, W1, W2, 2, O.ACT_RELU, O.GATE_SOFTMAX_TOPK, count_multiplies=True)
        rall = O.moe_forward(x, W_r, W1, W2, E_, O.ACT_RELU, O.GATE_SOFTMAX_TOPK, count_multiplies=True)
        assert round(100.0 * rk.multiplies / rall.multiplies, 1) == pct


def check_balance_uniform():
    """Uniform f and P give L = alpha exactly, for any N (the guide's 'Check
    yourself': N makes the minimum 1 independent of N).  Built as a cyclic
    layer: d = E, W_r = I, x_t = c * (e_{t mod E} + ... + e_{t+k-1 mod E})."""
    for E, k in ((4, 1), (8, 2), (6, 3), (16, 1)):
        T = 5 * E
        x = np.zeros((T, E))
        for t in range(T):
            for j in range(k):
                x[t, (t + j) % E] = 3.0
        r = O.moe_forward(x, np.eye(E), np.zeros((E, 2, E)), np.zeros((E, E, 2)), k,
                          O.ACT_RELU, O.GATE_SOFTMAX_TOPK, alpha=0.01)
        np.testing.assert_allclose(r.f, 1.0 / E, rtol=1e-14)
        np.testing.assert_allclose(r.P, 1.0 / E, rtol=1e-12)
        assert abs(r.aux_loss - 0.01) < 1e-14
        # sigmoid distribution, same symmetry
        r = O.moe_forward(x, np.eye(E), np.zeros((E, 2, E)), np.zeros((E, E, 2)), k,
                          O.ACT_RELU, O.GATE_SIGMOID_RENORM, alpha=1e-4)
        assert abs(r.aux_loss - 1e-4) < 1e-16


def check_balance_hand_and_collapse():
    """Hand-computed f, P, L for 4 tokens; collapsed routing costs more than
    balanced routing (chapter 11, exercise 3 and its demo)."""
    probs = np.array([[0.7, 0.2, 0.1], [0.1, 0.8, 0.1], [0.6, 0.3, 0.1], [0.2, 0.2, 0.6]])
    routed = np.array([2, 1, 1])
    f, P, L = O.balance_stats(routed, probs, T=4, k=1, alpha=0.01)
    np.testing.assert_allclose(f, [0.5, 0.25, 0.25], rtol=1e-15)
    np.testing.assert_allclose(P, [0.4, 0.375, 0.225], rtol=1e-14)
    assert abs(L - 0.01 * 3 * (0.5 * 0.4 + 0.25 * 0.375 + 0.25 * 0.225)) < 1e-16
    # k = 2: f divides by T*k
    f2, _, _ = O.balance_stats(np.array([3, 3, 2]), probs, T=4, k=2, alpha=0.01)
    np.testing.assert_allclose(f2, [3 / 8, 3 / 8, 2 / 8], rtol=1e-15)
    rng = _rng(0)
    E, T = 4, 100
    bal = rng.dirichlet([5.0] * E, size=T)
    col = rng.dirichlet([10.0, 0.1, 0.1, 0.1], size=T)
    Lb = O.balance_stats(np.bincount(bal.argmax(1), minlength=E), bal, T, 1, 0.01)[2]
    Lc = O.balance_stats(np.bincount(col.argmax(1), minlength=E), col, T, 1, 0.01)[2]
    assert Lc > Lb


def check_pipeline_stats_pre_drop():
    """In the full pipeline f counts assignments before drops (so sum f = 1
    even when capacity drops some), while kept counts drop."""
    T, d, E, f_, k = 40, 6, 4, 5, 2
    x, W_r, W1, W2, _ = _rand_layer(60, T, d, E, f_, False)
    off = np.array([2.0, 0.0, 0.0, -2.0])
    r = O.moe_forward(x, W_r, W1, W2, k, O.ACT_RELU, O.GATE_SOFTMAX_TOPK,
                      logit_offset=off, capacity_factor=1.0)
    assert int(r.asg.kept.sum()) < T * k
    np.testing.assert_allclose(r.f.sum(), 1.0, rtol=1e-15)
    np.testing.assert_allclose(r.f, r.asg.routed / (T * k), rtol=1e-15)
    np.testing.assert_allclose(r.P.sum(), 1.0, rtol=1e-14)


# ---------------------------------------------------------------- next rows
def check_z_loss_closed_forms():
    """Router z-loss, pinned to its reading (mean over tokens of the squared
    log-partition function): constant logits c give (c + ln E)^2; E = 1 gives
    the mean square of the logits; two experts give logaddexp; random rows
    agree with scipy's logsumexp; a per-token shift moves each term."""
    from scipy.special import logsumexp
    for E, c in ((1, 0.7), (4, 0.0), (64, -2.5), (256, 3.0)):
        s = np.full((5, E), c)
        assert abs(O.router_z_loss(s) - (c + math.log(E)) ** 2) < 1e-12 * max(1.0, (c + math.log(E)) ** 2)
    v = _rng(70).normal(size=(9, 1))
    assert abs(O.router_z_loss(v) - float(np.mean(v[:, 0] ** 2))) < 1e-14
    ab = _rng(71).normal(size=(7, 2)) * 4
    lse2 = np.logaddexp(ab[:, 0], ab[:, 1])
    assert abs(O.router_z_loss(ab) - float(np.mean(lse2 ** 2))) < 1e-13
    s = _rng(72).normal(size=(33, 17)) * 3
    ref = float(np.mean(logsumexp(s, axis=1) ** 2))
    assert abs(O.router_z_loss(s) - ref) < 1e-12 * ref
    shift = _rng(73).normal(size=(33, 1)) * 10
    ref_shift = float(np.mean((logsumexp(s, axis=1) + shift[:, 0]) ** 2))
    assert abs(O.router_z_loss(s + shift) - ref_shift) < 1e-12 * ref_shift
    # huge logits stay finite (the maximum is taken out first)
    big = np.array([[1000.0, 999.0, -1000.0]])
    assert abs(O.router_z_loss(big) - (1000.0 + math.log1p(math.exp(-1.0))) ** 2) < 1e-9
    assert O.router_z_loss(np.zeros((0, 8))) == 0.0


def check_bias_update_rule():
    """One balancing step of the per-expert selection bias (the guide's
    auxiliary-loss-free balancing): down by gamma above the mean load, up by
    gamma below it, unchanged at the mean; float32 state."""
    g = 0.25
    # T = 8, k = 1, E = 4: mean load 2
    np.testing.assert_array_equal(O.bias_update([0, 0, 0, 0], [5, 2, 1, 0], 8, 1, g),
                                  np.array([-0.25, 0.0, 0.25, 0.25], dtype=np.float32))
    # non-integer mean 4/3 (T = 4, k = 1, E = 3): nobody sits at the mean
    np.testing.assert_array_equal(O.bias_update([1, 1, 1], [2, 1, 1], 4, 1, g),
                                  np.array([0.75, 1.25, 1.25], dtype=np.float32))
    # k = 2 doubles the mean (T = 6, E = 4: mean 3)
    np.testing.assert_array_equal(O.bias_update([0, 0, 0, 0], [3, 4, 2, 3], 6, 2, g),
                                  np.array([0.0, -0.25, 0.25, 0.0], dtype=np.float32))
    # balanced loads keep every bias
    b0 = _rng(74).uniform(-0.05, 0.05, size=16).astype(np.float32)
    np.testing.assert_array_equal(O.bias_update(b0, [10] * 16, 40, 4, 1e-3), b0)
    # a collapsed router: n steps move the favourite down by n*gamma and the
    # rest up by n*gamma (exact in binary for gamma = 2^-6)
    b = np.zeros(8, dtype=np.float32)
    for _ in range(5):
        b = O.bias_update(b, [64, 0, 0, 0, 0, 0, 0, 0], 64, 1, 2.0 ** -6)
    np.testing.assert_array_equal(b, np.array([-5 / 64] + [5 / 64] * 7, dtype=np.float32))
    # float32 state: a step below half an ulp of 1.0 leaves 1.0
    assert O.bias_update([1.0, 1.0], [2, 0], 2, 1, 1e-8)[0] == np.float32(1.0)
    out = O.bias_update([0.1], [1], 2, 1, 0.3)   # E = 1, load 1 < mean 2
    assert out.dtype == np.float32 and out[0] == np.float32(np.float32(0.1) + np.float32(0.3))


# ---------------------------------------------------------------- fp8 variant
def check_e4m3_format():
    """e4m3 decoding and rounding against torch's float8_e4m3fn (a library
    routine) on all 256 codes and on sampled values, plus hand-checked ties."""
    codes = np.arange(256)
    ref = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    got = O.e4m3_decode(codes)
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[finite], ref[finite])
    rng = _rng(80)
    v = np.concatenate([rng.normal(size=20000) * rng.choice([1e-3, 0.05, 1.0, 30.0], 20000),
                        rng.uniform(-448, 448, 5000)]).astype(np.float32)
    r = O.e4m3_round(v)
    t = torch.tensor(v).to(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(r, t)
    # ties go to the even mantissa; subnormal spacing 2^-9; saturation at 448
    hand = {1.0625: 1.0, 1.1875: 1.25, 2.0 ** -10: 0.0, 3 * 2.0 ** -10: 2.0 ** -8,
            448.0: 448.0, 464.0: 448.0, 1000.0: 448.0, -0.6875: -0.6875, -0.71875: -0.75}
    for a, b in hand.items():
        assert O.e4m3_round(np.array([a]))[0] == b, (a, b)


def check_row_scale_rule():
    """The power-of-two row scale is the smallest with max|x| / s <= 448."""
    cases = {448.0: 0, 449.0: 1, 1.0: -8, 1.75: -8, 1.8: -7, 0.0: 0, 1e-40: -126,
             3.0e38: 120}
    for amax, e in cases.items():
        assert O.row_scale_exponent(amax) == e, (amax, e)
    for amax in _rng(81).lognormal(0.0, 6.0, size=2000):
        e = O.row_scale_exponent(amax)
        assert amax / 2.0 ** e <= 448.0 < amax / 2.0 ** (e - 1)
    vals, scales = O.quantize_rows_e4m3(np.array([[1.1, 0.5], [0.0, 0.0], [-448.0, 3.0]]))
    np.testing.assert_array_equal(scales, [2.0 ** -8, 1.0, 1.0])
    np.testing.assert_array_equal(vals, [[288.0, 128.0], [0.0, 0.0], [-448.0, 3.0]])


def check_fp8_layer():
    """The fp8 layer: a hand-computed one-expert case (the row 1.1, 0.5 is
    read as 1.125, 0.5), and rows that are already e4m3 values with max 448
    (scale 1: quantisation is the identity) reduce to the bf16 layer on the
    dequantised weights."""
    one = np.array([[[0x38, 0x00]]])          # e4m3 1.0 and 0.0
    r = O.moe_forward_fp8(np.array([[1.1, 0.5]]), np.ones((1, 2)), one, np.ones((1, 1)),
                          one, np.ones((1, 1)), np.ones((1, 2, 1)), 1, O.GATE_SOFTMAX_TOPK)
    g = 1.125
    assert abs(r.y[0, 0] - g * g / (1 + math.exp(-g))) < 1e-15
    assert abs(r.y[0, 1] - g * g / (1 + math.exp(-g))) < 1e-15
    rng = _rng(82)
    T, d, E, f, k = 12, 16, 4, 8, 2
    x = O.e4m3_decode(rng.integers(0, 0x7E, size=(T, d)))
    x[:, 0] = 448.0
    # codes of magnitudes 2^-5 .. 1 with either sign, small channel scales
    W1q = rng.integers(0x10, 0x38, size=(E, f, d)) | (rng.integers(0, 2, size=(E, f, d)) << 7)
    W3q = rng.integers(0x10, 0x38, size=(E, f, d))
    W1s = rng.uniform(1e-3, 2e-3, size=(E, f)).astype(np.float32)
    W3s = rng.uniform(1e-3, 2e-3, size=(E, f)).astype(np.float32)
    W2 = rng.normal(size=(E, d, f))
    W_r = rng.normal(size=(E, d))
    a = O.moe_forward_fp8(x, W_r, W1q, W1s, W3q, W3s, W2, k, O.GATE_SOFTMAX_TOPK)
    b = O.moe_forward(x, W_r, O.dequantize_weights(W1q, W1s), W2, k, O.ACT_SWIGLU,
                      O.GATE_SOFTMAX_TOPK, W3=O.dequantize_weights(W3q, W3s))
    np.testing.assert_array_equal(a.y, b.y)


def _e4m3_value_by_definition(code: int) -> float:
    """OCP e4m3 (fn): sign, 4 exponent bits with bias 7, 3 mantissa bits;
    exponent 0 is subnormal (2^-6 * m/8); 0x7F / 0xFF are NaN."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * 2.0 ** -6 * (m / 8.0)
    return sign * 2.0 ** (e - 7) * (1.0 + m / 8.0)


def check_fp8_down_weights():
    """e4m3 down weights: a hand-computed one-expert case (d = f = 2; the codes
    of the down matrix are 1, 1 / 4, 0 on two output channels with scales
    1/2 and 1/4: y = ((h0 + h1) / 2, h0)), and a square random case (d = f,
    so a scale applied along the wrong axis keeps the shapes) against weights
    decoded element by element from the e4m3 definition and scaled per output
    channel."""
    x = np.array([[1.1, 0.5]])
    W13 = np.array([[[0x38, 0x00], [0x00, 0x38]]])     # identity: gate = up = (1.125, 0.5)
    r = O.moe_forward_fp8(x, np.ones((1, 2)), W13, np.ones((1, 2)), W13, np.ones((1, 2)),
                          np.array([[[0x38, 0x38], [0x48, 0x00]]]), 1, O.GATE_SOFTMAX_TOPK,
                          W2s=np.array([[0.5, 0.25]], dtype=np.float32))
    h0, h1 = (g * g / (1 + math.exp(-g)) for g in (1.125, 0.5))
    assert abs(r.y[0, 0] - 0.5 * (h0 + h1)) < 1e-15 and abs(r.y[0, 1] - h0) < 1e-15
    rng = _rng(83)
    T, d, E, k = 10, 8, 3, 2
    f = d
    x = rng.normal(size=(T, d))
    W1q = rng.integers(0x10, 0x38, size=(E, f, d)) | (rng.integers(0, 2, size=(E, f, d)) << 7)
    W3q = rng.integers(0x10, 0x38, size=(E, f, d))
    W1s = rng.uniform(1e-2, 2e-2, size=(E, f)).astype(np.float32)
    W3s = rng.uniform(1e-2, 2e-2, size=(E, f)).astype(np.float32)
    W2q = rng.integers(0x00, 0x7F, size=(E, d, f)) | (rng.integers(0, 2, size=(E, d, f)) << 7)
    W2s = rng.uniform(0.5, 4.0, size=(E, d)).astype(np.float32)
    W2 = np.empty((E, d, f))
    for e in range(E):
        for n in range(d):
            for c in range(f):
                W2[e, n, c] = float(W2s[e, n]) * _e4m3_value_by_definition(int(W2q[e, n, c]))
    W_r = rng.normal(size=(E, d))
    a = O.moe_forward_fp8(x, W_r, W1q, W1s, W3q, W3s, W2q, k, O.GATE_SOFTMAX_TOPK, W2s=W2s)
    b = O.moe_forward_fp8(x, W_r, W1q, W1s, W3q, W3s, W2, k, O.GATE_SOFTMAX_TOPK)
    np.testing.assert_allclose(a.y, b.y, rtol=1e-13, atol=1e-13)


ALL_CHECKS = [
    check_router_onehot, check_topk_bruteforce, check_topk_ties, check_topk_gap, check_gates_closed_form,
    check_gates_invariants, check_router_probs, check_selection_bias,
    check_capacity_formula, check_capacity_drops, check_offsets_and_permutation,
    check_sparse_equals_dense, check_shared_expert_outside_routing,
    check_conditioning_and_token_sample,
    check_drop_is_identity_branch, check_dense_ffn_special_case,
    check_elementwise_primitives, check_expert_ffn_rows_bruteforce,
    check_multiply_counts, check_balance_uniform, check_balance_hand_and_collapse,
    check_pipeline_stats_pre_drop, check_z_loss_closed_forms, check_bias_update_rule,
    check_e4m3_format, check_row_scale_rule, check_fp8_layer, check_fp8_down_weights,
]
