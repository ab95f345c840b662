"""Plant plausible mistakes in the CPU oracle and show that a pin catches each.

Every mutation below replaces one oracle function (on the CPU, for the
duration of one test) with a wrong variant: a dropped term, a wrong sign or
index, a transposed operand, a wrong rounding.  The named pin must then fail.
"""
import math

import numpy as np
import pytest

import oracle as O
import oracle.moe_oracle as M
import oracle_pins as P

_orig = {name: getattr(M, name) for name in (
    "router_logits", "topk_indices", "topk_gap", "gate_values", "affinity", "expert_capacity",
    "assign_slots", "gelu_erf", "silu", "expert_ffn_rows", "balance_stats", "router_probs",
    "softmax_rows", "router_z_loss", "bias_update", "e4m3_round", "row_scale_exponent",
    "quantize_rows_e4m3", "moe_forward_fp8", "sigmoid", "near_tie_tokens", "selection_scores",
    "permutation_rows", "e4m3_decode", "moe_forward", "route")}


def _router_reversed(x, W_r, logit_offset=None):
    return _orig["router_logits"](x, W_r, logit_offset)[:, ::-1]


def _router_offset_sign(x, W_r, logit_offset=None):
    s = _orig["router_logits"](x, W_r, None)
    return s if logit_offset is None else s - np.asarray(logit_offset)[None, :]


def _topk_ascending(sel, k):
    return _orig["topk_indices"](-np.asarray(sel, dtype=float), k)


def _topk_ties_high(sel, k):
    sel = np.asarray(sel, dtype=float)
    E = sel.shape[1]
    return (E - 1) - _orig["topk_indices"](sel[:, ::-1], k)


def _gap_k_plus_2(sel, k):
    sel = np.asarray(sel, dtype=float)
    if k + 1 >= sel.shape[1]:
        return _orig["topk_gap"](sel, k)
    return _orig["topk_gap"](sel, k + 1)          # one score too many in the window


def _gap_ascending(sel, k):
    return _orig["topk_gap"](-np.asarray(sel, dtype=float), k)   # the smallest scores


def _gap_set_boundary_only(sel, k):
    sel = np.asarray(sel, dtype=float)
    E = sel.shape[1]
    if k >= E:
        return np.full(sel.shape[0], np.inf)
    srt = -np.sort(-sel, axis=1)
    return srt[:, k - 1] - srt[:, k]              # ignores the order inside the set


def _gates_full_softmax(s, idx, mode):
    if mode == M.GATE_SOFTMAX_TOPK:
        mode = M.GATE_SOFTMAX_FULL
    return _orig["gate_values"](s, idx, mode)


def _gates_sigmoid_unnormalised(s, idx, mode):
    g = _orig["gate_values"](s, idx, mode)
    if mode == M.GATE_SIGMOID_RENORM:
        return M.sigmoid(np.take_along_axis(np.asarray(s, dtype=float), np.asarray(idx), 1))
    return g


def _affinity_no_sigmoid(s, mode):
    return np.asarray(s, dtype=float)


def _capacity_floor(T, k, E, rho):
    if rho is None or rho <= 0:
        return None
    return int(math.floor(k * T * rho / E))


def _capacity_no_k(T, k, E, rho):
    return _orig["expert_capacity"](T, 1, E, rho)


def _assign_last_come(idx, E, capacity):
    idx = np.asarray(idx)
    a = _orig["assign_slots"](idx[::-1, ::-1], E, capacity)
    a.slot_pos = a.slot_pos[::-1, ::-1]
    a.pos = a.pos[::-1, ::-1]
    return a


def _gelu_tanh(z):
    z = np.asarray(z, dtype=float)
    return 0.5 * z * (1 + np.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))


def _silu_plain_sigmoid(z):
    return M.sigmoid(z)


def _ffn_swiglu_no_up(X, W1, W2, act, W3=None, counter=None):
    if act == M.ACT_SWIGLU:
        W3 = np.asarray(W1, dtype=float)
    return _orig["expert_ffn_rows"](X, W1, W2, act, W3, counter)


def _ffn_swapped_gate_up(X, W1, W2, act, W3=None, counter=None):
    if act == M.ACT_SWIGLU:
        return _orig["expert_ffn_rows"](X, W3, W2, act, W1, counter)
    return _orig["expert_ffn_rows"](X, W1, W2, act, W3, counter)


def _ffn_transposed_down(X, W1, W2, act, W3=None, counter=None):
    W2 = np.asarray(W2, dtype=float)
    if W2.shape[0] == W2.shape[1]:
        W2 = W2.T
    else:
        W2 = W2[::-1]
    return _orig["expert_ffn_rows"](X, W1, W2, act, W3, counter)


def _balance_no_k(routed, probs, T, k, alpha):
    return _orig["balance_stats"](routed, probs, T, 1, alpha)


def _balance_no_E(routed, probs, T, k, alpha):
    f, P, L = _orig["balance_stats"](routed, probs, T, k, alpha)
    return f, P, L / len(np.asarray(routed))


def _probs_unnormalised_sigmoid(s, mode):
    if mode == M.GATE_SIGMOID_RENORM:
        return M.sigmoid(s)
    return _orig["router_probs"](s, mode)


def _softmax_no_shift_bug(z):
    z = np.asarray(z, dtype=float)
    return np.exp(z) / np.exp(z).sum(axis=-1, keepdims=True) * 1.0000001


def _z_no_square(s):
    s = np.asarray(s, dtype=float)
    if s.shape[0] == 0:
        return 0.0
    m = s.max(axis=1)
    return float(np.mean(m + np.log(np.exp(s - m[:, None]).sum(axis=1))))


def _z_no_max_term(s):
    s = np.asarray(s, dtype=float)
    if s.shape[0] == 0:
        return 0.0
    m = s.max(axis=1)
    return float(np.mean(np.log(np.exp(s - m[:, None]).sum(axis=1)) ** 2))


def _bias_sign_flipped(sel_bias, routed, T, k, gamma):
    return _orig["bias_update"](sel_bias, routed, T, k, -gamma)


def _bias_mean_ignores_k(sel_bias, routed, T, k, gamma):
    return _orig["bias_update"](sel_bias, routed, T, 1, gamma)


def _bias_float64_state(sel_bias, routed, T, k, gamma):
    b = np.array(sel_bias, dtype=np.float64)
    E = b.shape[0]
    for i in range(E):
        if routed[i] * E > T * k:
            b[i] -= gamma
        elif routed[i] * E < T * k:
            b[i] += gamma
    return b


def _e4m3_truncate(v):
    v = np.asarray(v, dtype=float)
    a = np.abs(v)
    _, q = np.frexp(a)
    quantum = np.where(a >= 2.0 ** -6, np.exp2(q - 4.0), 2.0 ** -9)
    return np.sign(v) * np.minimum(np.floor(a / quantum) * quantum, 448.0)


def _e4m3_ties_away(v):
    v = np.asarray(v, dtype=float)
    a = np.abs(v)
    _, q = np.frexp(a)
    quantum = np.where(a >= 2.0 ** -6, np.exp2(q - 4.0), 2.0 ** -9)
    return np.sign(v) * np.minimum(np.floor(a / quantum + 0.5) * quantum, 448.0)


def _scale_no_mantissa_check(amax):
    if not amax > 0.0:
        return 0
    _, q = math.frexp(float(amax))
    return max(q - 9, -126)


def _quantize_rows_unit_scale(X):
    X = np.asarray(X, dtype=float)
    return _orig["e4m3_round"](X), np.ones(X.shape[0])


def _fp8_layer_unquantised_rows(x, W_r, W1q, W1s, W3q, W3s, W2, k, gate_mode, **kw):
    return M.moe_forward(x, W_r, M.dequantize_weights(W1q, W1s), W2, k, M.ACT_SWIGLU, gate_mode,
                         W3=M.dequantize_weights(W3q, W3s), **kw)


def _fp8_down_scale_on_input_axis(x, W_r, W1q, W1s, W3q, W3s, W2, k, gate_mode, W2s=None,
                                  **kw):
    if W2s is not None:
        W2 = M.e4m3_decode(W2) * np.asarray(W2s, dtype=float)[:, None, :]
    return _orig["moe_forward_fp8"](x, W_r, W1q, W1s, W3q, W3s, W2, k, gate_mode, **kw)



def _sigmoid_sign_flipped(z):
    return 1.0 / (1.0 + np.exp(np.asarray(z, dtype=float)))


def _affinity_sigmoid_everywhere(s, mode):
    return _orig["sigmoid"](s)


def _near_tie_reversed(sel, k, band=1e-5):
    return M.topk_gap(sel, k) >= band


def _bias_subtracted(s, mode, sel_bias=None):
    a = M.affinity(s, mode)
    return a if sel_bias is None else a - np.asarray(sel_bias, dtype=float)[None, :]


def _rows_reverse_key_order(asg, idx):
    rows = _orig["permutation_rows"](asg, idx)
    for e in range(len(asg.offsets) - 1):
        lo, hi = int(asg.offsets[e]), int(asg.offsets[e + 1])
        rows[lo:hi] = rows[lo:hi][::-1]
    return rows


def _e4m3_bias_8(codes):
    return _orig["e4m3_decode"](codes) * 0.5


def _relu_dropped(X, W1, W2, act, W3=None, counter=None):
    if act != O.ACT_RELU:
        return _orig["expert_ffn_rows"](X, W1, W2, act, W3, counter)
    X = np.asarray(X, dtype=float)
    return (X @ np.asarray(W1, dtype=float).T) @ np.asarray(W2, dtype=float).T


def _shared_only_where_kept(x, W_r, W1, W2, k, act, gate_mode, Ws1=None, Ws3=None, Ws2=None,
                            **kw):
    r = _orig["moe_forward"](x, W_r, W1, W2, k, act, gate_mode, **kw)
    if Ws1 is not None:
        kept = np.any(r.asg.slot_pos >= 0, axis=1)
        sh = M.expert_ffn_rows(np.asarray(x, dtype=float), Ws1, Ws2, O.ACT_SWIGLU, Ws3)
        r.y[kept] += sh[kept]
    return r


def _shared_scaled_by_kept_gates(x, W_r, W1, W2, k, act, gate_mode, Ws1=None, Ws3=None,
                                 Ws2=None, **kw):
    r = _orig["moe_forward"](x, W_r, W1, W2, k, act, gate_mode, **kw)
    if Ws1 is not None:
        w = np.where(r.asg.slot_pos >= 0, r.topk_w, 0.0).sum(axis=1)
        sh = M.expert_ffn_rows(np.asarray(x, dtype=float), Ws1, Ws2, O.ACT_SWIGLU, Ws3)
        r.y += w[:, None] * sh
    return r


def _route_ignores_forced_choice(*args, forced_idx=None, **kw):
    return _orig["route"](*args[:8], **kw)   # the ninth positional argument is forced_idx


def _sample_routed_alone(x, W_r, W1, W2, k, act, gate_mode, tokens=None, **kw):
    if tokens is None:
        return _orig["moe_forward"](x, W_r, W1, W2, k, act, gate_mode, **kw)
    tok = np.asarray(tokens)
    return _orig["moe_forward"](np.asarray(x)[tok], W_r, W1, W2, k, act, gate_mode, **kw)

MUTATIONS = [
    ("router expert order reversed", "router_logits", _router_reversed, P.check_router_onehot),
    ("router offset sign flipped", "router_logits", _router_offset_sign, P.check_router_onehot),
    ("top-k takes the smallest", "topk_indices", _topk_ascending, P.check_topk_bruteforce),
    ("ties go to the higher index", "topk_indices", _topk_ties_high, P.check_topk_ties),
    ("near-tie window reaches the (k+2)-th score", "topk_gap", _gap_k_plus_2, P.check_topk_gap),
    ("near-tie gap over the smallest scores", "topk_gap", _gap_ascending, P.check_topk_gap),
    ("near-tie gap ignores the order inside the set", "topk_gap", _gap_set_boundary_only,
     P.check_topk_gap),
    ("top-k gates use the full softmax", "gate_values", _gates_full_softmax, P.check_gates_closed_form),
    ("sigmoid gates not renormalised", "gate_values", _gates_sigmoid_unnormalised, P.check_gates_invariants),
    ("sigmoid affinity dropped", "affinity", _affinity_no_sigmoid, P.check_selection_bias),
    ("capacity rounded down", "expert_capacity", _capacity_floor, P.check_capacity_formula),
    ("capacity ignores k", "expert_capacity", _capacity_no_k, P.check_capacity_formula),
    ("last come kept instead of first", "assign_slots", _assign_last_come, P.check_capacity_drops),
    ("GELU tanh approximation", "gelu_erf", _gelu_tanh, P.check_dense_ffn_special_case),
    ("SiLU without the z factor", "silu", _silu_plain_sigmoid, P.check_dense_ffn_special_case),
    ("SwiGLU up projection replaced", "expert_ffn_rows", _ffn_swiglu_no_up, P.check_sparse_equals_dense),
    ("SwiGLU gate and up swapped", "expert_ffn_rows", _ffn_swapped_gate_up, P.check_dense_ffn_special_case),
    ("down projection transposed", "expert_ffn_rows", _ffn_transposed_down, P.check_sparse_equals_dense),
    ("f divides by T, not T*k", "balance_stats", _balance_no_k, P.check_balance_uniform),
    ("loss misses the factor N", "balance_stats", _balance_no_E, P.check_balance_uniform),
    ("sigmoid P not normalised", "router_probs", _probs_unnormalised_sigmoid, P.check_router_probs),
    ("softmax scaled wrongly", "softmax_rows", _softmax_no_shift_bug, P.check_gates_invariants),
    ("z-loss without the square", "router_z_loss", _z_no_square, P.check_z_loss_closed_forms),
    ("z-loss drops the row maximum", "router_z_loss", _z_no_max_term, P.check_z_loss_closed_forms),
    ("bias step has the wrong sign", "bias_update", _bias_sign_flipped, P.check_bias_update_rule),
    ("bias mean load ignores k", "bias_update", _bias_mean_ignores_k, P.check_bias_update_rule),
    ("bias state kept in float64", "bias_update", _bias_float64_state, P.check_bias_update_rule),
    ("e4m3 truncates", "e4m3_round", _e4m3_truncate, P.check_e4m3_format),
    ("e4m3 ties away from zero", "e4m3_round", _e4m3_ties_away, P.check_e4m3_format),
    ("row scale ignores the mantissa", "row_scale_exponent", _scale_no_mantissa_check,
     P.check_row_scale_rule),
    ("rows quantised without a scale", "quantize_rows_e4m3", _quantize_rows_unit_scale,
     P.check_row_scale_rule),
    ("fp8 layer skips the row quantisation", "moe_forward_fp8", _fp8_layer_unquantised_rows,
     P.check_fp8_layer),
    ("fp8 down scales along the input axis", "moe_forward_fp8", _fp8_down_scale_on_input_axis,
     P.check_fp8_down_weights),
    ("sigmoid sign flipped", "sigmoid", _sigmoid_sign_flipped, P.check_elementwise_primitives),
    ("sigmoid affinity in the softmax modes", "affinity", _affinity_sigmoid_everywhere,
     P.check_elementwise_primitives),
    ("near-tie test reversed", "near_tie_tokens", _near_tie_reversed, P.check_topk_gap),
    ("selection bias subtracted", "selection_scores", _bias_subtracted, P.check_selection_bias),
    ("rows inside an expert in reverse key order", "permutation_rows", _rows_reverse_key_order,
     P.check_offsets_and_permutation),
    ("e4m3 exponent bias 8", "e4m3_decode", _e4m3_bias_8, P.check_e4m3_format),
    ("ReLU dropped from the expert", "expert_ffn_rows", _relu_dropped,
     P.check_expert_ffn_rows_bruteforce),
    ("shared expert only for tokens with a kept slot", "moe_forward", _shared_only_where_kept,
     P.check_shared_expert_outside_routing),
    ("shared expert scaled by the kept gates", "moe_forward", _shared_scaled_by_kept_gates,
     P.check_shared_expert_outside_routing),
    ("forced choice ignored", "route", _route_ignores_forced_choice,
     P.check_conditioning_and_token_sample),
    ("sampled tokens routed on their own", "moe_forward", _sample_routed_alone,
     P.check_conditioning_and_token_sample),
]


@pytest.mark.parametrize("name,attr,bad,check", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pin_catches_mutation(monkeypatch, name, attr, bad, check):
    check()  # passes on the real oracle
    monkeypatch.setattr(M, attr, bad)
    with pytest.raises(AssertionError):
        check()
