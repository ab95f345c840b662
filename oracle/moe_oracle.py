"""Plain, slow CPU oracle for the forward pass of one sparse top-k MoE FFN layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` use it.  It shares no code, table or constant
with the CUDA path under ``sparse_mixture_experts_65_b300/``; the two meet
only through the seeded inputs that the tests hand to both.

Everything here is the plain definition written out in float64 numpy with the
loops the definition implies.  Inputs arrive as fp32 or bf16 values; the
upcast of either to float64 is exact.  Library primitives used as single
steps: ``numpy`` matrix-vector / matrix products (a plain inner product), and
``numpy.lexsort`` (a sort).

Sources (page title, then section):
  [MoE-ch11]   "Mixture of Experts" (llm-tutorial, chapter 11):
               § The mathematics; § Top-k routing: the gating function;
               § Top-1 vs top-2; § The auxiliary loss; § Expert capacity and
               dropped tokens; § Why MoE is hard (router precision, router
               z-loss); § Exercises.
  [MoE-guide]  "Mixture of experts" (inside-the-model guide, chapter 14):
               § The computation; § Auxiliary loss; § Fine-grained and shared
               experts; § Auxiliary-loss-free balancing; § Check yourself.
  [MoE-ch33]   "Chapter 33 — Mixture of Experts (MoE)": § The Router;
               § Load Balancing; § Simple MoE Layer Implementation.
  [MoE-visual] "Mixture-of-Experts" (neural networks visually, chapter 15):
               routing figure; § Show the math.
  [MoE-atlas]  "Mixture of experts (MoE)" (tech-atlas glossary entry).

Readings taken where the pages are silent or garbled (each one also appears,
with its reason, in the design notes of the repository):
  * top-k order: descending selection score, ties to the lower expert index;
  * capacity C = ceil(k*T*rho/E) evaluated in double, k*T first; rho <= 0
    means no limit; the drop test is "earlier keys routed to e" < C with the
    token-major key t*k + j (first come by token index);
  * f_i counts routed (pre-drop) assignments over T*k; P_i averages the full
    router distribution (softmax over all E, or sigmoid normalised over all E);
  * GELU is the exact erf form; SwiGLU is silu(W1 x) * (W3 x) then W2;
  * the shared expert is a SwiGLU expert added with weight 1, outside f/P and
    outside capacity;
  * a dropped slot contributes zero and the remaining gates are not
    renormalised; y is the MoE branch only (the caller adds the residual);
  * router z-loss: the ST-MoE form, mean over tokens of logsumexp(s_t)^2
    (the pages give no formula, so this function is pinned only to that
    reading: closed forms and a library logsumexp);
  * bias balancing step: load = routed count, overloaded iff
    routed_i * E > T * k, underloaded iff below, float32 state;
  * fp8 variant (not on the pages): e4m3 gate/up weights with per-channel
    scales, token rows quantised with a power-of-two scale (the smallest
    with max|x| / s <= 448), values rounded to nearest e4m3, ties to even.

Parity pins: every function below is pinned by ``tests/test_oracle_pins.py``
(brute force, closed forms, library special cases and page numbers under
``tests/golden/``).  What no page value fixes -- the absolute output values
for a given random seed -- is pinned only through those checks.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Optional

import numpy as np

GATE_SOFTMAX_TOPK = "softmax_topk"
GATE_SIGMOID_RENORM = "sigmoid_renorm"
GATE_SOFTMAX_FULL = "softmax_full"
GATE_MODES = (GATE_SOFTMAX_TOPK, GATE_SIGMOID_RENORM, GATE_SOFTMAX_FULL)

ACT_GELU = "gelu"
ACT_RELU = "relu"
ACT_SWIGLU = "swiglu"
ACTS = (ACT_GELU, ACT_RELU, ACT_SWIGLU)


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# Stage 1: router scores.
# [MoE-ch11] § The mathematics: the router W_r (N x d) gives one logit per
# expert, l = W_r x.  [MoE-guide] § The computation: s = W_r x.
# [MoE-ch33] § The Router: a bias-free linear map d_model -> n_experts.
# The optional per-expert logit offset o_e is added to every token's logits
# (a fixed skew of the router; it enters gates and P like any other logit).
# --------------------------------------------------------------------------
def router_logits(x, W_r, logit_offset=None) -> np.ndarray:
    """s[t, e] = sum_c x[t, c] * W_r[e, c] (+ o_e), float64.  x: [T, d], W_r: [E, d]."""
    x = _f64(x)
    W_r = _f64(W_r)
    s = x @ W_r.T
    if logit_offset is not None:
        s = s + _f64(logit_offset)[None, :]
    return s


def sigmoid(z) -> np.ndarray:
    z = _f64(z)
    return 1.0 / (1.0 + np.exp(-z))


def softmax_rows(z) -> np.ndarray:
    """Row softmax with the row maximum subtracted first ([MoE-ch11] demo code)."""
    z = _f64(z)
    m = z.max(axis=-1, keepdims=True)
    ez = np.exp(z - m)
    return ez / ez.sum(axis=-1, keepdims=True)


# --------------------------------------------------------------------------
# Stage 2: top-k selection and gates.
# [MoE-ch11] § Top-k routing: the k largest logits are kept; softmax is taken
# over only those k values, so the gates sum to 1 over the chosen experts.
# [MoE-ch11] § Top-1 vs top-2: a top-1 gate is the softmax probability of the
# chosen expert over all experts (or 1.0 in some variants).
# [MoE-guide] § The computation: gates are a softmax over the chosen scores
# or renormalised sigmoids.  [MoE-guide] § Auxiliary-loss-free balancing:
# a per-expert bias b_i is added to the affinity only when choosing experts;
# the gate values use the original affinity.
# --------------------------------------------------------------------------
def affinity(s, gate_mode: str) -> np.ndarray:
    """Affinity per (token, expert): the logit itself, or its sigmoid."""
    if gate_mode == GATE_SIGMOID_RENORM:
        return sigmoid(s)
    if gate_mode in (GATE_SOFTMAX_TOPK, GATE_SOFTMAX_FULL):
        return _f64(s)
    raise ValueError(gate_mode)


def selection_scores(s, gate_mode: str, sel_bias=None) -> np.ndarray:
    """sel = affinity + b (b only steers the choice, never the gate value)."""
    a = affinity(s, gate_mode)
    if sel_bias is not None:
        a = a + _f64(sel_bias)[None, :]
    return a


def topk_indices(sel, k: int) -> np.ndarray:
    """Indices of the k largest selection scores per row, in descending order;
    equal scores go to the lower expert index.  [T, E] -> int64 [T, k]."""
    sel = _f64(sel)
    T, E = sel.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    out = np.empty((T, k), dtype=np.int64)
    order_key = np.arange(E)
    for t in range(T):
        # lexsort: last key is primary -> by -sel ascending, then by index.
        perm = np.lexsort((order_key, -sel[t]))
        out[t] = perm[:k]
    return out


def topk_gap(sel, k: int) -> np.ndarray:
    """Per token: the smallest difference between neighbouring scores among its
    k+1 largest selection scores (all E of them when k == E); +inf when E == 1.

    The chosen list (which experts, and their descending order) of a token is
    decided by exactly those neighbouring comparisons: the k-th against the
    (k+1)-th decides the set, the pairs inside the first k decide the order.
    So if every score moves by less than half of this gap the list cannot
    change, while moving the closest pair toward each other by more than half
    of it swaps them.  A token whose gap lies below the near-tie band may
    therefore legitimately be routed differently by another, equally valid,
    rounding of its scores ([MoE-ch11] § Top-k routing: the k largest)."""
    sel = _f64(sel)
    T, E = sel.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    m = min(k + 1, E)
    gap = np.full(T, np.inf)
    for t in range(T):
        best = np.sort(sel[t])[::-1][:m]          # the m largest, descending
        for i in range(m - 1):
            gap[t] = min(gap[t], best[i] - best[i + 1])
    return gap


def near_tie_tokens(sel, k: int, band: float = 1e-5) -> np.ndarray:
    """Boolean [T]: tokens whose top-k list sits within `band` of a tie
    (topk_gap below the band).  Such tokens are counted and reported when two
    implementations route them differently."""
    return topk_gap(sel, k) < band


def gate_values(s, idx, gate_mode: str) -> np.ndarray:
    """Gate g[t, j] for chosen expert idx[t, j], from the unbiased logits s."""
    s = _f64(s)
    idx = np.asarray(idx)
    T, k = idx.shape
    g = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        chosen = s[t, idx[t]]
        if gate_mode == GATE_SOFTMAX_TOPK:
            m = chosen.max()
            e = np.exp(chosen - m)
            g[t] = e / e.sum()
        elif gate_mode == GATE_SIGMOID_RENORM:
            a = sigmoid(chosen)
            g[t] = a / a.sum()
        elif gate_mode == GATE_SOFTMAX_FULL:
            m = s[t].max()
            e_all = np.exp(s[t] - m)
            g[t] = np.exp(chosen - m) / e_all.sum()
        else:
            raise ValueError(gate_mode)
    return g


def router_probs(s, gate_mode: str) -> np.ndarray:
    """Full per-token router distribution over all E experts (for P_i):
    softmax of the logits, or sigmoid affinities normalised over all E."""
    if gate_mode == GATE_SIGMOID_RENORM:
        a = sigmoid(s)
        return a / a.sum(axis=1, keepdims=True)
    return softmax_rows(s)


# --------------------------------------------------------------------------
# Stage 3: expert capacity and drops.
# [MoE-ch11] § Expert capacity and dropped tokens: capacity is the fair share
# T/N scaled by rho; excess tokens skip the expert and pass on through the
# residual.  [MoE-guide] § Auxiliary loss: capacity = (tokens per batch / N) x
# capacity factor.  [MoE-ch11] § Exercises (exercise 4): drops per expert are
# max(0, count - capacity).
# --------------------------------------------------------------------------
def expert_capacity(T: int, k: int, E: int, capacity_factor: float) -> Optional[int]:
    """C = ceil(k*T*rho/E) in double precision (k*T formed first); None = no limit."""
    if capacity_factor is None or capacity_factor <= 0:
        return None
    return int(math.ceil((k * T) * float(capacity_factor) / E))


@dataclass
class Assignment:
    routed: np.ndarray          # [E] assignments per expert before drops
    kept: np.ndarray            # [E] assignments per expert after drops
    pos: np.ndarray             # [T, k] earlier keys routed to the same expert
    slot_pos: np.ndarray        # [T, k] row in expert-contiguous order, -1 = dropped
    offsets: np.ndarray         # [E+1] exclusive scan of kept
    capacity: Optional[int]


def assign_slots(idx, E: int, capacity: Optional[int]) -> Assignment:
    """Walk the keys t*k + j in increasing order.  An assignment to expert e is
    kept iff the number of earlier keys routed to e is below the capacity."""
    idx = np.asarray(idx)
    T, k = idx.shape
    routed = np.zeros(E, dtype=np.int64)
    kept = np.zeros(E, dtype=np.int64)
    pos = np.empty((T, k), dtype=np.int64)
    keep = np.empty((T, k), dtype=bool)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            p = int(routed[e])
            routed[e] += 1
            pos[t, j] = p
            if capacity is None or p < capacity:
                keep[t, j] = True
                kept[e] += 1
            else:
                keep[t, j] = False
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + kept[e]
    slot_pos = np.full((T, k), -1, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            if keep[t, j]:
                slot_pos[t, j] = offsets[int(idx[t, j])] + pos[t, j]
    return Assignment(routed, kept, pos, slot_pos, offsets, capacity)


def permutation_rows(asg: Assignment, idx) -> np.ndarray:
    """Stage 4 as data: row_token[r] = token whose copy sits at expert-contiguous
    row r (rows within one expert in increasing key order)."""
    idx = np.asarray(idx)
    T, k = idx.shape
    n = int(asg.offsets[-1])
    row_token = np.full(n, -1, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            r = asg.slot_pos[t, j]
            if r >= 0:
                row_token[r] = t
    return row_token


# --------------------------------------------------------------------------
# Stage 5: expert MLPs.
# [MoE-ch11] § The mathematics: an expert is a full FFN W2 sigma(W1 x), GeLU in
# most production transformers, ReLU in the demo; no biases in the demo code.
# [MoE-ch11] § Active vs total parameters and [MoE-ch33] § Simple MoE Layer
# Implementation: SwiGLU experts with gate W1, up W3, down W2.
# [MoE-guide] § Fine-grained and shared experts: shared experts run for every
# token.
# --------------------------------------------------------------------------
class MultiplyCounter:
    """Counts scalar multiplies performed by expert evaluations ([MoE-visual]
    routing figure: 65,536 per token at top-2 versus 262,144 if all fire)."""

    def __init__(self):
        self.count = 0


def gelu_erf(z) -> np.ndarray:
    z = _f64(z)
    erf = np.vectorize(math.erf, otypes=[np.float64])
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def silu(z) -> np.ndarray:
    z = _f64(z)
    return z * sigmoid(z)


def _matmul_rows(X, W, counter: Optional[MultiplyCounter]) -> np.ndarray:
    """Rows of X times W^T: each row is one token's matrix-vector product."""
    W = _f64(W)
    if counter is not None:
        counter.count += X.shape[0] * W.shape[0] * W.shape[1]
    return X @ W.T


def expert_ffn_rows(X, W1, W2, act: str, W3=None, counter: Optional[MultiplyCounter] = None) -> np.ndarray:
    """One expert applied to each row of X ([n, d]) independently.
    W1, W3: [f, d]; W2: [d, f].  Returns [n, d]."""
    X = _f64(X)
    a = _matmul_rows(X, W1, counter)
    if act == ACT_GELU:
        h = gelu_erf(a)
    elif act == ACT_RELU:
        h = np.maximum(a, 0.0)
    elif act == ACT_SWIGLU:
        if W3 is None:
            raise ValueError("SwiGLU needs W3")
        b = _matmul_rows(X, W3, counter)
        h = silu(a) * b
    else:
        raise ValueError(act)
    return _matmul_rows(h, W2, counter)


def expert_ffn(xt, W1, W2, act: str, W3=None, counter: Optional[MultiplyCounter] = None) -> np.ndarray:
    """One expert on one token.  W1, W3: [f, d]; W2: [d, f]; xt: [d]."""
    return expert_ffn_rows(_f64(xt)[None, :], W1, W2, act, W3, counter)[0]


# --------------------------------------------------------------------------
# Stage 6: combine and balance statistics.
# [MoE-ch11] § The mathematics / [MoE-guide] § The computation /
# [MoE-visual] § Show the math: y = sum over chosen i of g_i * Expert_i(x);
# unselected experts contribute exactly zero because they never run.
# [MoE-guide] § Auxiliary loss: L = alpha * N * sum_i f_i * P_i with f_i the
# fraction of tokens sent to i and P_i the average router probability of i.
# --------------------------------------------------------------------------
def balance_stats(routed, probs, T: int, k: int, alpha: float):
    """f_i = routed_i / (T*k); P_i = mean over tokens of probs[:, i];
    L = alpha * E * sum_i f_i * P_i.  Returns (f, P, L)."""
    routed = _f64(routed)
    probs = _f64(probs)
    E = routed.shape[0]
    if T == 0:
        return np.zeros(E), np.zeros(E), 0.0
    f = routed / float(T * k)
    P = probs.sum(axis=0) / float(T)
    L = float(alpha) * E * float(np.sum(f * P))
    return f, P, L


# [MoE-ch11] § Why MoE is hard: the router z-loss (from ST-MoE) penalises
# large router logits so that the softmax stays well conditioned.  The pages
# name it and its purpose but print no formula; the reading taken is the
# ST-MoE form, the batch mean of the squared log-partition function of each
# token's logits, without its coefficient:  z = (1/T) sum_t (log sum_e
# exp s_te)^2.  The logits are those the layer routes with (offset included).
# --------------------------------------------------------------------------
def router_z_loss(s) -> float:
    """z = mean over tokens of logsumexp(s_t)^2, in float64 with the row
    maximum taken out before the exponentials.  T = 0 gives 0."""
    s = _f64(s)
    T = s.shape[0]
    if T == 0:
        return 0.0
    z = 0.0
    for t in range(T):
        m = float(np.max(s[t]))
        lse = m + math.log(float(np.sum(np.exp(s[t] - m))))
        z += lse * lse
    return z / T


# [MoE-guide] § Auxiliary-loss-free balancing: every expert keeps a bias that
# only steers the choice; after each step it goes down by a small gamma for an
# overloaded expert and up by gamma for an underloaded one.  Readings (the
# pages fix neither): the load of expert i is its routed (pre-drop) count,
# "overloaded" means above the mean load T*k/E and "underloaded" below it,
# compared exactly as routed_i * E against T * k; an expert at the mean keeps
# its bias.  The bias is float32 state and each step is one float32 add.
# --------------------------------------------------------------------------
def bias_update(sel_bias, routed, T: int, k: int, gamma: float) -> np.ndarray:
    """The biases after one balancing step (float32 [E])."""
    b = np.array(sel_bias, dtype=np.float32, copy=True).reshape(-1)
    E = b.shape[0]
    g = np.float32(gamma)
    mean_scaled = int(T) * int(k)
    for i in range(E):
        load_scaled = int(routed[i]) * E
        if load_scaled > mean_scaled:
            b[i] = np.float32(b[i] - g)
        elif load_scaled < mean_scaled:
            b[i] = np.float32(b[i] + g)
    return b


# Variant with fp8 (e4m3) gate and up expert weights.  The pages use no 8-bit
# formats: this is the plain definition of that variant of the same layer.
# The weights arrive as e4m3 codes with one float32 scale per output channel
# (W[e][n][c] = scale[e][n] * e4m3(code[e][n][c])); every token row entering the
# up projection is quantised with a power-of-two scale s_t = 2^q, q the
# smallest integer (not below -126) with max|x_t| / 2^q <= 448 (s_t = 1 for an
# all-zero row), its values rounded to the nearest e4m3 value (ties to even);
# the products are then exact and summed in float64.  The down projection
# reads the same h as the bf16 layer.
# --------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Values of e4m3 codes (sign bit, 4 exponent bits with bias 7, 3 mantissa
    bits; exponent 0 is subnormal, m * 2^-9; code S.1111.111 is NaN)."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    man = (c & 0x7).astype(np.float64)
    val = np.where(ex == 0, man * 2.0 ** -9, (1.0 + man / 8.0) * np.exp2(ex - 7.0))
    val = np.where((ex == 15) & ((c & 0x7) == 7), np.nan, val)
    return sign * val


def e4m3_round(v) -> np.ndarray:
    """Nearest e4m3 value (ties to even), magnitudes above 448 saturated."""
    v = _f64(v)
    a = np.abs(v)
    _, q = np.frexp(a)                       # a = f * 2^q, f in [0.5, 1)
    # spacing of e4m3 values around a: 2^(exponent - 3) for normals
    # (|a| >= 2^-6), 2^-9 in the subnormal range
    quantum = np.where(a >= 2.0 ** -6, np.exp2(q - 1.0 - 3.0), 2.0 ** -9)
    r = np.rint(a / quantum) * quantum       # rint: half to even
    r = np.minimum(r, E4M3_MAX)
    return np.sign(v) * r


def row_scale_exponent(amax: float) -> int:
    """The q of s = 2^q: smallest integer >= -126 with amax / 2^q <= 448."""
    if not amax > 0.0:
        return 0
    f, q = math.frexp(float(amax))          # amax = f * 2^q, f in [0.5, 1)
    e = q - 9 + (1 if f > 0.875 else 0)     # 448 = 1.75 * 2^8
    return max(e, -126)


def quantize_rows_e4m3(X):
    """(values, scales): each row of X as e4m3 values times its power-of-two
    scale; values * scale[:, None] is the row the fp8 up projection reads."""
    X = _f64(X)
    scales = np.empty(X.shape[0])
    vals = np.empty_like(X)
    for t in range(X.shape[0]):
        s = 2.0 ** row_scale_exponent(float(np.max(np.abs(X[t]))) if X.shape[1] else 0.0)
        scales[t] = s
        vals[t] = e4m3_round(X[t] / s)
    return vals, scales


def dequantize_weights(codes, scales) -> np.ndarray:
    """[E, n, c] e4m3 codes and [E, n] float32 scales -> float64 weights."""
    return e4m3_decode(codes) * _f64(scales)[..., None]


def moe_forward_fp8(x, W_r, W1q, W1s, W3q, W3s, W2, k: int, gate_mode: str,
                    logit_offset=None, sel_bias=None, capacity_factor=None,
                    alpha: float = 0.01, tokens=None, forced_idx=None,
                    W2s=None) -> OracleResult:
    """The SwiGLU layer with e4m3 gate/up weights (codes + per-channel scales):
    routing on x, the up projection on the quantised rows of x.  With W2s
    given, W2 holds e4m3 codes [E, d, f] too and W2s [E, d] one scale per
    output channel: the down weights are those codes times their channel's
    scale (the activations h are not quantised)."""
    vals, scales = quantize_rows_e4m3(x)
    xq = vals * scales[:, None]
    W1 = dequantize_weights(W1q, W1s)
    W3 = dequantize_weights(W3q, W3s)
    if W2s is not None:
        W2 = dequantize_weights(W2, W2s)
    return moe_forward(x, W_r, W1, W2, k, ACT_SWIGLU, gate_mode, W3=W3,
                       logit_offset=logit_offset, sel_bias=sel_bias,
                       capacity_factor=capacity_factor, alpha=alpha, tokens=tokens,
                       forced_idx=forced_idx, x_experts=xq)


class _Indexable:
    """Per-expert weight access; lets callers stream experts lazily."""

    def __init__(self, arr):
        self.arr = arr

    def __getitem__(self, e):
        return self.arr[e]


@dataclass
class OracleResult:
    s: np.ndarray
    sel: np.ndarray
    topk_idx: np.ndarray
    topk_w: np.ndarray
    probs: np.ndarray
    gap: np.ndarray
    asg: Assignment
    f: np.ndarray
    P: np.ndarray
    aux_loss: float
    y: Optional[np.ndarray]            # [T, d], or rows for `tokens` only
    tokens: Optional[np.ndarray] = None
    multiplies: int = 0
    extras: dict = field(default_factory=dict)


def route(x, W_r, k: int, gate_mode: str, logit_offset=None, sel_bias=None,
          capacity_factor=None, alpha: float = 0.01, forced_idx=None):
    """Stages 1-3 and the balance statistics.  If forced_idx is given, the
    selection is taken from it instead of being computed (used to condition
    the later stages on another implementation's choice)."""
    s = router_logits(x, W_r, logit_offset)
    T, E = s.shape
    sel = selection_scores(s, gate_mode, sel_bias)
    idx = topk_indices(sel, k) if forced_idx is None else np.asarray(forced_idx, dtype=np.int64)
    g = gate_values(s, idx, gate_mode)
    probs = router_probs(s, gate_mode)
    cap = expert_capacity(T, k, E, capacity_factor)
    asg = assign_slots(idx, E, cap)
    f, P, L = balance_stats(asg.routed, probs, T, k, alpha)
    return s, sel, idx, g, probs, asg, f, P, L


def moe_forward(x, W_r, W1, W2, k: int, act: str, gate_mode: str, W3=None,
                logit_offset=None, sel_bias=None, capacity_factor=None,
                alpha: float = 0.01, Ws1=None, Ws3=None, Ws2=None,
                tokens=None, forced_idx=None, count_multiplies=False,
                x_experts=None) -> OracleResult:
    """The whole layer.  W1/W3/W2 may be arrays [E, ...] or any object whose
    [e] returns expert e's matrix.  tokens: optional subset of token indices for
    which y is evaluated (routing always runs on the whole batch, since capacity
    is a property of the whole batch).  x_experts: optional [T, d] rows that
    the routed experts read instead of x (the fp8 variant's quantised rows);
    routing always reads x."""
    x = _f64(x)
    xe = x if x_experts is None else _f64(x_experts)
    T = x.shape[0]
    s, sel, idx, g, probs, asg, f, P, L = route(
        x, W_r, k, gate_mode, logit_offset, sel_bias, capacity_factor, alpha, forced_idx)
    gap = topk_gap(sel, k)
    counter = MultiplyCounter() if count_multiplies else None
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    d = x.shape[1]
    y = np.zeros((len(tok), d), dtype=np.float64)
    W1i, W2i = _Indexable(W1), _Indexable(W2)
    W3i = _Indexable(W3) if W3 is not None else None
    # Group the kept (token, slot) pairs by expert so that lazily streamed
    # weights are fetched once per expert.
    work = {}
    for r, t in enumerate(tok):
        for j in range(k):
            if asg.slot_pos[t, j] >= 0:
                work.setdefault(int(idx[t, j]), []).append((r, int(t), j))
    for e in sorted(work):
        w1, w2 = W1i[e], W2i[e]
        w3 = W3i[e] if W3i is not None else None
        items = work[e]
        out = expert_ffn_rows(xe[[t for _, t, _ in items]], w1, w2, act, w3, counter)
        for i, (r, t, j) in enumerate(items):
            y[r] += g[t, j] * out[i]
    if Ws1 is not None and len(tok):
        y += expert_ffn_rows(x[tok], Ws1, Ws2, ACT_SWIGLU, Ws3, counter)
    return OracleResult(s=s, sel=sel, topk_idx=idx, topk_w=g, probs=probs, gap=gap,
                        asg=asg, f=f, P=P, aux_loss=L, y=y,
                        tokens=None if tokens is None else tok,
                        multiplies=counter.count if counter else 0)
