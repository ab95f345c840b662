"""Seeded synthetic workloads for the MoE layer: shapes, modes and input draws.

This module holds no arithmetic of the method.  It only names the layer
shapes (taken from the models the MoE pages describe) and draws seeded random
tensors with the stated distributions.  Both the CUDA path and the CPU oracle
receive the very same tensors from here.

Distribution convention: N(mu, v) names a normal with VARIANCE v, so weights
drawn "N(0, 1/fan_in)" have standard deviation 1/sqrt(fan_in) and the Switch
logit skew "N(0, 1.5)" has standard deviation sqrt(1.5).

Seeds: tensor number i of workload number c uses a generator seeded with
1000*c + i (+ the caller's extra seed), drawn in the fixed order below.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

ACT_GELU, ACT_RELU, ACT_SWIGLU = "gelu", "relu", "swiglu"
GATE_SOFTMAX_TOPK, GATE_SIGMOID_RENORM, GATE_SOFTMAX_FULL = (
    "softmax_topk", "sigmoid_renorm", "softmax_full")


@dataclass(frozen=True)
class LayerShape:
    name: str
    cid: int                    # workload number (seed base)
    T: int                      # tokens in the batch
    d: int                      # model width
    E: int                      # routed experts
    k: int                      # experts per token
    f: int                      # routed expert width
    act: str
    gate: str
    dtype: str                  # "f32" or "bf16"
    capacity_factor: float = 0.0        # <= 0: no capacity limit
    alpha: float = 0.01
    n_shared: int = 0
    f_shared: int = 0
    logit_offset_var: float = 0.0       # variance of a per-expert logit skew
    sel_bias_halfwidth: float = 0.0     # sel bias ~ U(-h, h)
    w_fp8: bool = False                 # gate/up expert weights as e4m3 codes + channel scales
    w2_fp8: bool = False                # down expert weights as e4m3 codes + channel scales too

    def with_T(self, T: int) -> "LayerShape":
        return replace(self, T=T)


# The layer shapes of the models the pages discuss.
TOY = LayerShape("toy", 0, T=256, d=64, E=8, k=2, f=256, act=ACT_GELU,
                 gate=GATE_SOFTMAX_TOPK, dtype="f32", alpha=0.01)
SWITCH = LayerShape("switch", 1, T=4096, d=768, E=64, k=1, f=3072, act=ACT_RELU,
                    gate=GATE_SOFTMAX_FULL, dtype="bf16", capacity_factor=1.25,
                    alpha=0.01, logit_offset_var=1.5)
MIXTRAL = LayerShape("mixtral", 2, T=8192, d=4096, E=8, k=2, f=14336, act=ACT_SWIGLU,
                     gate=GATE_SOFTMAX_TOPK, dtype="bf16", alpha=0.01)
DSV3 = LayerShape("dsv3", 3, T=4096, d=7168, E=256, k=8, f=2048, act=ACT_SWIGLU,
                  gate=GATE_SIGMOID_RENORM, dtype="bf16", alpha=1e-4,
                  n_shared=1, f_shared=2048, sel_bias_halfwidth=0.05)
GPTOSS = LayerShape("gptoss", 4, T=256, d=2880, E=128, k=4, f=2880, act=ACT_SWIGLU,
                    gate=GATE_SOFTMAX_TOPK, dtype="bf16", alpha=0.01)
GPTOSS_SWEEP_T = (1, 16, 64, 256)

WORKLOADS = {w.name: w for w in (TOY, SWITCH, MIXTRAL, DSV3, GPTOSS)}


def get(name: str) -> LayerShape:
    """A named workload; the suffix "_fp8" gives the same layer with e4m3
    gate/up expert weights (SwiGLU layers), "_fp8all" with e4m3 down expert
    weights as well."""
    if name.endswith("_fp8all"):
        base = get(name[:-len("_fp8all")])
        return replace(base, name=base.name + "_fp8all", w_fp8=True, w2_fp8=True)
    if name.endswith("_fp8"):
        base = get(name[:-len("_fp8")])
        return replace(base, name=base.name + "_fp8", w_fp8=True)
    if name.startswith("gptoss") and name != "gptoss":
        return GPTOSS.with_T(int(name[len("gptoss"):].lstrip("_T")))
    if name == "dsv3_e32":
        # the DeepSeek-V3-shaped layer with 32 routed experts and T = 640 (160
        # rows per expert on average against the full layer's 128, 2 GB of
        # weights): a case small enough for multi-pass counter captures of the
        # same kernels
        return replace(DSV3, name="dsv3_e32", T=640, E=32)
    return WORKLOADS[name]


def torch_dtype(shape: LayerShape) -> torch.dtype:
    return torch.float32 if shape.dtype == "f32" else torch.bfloat16


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device, dtype, chunk_dim0=False):
    """std * N(0,1) drawn in fp32 and rounded once to `dtype`.  With
    chunk_dim0 the leading dimension is drawn slice by slice (same stream)."""
    if not chunk_dim0:
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        return (t * std).to(dtype)
    out = torch.empty(shape, device=device, dtype=dtype)
    for i in range(shape[0]):
        t = torch.randn(shape[1:], generator=g, device=device, dtype=torch.float32)
        out[i] = (t * std).to(dtype)
    return out


@dataclass
class LayerInputs:
    shape: LayerShape
    x: torch.Tensor                      # [T, d]
    W_r: torch.Tensor                    # [E, d]
    W1: torch.Tensor                     # [E, f, d]
    W2: torch.Tensor                     # [E, d, f]
    W3: Optional[torch.Tensor] = None    # [E, f, d] (SwiGLU only)
    logit_offset: Optional[torch.Tensor] = None   # [E] fp32
    sel_bias: Optional[torch.Tensor] = None       # [E] fp32
    Ws1: Optional[torch.Tensor] = None   # [f_s, d]
    Ws3: Optional[torch.Tensor] = None   # [f_s, d]
    Ws2: Optional[torch.Tensor] = None   # [d, f_s]
    # e4m3 gate/up weights (W1, W3 are None then): codes [E, f, d] uint8 and
    # one float32 scale per output channel [E, f]
    W1q: Optional[torch.Tensor] = None
    W1s: Optional[torch.Tensor] = None
    W3q: Optional[torch.Tensor] = None
    W3s: Optional[torch.Tensor] = None
    # e4m3 down weights (W2 is None then): codes [E, d, f] uint8 and one
    # float32 scale per output channel [E, d]
    W2q: Optional[torch.Tensor] = None
    W2s: Optional[torch.Tensor] = None

    def weight_bytes(self) -> int:
        n = 0
        for t in (self.W_r, self.W1, self.W2, self.W3, self.Ws1, self.Ws3, self.Ws2, self.W1q,
                  self.W1s, self.W3q, self.W3s, self.W2q, self.W2s):
            if t is not None:
                n += t.numel() * t.element_size()
        return n


def _fp8_channels(shape3, std, g, device):
    """std * N(0,1) drawn in fp32 (slice by slice, the stream of _normal with
    chunk_dim0), then stored per output channel (row) as e4m3 codes and a
    float32 scale amax / 448, the codes rounded to nearest by torch's float8
    conversion: input preparation, not the layer's arithmetic."""
    E, n, c = shape3
    codes = torch.empty(shape3, device=device, dtype=torch.uint8)
    scales = torch.empty((E, n), device=device, dtype=torch.float32)
    for i in range(E):
        w = torch.randn((n, c), generator=g, device=device, dtype=torch.float32) * std
        s = w.abs().amax(dim=1).clamp_min(1e-30) / 448.0
        scales[i] = s
        codes[i] = (w / s[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scales


def make_x(shape: LayerShape, device="cpu", seed: int = 0) -> torch.Tensor:
    """Activations only: x ~ N(0, 1), [T, d]."""
    base = 1000 * shape.cid + seed * 100003
    return _normal((shape.T, shape.d), 1.0, _gen(device, base + 0), device, torch_dtype(shape))


def make_inputs(shape: LayerShape, device="cpu", seed: int = 0) -> LayerInputs:
    """All tensors of one layer: x ~ N(0,1); W_r ~ N(0, 1/d); W1, W3 ~ N(0, 1/d);
    W2 ~ N(0, 1/f); shared weights likewise; optional logit skew ~ N(0, v) and
    selection bias ~ U(-h, h) in fp32."""
    dt = torch_dtype(shape)
    base = 1000 * shape.cid + seed * 100003
    T, d, E, f = shape.T, shape.d, shape.E, shape.f
    big = E * f * d > (1 << 26)
    x = make_x(shape, device, seed)
    W_r = _normal((E, d), 1.0 / math.sqrt(d), _gen(device, base + 1), device, dt)
    W1 = W3 = W1q = W1s = W3q = W3s = None
    if shape.w_fp8:
        W1q, W1s = _fp8_channels((E, f, d), 1.0 / math.sqrt(d), _gen(device, base + 2), device)
    else:
        W1 = _normal((E, f, d), 1.0 / math.sqrt(d), _gen(device, base + 2), device, dt, big)
    W2 = W2q = W2s = None
    if shape.w2_fp8:
        W2q, W2s = _fp8_channels((E, d, f), 1.0 / math.sqrt(f), _gen(device, base + 3), device)
    else:
        W2 = _normal((E, d, f), 1.0 / math.sqrt(f), _gen(device, base + 3), device, dt, big)
    if shape.act == ACT_SWIGLU and shape.w_fp8:
        W3q, W3s = _fp8_channels((E, f, d), 1.0 / math.sqrt(d), _gen(device, base + 4), device)
    elif shape.act == ACT_SWIGLU:
        W3 = _normal((E, f, d), 1.0 / math.sqrt(d), _gen(device, base + 4), device, dt, big)
    logit_offset = None
    if shape.logit_offset_var > 0:
        logit_offset = torch.randn(E, generator=_gen(device, base + 5), device=device,
                                   dtype=torch.float32) * math.sqrt(shape.logit_offset_var)
    sel_bias = None
    if shape.sel_bias_halfwidth > 0:
        u = torch.rand(E, generator=_gen(device, base + 6), device=device, dtype=torch.float32)
        sel_bias = (u * 2.0 - 1.0) * shape.sel_bias_halfwidth
    Ws1 = Ws3 = Ws2 = None
    if shape.n_shared:
        fs = shape.f_shared
        Ws1 = _normal((fs, d), 1.0 / math.sqrt(d), _gen(device, base + 7), device, dt)
        Ws3 = _normal((fs, d), 1.0 / math.sqrt(d), _gen(device, base + 8), device, dt)
        Ws2 = _normal((d, fs), 1.0 / math.sqrt(fs), _gen(device, base + 9), device, dt)
    return LayerInputs(shape, x, W_r, W1, W2, W3, logit_offset, sel_bias, Ws1, Ws3, Ws2,
                       W1q, W1s, W3q, W3s, W2q, W2s)


def make_logits(T: int, E: int, seed: int, scale: float = 1.0, shift: float = 0.0,
                device="cpu") -> torch.Tensor:
    """Router-logit-shaped float32 [T, E]: scale * N(0, 1) + shift."""
    g = _gen(device, 7_000_003 + seed)
    return torch.randn((T, E), generator=g, device=device, dtype=torch.float32) * scale + shift


def make_routed_counts(E: int, T: int, k: int, seed: int, skew: float = 1.0,
                       device="cpu") -> torch.Tensor:
    """Per-expert routed counts int32 [E] summing to T*k: the T*k assignments
    are dealt by a seeded multinomial over E experts with weights exp(skew * N(0,1)).
    When E divides T*k, every third expert is then set to the exact mean load
    where the last expert can absorb the difference (so the 'at the mean' case
    occurs); the total stays T*k."""
    g = _gen("cpu", 8_000_009 + seed)
    w = torch.exp(skew * torch.randn(E, generator=g, dtype=torch.float64))
    counts = torch.zeros(E, dtype=torch.int64)
    if T * k > 0:
        draws = torch.multinomial(w, T * k, replacement=True, generator=g)
        counts = torch.bincount(draws, minlength=E)
    if E > 1 and (T * k) % E == 0:
        mean = (T * k) // E
        for i in range(0, E - 1, 3):
            delta = int(counts[i]) - mean
            if int(counts[E - 1]) + delta >= 0:   # the last expert absorbs the difference
                counts[i] = mean
                counts[E - 1] += delta
    return counts.to(torch.int32).to(device)
