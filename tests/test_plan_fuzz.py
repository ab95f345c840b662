"""The library's host-side planning over many layer descriptions (no GPU).

Every call first plans the layer on the host: argument checks, the kernel
path, tile widths and the workspace layout.  Random configurations, valid
and invalid, must never crash that code; they must come back with a
documented status; and the path it picks must respect the documented limits
of each routing kernel (include/moe.h, moe_plan_flags).
"""
import ctypes
import math

from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

from sparse_mixture_experts_65_b300 import _native as N
from sparse_mixture_experts_65_b300 import layer as L

ROUTE_BITS = (N.MOE_PLAN_ROUTE_ONE_LAUNCH | N.MOE_PLAN_ROUTE_CLUSTER | N.MOE_PLAN_ROUTE_DECODE)
CODES = {N.MOE_OK, N.MOE_ERR_ARG, N.MOE_ERR_UNSUPPORTED}
SETTINGS = settings(max_examples=400, derandomize=True, deadline=None,
                    suppress_health_check=[HealthCheck.too_slow])


def _cfg(T, d, E, k, f, n_shared, f_shared, dtype, act, gate, rho, reserved=0, alpha=0.01):
    return N.MoeConfig(T=T, d=d, E=E, k=k, f=f, n_shared=n_shared, f_shared=f_shared,
                       dtype=dtype, act=act, gate=gate, capacity_factor=rho, alpha=alpha,
                       reserved=reserved)


def _query(cfg):
    lib = N.lib()
    out = {}
    for name, fn, val in (("ws", lib.moe_workspace_size, ctypes.c_size_t),
                          ("ws_route", lib.moe_route_workspace_size, ctypes.c_size_t),
                          ("ws_hio", lib.moe_host_io_workspace_size, ctypes.c_size_t),
                          ("ws_fp8", lib.moe_workspace_size_fp8, ctypes.c_size_t),
                          ("flags", lib.moe_plan_flags, ctypes.c_uint32),
                          ("flags_fp8", lib.moe_plan_flags_fp8, ctypes.c_uint32),
                          ("launches", lib.moe_launch_count, ctypes.c_int32),
                          ("launches_fp8", lib.moe_launch_count_fp8, ctypes.c_int32)):
        v = val(0)
        rc = fn(ctypes.byref(cfg), ctypes.byref(v))
        assert rc in CODES, (name, rc)
        out[name] = (rc, v.value)
    return out


# valid-looking layers: sizes the kernels take (multiples of 8 / 16), all modes
valid_layers = st.builds(
    lambda T, d8, E, kf, f8, sh, fs8, dt, act, gate, rho: _cfg(
        T, 8 * d8, E, max(1, min(E, 32, int(kf * E) or 1)), 16 * f8, sh, 16 * fs8 if sh else 0,
        dt, act, gate, rho),
    st.integers(0, 70000), st.integers(1, 1024), st.integers(1, 512), st.floats(0, 1),
    st.integers(1, 1024), st.integers(0, 1), st.integers(1, 256),
    st.sampled_from([N.MOE_F32, N.MOE_BF16]),
    st.sampled_from([N.MOE_ACT_GELU, N.MOE_ACT_RELU, N.MOE_ACT_SWIGLU]),
    st.sampled_from([N.MOE_GATE_SOFTMAX_TOPK, N.MOE_GATE_SIGMOID_RENORM,
                     N.MOE_GATE_SOFTMAX_FULL]),
    st.sampled_from([0.0, -1.0, 0.05, 1.0, 1.25, 2.0, 1e9]))


@SETTINGS
@given(valid_layers)
def test_valid_layers_plan_within_the_documented_limits(cfg):
    q = _query(cfg)
    rc, ws = q["ws"]
    if cfg.dtype == N.MOE_BF16 and cfg.n_shared and cfg.act != N.MOE_ACT_SWIGLU:
        assert rc == N.MOE_ERR_UNSUPPORTED     # a bf16 shared expert needs SwiGLU experts
        return
    assert rc == N.MOE_OK, rc
    assert ws >= 4096 and ws % 256 == 0        # header, 256-byte regions
    rc_r, ws_r = q["ws_route"]
    assert rc_r == N.MOE_OK and 4096 <= ws_r <= ws
    rc_h, ws_h = q["ws_hio"]
    assert rc_h == N.MOE_OK and ws_h >= ws
    rc_f, flags = q["flags"]
    assert rc_f == N.MOE_OK
    assert bin(flags & ROUTE_BITS).count("1") <= 1, flags
    if flags & N.MOE_PLAN_ROUTE_DECODE:
        assert 1 <= cfg.T <= 16 and cfg.E <= 256
    if flags & N.MOE_PLAN_ROUTE_ONE_LAUNCH:
        assert cfg.dtype == N.MOE_BF16 and cfg.E <= 64 and cfg.k <= 8
    if flags & N.MOE_PLAN_ROUTE_CLUSTER:
        assert cfg.dtype == N.MOE_BF16 and 64 < cfg.E <= 256 and cfg.k <= 8
    if flags & (N.MOE_PLAN_GATHER_ROWS | N.MOE_PLAN_FUSED_PROJECTIONS):
        assert cfg.dtype == N.MOE_BF16           # tensor-core path only
    if flags & N.MOE_PLAN_COMBINE_IN_DOWN:       # by default: top-1 without a shared expert
        assert cfg.dtype == N.MOE_BF16 and cfg.k == 1 and cfg.n_shared == 0
    if flags & N.MOE_PLAN_FUSED_PROJECTIONS:     # by default: the ReLU form with the combine
        assert cfg.act == N.MOE_ACT_RELU and flags & N.MOE_PLAN_COMBINE_IN_DOWN
    rc_l, launches = q["launches"]
    assert rc_l == N.MOE_OK
    assert launches == 0 if cfg.T == 0 else 2 <= launches <= 6, launches
    if cfg.T and flags & (N.MOE_PLAN_ROUTE_ONE_LAUNCH | N.MOE_PLAN_ROUTE_CLUSTER |
                          N.MOE_PLAN_ROUTE_DECODE):
        assert launches <= 5
    # the e4m3 variant: bf16 SwiGLU layers without a shared expert, d % 16 == 0
    rc8, ws8 = q["ws_fp8"]
    fp8_ok = (cfg.dtype == N.MOE_BF16 and cfg.act == N.MOE_ACT_SWIGLU and cfg.n_shared == 0
              and cfg.d % 16 == 0)
    assert (rc8 == N.MOE_OK) == fp8_ok, (rc8, fp8_ok)
    if fp8_ok:
        assert ws8 >= 4096 and ws8 % 256 == 0
        f8 = q["flags_fp8"][1]
        assert not f8 & (N.MOE_PLAN_GATHER_ROWS | N.MOE_PLAN_FUSED_PROJECTIONS)
        assert bin(f8 & ROUTE_BITS).count("1") <= 1
        l8 = q["launches_fp8"][1]
        assert l8 == 0 if cfg.T == 0 else 4 <= l8 <= 7, l8


# anything at all in the fields, including nonsense
any_layers = st.builds(
    _cfg, st.integers(-5, (1 << 31) - 1), st.integers(-5, 1 << 20), st.integers(-5, 2048),
    st.integers(-5, 64), st.integers(-5, 1 << 20), st.integers(-2, 3), st.integers(-5, 1 << 16),
    st.integers(-2, 3), st.integers(-2, 4), st.integers(-2, 4),
    st.sampled_from([0.0, -1.0, 1.25, 1e30, float("inf"), float("nan")]), st.integers(0, 1),
    st.sampled_from([0.01, 0.0, float("inf"), float("nan")]))


@SETTINGS
@given(any_layers)
def test_any_description_gets_a_documented_status(cfg):
    q = _query(cfg)
    bad = (cfg.reserved != 0 or cfg.T < 0 or cfg.d < 1 or cfg.E < 1 or cfg.k < 1 or cfg.k > cfg.E
           or cfg.f < 1 or cfg.n_shared not in (0, 1) or (cfg.n_shared == 1 and cfg.f_shared < 1)
           or cfg.dtype not in (0, 1) or cfg.act not in (0, 1, 2) or cfg.gate not in (0, 1, 2)
           or not math.isfinite(cfg.capacity_factor) or not math.isfinite(cfg.alpha))
    if bad:
        assert q["ws"][0] == N.MOE_ERR_ARG, q["ws"]
        assert q["flags"][0] == N.MOE_ERR_ARG and q["launches"][0] == N.MOE_ERR_ARG


def test_null_outputs_are_refused():
    cfg = L.make_config(T=16, d=64, E=8, k=2, f=64)
    lib = N.lib()
    for fn in (lib.moe_workspace_size, lib.moe_route_workspace_size,
               lib.moe_host_io_workspace_size, lib.moe_workspace_size_fp8, lib.moe_plan_flags,
               lib.moe_plan_flags_fp8, lib.moe_launch_count, lib.moe_launch_count_fp8):
        assert fn(ctypes.byref(cfg), None) == N.MOE_ERR_ARG, fn.__name__
        assert fn(None, None) == N.MOE_ERR_ARG, fn.__name__
