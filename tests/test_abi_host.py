"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/moe.h declares, sizes workspaces and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

from sparse_mixture_experts_65_b300 import _native as N
from sparse_mixture_experts_65_b300 import layer as L
from sparse_mixture_experts_65_b300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(moe_\w+)\s*\(", text, re.M))
    return names


@pytest.mark.parametrize("path", [N.LIB_PATH, N.CHECK_LIB_PATH], ids=["libmoe", "libmoe_check"])
def test_library_exports_every_declared_function(path):
    """Both builds (the normal one and the bounds-checked one) load and export
    every function the header declares."""
    declared = _declared()
    assert {"moe_forward", "moe_workspace_size", "moe_error_string"} <= declared
    lib = N._load(path)
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert set(N.EXPORTS) <= declared


def test_fp8_host_io_checks_arguments_without_gpu():
    cfg = L.config_for(W.get("gptoss16_fp8"))
    fp8 = L.workspace_size(cfg, "fp8")
    hio = L.workspace_size(cfg, "host_io_fp8")
    assert hio > fp8
    fake = ctypes.c_void_p(4096)
    lib = N.lib()
    args = [ctypes.byref(cfg)] + [fake] * 12 + [ctypes.c_size_t(hio), None]
    bad = list(args)
    bad[1] = None                                      # no host x
    assert lib.moe_forward_fp8_host_io(*bad) == N.MOE_ERR_ARG
    bad = list(args)
    bad[6] = None                                      # no W1 scales
    assert lib.moe_forward_fp8_host_io(*bad) == N.MOE_ERR_ARG
    bad = list(args)
    bad[11] = None                                     # no host loss
    assert lib.moe_forward_fp8_host_io(*bad) == N.MOE_ERR_ARG


def test_host_io_batches_check_arguments_without_gpu():
    cfg = L.config_for(W.get("gptoss16"))
    n = L.workspace_size(cfg, "host_io")
    fake = ctypes.c_void_p(4096)
    arr = (ctypes.c_void_p * 2)(4096, 8192)
    lib = N.lib()
    s1, s2 = ctypes.c_void_p(1), ctypes.c_void_p(2)

    def call(count=2, xs=arr, ys=arr, aux=fake, st=s1, cs=s2):
        return lib.moe_forward_host_io_batches(ctypes.byref(cfg), count, xs, fake, None, None,
                                               fake, fake, fake, None, None, None, ys, aux, fake,
                                               ctypes.c_size_t(n), st, cs, cs)
    assert call(count=-1) == N.MOE_ERR_ARG
    assert call(xs=None) == N.MOE_ERR_ARG
    assert call(ys=None) == N.MOE_ERR_ARG
    assert call(aux=None) == N.MOE_ERR_ARG
    assert call(cs=s1) == N.MOE_ERR_ARG               # the copies need their own stream
    bad = (ctypes.c_void_p * 2)(4096, None)
    assert call(xs=bad) == N.MOE_ERR_ARG
    assert call(count=0) == N.MOE_OK                  # nothing to do, nothing enqueued


def test_tuning_knobs_check_their_arguments():
    lib = N.lib()
    assert lib.moe_set_tuning(99, 0) == N.MOE_ERR_ARG
    assert lib.moe_set_tuning(N.MOE_TUNE_ROUTER, 9) == N.MOE_ERR_ARG
    assert lib.moe_set_tuning(N.MOE_TUNE_GATHER, 3) == N.MOE_ERR_ARG
    assert lib.moe_set_tuning(N.MOE_TUNE_TILE_N_UP, -2) == N.MOE_ERR_ARG
    assert lib.moe_set_tuning(N.MOE_TUNE_FUSED_COMBINE, 2) == N.MOE_ERR_ARG
    with L.tuning(router="simt", tile_n_up=64):
        pass                                        # set, then restored
    assert lib.moe_set_tuning(N.MOE_TUNE_ROUTER, -1) == N.MOE_OK


def test_config_struct_layout():
    assert ctypes.sizeof(N.MoeConfig) == 56
    assert N.MoeConfig.capacity_factor.offset == 40


def test_error_strings():
    for code in range(8):
        assert N.error_string(code).startswith("MOE_")
    assert "BOUNDS" in N.error_string(N.MOE_ERR_BOUNDS)
    assert "UNKNOWN" in N.error_string(99)


@pytest.mark.parametrize("name", ["toy", "switch", "mixtral", "dsv3", "gptoss"])
def test_workspace_sizes(name):
    s = W.get(name)
    cfg = L.config_for(s)
    fw = L.workspace_size(cfg)
    rt = L.workspace_size(cfg, "route")
    io = L.workspace_size(cfg, "host_io")
    assert 0 < rt < fw < io
    assert fw % 256 == 0
    elem = 4 if s.dtype == "f32" else 2
    # the expert-ordered buffers alone: at least T*k rows of h and o, both in
    # the layer dtype (and of x unless the up projection gathers rows: the
    # Switch layer, and the gpt-oss-shaped batch of 8 rows per expert)
    x_rows = 0 if name in ("switch", "gptoss") else s.d * elem
    assert fw >= s.T * s.k * (x_rows + s.f * elem + s.d * elem)
    # routing: one tensor-core launch for bf16 layers with E <= 64 and k <= 8
    # (plus a row copy unless the up projection gathers rows: Mixtral copies),
    # one launch with the row copy inside for bf16 layers with 64 < E <= 256
    # and k <= 8 (DeepSeek-V3- and gpt-oss-shaped), else three (logits, top-k,
    # permute: the float32 toy layer); two projections, or one launch for
    # both (by default the Switch layer's form; every compiled form on
    # request); the combine unless a top-1 bf16 layer without a shared expert
    # folds it into the down projection (the other bf16 layers do so only on
    # request)
    expected = {"toy": 6, "switch": 2, "mixtral": 5, "dsv3": 4, "gptoss": 4}
    with L.tuning(fused_combine=1):
        fused = {"toy": 6, "switch": 2, "mixtral": 4, "dsv3": 3, "gptoss": 3}
        assert L.launch_count(cfg) == fused[name]
    with L.tuning(fused_proj=0):
        two = {"toy": 6, "switch": 3, "mixtral": 5, "dsv3": 4, "gptoss": 4}
        assert L.launch_count(cfg) == two[name]
        assert "fused_projections" not in L.plan_flags(cfg)
    with L.tuning(fused_proj=1):
        one = {"toy": 6, "switch": 2, "mixtral": 4, "dsv3": 3, "gptoss": 3}
        assert L.launch_count(cfg) == one[name]
        assert ("fused_projections" in L.plan_flags(cfg)) == (name != "toy")
    assert L.launch_count(cfg) == expected[name]
    flags = L.plan_flags(cfg)
    route = {"toy": set(), "switch": {"route_one_launch", "gather_rows", "combine_in_down",
                                      "fused_projections"},
             "mixtral": {"route_one_launch"}, "dsv3": {"route_cluster"},
             "gptoss": {"route_cluster", "gather_rows"}}
    assert flags == route[name], flags


def _rc_size(cfg):
    n = ctypes.c_size_t()
    return N.lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n))


@pytest.mark.parametrize("field,value,code", [
    ("k", 9, N.MOE_ERR_ARG), ("k", 0, N.MOE_ERR_ARG), ("E", 0, N.MOE_ERR_ARG),
    ("T", -1, N.MOE_ERR_ARG), ("dtype", 7, N.MOE_ERR_ARG), ("gate", 3, N.MOE_ERR_ARG),
    ("act", -1, N.MOE_ERR_ARG), ("reserved", 1, N.MOE_ERR_ARG), ("n_shared", 2, N.MOE_ERR_ARG),
    ("E", 600, N.MOE_ERR_UNSUPPORTED), ("d", 100, N.MOE_ERR_UNSUPPORTED),
])
def test_bad_configs(field, value, code):
    cfg = L.make_config(T=16, d=64, E=8, k=2, f=64)
    if field == "E" and value == 600:
        cfg.k = 2
    setattr(cfg, field, value)
    assert _rc_size(cfg) == code


def test_bf16_shared_expert_needs_swiglu_layers():
    """The tensor-core path runs the SwiGLU shared expert inside the routed
    experts' launches: a plain (ReLU / GELU) bf16 layer with a shared expert
    is reported unsupported; float32 layers and SwiGLU layers take it."""
    cfg = L.make_config(T=16, d=64, E=8, k=2, f=64, act=N.MOE_ACT_RELU, dtype="bf16")
    cfg.n_shared, cfg.f_shared = 1, 64
    assert _rc_size(cfg) == N.MOE_ERR_UNSUPPORTED
    cfg.dtype = N.MOE_F32
    assert _rc_size(cfg) == N.MOE_OK
    cfg = L.make_config(T=16, d=64, E=8, k=2, f=64, dtype="bf16")
    cfg.n_shared, cfg.f_shared = 1, 64
    assert _rc_size(cfg) == N.MOE_OK


def test_forward_rejects_null_and_small_workspace_without_gpu():
    cfg = L.make_config(T=16, d=64, E=8, k=2, f=64)
    lib = N.lib()
    nulls = [None] * 20
    rc = lib.moe_forward(ctypes.byref(cfg), *nulls, None, ctypes.c_size_t(0), None)
    assert rc == N.MOE_ERR_ARG
    # all required pointers present (fake, never dereferenced) but no workspace
    fake = ctypes.c_void_p(1 << 20)
    args = [fake, fake, None, None, fake, fake, fake, None, None, None,
            fake, fake, fake, fake, fake, None, None, None, None, None]
    rc = lib.moe_forward(ctypes.byref(cfg), *args, None, ctypes.c_size_t(0), None)
    assert rc == N.MOE_ERR_WORKSPACE
    misaligned = ctypes.c_void_p((1 << 20) + 2)
    args[0] = misaligned
    rc = lib.moe_forward(ctypes.byref(cfg), *args, None, ctypes.c_size_t(0), None)
    assert rc == N.MOE_ERR_ARG


def test_capacity_formula_matches_documented_rounding():
    # capacity is visible through the tile planning only on the device; here we
    # check that huge factors do not overflow the size computation
    cfg = L.make_config(T=4096, d=768, E=64, k=1, f=3072, act=W.ACT_RELU, capacity_factor=1e12)
    assert _rc_size(cfg) == N.MOE_OK


def test_balance_controls_check_arguments_without_gpu():
    """moe_router_z_loss and moe_bias_update reject bad sizes, NULL and
    unaligned pointers before any device work."""
    lib = N.lib()
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert lib.moe_router_z_loss(fake, -1, 8, fake, None) == N.MOE_ERR_ARG
    assert lib.moe_router_z_loss(fake, 4, 0, fake, None) == N.MOE_ERR_ARG
    assert lib.moe_router_z_loss(fake, 4, 513, fake, None) == N.MOE_ERR_ARG
    assert lib.moe_router_z_loss(None, 4, 8, fake, None) == N.MOE_ERR_ARG
    assert lib.moe_router_z_loss(odd, 4, 8, fake, None) == N.MOE_ERR_ARG
    assert lib.moe_router_z_loss(fake, 4, 8, None, None) == N.MOE_ERR_ARG
    f = ctypes.c_float
    assert lib.moe_bias_update(fake, 0, 4, 1, f(1e-3), fake, None) == N.MOE_ERR_ARG
    assert lib.moe_bias_update(fake, 8, 4, 9, f(1e-3), fake, None) == N.MOE_ERR_ARG
    assert lib.moe_bias_update(fake, 8, -1, 1, f(1e-3), fake, None) == N.MOE_ERR_ARG
    assert lib.moe_bias_update(fake, 8, 4, 1, f(-1.0), fake, None) == N.MOE_ERR_ARG
    assert lib.moe_bias_update(fake, 8, 4, 1, f(float("nan")), fake, None) == N.MOE_ERR_ARG
    assert lib.moe_bias_update(None, 8, 4, 1, f(1e-3), fake, None) == N.MOE_ERR_ARG
    assert lib.moe_bias_update(fake, 8, 4, 1, f(1e-3), odd, None) == N.MOE_ERR_ARG


def test_fp8_entry_point_checks_without_gpu():
    """moe_forward_fp8: unsupported layers and missing or misaligned scale
    arrays are rejected before any device work; launch counts add the row
    quantisation and drop the bf16 row copy."""
    lib = N.lib()
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)
    size = ctypes.c_size_t(0)

    def call(cfg, W1s=fake, W3s=fake):
        args = [fake, fake, None, None, fake, W1s, fake, W3s, fake,
                fake, fake, fake, fake, fake, None, None, None, None, None]
        return lib.moe_forward_fp8(ctypes.byref(cfg), *args, None, ctypes.c_size_t(0), None)

    ok = L.make_config(T=16, d=256, E=8, k=2, f=64)
    assert lib.moe_workspace_size_fp8(ctypes.byref(ok), ctypes.byref(size)) == N.MOE_OK
    plain = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(ok), ctypes.byref(plain)) == N.MOE_OK
    assert size.value > 0
    for bad in (L.make_config(T=16, d=256, E=8, k=2, f=64, act=L.ACT_GELU),
                L.make_config(T=16, d=264, E=8, k=2, f=64),
                L.make_config(T=16, d=256, E=8, k=2, f=64, dtype="f32"),
                L.make_config(T=16, d=256, E=8, k=2, f=64, n_shared=1, f_shared=64)):
        assert call(bad) == N.MOE_ERR_UNSUPPORTED
        assert lib.moe_workspace_size_fp8(ctypes.byref(bad), ctypes.byref(size)) == \
            N.MOE_ERR_UNSUPPORTED
    assert call(ok, W1s=None) == N.MOE_ERR_ARG
    assert call(ok, W3s=None) == N.MOE_ERR_ARG
    assert call(ok, W1s=odd) == N.MOE_ERR_ARG
    assert call(ok) == N.MOE_ERR_WORKSPACE          # everything else valid, no workspace
    # decode batch: router, row quantisation, the two projections, combine;
    # larger batches route in one launch as well (64 < E <= 256), the bf16
    # layer with its row copy inside it
    assert L.launch_count(L.config_for(W.get("gptoss16_fp8")), fp8=True) == 5
    assert L.launch_count(L.config_for(W.get("gptoss256")), fp8=False) == 4
    assert L.launch_count(L.config_for(W.get("gptoss256_fp8")), fp8=True) == 5
    # the fp8 plan: the row quantisation replaces the gather and the fused
    # projections (compiled for the bf16 decode layer's tiling, opt-in)
    dec = L.config_for(W.get("gptoss1"))
    assert "fused_projections" not in L.plan_flags(dec)
    with L.tuning(fused_proj=1):
        assert "fused_projections" in L.plan_flags(dec)
        assert not {"fused_projections", "gather_rows"} & L.plan_flags(dec, fp8=True)
    assert "route_decode" in L.plan_flags(dec, fp8=True)
    # the knob of the e4m3 down projection's form takes 0 and 1 only
    assert N.lib().moe_set_tuning(N.MOE_TUNE_F8_DOWN_FORM, 2) == N.MOE_ERR_ARG
    with L.tuning(f8_down_form=1):
        assert L.launch_count(L.config_for(W.get("gptoss16_fp8")), fp8=True) == 5
    # forcing the split router (tensor-core logits, top-k, permute)
    with L.tuning(router="tc"):
        assert L.launch_count(L.config_for(W.get("gptoss256")), fp8=False) == 6
        assert L.launch_count(L.config_for(W.get("gptoss256_fp8")), fp8=True) == 7


def test_fp8_all_entry_point_checks_without_gpu():
    """moe_forward_fp8_all (e4m3 down weights as well): missing or misaligned
    down scales and the layers moe_forward_fp8 rejects are refused before any
    device work."""
    lib = N.lib()
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)

    def call(cfg, W2s=fake, W1s=fake):
        args = [fake, fake, None, None, fake, W1s, fake, fake, fake, W2s,
                fake, fake, fake, fake, fake, None, None, None, None, None]
        return lib.moe_forward_fp8_all(ctypes.byref(cfg), *args, None, ctypes.c_size_t(0), None)

    ok = L.make_config(T=16, d=256, E=8, k=2, f=64)
    assert call(ok, W2s=None) == N.MOE_ERR_ARG
    assert call(ok, W1s=None) == N.MOE_ERR_ARG
    assert call(ok, W2s=odd) == N.MOE_ERR_ARG
    assert call(ok) == N.MOE_ERR_WORKSPACE           # everything else valid, no workspace
    for bad in (L.make_config(T=16, d=256, E=8, k=2, f=64, act=L.ACT_GELU),
                L.make_config(T=16, d=264, E=8, k=2, f=64)):
        assert call(bad) == N.MOE_ERR_UNSUPPORTED
    fake_hosts = (ctypes.c_void_p * 2)(fake.value, fake.value)
    n = L.workspace_size(ok, "host_io_fp8")
    args = ([ctypes.byref(ok), ctypes.c_int32(2), fake_hosts, fake, None, None, fake, fake, fake,
             fake, fake, None, fake_hosts, fake, fake, ctypes.c_size_t(n)] + [None] * 3)
    assert lib.moe_forward_fp8_all_host_io_batches(*args) == N.MOE_ERR_ARG   # no W2s
