"""The Python binding refuses tensors the library would misread, before any
library call (no GPU needed).

The C ABI takes bare pointers, so a host tensor where device memory is
expected, or a buffer of the wrong dtype or shape, would be read or written
out of bounds on the GPU.  The binding checks memory, dtype and exact shape of
every tensor first.  Here the library is replaced by a stub that records the
entry points it receives, so that no host pointer ever reaches a kernel; the
"device" of these tests is the host (the binding's device test is patched to
accept it), and a tensor on the meta device stands for one on another device.
"""
import dataclasses

import pytest
import torch

from sparse_mixture_experts_65_b300 import _native as N
from sparse_mixture_experts_65_b300 import layer as L
from sparse_mixture_experts_65_b300 import workloads as W

SHAPE = W.LayerShape("check_bf16", 90, T=6, d=32, E=4, k=2, f=16, act=W.ACT_SWIGLU,
                     gate=W.GATE_SIGMOID_RENORM, dtype="bf16", n_shared=1, f_shared=8,
                     logit_offset_var=1.0, sel_bias_halfwidth=0.05)
FP8_ALL = W.LayerShape("check_fp8all", 91, T=6, d=32, E=4, k=2, f=16, act=W.ACT_SWIGLU,
                       gate=W.GATE_SOFTMAX_TOPK, dtype="bf16", w_fp8=True, w2_fp8=True)


class _StubLib:
    """Stands in for libmoe.so: every entry point returns MOE_OK and is
    recorded; nothing is dereferenced."""

    def __init__(self):
        self.called = []

    def __getattr__(self, name):
        def fn(*args):
            self.called.append(name)
            return N.MOE_OK
        fn.__name__ = name
        return fn


@pytest.fixture
def stub(monkeypatch):
    lib = _StubLib()
    monkeypatch.setattr(N, "lib", lambda: lib)
    monkeypatch.setattr(L, "_cuda_device", lambda t, name: t.device)
    monkeypatch.setattr(L, "_stream_handle", lambda stream: None)
    return lib


def _ws():
    return torch.zeros(4096, dtype=torch.uint8)


def _forward(inp, **over):
    a = dict(x=inp.x, W_r=inp.W_r, W1=inp.W1, W2=inp.W2, W3=inp.W3,
             logit_offset=inp.logit_offset, sel_bias=inp.sel_bias, Ws1=inp.Ws1, Ws3=inp.Ws3,
             Ws2=inp.Ws2, workspace=_ws())
    a.update(over)
    return L.forward(L.config_for(inp.shape), **a)


# ------------------------------------------------------------ host memory
def test_host_tensors_are_refused_where_device_memory_is_expected():
    """Without the patch: every device-memory call refuses host x (or host
    logits, bias, workspace) before reaching the library."""
    inp = W.make_inputs(SHAPE, "cpu")
    cfg = L.config_for(SHAPE)
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.forward(cfg, inp.x, inp.W_r, inp.W1, inp.W2, inp.W3, workspace=_ws())
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.route(cfg, inp.x, inp.W_r, workspace=_ws())
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.router_scores(cfg, inp.x, inp.W_r, workspace=_ws())
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.BoundForward(cfg, inp.x, inp.W_r, inp.W1, inp.W2, inp.W3, workspace=_ws())
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.router_z_loss(torch.zeros((3, 4)))
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.bias_update(torch.zeros(4), torch.zeros(4, dtype=torch.int32), 3, 1, 1e-3)
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.check_status(_ws())
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.selftest_wait_timeout(_ws(), 1000)
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.forward_host_io(cfg, inp.x, torch.empty_like(inp.x), torch.empty(1), inp.W_r,
                          inp.W1, inp.W2, inp.W3, workspace=_ws())
    f8 = W.make_inputs(FP8_ALL, "cpu")
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.forward_fp8(L.config_for(FP8_ALL), f8.x, f8.W_r, f8.W1q, f8.W1s, f8.W3q, f8.W3s,
                      f8.W2q, workspace=_ws(), W2s=f8.W2s)


# ------------------------------------------------------------ device calls
def test_valid_arguments_reach_the_library(stub):
    inp = W.make_inputs(SHAPE, "cpu")
    out = _forward(inp)
    assert stub.called == ["moe_forward"]
    assert out.y.shape == (SHAPE.T, SHAPE.d) and out.y.dtype == torch.bfloat16
    _forward(inp, out=out)
    L.route(L.config_for(SHAPE), inp.x, inp.W_r, inp.logit_offset, inp.sel_bias,
            workspace=_ws())
    L.router_scores(L.config_for(SHAPE), inp.x, inp.W_r, inp.logit_offset, workspace=_ws())
    L.bias_update(inp.sel_bias, torch.zeros(SHAPE.E, dtype=torch.int32), SHAPE.T, SHAPE.k, 1e-3)
    f8 = W.make_inputs(FP8_ALL, "cpu")
    cfg8 = L.config_for(FP8_ALL)
    L.forward_fp8(cfg8, f8.x, f8.W_r, f8.W1q, f8.W1s, f8.W3q, f8.W3s, f8.W2q, workspace=_ws(),
                  W2s=f8.W2s)
    # codes may also arrive as torch's float8 type (the same bytes)
    L.forward_fp8(cfg8, f8.x, f8.W_r, f8.W1q.view(torch.float8_e4m3fn), f8.W1s,
                  f8.W3q.view(torch.float8_e4m3fn), f8.W3s, f8.W2q, workspace=_ws(), W2s=f8.W2s)
    bf16_down = W.make_inputs(dataclasses.replace(FP8_ALL, w2_fp8=False), "cpu")
    L.forward_fp8(cfg8, f8.x, f8.W_r, f8.W1q, f8.W1s, f8.W3q, f8.W3s, bf16_down.W2,
                  workspace=_ws())
    assert stub.called == ["moe_forward", "moe_forward", "moe_route", "moe_router_scores",
                           "moe_bias_update", "moe_forward_fp8_all", "moe_forward_fp8_all",
                           "moe_forward_fp8"]


def _bad_cases(inp):
    meta = torch.empty(inp.W_r.shape, dtype=inp.W_r.dtype, device="meta")
    return {
        "x in float32 for a bf16 layer": dict(x=inp.x.float()),
        "x with one token too many": dict(x=torch.cat([inp.x, inp.x[:1]])),
        "x transposed (not contiguous)": dict(x=inp.x.t().contiguous().t()),
        "W_r on another device": dict(W_r=meta),
        "W1 of a wider expert": dict(W1=torch.zeros((4, 32, 32), dtype=torch.bfloat16)),
        "W2 stored as W1 (transposed shape)": dict(W2=inp.W1),
        "W3 in float32": dict(W3=inp.W3.float()),
        "logit offset in float64": dict(logit_offset=inp.logit_offset.double()),
        "selection bias one entry short": dict(sel_bias=inp.sel_bias[:-1].contiguous()),
        "shared down weights transposed": dict(Ws2=inp.Ws1),
        "workspace of int32 words": dict(workspace=torch.zeros(1024, dtype=torch.int32)),
        "workspace not a tensor": dict(workspace=bytearray(4096)),
        "W1 not a tensor": dict(W1=[[0.0]]),
    }


@pytest.mark.parametrize("case", list(_bad_cases(W.make_inputs(SHAPE, "cpu"))))
def test_wrong_tensors_are_refused_before_the_library(stub, case):
    inp = W.make_inputs(SHAPE, "cpu")
    with pytest.raises((ValueError, TypeError)):
        _forward(inp, **_bad_cases(inp)[case])
    assert stub.called == []


def test_wrong_outputs_are_refused(stub):
    inp = W.make_inputs(SHAPE, "cpu")
    cfg = L.config_for(SHAPE)
    good = L.alloc_outputs(cfg, "cpu", torch.bfloat16)
    for field, bad in (("y", torch.empty((SHAPE.T, SHAPE.d), dtype=torch.float32)),
                       ("topk_idx", torch.empty((SHAPE.T, SHAPE.k), dtype=torch.int64)),
                       ("offsets", torch.empty(SHAPE.E, dtype=torch.int32)),
                       ("aux_loss", torch.empty(2, dtype=torch.float32)),
                       ("P", torch.empty(SHAPE.E, dtype=torch.float16))):
        with pytest.raises(ValueError, match="out." + field):
            _forward(inp, out=dataclasses.replace(good, **{field: bad}))
    assert stub.called == []


def test_fp8_calls_check_codes_and_scales(stub):
    f8 = W.make_inputs(FP8_ALL, "cpu")
    cfg = L.config_for(FP8_ALL)
    base = dict(x=f8.x, W_r=f8.W_r, W1q=f8.W1q, W1s=f8.W1s, W3q=f8.W3q, W3s=f8.W3s, W2=f8.W2q,
                workspace=_ws(), W2s=f8.W2s)
    bad = {
        "gate codes as bf16 values": dict(W1q=f8.W1q.to(torch.bfloat16)),
        "up scales per expert only": dict(W3s=f8.W3s[:, :1].contiguous()),
        "down scales along the input axis": dict(W2s=torch.ones((4, 16))),
        "down codes without their layout": dict(W2=f8.W2q.transpose(1, 2).contiguous()),
        "bf16 down weights with down scales": dict(W2=f8.W2q.to(torch.bfloat16)),
    }
    for name, over in bad.items():
        a = dict(base, **over)
        with pytest.raises(ValueError):
            L.forward_fp8(cfg, **a)
    assert stub.called == []


# ------------------------------------------------------------ host-memory calls
def test_host_memory_calls_check_their_host_buffers(stub):
    inp = W.make_inputs(SHAPE, "cpu")
    cfg = L.config_for(SHAPE)
    x_h, y_h, aux_h = inp.x.clone(), torch.empty_like(inp.x), torch.empty(1)

    def call(**over):
        a = dict(x_host=x_h, y_host=y_h, aux_host=aux_h, W_r=inp.W_r, W1=inp.W1, W2=inp.W2,
                 W3=inp.W3, logit_offset=inp.logit_offset, sel_bias=inp.sel_bias, Ws1=inp.Ws1,
                 Ws3=inp.Ws3, Ws2=inp.Ws2, workspace=_ws())
        a.update(over)
        return L.forward_host_io(cfg, **a)

    call()
    assert stub.called == ["moe_forward_host_io"]
    for over in (dict(x_host=x_h[:-1].contiguous()), dict(y_host=y_h.float()),
                 dict(aux_host=torch.empty(1, dtype=torch.float64)),
                 dict(x_host=torch.empty(x_h.shape, dtype=x_h.dtype, device="meta"))):
        with pytest.raises(ValueError):
            call(**over)
    assert stub.called == ["moe_forward_host_io"]
    # a sequence of batches: every x and y buffer, and one loss entry per batch
    xs = [x_h.clone() for _ in range(3)]
    ys = [torch.empty_like(x_h) for _ in range(3)]
    kw = dict(workspace=_ws(), copy_in_stream=object(), copy_out_stream=object())
    with pytest.raises(ValueError):
        L.BoundHostIOBatches(cfg, xs, ys[:2] + [ys[2][:-1]], torch.empty(3), inp, **kw)
    with pytest.raises(ValueError):
        L.BoundHostIOBatches(cfg, xs, ys, torch.empty(2), inp, **kw)
    with pytest.raises(ValueError):
        L.BoundHostIOBatches(cfg, xs, ys, torch.empty(3, dtype=torch.float64), inp, **kw)
    b = L.BoundHostIOBatches(cfg, xs, ys, torch.empty(3), inp, **kw)
    b()
    assert stub.called == ["moe_forward_host_io", "moe_forward_host_io_batches"]


# ------------------------------------------------------------ the GPU tests' own inputs
def _gpu_test_shapes():
    """Every layer shape the GPU test modules and the named workloads define,
    up to 60 MB of expert weights (the larger ones are the same kinds of layer)."""
    import importlib
    shapes = {}
    for mod in ("test_gpu_parity", "test_gpu_fp8", "test_gpu_bounds", "test_gpu_balance"):
        for v in vars(importlib.import_module(mod)).values():
            for it in (v if isinstance(v, (list, tuple)) else [v]):
                if isinstance(it, tuple):
                    it = next((x for x in it if isinstance(x, W.LayerShape)), None)
                if isinstance(it, W.LayerShape):
                    shapes[it.name] = it
    for s in W.WORKLOADS.values():
        shapes[s.name] = s
    return [s for _, s in sorted(shapes.items()) if s.E * s.f * s.d * 6 <= 6e7]


def test_the_gpu_tests_inputs_pass_the_checks(stub):
    """The checks refuse nothing the GPU tests, the bench or smoke() pass: the
    calls those make, on every shape they use, reach the library."""
    shapes = _gpu_test_shapes()
    kinds = {(s.dtype, s.act, bool(s.n_shared), s.w_fp8, s.w2_fp8) for s in shapes}
    assert len(shapes) >= 30 and len(kinds) >= 6
    for s in shapes:
        inp = W.make_inputs(s, "cpu")
        cfg = L.config_for(s)
        n = len(stub.called)
        L.bound_forward(cfg, inp, workspace=_ws())()
        xs = [inp.x.clone(), inp.x.clone()]
        L.BoundHostIOBatches(cfg, xs, [torch.empty_like(x) for x in xs], torch.empty(4), inp,
                             workspace=_ws(), copy_in_stream=object(),
                             copy_out_stream=object())()
        if inp.W1q is None:
            L.forward(cfg, inp.x, inp.W_r, inp.W1, inp.W2, inp.W3, inp.logit_offset,
                      inp.sel_bias, inp.Ws1, inp.Ws3, inp.Ws2, workspace=_ws())
            L.route(cfg, inp.x, inp.W_r, inp.logit_offset, inp.sel_bias, workspace=_ws())
            L.router_scores(cfg, inp.x, inp.W_r, inp.logit_offset, workspace=_ws())
            L.forward_host_io(cfg, inp.x.clone(), torch.empty_like(inp.x), torch.empty(1),
                              inp.W_r, inp.W1, inp.W2, inp.W3, inp.logit_offset, inp.sel_bias,
                              inp.Ws1, inp.Ws3, inp.Ws2, workspace=_ws())
        elif inp.W2q is None:
            L.BoundHostIOFp8(cfg, inp.x.clone(), torch.empty_like(inp.x), torch.empty(1),
                             inp.W_r, inp.W1q, inp.W1s, inp.W3q, inp.W3s, inp.W2,
                             inp.logit_offset, inp.sel_bias, workspace=_ws())()
        assert len(stub.called) > n + 1, s.name
