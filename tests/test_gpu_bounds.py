"""The bounds-checked build (libmoe_check.so: every index routing produces is
range-tested on the device before the access it drives; a failure is recorded
as MOE_ERR_BOUNDS and the access skipped, never a trap).  Over the parity
shapes -- ragged tiles, capacity drops, many experts, every routing path
(including the cluster router for 64 < E <= 256), the decode batches, the
projections as one launch, the e4m3 weight layers and a full-size layer -- it must report no
out-of-range index and still match the oracle."""
import pytest
import torch

from sparse_mixture_experts_65_b300 import _native as N
from sparse_mixture_experts_65_b300 import layer as L
from sparse_mixture_experts_65_b300 import workloads as W

from gpu_harness import check_layer, run_gpu
import test_gpu_fp8 as TF
import test_gpu_parity as TP

pytestmark = pytest.mark.gpu

SHAPES = TP.SMALL + TP.ONE_LAUNCH + TP.DECODE + TP.ROUTE_WIDE


@pytest.fixture
def checked_library():
    N.use_library("check")
    try:
        yield
    finally:
        N.use_library("default")


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_checked_build_finds_no_out_of_range_index(checked_library, shape):
    inp = W.make_inputs(shape, "cuda", seed=21)
    cfg = L.config_for(shape)
    ws = L.alloc_workspace(cfg)
    _, out = run_gpu(inp, cfg, ws)
    assert L.check_status(ws) == N.MOE_OK
    check_layer(inp, out)


@pytest.mark.parametrize("router", ["simt", "tc"])
def test_checked_build_on_the_split_router_paths(checked_library, router):
    for shape in (TP.SMALL[1], TP.SMALL[4], TP.DECODE[2]):
        inp = W.make_inputs(shape, "cuda", seed=22)
        with L.tuning(router=router):
            cfg = L.config_for(shape)
            ws = L.alloc_workspace(cfg)
            _, out = run_gpu(inp, cfg, ws)
        assert L.check_status(ws) == N.MOE_OK
        check_layer(inp, out)


def test_checked_build_full_switch_layer(checked_library):
    inp = W.make_inputs(W.SWITCH, "cuda")
    cfg = L.config_for(W.SWITCH)
    ws = L.alloc_workspace(cfg)
    _, out = run_gpu(inp, cfg, ws)
    assert L.check_status(ws) == N.MOE_OK
    rep = check_layer(inp, out)
    assert rep["dropped"] > 0
    del inp, out, ws
    torch.cuda.empty_cache()


@pytest.mark.parametrize("case", TP.FUSED_CASES, ids=lambda c: c[0].name)
def test_checked_build_on_the_one_launch_projections(checked_library, case):
    shape, tiles, _ = case
    inp = W.make_inputs(shape, "cuda", seed=29)
    with L.tuning(fused_proj=1, **tiles):
        cfg = L.config_for(shape)
        ws = L.alloc_workspace(cfg)
        _, out = run_gpu(inp, cfg, ws)
    assert L.check_status(ws) == N.MOE_OK
    check_layer(inp, out)


@pytest.mark.parametrize("shape", TF.FP8 + TF.FP8_ALL, ids=lambda s: s.name)
def test_checked_build_on_the_fp8_layers(checked_library, shape):
    """e4m3 gate/up weights (and e4m3 down weights): the row quantisation,
    the e4m3 projections and the on-chip expansion of the down codes."""
    inp = W.make_inputs(shape, "cuda", seed=23)
    cfg = L.config_for(shape)
    ws = L.alloc_workspace(cfg, kind="fp8")
    _, out = run_gpu(inp, cfg, ws)
    assert L.check_status(ws) == N.MOE_OK
    check_layer(inp, out)
