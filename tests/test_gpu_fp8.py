"""The layer with fp8 (e4m3) gate/up expert weights (moe_forward_fp8) against
the oracle's fp8 variant on the same seeded inputs: routing bit-exact (or a
counted near tie), integers exact given the GPU's choice, y within the bf16
tolerance.  The row quantisation is exact on both sides (power-of-two scales),
so only the float32 accumulation and the bf16 roundings of h, o and y differ.
"""
import dataclasses
import gc

import pytest
import torch

from sparse_mixture_experts_65_b300 import layer as L
from sparse_mixture_experts_65_b300 import workloads as W
from sparse_mixture_experts_65_b300.workloads import LayerShape

from gpu_harness import check_layer, run_gpu

pytestmark = pytest.mark.gpu

SW = W.ACT_SWIGLU
TOPK, SIG, FULL = W.GATE_SOFTMAX_TOPK, W.GATE_SIGMOID_RENORM, W.GATE_SOFTMAX_FULL

FP8 = [
    # decode batches (one-launch small-batch router)
    LayerShape("fp8_decode_t1", 70, T=1, d=256, E=16, k=4, f=192, act=SW, gate=TOPK,
               dtype="bf16", w_fp8=True),
    LayerShape("fp8_decode_ragged", 71, T=13, d=272, E=40, k=3, f=200, act=SW, gate=SIG,
               dtype="bf16", sel_bias_halfwidth=0.05, w_fp8=True),
    # tensor-core one-launch router; K (d) not a multiple of 128, N (f) ragged
    LayerShape("fp8_one_launch", 72, T=700, d=400, E=24, k=2, f=328, act=SW, gate=TOPK,
               dtype="bf16", w_fp8=True),
    # split router (E > 64)
    LayerShape("fp8_split_many", 73, T=300, d=256, E=100, k=4, f=128, act=SW, gate=SIG,
               dtype="bf16", sel_bias_halfwidth=0.05, w_fp8=True),
    # top-1 with capacity drops: the combine runs inside the down projection
    LayerShape("fp8_capacity_top1", 74, T=517, d=192, E=16, k=1, f=256, act=SW, gate=FULL,
               dtype="bf16", capacity_factor=1.0, logit_offset_var=1.5, w_fp8=True),
]


def _free():
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("shape", FP8, ids=lambda s: s.name)
def test_fp8_layers(shape):
    inp = W.make_inputs(shape, "cuda", seed=2)
    _, out = run_gpu(inp)
    rep = check_layer(inp, out)
    print(shape.name, rep)


@pytest.mark.parametrize("T", [1, 16])
def test_fp8_gptoss_decode(T):
    shape = W.get(f"gptoss{T}_fp8")
    inp = W.make_inputs(shape, "cuda")
    _, out = run_gpu(inp)
    sample = None if T <= 16 else list(range(0, T, max(1, T // 32)))
    rep = check_layer(inp, out, sample=sample)
    print("gptoss_fp8", T, rep)
    del inp, out
    _free()


def test_fp8_repeat_calls_bitwise_identical():
    inp = W.make_inputs(FP8[2], "cuda", seed=3)
    cfg = L.config_for(inp.shape)
    ws = L.alloc_workspace(cfg, kind="fp8")
    _, a = run_gpu(inp, cfg, ws)
    _, b = run_gpu(inp, cfg, ws)
    for name in ("y", "topk_idx", "topk_w", "expert_counts", "aux_loss", "slot_pos"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert L.check_status(ws) == L.N.MOE_OK


def test_fp8_zero_token_rows():
    """An all-zero token row takes scale 1 and codes 0: its expert outputs are
    the down projection of silu(0) * 0 = 0."""
    inp = W.make_inputs(FP8[0], "cuda", seed=4)
    inp.x.zero_()
    _, out = run_gpu(inp)
    assert torch.count_nonzero(out.y) == 0


@pytest.mark.parametrize("shape", [FP8[1], FP8[2]], ids=lambda s: s.name)
def test_fp8_host_io_entry_point_matches_device_entry_point(shape):
    """moe_forward_fp8_host_io (x from pinned host memory, y and the loss back
    to the host) gives exactly moe_forward_fp8's y and loss."""
    inp = W.make_inputs(shape, "cuda", seed=6)
    cfg, dev = run_gpu(inp)
    x_h = inp.x.cpu().pin_memory()
    y_h = torch.empty_like(x_h).pin_memory()
    aux_h = torch.empty(1, dtype=torch.float32).pin_memory()
    hio = L.BoundHostIOFp8(cfg, x_h, y_h, aux_h, inp.W_r, inp.W1q, inp.W1s, inp.W3q, inp.W3s,
                           inp.W2, inp.logit_offset, inp.sel_bias)
    hio()
    torch.cuda.synchronize()
    assert L.check_status(hio.workspace) == 0
    assert torch.equal(y_h, dev.y.cpu())
    assert torch.equal(aux_h, dev.aux_loss.cpu())


def test_fp8_host_io_batches_match_device_entry_point():
    shape = FP8[1]
    inp = W.make_inputs(shape, "cuda", seed=7)
    cfg, dev = run_gpu(inp)
    x_h = [inp.x.cpu().pin_memory() for _ in range(3)]
    y_h = [torch.empty_like(x).pin_memory() for x in x_h]
    aux_h = torch.empty(3, dtype=torch.float32).pin_memory()
    b = L.BoundHostIOBatches(cfg, x_h, y_h, aux_h, inp)
    b()
    torch.cuda.synchronize()
    for y in y_h:
        assert torch.equal(y, dev.y.cpu())
    assert torch.all(aux_h == dev.aux_loss.cpu()[0])


# e4m3 down weights as well (moe_forward_fp8_all): f a multiple of 16
FP8_ALL = [
    LayerShape("fp8all_decode_t1", 75, T=1, d=256, E=16, k=4, f=192, act=SW, gate=TOPK,
               dtype="bf16", w_fp8=True, w2_fp8=True),
    LayerShape("fp8all_decode_ragged", 76, T=13, d=272, E=40, k=3, f=208, act=SW, gate=SIG,
               dtype="bf16", sel_bias_halfwidth=0.05, w_fp8=True, w2_fp8=True),
    # d = 400: a ragged last down tile of output channels (their scales are
    # not read); f = 336: a ragged last K block of codes
    LayerShape("fp8all_one_launch", 77, T=700, d=400, E=24, k=2, f=336, act=SW, gate=TOPK,
               dtype="bf16", w_fp8=True, w2_fp8=True),
    LayerShape("fp8all_split_many", 78, T=300, d=256, E=100, k=4, f=128, act=SW, gate=SIG,
               dtype="bf16", sel_bias_halfwidth=0.05, w_fp8=True, w2_fp8=True),
    # top-1 with capacity drops: the combine in the down epilogue
    LayerShape("fp8all_capacity_top1", 79, T=517, d=192, E=16, k=1, f=256, act=SW, gate=FULL,
               dtype="bf16", capacity_factor=1.0, logit_offset_var=1.5, w_fp8=True,
               w2_fp8=True),
]


@pytest.mark.parametrize("shape", FP8_ALL, ids=lambda s: s.name)
def test_fp8_down_weight_layers(shape):
    inp = W.make_inputs(shape, "cuda", seed=2)
    assert inp.W2 is None and inp.W2q is not None
    _, out = run_gpu(inp)
    rep = check_layer(inp, out)
    print(shape.name, rep)


@pytest.mark.parametrize("T", [1, 16, 256])
def test_fp8_down_weight_gptoss(T):
    shape = W.get(f"gptoss{T}_fp8all")
    inp = W.make_inputs(shape, "cuda")
    _, out = run_gpu(inp)
    sample = None if T <= 16 else list(range(0, T, max(1, T // 32)))
    rep = check_layer(inp, out, sample=sample)
    print("gptoss_fp8all", T, rep)
    del inp, out
    _free()


def test_fp8_down_weight_repeat_calls_bitwise_identical():
    inp = W.make_inputs(FP8_ALL[2], "cuda", seed=3)
    cfg = L.config_for(inp.shape)
    ws = L.alloc_workspace(cfg, kind="fp8")
    _, a = run_gpu(inp, cfg, ws)
    _, b = run_gpu(inp, cfg, ws)
    for name in ("y", "topk_idx", "topk_w", "expert_counts", "aux_loss", "slot_pos"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def test_fp8_down_weight_routing_matches_fp8_layer():
    """The down weights' format changes only the down projection: routing,
    gates and counts are those of moe_forward_fp8 on the same x."""
    shape = FP8_ALL[3]
    inp = W.make_inputs(shape, "cuda", seed=5)
    ref = W.make_inputs(dataclasses.replace(shape, w2_fp8=False), "cuda", seed=5)
    assert torch.equal(inp.x, ref.x) and torch.equal(inp.W1q, ref.W1q)
    _, a = run_gpu(inp)
    _, b = run_gpu(ref)
    for name in ("topk_idx", "topk_w", "expert_counts", "aux_loss", "slot_pos"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def test_fp8_down_weight_unsupported_width():
    """f not a multiple of 16: a row of down codes is no TMA row."""
    shape = LayerShape("fp8all_f200", 80, T=64, d=256, E=8, k=2, f=200, act=SW, gate=TOPK,
                       dtype="bf16", w_fp8=True, w2_fp8=True)
    inp = W.make_inputs(shape, "cuda")
    with pytest.raises(L.N.MoeError) as e:
        run_gpu(inp)
    assert e.value.code == L.N.MOE_ERR_UNSUPPORTED


def test_fp8_down_weight_host_io_batches_match_device_entry_point():
    shape = FP8_ALL[1]
    inp = W.make_inputs(shape, "cuda", seed=7)
    cfg, dev = run_gpu(inp)
    x_h = [inp.x.cpu().pin_memory() for _ in range(3)]
    y_h = [torch.empty_like(x).pin_memory() for x in x_h]
    aux_h = torch.empty(3, dtype=torch.float32).pin_memory()
    b = L.BoundHostIOBatches(cfg, x_h, y_h, aux_h, inp)
    assert b._fn.__name__ == "moe_forward_fp8_all_host_io_batches"
    b()
    torch.cuda.synchronize()
    assert L.check_status(b.workspace) == 0
    for y in y_h:
        assert torch.equal(y, dev.y.cpu())
    assert torch.all(aux_h == dev.aux_loss.cpu()[0])


@pytest.mark.parametrize("codes", ["subnormal", "every"])
def test_fp8_down_weight_code_ranges(codes):
    """Down codes drawn only from the e4m3 subnormals (exponent field 0: a
    kernel that flushed them would return y = 0), or uniformly from every
    non-NaN code (exponents 2^-9 .. 2^8 in one matrix), against the oracle."""
    shape = FP8_ALL[2]
    inp = W.make_inputs(shape, "cuda", seed=8)
    g = torch.Generator(device="cuda")
    g.manual_seed(808)
    n = inp.W2q.numel()
    if codes == "subnormal":
        mag = torch.randint(1, 8, (n,), generator=g, device="cuda")
        unit = 2.0 ** -9                 # the smallest subnormal step
    else:
        mag = torch.randint(0, 0x7F, (n,), generator=g, device="cuda")
        unit = 64.0                      # a typical magnitude of a uniform code
    sign = torch.randint(0, 2, (n,), generator=g, device="cuda") << 7
    inp.W2q.copy_((mag | sign).to(torch.uint8).view_as(inp.W2q))
    inp.W2s.fill_(1.0 / (unit * 4.0 * shape.f ** 0.5))
    _, out = run_gpu(inp)
    assert torch.count_nonzero(out.y) > out.y.numel() // 2
    rep = check_layer(inp, out)
    print(codes, rep)


@pytest.mark.parametrize("form", [0, 1], ids=["weights_as_n", "weights_as_m"])
@pytest.mark.parametrize("shape", FP8_ALL, ids=lambda s: s.name)
def test_fp8_down_weight_both_kernel_forms(shape, form):
    """Both down-projection forms (weights as the MMA's N operand, or as its M
    operand with 32 token rows per pass: segments of more than 32 rows take
    several passes) on every shape, whichever the plan would pick."""
    inp = W.make_inputs(shape, "cuda", seed=9)
    with L.tuning(f8_down_form=form):
        cfg = L.config_for(shape)
        _, out = run_gpu(inp, cfg)
    rep = check_layer(inp, out)
    print(shape.name, form, rep)


def test_fp8_down_weight_many_rows_per_segment_weights_as_m():
    """Weights as M with segments of up to ~200 rows (several 32-row passes
    and several 128-row M tiles per expert), a ragged d and f."""
    shape = LayerShape("fp8all_long_segments", 81, T=1500, d=336, E=8, k=1, f=272, act=SW,
                       gate=TOPK, dtype="bf16", w_fp8=True, w2_fp8=True)
    inp = W.make_inputs(shape, "cuda", seed=10)
    with L.tuning(f8_down_form=1):
        cfg = L.config_for(shape)
        _, out = run_gpu(inp, cfg)
    rep = check_layer(inp, out)
    print(rep)


def test_fp8_down_weight_empty_batch_and_combine_override():
    """T = 0 gives empty outputs and zero counts; the k-slot combine override
    (no form with e4m3 down weights) is refused before any launch."""
    shape = FP8_ALL[2]
    empty = dataclasses.replace(shape, T=0)
    inp = W.make_inputs(empty, "cuda", seed=12)
    cfg, out = run_gpu(inp)
    assert torch.count_nonzero(out.expert_counts) == 0
    assert float(out.aux_loss.cpu()[0]) == 0.0
    inp = W.make_inputs(shape, "cuda", seed=12)
    with L.tuning(fused_combine=1):
        cfg = L.config_for(shape)
        with pytest.raises(L.N.MoeError) as e:
            run_gpu(inp, cfg)
    assert e.value.code == L.N.MOE_ERR_UNSUPPORTED
