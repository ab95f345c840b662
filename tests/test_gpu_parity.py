"""CUDA layer versus the CPU oracle on seeded inputs, through the C ABI.

Small cases span several tiles with ragged tails (rows, N columns and the K
reduction); the named layers run at full size with routing checked over the
whole batch and y on every token or on a seeded sample the oracle can afford.
"""
import gc

import numpy as np
import pytest
import torch

from sparse_mixture_experts_65_b300 import layer as L
from sparse_mixture_experts_65_b300 import workloads as W
from sparse_mixture_experts_65_b300.workloads import LayerShape

from gpu_harness import check_layer, host64, run_gpu

pytestmark = pytest.mark.gpu

SW, RE, GE = W.ACT_SWIGLU, W.ACT_RELU, W.ACT_GELU
TOPK, SIG, FULL = W.GATE_SOFTMAX_TOPK, W.GATE_SIGMOID_RENORM, W.GATE_SOFTMAX_FULL

SMALL = [
    LayerShape("bf16_swiglu_ragged", 10, T=300, d=256, E=8, k=2, f=384, act=SW, gate=TOPK,
               dtype="bf16"),
    LayerShape("bf16_relu_capacity_skew", 11, T=517, d=192, E=16, k=1, f=256, act=RE, gate=FULL,
               dtype="bf16", capacity_factor=1.0, logit_offset_var=1.5),
    LayerShape("bf16_sigmoid_bias_shared", 12, T=130, d=136, E=32, k=4, f=160, act=SW, gate=SIG,
               dtype="bf16", alpha=1e-4, n_shared=1, f_shared=96, sel_bias_halfwidth=0.05),
    LayerShape("bf16_gelu_ntail", 13, T=77, d=64, E=4, k=2, f=200, act=GE, gate=TOPK, dtype="bf16"),
    LayerShape("bf16_many_experts", 16, T=64, d=128, E=300, k=6, f=64, act=SW, gate=SIG,
               dtype="bf16", sel_bias_halfwidth=0.05),
    LayerShape("f32_swiglu_shared_cap", 14, T=150, d=48, E=6, k=3, f=80, act=SW, gate=SIG,
               dtype="f32", capacity_factor=1.1, n_shared=1, f_shared=40),
    LayerShape("f32_relu_full", 15, T=99, d=36, E=5, k=1, f=52, act=RE, gate=FULL, dtype="f32",
               capacity_factor=0.9, logit_offset_var=1.5),
]


def _free():
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_small_layers(shape):
    inp = W.make_inputs(shape, "cuda", seed=1)
    _, out = run_gpu(inp)
    rep = check_layer(inp, out)
    print(shape.name, rep)


@pytest.mark.parametrize("up_bn,dn_bn", [(32, 64), (64, 96), (96, 128), (128, 192), (128, 256)])
def test_every_swiglu_tile_width(up_bn, dn_bn):
    """Force each tile width of the tensor-core kernels on a ragged layer."""
    shape = LayerShape("tiles", 20, T=211, d=200, E=6, k=2, f=416, act=SW, gate=TOPK,
                       dtype="bf16", n_shared=1, f_shared=136)
    inp = W.make_inputs(shape, "cuda", seed=2)
    with L.tuning(tile_n_up=up_bn, tile_n_down=dn_bn):
        _, out = run_gpu(inp)
    check_layer(inp, out)


@pytest.mark.parametrize("act", [RE, GE])
@pytest.mark.parametrize("up_bn", [64, 96, 128, 256])
def test_every_plain_tile_width(act, up_bn):
    shape = LayerShape("plain", 21, T=190, d=96, E=5, k=2, f=328, act=act, gate=TOPK, dtype="bf16")
    inp = W.make_inputs(shape, "cuda", seed=3)
    with L.tuning(tile_n_up=up_bn):
        _, out = run_gpu(inp)
    check_layer(inp, out)


def test_toy_layer_full():
    inp = W.make_inputs(W.TOY, "cuda")
    _, out = run_gpu(inp)
    rep = check_layer(inp, out)
    assert rep["flipped_tokens"] == 0
    print("toy", rep)


def test_switch_layer_full():
    inp = W.make_inputs(W.SWITCH, "cuda")
    _, out = run_gpu(inp)
    rep = check_layer(inp, out)
    assert rep["dropped"] > 0       # the logit skew overflows some experts at rho = 1.25
    print("switch", rep)
    del inp, out
    _free()


def test_mixtral_layer_sampled():
    inp = W.make_inputs(W.MIXTRAL, "cuda")
    _, out = run_gpu(inp)
    sample = np.sort(np.random.default_rng(7).choice(W.MIXTRAL.T, 1024, replace=False))
    rep = check_layer(inp, out, sample=sample)
    print("mixtral", rep)
    del inp, out
    _free()


def test_dsv3_layer_sampled():
    inp = W.make_inputs(W.DSV3, "cuda")
    _, out = run_gpu(inp)
    sample = np.sort(np.random.default_rng(8).choice(W.DSV3.T, 512, replace=False))
    rep = check_layer(inp, out, sample=sample)
    print("dsv3", rep)
    del inp, out
    _free()


@pytest.mark.parametrize("T", W.GPTOSS_SWEEP_T)
def test_gptoss_decode_sweep(T):
    shape = W.GPTOSS.with_T(T)
    inp = W.make_inputs(shape, "cuda")
    _, out = run_gpu(inp)
    sample = None if T <= 64 else np.sort(np.random.default_rng(9).choice(T, 48, replace=False))
    rep = check_layer(inp, out, sample=sample)
    print("gptoss", T, rep)
    del inp, out
    _free()


# ---------------------------------------------------------------- edge cases
def test_empty_batch():
    shape = LayerShape("empty", 30, T=0, d=64, E=4, k=2, f=64, act=SW, gate=TOPK, dtype="bf16")
    inp = W.make_inputs(shape, "cuda")
    cfg, out = run_gpu(inp)
    assert out.expert_counts.sum().item() == 0
    assert out.offsets.cpu().tolist() == [0] * 5
    assert float(out.aux_loss.cpu()[0]) == 0.0
    assert L.launch_count(cfg) == 0


@pytest.mark.parametrize("T", [1, 2, 129])
def test_tiny_batches(T):
    shape = LayerShape("tiny", 31, T=T, d=128, E=8, k=2, f=128, act=SW, gate=TOPK, dtype="bf16",
                       n_shared=1, f_shared=64)
    inp = W.make_inputs(shape, "cuda")
    _, out = run_gpu(inp)
    check_layer(inp, out)


def test_single_expert_is_dense_ffn():
    shape = LayerShape("dense", 32, T=200, d=64, E=1, k=1, f=192, act=GE, gate=TOPK, dtype="bf16")
    inp = W.make_inputs(shape, "cuda")
    _, out = run_gpu(inp)
    np.testing.assert_array_equal(out.topk_w.cpu().numpy(), 1.0)
    check_layer(inp, out)


def test_k_equals_E():
    shape = LayerShape("allk", 33, T=70, d=64, E=4, k=4, f=64, act=SW, gate=TOPK, dtype="bf16")
    inp = W.make_inputs(shape, "cuda")
    _, out = run_gpu(inp)
    check_layer(inp, out)


def test_all_tokens_to_one_expert_with_drops():
    shape = LayerShape("onehot", 34, T=400, d=64, E=8, k=1, f=128, act=RE, gate=FULL,
                       dtype="bf16", capacity_factor=1.25)
    inp = W.make_inputs(shape, "cuda")
    inp.logit_offset = torch.zeros(8, device="cuda")
    inp.logit_offset[5] = 100.0
    _, out = run_gpu(inp)
    counts = out.routed_counts.cpu().numpy()
    assert counts[5] == 400
    C = int(np.ceil(400 * 1.25 / 8))
    assert out.expert_counts.cpu().numpy()[5] == C
    slot = out.slot_pos.cpu().numpy()[:, 0]
    assert np.all(slot[:C] == np.arange(C)) and np.all(slot[C:] == -1)   # first come by token
    assert torch.all(out.y[C:] == 0)                                     # dropped tokens: y = 0
    check_layer(inp, out)


def test_tiny_capacity():
    shape = LayerShape("tinycap", 35, T=333, d=64, E=8, k=2, f=64, act=SW, gate=TOPK,
                       dtype="bf16", capacity_factor=0.05)
    inp = W.make_inputs(shape, "cuda")
    _, out = run_gpu(inp)
    C = int(np.ceil(333 * 2 * 0.05 / 8))
    assert out.expert_counts.cpu().numpy().max() <= C
    check_layer(inp, out)


def test_selection_bias_moves_choice_not_gates():
    shape = LayerShape("bias", 36, T=256, d=64, E=16, k=2, f=64, act=SW, gate=SIG, dtype="bf16")
    inp = W.make_inputs(shape, "cuda")
    _, out0 = run_gpu(inp)
    inp.sel_bias = torch.zeros(16, device="cuda")
    inp.sel_bias[3] = 2.0                 # sigmoid <= 1, so expert 3 always wins
    _, out1 = run_gpu(inp)
    assert torch.all(out1.topk_idx[:, 0] == 3)
    check_layer(inp, out1)
    # the same bias on every expert changes nothing
    inp.sel_bias = torch.full((16,), 0.3, device="cuda")
    _, out2 = run_gpu(inp)
    assert torch.equal(out2.topk_idx, out0.topk_idx)
    assert torch.equal(out2.y, out0.y)


# ---------------------------------------------------------------- properties
def test_repeat_calls_bitwise_identical():
    inp = W.make_inputs(SMALL[2], "cuda", seed=4)
    cfg = L.config_for(inp.shape)
    ws = L.alloc_workspace(cfg)
    _, a = run_gpu(inp, cfg, ws)
    _, b = run_gpu(inp, cfg, ws)
    for name in ("y", "topk_idx", "topk_w", "expert_counts", "aux_loss", "slot_pos", "P"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def test_route_entry_point_matches_forward():
    shape = SMALL[1]
    inp = W.make_inputs(shape, "cuda", seed=5)
    cfg, fw = run_gpu(inp)
    rt = L.route(cfg, inp.x, inp.W_r, inp.logit_offset, inp.sel_bias)
    torch.cuda.synchronize()
    for name in ("topk_idx", "topk_w", "expert_counts", "aux_loss", "routed_counts", "offsets",
                 "slot_pos", "f", "P"):
        assert torch.equal(getattr(rt, name), getattr(fw, name)), name


def test_host_io_entry_point_matches_forward():
    shape = SMALL[0]
    inp = W.make_inputs(shape, "cuda", seed=6)
    cfg, fw = run_gpu(inp)
    x_h = inp.x.cpu().pin_memory()
    y_h = torch.empty_like(x_h).pin_memory()
    aux_h = torch.empty(1, dtype=torch.float32).pin_memory()
    L.forward_host_io(cfg, x_h, y_h, aux_h, inp.W_r, inp.W1, inp.W2, inp.W3)
    torch.cuda.synchronize()
    assert torch.equal(y_h, fw.y.cpu())
    assert torch.equal(aux_h, fw.aux_loss.cpu())


def test_bounded_wait_reports_timeout():
    """A wait on a barrier nothing completes gives up after ~1 ms and the host
    reads MOE_ERR_TIMEOUT; the context stays usable afterwards."""
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert L.check_status(ws) == L.N.MOE_OK
    L.selftest_wait_timeout(ws, 1_000_000)
    assert L.check_status(ws) == L.N.MOE_ERR_TIMEOUT
    assert L.check_status(ws) == L.N.MOE_OK          # cleared by the first check
    inp = W.make_inputs(SMALL[3], "cuda")
    _, out = run_gpu(inp)
    check_layer(inp, out)


def test_status_clean_after_full_layer():
    inp = W.make_inputs(SMALL[0], "cuda", seed=9)
    cfg = L.config_for(inp.shape)
    ws = L.alloc_workspace(cfg)
    run_gpu(inp, cfg, ws)
    assert L.check_status(ws) == L.N.MOE_OK


def test_bad_arguments_rejected_on_device():
    inp = W.make_inputs(SMALL[0], "cuda", seed=10)
    cfg = L.config_for(inp.shape)
    ws = L.alloc_workspace(cfg)
    with pytest.raises(L.N.MoeError) as e:
        L.forward(cfg, inp.x, inp.W_r, inp.W1, inp.W2, None, workspace=ws)   # SwiGLU needs W3
    assert e.value.code == L.N.MOE_ERR_ARG
    with pytest.raises(L.N.MoeError) as e:
        L.forward(cfg, inp.x, inp.W_r, inp.W1, inp.W2, inp.W3, workspace=ws[:1024])
    assert e.value.code == L.N.MOE_ERR_WORKSPACE
    xbig = torch.empty(inp.x.numel() + 8, dtype=inp.x.dtype, device="cuda")
    xmis = xbig[1:1 + inp.x.numel()].view_as(inp.x)     # 2-byte offset: not 16-byte aligned
    with pytest.raises(L.N.MoeError) as e:
        L.forward(cfg, xmis, inp.W_r, inp.W1, inp.W2, inp.W3, workspace=ws)
    assert e.value.code == L.N.MOE_ERR_ARG


# ---------------------------------------------------------------- router precision
@pytest.mark.parametrize("path", ["simt", "fused", "tc"])
@pytest.mark.parametrize("name", ["dsv3", "mixtral", "switch"])
def test_router_logits_within_half_the_near_tie_band(path, name):
    """Every float32 logit lies within 5e-6 of the float64 value, half the
    1e-5 near-tie band, on each router path (float32 FMA split-K; fused float32
    FMA; tensor cores with 128-wide float32 chunks): two experts can then only
    swap order when their float64 scores are closer than the band."""
    shape = W.get(name)
    x = W.make_x(shape, "cuda")
    inp = W.make_inputs(shape.with_T(1), "cuda")      # W_r etc.; x replaced below
    cfg = L.config_for(shape)
    with L.tuning(router=path):
        s = L.router_scores(cfg, x, inp.W_r, inp.logit_offset)
    torch.cuda.synchronize()
    ref = host64(x) @ host64(inp.W_r).T
    if inp.logit_offset is not None:
        ref = ref + host64(inp.logit_offset)[None, :]
    err = np.abs(s.cpu().numpy().astype(np.float64) - ref)
    print(name, path, "max |err|", err.max(), "mean", err.mean(), "max |s|", np.abs(ref).max())
    assert err.max() < 5e-6


ONE_LAUNCH = [
    # 150 tiles of 128 tokens on 148 SMs: two routing CTAs own two tiles each
    LayerShape("route_multi_tile", 40, T=19200, d=64, E=64, k=1, f=64, act=RE, gate=FULL,
               dtype="bf16", capacity_factor=1.25, logit_offset_var=1.5),
    # the largest k of the one-launch router, with sigmoid gates and a bias
    LayerShape("route_k8_sigmoid", 41, T=300, d=128, E=64, k=8, f=64, act=SW, gate=SIG,
               dtype="bf16", sel_bias_halfwidth=0.05, capacity_factor=1.5),
    # a wider model: 16 k-blocks per row gathered by the up projection
    LayerShape("route_wide_rows", 42, T=1024, d=1024, E=8, k=2, f=64, act=SW, gate=TOPK,
               dtype="bf16"),
    # E = 33: the 64-wide expert tile with a ragged tail, k = 3
    LayerShape("route_e33", 43, T=700, d=96, E=33, k=3, f=64, act=GE, gate=FULL, dtype="bf16",
               capacity_factor=1.0, logit_offset_var=1.5),
]


@pytest.mark.parametrize("shape", ONE_LAUNCH, ids=lambda s: s.name)
def test_one_launch_router_layers(shape):
    """Layers routed by the one-launch tensor-core router (bf16, E <= 64,
    k <= 8): several tiles per CTA, k = 8, wide rows, a ragged E."""
    inp = W.make_inputs(shape, "cuda", seed=2)
    _, out = run_gpu(inp)
    rep = check_layer(inp, out)
    print(shape.name, rep)


DECODE = [
    LayerShape("small_f32_sigmoid_cap", 50, T=5, d=72, E=6, k=3, f=40, act=SW, gate=SIG,
               dtype="f32", capacity_factor=0.8, sel_bias_halfwidth=0.05),
    LayerShape("small_bf16_dsv3_like", 51, T=16, d=256, E=256, k=8, f=64, act=SW, gate=SIG,
               dtype="bf16", n_shared=1, f_shared=64, sel_bias_halfwidth=0.05),
    LayerShape("small_bf16_e200_full", 52, T=11, d=200, E=200, k=2, f=96, act=GE, gate=FULL,
               dtype="bf16", capacity_factor=1.0, logit_offset_var=1.5),
    LayerShape("small_bf16_top1", 53, T=1, d=640, E=16, k=1, f=128, act=RE, gate=FULL,
               dtype="bf16"),
]


@pytest.mark.parametrize("shape", DECODE, ids=lambda s: s.name)
def test_decode_batch_router(shape):
    """Decode batches (T <= 16) route in one launch: split-K partial logits,
    the last block's top-k, capacity scan and positions."""
    inp = W.make_inputs(shape, "cuda", seed=3)
    _, out = run_gpu(inp)
    rep = check_layer(inp, out)
    print(shape.name, rep)


@pytest.mark.parametrize("gather", ["0", "1", "2"])
def test_up_projection_row_source(gather):
    """Every row source of the tensor-core up projection, on layers of every
    routing path (one-launch tensor-core router, split router with E > 64,
    decode-batch router): an expert-ordered copy read through TMA (0), rows
    gathered from x inside the GEMM with cp.async (1) or with the TMA row
    gather, four rows per instruction (2)."""
    for shape in (SMALL[0], SMALL[1], SMALL[2], SMALL[3], SMALL[4], ONE_LAUNCH[1], ONE_LAUNCH[3],
                  DECODE[1], DECODE[3]):
        inp = W.make_inputs(shape, "cuda", seed=12)
        with L.tuning(gather=int(gather)):
            _, out = run_gpu(inp)
        check_layer(inp, out)


@pytest.mark.parametrize("shape", [SMALL[0], SMALL[2], SMALL[3], SMALL[4], ONE_LAUNCH[1],
                                   ONE_LAUNCH[3], DECODE[1], DECODE[2]], ids=lambda s: s.name)
def test_fused_combine_matches_the_separate_kernel_bitwise(shape):
    """The down projection's epilogue combine (the last row of each token's
    column slice sums it, fixed slot order) gives the separate combine
    kernel's y bit for bit, with drops, shared experts and many experts."""
    inp = W.make_inputs(shape, "cuda", seed=13)
    with L.tuning(fused_combine=1):
        _, fused = run_gpu(inp)
    _, separate = run_gpu(inp)
    assert torch.equal(fused.y, separate.y)
    check_layer(inp, fused)


def test_fused_combine_with_most_slots_dropped():
    """k = 2 with a tiny capacity: most tokens lose both slots and get y = 0,
    some keep one; every token's counters still complete."""
    shape = LayerShape("drops_k2", 37, T=700, d=128, E=8, k=2, f=64, act=SW, gate=TOPK,
                       dtype="bf16", capacity_factor=0.1)
    inp = W.make_inputs(shape, "cuda", seed=14)
    with L.tuning(fused_combine=1):
        _, out = run_gpu(inp)
    slot = out.slot_pos.cpu()
    none = (slot < 0).all(dim=1)
    assert none.any() and (~none).any()
    assert torch.all(out.y[none.cuda()] == 0)
    check_layer(inp, out)


@pytest.mark.parametrize("path", ["simt", "fused", "tc"])
def test_forced_router_path_parity(path):
    """The split router paths (split-K float32 logits, the fused float32
    router, tensor-core logits; each followed by the top-k and permute
    kernels) on small ragged layers, each routing as the oracle does."""
    shapes = (SMALL[0], SMALL[1], SMALL[2], SMALL[3], SMALL[4], SMALL[5], SMALL[6])
    for shape in shapes:
        if path == "fused" and shape.E > 256:
            continue
        inp = W.make_inputs(shape, "cuda", seed=11)
        with L.tuning(router=path):
            _, out = run_gpu(inp)
        check_layer(inp, out)


@pytest.mark.parametrize("one_copy_stream", [False, True], ids=["in_out_streams", "one_stream"])
@pytest.mark.parametrize("shape", [SMALL[0], SMALL[2], DECODE[1]], ids=lambda s: s.name)
def test_host_io_batches_match_forward_per_batch(shape, one_copy_stream):
    """moe_forward_host_io_batches: five host batches (different x), the copies
    of one overlapping the layer of another through two staging slots (copies
    in and out on two streams, or taking turns on one), give exactly what
    moe_forward gives for each batch."""
    base = W.make_inputs(shape, "cuda", seed=15)
    cfg = L.config_for(shape)
    xs = [W.make_x(shape, "cuda", seed=40 + i) for i in range(5)]
    refs = []
    for x in xs:
        inp = W.make_inputs(shape, "cuda", seed=15)
        inp.x = x
        _, out = run_gpu(inp, cfg)
        refs.append((out.y.cpu(), out.aux_loss.cpu()))
    x_h = [x.cpu().pin_memory() for x in xs]
    y_h = [torch.empty_like(x).pin_memory() for x in x_h]
    aux_h = torch.empty(5, dtype=torch.float32).pin_memory()
    cs = torch.cuda.Stream() if one_copy_stream else None
    b = L.BoundHostIOBatches(cfg, x_h, y_h, aux_h, base, copy_in_stream=cs, copy_out_stream=cs)
    b()
    torch.cuda.synchronize()
    assert L.check_status(b.workspace) == 0
    for i, (y, aux) in enumerate(refs):
        assert torch.equal(y_h[i], y), i
        assert aux_h[i].item() == aux.item(), i
    b()                                       # a second call on the same workspace
    torch.cuda.synchronize()
    assert torch.equal(y_h[4], refs[4][0])


# ---------------------------------------------------------------- limits
LIMITS = [
    # the largest expert count and k the ABI takes (split router, sigmoid gates, bias)
    LayerShape("max_e512_k32", 60, T=100, d=128, E=512, k=32, f=64, act=SW, gate=SIG,
               dtype="bf16", sel_bias_halfwidth=0.05),
    LayerShape("max_e512_k32_f32", 61, T=40, d=32, E=512, k=32, f=16, act=GE, gate=TOPK,
               dtype="f32"),
    # either side of the decode-batch threshold (16 tokens) and of the
    # tensor-core router threshold (256 tokens), with E > 64
    LayerShape("decode_edge_t16", 62, T=16, d=192, E=96, k=4, f=64, act=SW, gate=TOPK,
               dtype="bf16"),
    LayerShape("decode_edge_t17", 63, T=17, d=192, E=96, k=4, f=64, act=SW, gate=TOPK,
               dtype="bf16"),
    LayerShape("router_tc_edge_t255", 64, T=255, d=256, E=80, k=2, f=64, act=RE, gate=FULL,
               dtype="bf16", capacity_factor=1.25, logit_offset_var=1.5),
    LayerShape("router_tc_edge_t256", 65, T=256, d=256, E=80, k=2, f=64, act=RE, gate=FULL,
               dtype="bf16", capacity_factor=1.25, logit_offset_var=1.5),
]


@pytest.mark.parametrize("shape", LIMITS, ids=lambda s: s.name)
def test_limits_and_thresholds(shape):
    inp = W.make_inputs(shape, "cuda", seed=17)
    _, out = run_gpu(inp)
    check_layer(inp, out)


def test_one_launch_router_largest_batch():
    """65 536 tokens: the largest batch of the one-launch router (512 tiles on
    at most 148 CTAs, several tiles per CTA), Switch-like skew and drops;
    routing over the whole batch, y on a sample."""
    shape = LayerShape("route_t65536", 66, T=65536, d=128, E=64, k=1, f=128, act=RE, gate=FULL,
                       dtype="bf16", capacity_factor=1.25, logit_offset_var=1.5)
    inp = W.make_inputs(shape, "cuda", seed=18)
    _, out = run_gpu(inp)
    sample = np.sort(np.random.default_rng(19).choice(shape.T, 256, replace=False))
    rep = check_layer(inp, out, sample=sample)
    assert rep["dropped"] > 0


CLUSTER_SHAPES = [SMALL[0], SMALL[2], ONE_LAUNCH[2], DECODE[1], LIMITS[4],
                  LayerShape("cluster_odd_ntiles", 67, T=600, d=256, E=6, k=2, f=640, act=SW,
                             gate=TOPK, dtype="bf16", n_shared=1, f_shared=384)]


@pytest.mark.parametrize("shape", CLUSTER_SHAPES, ids=lambda s: s.name)
def test_two_cta_cluster_projections(shape):
    """The projections as clusters of two CTAs sharing a multicast A tile
    (odd column-tile counts leave a phantom tile that stores nothing; M = 64
    tails load one half): the same parity as single CTAs, and the same y."""
    inp = W.make_inputs(shape, "cuda", seed=23)
    with L.tuning(tile_n_up=128, tile_n_down=256):     # the compiled cluster forms
        _, single = run_gpu(inp)
        with L.tuning(cluster=1):
            _, pair = run_gpu(inp)
    check_layer(inp, pair)
    assert torch.equal(pair.y, single.y)


# ---------------------------------------------------------------- one-launch router, 64 < E <= 256
# Clusters of KS CTAs per 128-token tile, each CTA on a share of the model
# width; KS = 8, 4, 2, 1 by tile count and width (tiles x KS within one wave
# of 148 SMs, at least one 128-wide chunk per CTA).
ROUTE_WIDE = [
    # KS = 4 (6 tiles, 4 chunks), sigmoid gates with a selection bias, drops,
    # the shared expert
    LayerShape("wide_e256_k8_sig_cap", 70, T=700, d=512, E=256, k=8, f=64, act=SW, gate=SIG,
               dtype="bf16", capacity_factor=1.0, sel_bias_halfwidth=0.05, n_shared=1,
               f_shared=64),
    # KS = 1 (one chunk), E = 130: 256-wide expert tile with a ragged tail and
    # a histogram row stride of 132; full-softmax gates, skewed offsets
    LayerShape("wide_e130_ks1_full", 71, T=1000, d=96, E=130, k=3, f=64, act=GE, gate=FULL,
               dtype="bf16", capacity_factor=1.0, logit_offset_var=1.5),
    # KS = 8 (3 tiles, 8 chunks), E = 100 (128-wide expert tile), a ragged
    # last k-block (d = 1000), top-k softmax gates
    LayerShape("wide_e100_ks8_ragged_d", 72, T=333, d=1000, E=100, k=2, f=64, act=SW,
               gate=TOPK, dtype="bf16"),
    # KS = 8 with 18 tiles: more tiles than clusters of 8 that fit at once,
    # so some clusters take two tiles (both partial-logit slots)
    LayerShape("wide_e160_ks8_two_tiles", 73, T=2200, d=2048, E=160, k=4, f=64, act=RE,
               gate=TOPK, dtype="bf16", capacity_factor=1.25),
    # KS = 1 with 313 tiles on at most 148 clusters: several tiles per CTA,
    # Switch-like skew and drops, k = 1
    LayerShape("wide_e72_persistent", 74, T=40000, d=64, E=72, k=1, f=64, act=RE, gate=FULL,
               dtype="bf16", capacity_factor=1.25, logit_offset_var=1.5),
    # KS = 2 (71 tiles, 2 chunks)
    LayerShape("wide_e192_ks2", 75, T=9000, d=256, E=192, k=6, f=64, act=SW, gate=SIG,
               dtype="bf16", sel_bias_halfwidth=0.05),
]


@pytest.mark.parametrize("shape", ROUTE_WIDE, ids=lambda s: s.name)
def test_wide_router_layers(shape):
    """Layers routed by the one-launch cluster router: routing over the whole
    batch (indices, gates, counts, positions, f, P, L) and y against the
    oracle (sampled for the largest batch)."""
    inp = W.make_inputs(shape, "cuda", seed=24)
    cfg = L.config_for(shape)
    assert L.launch_count(cfg) == 4 - (shape.k == 1)       # router, up, down (+ combine)
    _, out = run_gpu(inp)
    sample = None
    if shape.T > 5000:
        sample = np.sort(np.random.default_rng(25).choice(shape.T, 384, replace=False))
    rep = check_layer(inp, out, sample=sample)
    print(shape.name, rep)
    if shape.capacity_factor > 0 and shape.k == 1:
        assert rep["dropped"] > 0
    del inp, out
    _free()


def test_wide_router_repeat_and_route_entry_point():
    """Bitwise repeatable (same workspace, twice), and moe_route gives the
    forward pass's routing outputs bit for bit."""
    shape = ROUTE_WIDE[0]
    inp = W.make_inputs(shape, "cuda", seed=26)
    cfg = L.config_for(shape)
    ws = L.alloc_workspace(cfg)
    _, a = run_gpu(inp, cfg, ws)
    _, b = run_gpu(inp, cfg, ws)
    for name in ("y", "topk_idx", "topk_w", "expert_counts", "aux_loss", "slot_pos", "P"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert L.check_status(ws) == 0
    rt = L.route(cfg, inp.x, inp.W_r, inp.logit_offset, inp.sel_bias)
    torch.cuda.synchronize()
    for name in ("topk_idx", "topk_w", "expert_counts", "aux_loss", "routed_counts", "offsets",
                 "slot_pos", "f", "P"):
        assert torch.equal(getattr(rt, name), getattr(a, name)), name


def test_wide_router_agrees_with_split_router():
    """The one-launch router and the split tensor-core router (logits GEMM,
    top-k kernel, permute) add the same 128-wide float32 chunks in different
    groupings: the same choices away from near-ties, gates within float32
    rounding, and the same y within the layer tolerance."""
    shape = ROUTE_WIDE[1]
    inp = W.make_inputs(shape, "cuda", seed=27)
    _, wide = run_gpu(inp)
    with L.tuning(router="tc"):
        _, split = run_gpu(inp)
    same = (wide.topk_idx == split.topk_idx).all(dim=1)
    assert same.float().mean().item() > 0.99
    g = (wide.topk_w - split.topk_w)[same].abs().max().item()
    assert g < 1e-5, g
    check_layer(inp, split)


# ---------------------------------------------------------------- up + down in one launch
FUSED_CASES = [
    # (shape, tile widths forced so that a compiled fused form applies, one launch?)
    (SMALL[0], dict(tile_n_up=128, tile_n_down=256), True),    # SwiGLU, TMA rows
    (SMALL[2], dict(tile_n_up=128, tile_n_down=192), True),    # + shared expert, sigmoid gates
    (SMALL[1], dict(tile_n_up=256, tile_n_down=192), True),    # ReLU top-1: gathered rows, combine in down
    (ROUTE_WIDE[0], dict(tile_n_up=128, tile_n_down=256), True),  # cluster router, shared expert, drops
    (ROUTE_WIDE[3], dict(tile_n_up=128, tile_n_down=192), False),  # ReLU k = 4: no compiled form
    (DECODE[1], dict(tile_n_up=96, tile_n_down=96), True),     # decode batch, E = 256, shared expert
    (ONE_LAUNCH[0], dict(tile_n_up=256, tile_n_down=256), False),  # ReLU rows by TMA: not compiled
    # 512 up and 128 down tiles on at most 148 CTAs: several of each per CTA
    (LayerShape("fused_many_tiles", 76, T=4096, d=512, E=16, k=2, f=1024, act=SW, gate=TOPK,
                dtype="bf16", capacity_factor=1.25),
     dict(tile_n_up=128, tile_n_down=256), True),
]


@pytest.mark.parametrize("case", FUSED_CASES, ids=lambda c: c[0].name)
def test_fused_projections_match_two_launches_bitwise(case):
    """The up and down projections as one persistent launch (down tiles wait
    for their M tile's up tiles through counters) give y bit for bit equal to
    the two launches, and pass the oracle comparison; the counters are back at
    zero afterwards (a second call on the same workspace agrees)."""
    shape, tiles, expect = case
    inp = W.make_inputs(shape, "cuda", seed=28)
    cfg = L.config_for(shape)
    with L.tuning(fused_proj=1, **tiles):
        fused = "fused_projections" in L.plan_flags(cfg)
        assert fused == expect, L.plan_flags(cfg)
        ws = L.alloc_workspace(cfg)
        _, one = run_gpu(inp, cfg, ws)
        _, again = run_gpu(inp, cfg, ws)
        with L.tuning(fused_proj=0):
            assert "fused_projections" not in L.plan_flags(cfg)
            _, two = run_gpu(inp, cfg)
    assert torch.equal(one.y, two.y)
    assert torch.equal(again.y, one.y)
    check_layer(inp, one)


@pytest.mark.parametrize("shape", [SMALL[2], ONE_LAUNCH[0], DECODE[1], ROUTE_WIDE[0]],
                         ids=lambda s: s.name)
def test_layer_call_replays_from_a_cuda_graph(shape):
    """One layer call captured in a CUDA graph (kernels only: no host
    synchronisation or allocation inside a call) replays to the direct call's
    outputs bit for bit, with the device status clean."""
    inp = W.make_inputs(shape, "cuda", seed=31)
    cfg = L.config_for(shape)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        direct = L.bound_forward(cfg, inp, stream=stream)
        direct()
        stream.synchronize()
        ref = {n: getattr(direct.out, n).clone()
               for n in ("y", "topk_idx", "topk_w", "expert_counts", "aux_loss", "slot_pos")}
        bound = L.bound_forward(cfg, inp, stream=stream)
        bound()
        stream.synchronize()
        g = L.capture_graph(bound, stream)
        for n in ("y", "topk_w"):
            getattr(bound.out, n).zero_()
        for _ in range(3):
            g.replay()
        stream.synchronize()
    assert L.check_status(bound.workspace) == 0
    for n, t in ref.items():
        assert torch.equal(getattr(bound.out, n), t), n
