"""Host-side logic of bench.py, no GPU: the max-over-ranks job time on a
world-size-2 gloo group, the reference arm's rank behaviour, the algorithmic
byte / FLOP accounting behind the roofline numbers."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from sparse_mixture_experts_65_b300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [3.5, 7.25][rank]
        out[rank] = bench.max_over_ranks(mine, dist)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_time_is_max_over_ranks_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert dict(out) == {0: 7.25, 1: 7.25}


def test_single_rank_max_is_identity():
    assert bench.max_over_ranks(1.5) == 1.5


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        workload = "toy"
        steps = 3
        warmup = 3
    assert bench.run_reference(A()) is None
    assert capsys.readouterr().out == ""


def test_accounting_switch_shape():
    s = W.SWITCH
    kept = [0] * 64
    kept[3], kept[7] = 80, 50
    acc, layer = bench.accounting(s, kept)
    el = 2
    w1 = 2 * s.f * s.d * el          # two active experts, plain (ReLU) up projection
    assert acc["up"]["bytes"] == w1 + 130 * s.d * el          # weights + input rows only
    assert acc["up"]["extra"] == 130 * s.f * el                 # h, an intermediate
    assert acc["up"]["flops"] == 2 * 130 * s.d * s.f
    assert acc["down"]["flops"] == 2 * 130 * s.f * s.d
    assert layer["active_experts"] == 2 and layer["kept_rows"] == 130
    assert layer["bytes"] == (2 * 2 * s.f * s.d + s.E * s.d + 2 * s.T * s.d) * el


def test_roofline_bound_selection():
    peaks = dict(bench.FALLBACK_PEAKS)
    acc = {"k": {"bytes": 1e9, "flops": 1e9}}
    r = bench.roofline_for("k", acc, 1.0, peaks, "fallback")
    assert r["bound"] == "hbm" and abs(r["achieved"] - 1000.0) < 1e-6
    acc = {"k": {"bytes": 1e6, "flops": 1e12}}
    r = bench.roofline_for("k", acc, 1.0, peaks, "fallback")
    assert r["bound"] == "tensor" and abs(r["achieved"] - 1000.0) < 1e-6


def test_accounting_fp8_gate_up_weights():
    """e4m3 gate/up weights count one byte each plus a float32 scale per
    channel; the up projection reads one-byte rows; the down projection and
    the layer's other bytes are those of the bf16 layer."""
    bf = W.get("gptoss16")
    f8 = W.get("gptoss16_fp8")
    kept = [0] * bf.E
    for e in range(0, 64, 4):
        kept[e] = 4                   # 16 active experts, 64 kept rows
    acc_b, lay_b = bench.accounting(bf, kept)
    acc_f, lay_f = bench.accounting(f8, kept)
    act, rows, d, f = 16, 64, bf.d, bf.f
    assert acc_f["up"]["bytes"] == act * 2 * f * (d + 4) + rows * d
    assert acc_b["up"]["bytes"] == act * 2 * f * d * 2 + rows * d * 2
    assert acc_f["down"] == acc_b["down"]
    assert acc_f["up"]["flops"] == acc_b["up"]["flops"]
    assert lay_b["bytes"] - lay_f["bytes"] == act * 2 * f * d * 2 - act * 2 * f * (d + 4)


def test_accounting_fp8_down_weights():
    """e4m3 down weights count one byte each plus a float32 scale per output
    channel; the up projection's figures are those of the fp8 gate/up layer;
    the down projection's flops are unchanged."""
    f8 = W.get("gptoss16_fp8")
    fa = W.get("gptoss16_fp8all")
    assert fa.w_fp8 and fa.w2_fp8 and not f8.w2_fp8
    kept = [0] * f8.E
    for e in range(0, 64, 4):
        kept[e] = 4
    acc_f, lay_f = bench.accounting(f8, kept)
    acc_a, lay_a = bench.accounting(fa, kept)
    act, d, f = 16, f8.d, f8.f
    assert acc_a["up"] == acc_f["up"]
    assert acc_a["down"]["bytes"] == act * d * (f + 4)
    assert acc_f["down"]["bytes"] == act * d * f * 2
    assert acc_a["down"]["flops"] == acc_f["down"]["flops"]
    assert lay_f["bytes"] - lay_a["bytes"] == act * d * f * 2 - act * d * (f + 4)
    assert bench.workload_config(fa)["expert_weights"].startswith("gate/up/down e4m3")


def test_fp8_up_projection_uses_the_fp8_tensor_peak():
    peaks = dict(bench.FALLBACK_PEAKS)
    acc = {"up": {"bytes": 1e6, "flops": 1e12}}
    r8 = bench.roofline_for("up", acc, 1.0, peaks, "fallback", fp8=True)
    r16 = bench.roofline_for("up", acc, 1.0, peaks, "fallback")
    assert r8["bound"] == r16["bound"] == "tensor"
    assert abs(r8["peak"] - 2 * r16["peak"]) < 0.2 and abs(r8["frac"] * 2 - r16["frac"]) < 1e-3


def test_default_arguments_finish_within_minutes(monkeypatch):
    monkeypatch.setattr("sys.argv", ["bench.py"])
    a = bench.parse()
    assert a.gpus == 1 and a.impl == "b300" and a.workload == "dsv3" and a.targets
    assert a.warmup >= 3 and a.steps >= 1


def test_combine_in_down_counts_y_as_output():
    s = W.SWITCH
    kept = [0] * 64
    kept[1] = 80
    acc, _ = bench.accounting(s, kept, combine_in_down=True)
    assert acc["down"]["bytes"] == s.d * s.f * 2 + s.T * s.d * 2
    assert acc["down"]["extra"] == 80 * s.f * 2


def test_cpu_baseline_and_routing_block_on_the_toy_layer():
    """The oracle legs of the bench on a small CPU layer: routing over the whole
    batch, whole experts timed, an all-core and a one-core figure, and the
    routing comparison (the oracle's own choice has no flips)."""
    import oracle.moe_oracle as O
    inp = W.make_inputs(W.TOY, "cpu")
    cb = bench.cpu_baseline(inp, 0.2)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["one_core"]["cores"] == 1
    assert cb["cpu_model"] and cb["host_cores"] >= 1
    sel = O.selection_scores(O.router_logits(bench._h64(inp.x), bench._h64(inp.W_r)),
                             W.TOY.gate)
    idx = torch.from_numpy(O.topk_indices(sel, W.TOY.k)).to(torch.int32)
    r = bench.routing_parity(inp, idx)
    assert r["tokens"] == 256 and r["flipped_tokens"] == 0 and r["flipped_outside_band"] == 0
    idx[0] = idx[0].flip(0)                      # a swapped order counts as a flip
    r = bench.routing_parity(inp, idx)
    assert r["flipped_tokens"] == 1


def test_fused_projections_count_as_one_kernel():
    """With the up and down projections in one launch, the "up" kernel's
    algorithmic bytes and FLOPs are the two projections' sums and "down" is
    empty; the layer's figures do not change."""
    s = W.SWITCH
    kept = [0] * 64
    kept[3], kept[7] = 80, 50
    two, lay2 = bench.accounting(s, kept, combine_in_down=True)
    one, lay1 = bench.accounting(s, kept, combine_in_down=True, fused=True)
    assert one["up"]["bytes"] == two["up"]["bytes"] + two["down"]["bytes"]
    assert one["up"]["flops"] == two["up"]["flops"] + two["down"]["flops"]
    assert one["down"]["bytes"] == 0 and lay1 == lay2


def test_roofline_reports_the_nominal_peaks_beside_the_measured_ones():
    peaks = dict(bench.FALLBACK_PEAKS)
    hbm = bench.roofline_for("down", {"down": {"bytes": 7.7e9, "flops": 1.0}}, 1000.0, peaks,
                             "fallback")
    assert hbm["bound"] == "hbm" and abs(hbm["frac_of_nominal"] - 1e-3) < 1e-9
    ten = bench.roofline_for("up", {"up": {"bytes": 1.0, "flops": 2.25e15}}, 1000.0, peaks,
                             "fallback")
    assert ten["bound"] == "tensor" and abs(ten["frac_of_nominal"] - 1.0) < 1e-9
    f8 = bench.roofline_for("up", {"up": {"bytes": 1.0, "flops": 2.25e15}}, 1000.0, peaks,
                            "fallback", fp8=True)
    assert abs(f8["frac_of_nominal"] - 0.5) < 1e-9


def test_workload_names():
    """Every name the bench and the profiles use resolves to the shape it
    names: the e4m3 suffixes, the decode sweep and the reduced DeepSeek-V3
    capture case (160 rows per expert on average, the full layer 128)."""
    full, small = W.get("dsv3"), W.get("dsv3_e32")
    assert (small.E, small.T) == (32, 640) and small.d == full.d and small.f == full.f
    assert small.T * small.k / small.E == 160 and full.T * full.k / full.E == 128
    assert small.n_shared == full.n_shared and small.gate == full.gate
    for T in (1, 16, 64, 256):
        g = W.get(f"gptoss{T}")
        assert g.T == T and not g.w_fp8
        f8 = W.get(f"gptoss{T}_fp8")
        assert f8.w_fp8 and not f8.w2_fp8 and f8.T == T
        fa = W.get(f"gptoss{T}_fp8all")
        assert fa.w_fp8 and fa.w2_fp8 and fa.T == T and fa.name == "gptoss_fp8all"
    m = W.get("mixtral_fp8all")
    assert m.w2_fp8 and m.f % 16 == 0
