#!/usr/bin/env python
"""Throughput of the B300 MoE layer forward pass (tokens/s), one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl b300|reference]
                    [--workload dsv3|switch|mixtral|gptoss<T>|toy|<name>_fp8|<name>_fp8all]
                    [--no-targets] [--no-cpu-baseline] [--no-e2e]

The default workload is the largest single-GPU layer, the DeepSeek-V3-shaped
one (256 routed SwiGLU experts of width 2048 on d = 7168, top-8 sigmoid
routing with a selection bias, one shared expert; T = 4096).

A step is one call of the whole layer (router, top-k, capacity, permute,
expert MLPs, combine and balance statistics) on one batch of seeded
synthetic input already resident in HBM.  K steps run back to back between
a barrier and a device synchronisation on each side, timed with CUDA
events on the launching stream; the job time is the maximum over ranks.
Each rank of a torchrun launch runs an independent replica on its own GPU
(weak scaling; the layer has no exchange step between replicas).

Also reported:
  roofline     the dominant kernel's algorithmic bytes (or FLOPs) per launch
               over its average duration, from per-stage CUDA events recorded
               inside the timed region, against the measured peak;
  e2e          the same metric through moe_forward_host_io_batches: every step's
               x copied from pinned host memory and its y and loss copied back,
               the copies overlapping the neighbouring steps' layers;
  cpu_baseline the fp64 CPU oracle on the host cores, all BLAS threads and one
               (rank 0, N = 1 only): routing of the whole batch, whole experts
               timed on a seeded sample, the whole-layer time scaled from it;
  routing      near-tie and flipped tokens of the GPU's routing against the
               oracle over the whole batch;
  targets      (default run) the Mixtral-shaped prefill layer's grouped GEMM
               against the bf16 tensor peak and the gpt-oss-shaped decode
               sweep's weight streaming against HBM;
  clocks       SM clocks and throttle reasons sampled during the timed region.

--impl reference times the CPU oracle itself on the same workload (bounded
per-step samples), the way the pages' own numpy / PyTorch loops would run.
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/sec on 1 B300 (bf16); % of tensor-core or HBM roofline"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
STAGES = ("router", "topk", "permute", "up", "down", "combine")
DEFAULT_STEPS = {"switch": 5000, "toy": 5000, "mixtral": 300, "dsv3": 300, "gptoss": 3000}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="b300", choices=["b300", "reference"])
    ap.add_argument("--workload", default="dsv3")
    ap.add_argument("--no-targets", dest="targets", action="store_false",
                    help="skip the prefill / decode target layers measured beside the headline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="target CPU time of the oracle baseline sample")
    a = ap.parse_args()
    base = a.workload.rstrip("0123456789_T") or a.workload
    if a.steps is None:
        a.steps = DEFAULT_STEPS.get(base, 200)
    if a.warmup is None:
        a.warmup = max(3, min(20, a.steps // 10))
    a.warmup = max(3, a.warmup)
    return a


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, dist=None, device="cpu"):
    """Largest value over all ranks of the job (the job time is the slowest
    rank's).  `dist` is torch.distributed when the job has several ranks."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha():
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "sparse_mixture_experts_65_b300", "csrc", "*"))):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + fh.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------- accounting
def accounting(shape, kept, combine_in_down=False, fused=False):
    """Algorithmic bytes and FLOPs per launch of each kernel and of the layer,
    from the kept assignments per expert.  With `fused` the up and down
    projections are one launch: its figures are their sum, under "up".

    "bytes" counts only what the definition must move: the weights of the
    experts with at least one kept row (e4m3 gate/up, and with w2_fp8 down,
    weights at one byte plus a float32 scale per channel), the router weights, the kernel's input rows of
    x and the layer's outputs.  Intermediates that this implementation stores
    between kernels (the expert-ordered row copy, h, the expert outputs o, the
    float32 logits of the split router) are reported apart as "extra"."""
    T, d, E, k, f = shape.T, shape.d, shape.E, shape.k, shape.f
    el = 2 if shape.dtype == "bf16" else 4
    rows = int(sum(kept))
    active = int(sum(1 for c in kept if c > 0))
    sw = shape.act == "swiglu"
    m_up = 2 if sw else 1
    S, fs = shape.n_shared, shape.f_shared
    fp8 = getattr(shape, "w_fp8", False)
    w_el = 1 if fp8 else el                      # bytes per gate/up weight
    w_up = active * m_up * f * (d * w_el + (4 if fp8 else 0)) + S * 2 * fs * d * el
    fp8_dn = getattr(shape, "w2_fp8", False)
    w_dn = active * d * (f * (1 if fp8_dn else el) + (4 if fp8_dn else 0)) + S * d * fs * el
    a_el = 1 if fp8 else el                      # bytes per up-projection input element
    h_bytes = (rows * f + S * T * fs) * el
    o_bytes = (rows + S * T) * d * el
    y_bytes = T * d * el
    acc = {
        "router": {"bytes": T * d * el + E * d * el + T * k * 8, "flops": 2 * T * d * E,
                   "extra": 0},
        "topk": {"bytes": T * k * 8, "flops": 0, "extra": 2 * T * E * 4},
        # reads the kept rows of x; writes their expert-ordered copy (or, fp8,
        # their quantised form)
        "permute": {"bytes": rows * d * el, "flops": 0,
                    "extra": rows * (d * a_el + (4 if fp8 else 0))},
        "up": {"bytes": w_up + (rows + S * T) * d * a_el,
               "flops": 2 * rows * d * f * m_up + S * 2 * T * d * fs * 2, "extra": h_bytes},
        "down": {"bytes": w_dn + (y_bytes if combine_in_down else 0),
                 "flops": 2 * rows * f * d + S * 2 * T * fs * d,
                 "extra": h_bytes + (0 if combine_in_down else o_bytes)},
        "combine": {"bytes": y_bytes, "flops": 2 * rows * d, "extra": o_bytes},
    }
    if fused:
        up, dn = acc["up"], acc["down"]
        acc["up"] = {"bytes": up["bytes"] + dn["bytes"], "flops": up["flops"] + dn["flops"],
                     "extra": up["extra"] + dn["extra"]}
        acc["down"] = {"bytes": 0, "flops": 0, "extra": 0}
    layer_bytes = (w_up + w_dn + E * d * el + 2 * T * d * el)
    layer_flops = 2 * rows * (m_up + 1) * d * f + S * 2 * T * 3 * d * fs + 2 * T * d * E
    return acc, {"bytes": layer_bytes, "flops": layer_flops, "active_experts": active,
                 "kept_rows": rows, "active_weight_bytes": w_up + w_dn, "w_up": w_up,
                 "w_dn": w_dn}


# dense fp8 over dense bf16 tensor-core rate, nominal (4.5 / 2.25 PFLOP/s)
FP8_OVER_BF16 = 2.0
# B300 datasheet figures, reported beside the measured denominators: HBM3e
# bandwidth and the dense bf16 tensor-core rate
NOMINAL_HBM_GBS = 7700.0
NOMINAL_BF16_TFLOPS = 2250.0


def roofline_for(stage, acc, ms, peaks, peak_kind, fp8=False):
    """The binding roof of one kernel.  The fp8 variant's up projection
    multiplies e4m3 operands: its tensor peak is the measured bf16 peak times
    the nominal fp8/bf16 ratio."""
    a = acc[stage]
    sec = ms / 1e3
    mult = FP8_OVER_BF16 if (fp8 and stage == "up") else 1.0
    ridge = mult * peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    ai = a["flops"] / a["bytes"] if a["bytes"] else float("inf")
    if a["flops"] and ai > ridge:
        peak = round(mult * peaks["bf16_tflops_sustained"], 1)
        ach = a["flops"] / sec / 1e12
        what = ("e4m3 sustained (measured bf16 sustained x 2, the nominal fp8/bf16 ratio)"
                if mult != 1.0 else "bf16 sustained")
        return {"bound": "tensor", "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4),
                "frac_of_nominal": round(ach / (mult * NOMINAL_BF16_TFLOPS), 4),
                "kernel": stage,
                "peak_source": f"{peak_kind} {what} (kernel runs inside a seconds-long loop)",
                "flops_per_launch": a["flops"], "ms_per_launch": round(ms, 5)}
    ach = a["bytes"] / sec / 1e9
    peak = peaks["hbm_gbs"]
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
            "frac": round(ach / peak, 4), "frac_of_nominal": round(ach / NOMINAL_HBM_GBS, 4),
            "kernel": stage, "peak_source": f"{peak_kind} HBM copy",
            "bytes_per_launch": a["bytes"], "traffic_extra": a.get("extra", 0),
            "ms_per_launch": round(ms, 5)}


def ncu_traffic(stage, workload):
    """dram bytes per launch of a kernel from the committed ncu summary, or
    None when no capture exists for the current sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    ent = d.get(f"{workload}:{stage}")
    if not ent or ent.get("source_sha") != source_sha():
        return None
    return ent.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock and throttle reasons during the timed region: NVML when the
    Python bindings are installed, else `nvidia-smi -lms` in the background."""
    REASONS = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
               "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}
    SMI_FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index, period_s=0.005):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self._raw = []
        self.period = period_s
        self._stop = threading.Event()
        self._h = None
        self._smi = None
        self.error = None
        self._uuid = None
        try:
            import torch
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            self._uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nv = pynvml
            try:   # CUDA and NVML number devices differently: match by UUID
                self._h = pynvml.nvmlDeviceGetHandleByUUID(self._uuid)
            except Exception:
                self._h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
        except Exception as e:  # pragma: no cover - reported in the JSON line
            self.error = repr(e)

    window = (0.0, float("inf"))

    def mark(self, t0, t1):
        """Wall-clock bounds of the timed region (used to filter samples)."""
        self.window = (t0, t1)

    def _sample(self):
        nv = self._nv
        mhz = nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM)
        r = nv.nvmlDeviceGetCurrentClocksEventReasons(self._h)
        self._raw.append((time.time(), mhz, r))

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def start(self):
        if self._h is None:
            import subprocess
            try:
                cmd = ["nvidia-smi", f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                       "-lms", "20"]
                if self._uuid:
                    cmd += ["-i", self._uuid]
                self._smi = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                             text=True)
                time.sleep(0.1)
            except Exception as e:
                self.error = repr(e)
            return
        self._sample()
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def stop(self):
        if self._h is None:
            if self._smi is not None:
                time.sleep(0.05)
                self._smi.terminate()
                out, _ = self._smi.communicate(timeout=10)
                names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
                import datetime
                rows = []
                for line in out.strip().splitlines():
                    f = [v.strip() for v in line.split(",")]
                    if len(f) < 7 or not f[1].isdigit():
                        continue
                    try:
                        ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    except ValueError:
                        ts = None
                    rows.append((ts, f))
                lo, hi = self.window
                inside = [f for ts, f in rows if ts is None or lo - 0.05 <= ts <= hi + 0.05]
                if not inside and rows:       # timed region shorter than one sample period
                    inside = [min(rows, key=lambda r: abs((r[0] or lo) - (lo + hi) / 2))[1]]
                for f in inside:
                    self.samples.append(int(f[1]))
                    self.max_mhz = int(f[2]) if f[2].isdigit() else self.max_mhz
                    for n, v in zip(names, f[3:7]):
                        if v.lower() == "active":
                            self.reasons.add(n)
            return
        self._sample()
        self._stop.set()
        self._t.join()
        lo, hi = self.window
        inside = [r for r in self._raw if lo <= r[0] <= hi] or self._raw[-1:]
        for _, mhz, r in inside:
            self.samples.append(mhz)
            for name, bit in self.REASONS.items():
                if r & bit:
                    self.reasons.add(name)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "samples": 0, "error": self.error}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": "nvml" if self._h is not None else "nvidia-smi"}


# ----------------------------------------------------------------- CPU oracle
def cpu_model():
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _openblas():
    """numpy's OpenBLAS and its thread-count getter / setter, found among the
    libraries this process has loaded (None when numpy uses another BLAS)."""
    import ctypes

    import numpy as np
    np.ones((2, 2)) @ np.ones((2, 2))            # make sure the BLAS is loaded
    try:
        with open("/proc/self/maps") as fh:
            paths = {ln.split()[-1] for ln in fh if "openblas" in ln.lower()}
    except OSError:
        return None
    for p in sorted(paths):
        try:
            lib = ctypes.CDLL(p)
        except OSError:
            continue
        for pre in ("scipy_openblas", "openblas"):
            for suf in ("64_", ""):
                get = getattr(lib, f"{pre}_get_num_threads{suf}", None)
                put = getattr(lib, f"{pre}_set_num_threads{suf}", None)
                if get is not None and put is not None:
                    get.restype = ctypes.c_int
                    put.argtypes = [ctypes.c_int]
                    return get, put
    return None


def blas_threads():
    ob = _openblas()
    return int(ob[0]()) if ob else (os.cpu_count() or 1)


class blas_limit:
    """Limits numpy's BLAS to `n` threads inside a `with` block (a no-op that
    reports False when the BLAS library offers no setter)."""

    def __init__(self, n):
        self.n, self.ob, self.old = n, _openblas(), None

    def __enter__(self):
        if self.ob:
            self.old = int(self.ob[0]())
            self.ob[1](self.n)
        return self.ob is not None

    def __exit__(self, *exc):
        if self.ob and self.old:
            self.ob[1](self.old)
        return False


def _h64(t):
    import numpy as np
    return None if t is None else t.detach().float().cpu().numpy().astype(np.float64)


class OracleLayer:
    """The CPU oracle on one workload's tensors: routing of the whole batch,
    then the expert stage expert by expert (the oracle groups its work by
    expert), so that a timed sample can cover whole experts."""

    def __init__(self, inp):
        import numpy as np
        self.np = np
        self.inp, self.s = inp, inp.shape
        self.x = _h64(inp.x)
        self.Wr, self.off, self.bias = _h64(inp.W_r), _h64(inp.logit_offset), _h64(inp.sel_bias)
        self.xe = self.x
        if inp.W1q is not None:           # e4m3 gate/up weights: quantised rows
            import oracle.moe_oracle as O
            vals, scales = O.quantize_rows_e4m3(self.x)
            self.xe = vals * scales[:, None]

    def route(self):
        import oracle.moe_oracle as O
        s = self.s
        return O.route(self.x, self.Wr, s.k, s.gate, self.off, self.bias, s.capacity_factor,
                       s.alpha)

    def expert_weights(self, e):
        """Expert e's matrices as float64 on the host (not timed)."""
        import oracle.moe_oracle as O
        inp = self.inp
        if inp.W1q is not None:
            w1 = O.dequantize_weights(inp.W1q[e].cpu().numpy(), inp.W1s[e].cpu().numpy())
            w3 = O.dequantize_weights(inp.W3q[e].cpu().numpy(), inp.W3s[e].cpu().numpy())
        else:
            w1 = _h64(inp.W1[e])
            w3 = _h64(inp.W3[e]) if inp.W3 is not None else None
        if getattr(inp, "W2q", None) is not None:
            w2 = O.dequantize_weights(inp.W2q[e].cpu().numpy(), inp.W2s[e].cpu().numpy())
        else:
            w2 = _h64(inp.W2[e])
        return w1, w3, w2

    def estimate(self, seconds, seed=0):
        """Seconds the oracle needs for the whole layer on this batch: routing
        timed in full; the routed experts timed on a seeded sample of whole
        experts (all their kept rows) until about `seconds` of CPU time, scaled
        by kept rows; the shared expert timed on a leading sample of tokens,
        scaled by tokens.  Returns (seconds, description)."""
        import oracle.moe_oracle as O
        np = self.np
        s = self.s
        t0 = time.perf_counter()
        _, _, idx, g, _, asg, _, _, _ = self.route()
        t_route = time.perf_counter() - t0
        rows_of = {}
        for t in range(s.T):
            for j in range(s.k):
                if asg.slot_pos[t, j] >= 0:
                    rows_of.setdefault(int(idx[t, j]), []).append((t, j))
        total = sum(len(v) for v in rows_of.values())
        order = np.random.default_rng(seed).permutation(sorted(rows_of))
        t_exp, done, n_exp = 0.0, 0, 0
        y = np.zeros((s.T, s.d))
        for e in order:
            w1, w3, w2 = self.expert_weights(int(e))
            items = rows_of[int(e)]
            tok = [t for t, _ in items]
            t0 = time.perf_counter()
            out = O.expert_ffn_rows(self.xe[tok], w1, w2, s.act, w3)
            for i, (t, j) in enumerate(items):
                y[t] += g[t, j] * out[i]
            t_exp += time.perf_counter() - t0
            done += len(items)
            n_exp += 1
            if t_exp >= 0.8 * seconds:
                break
        est = t_route + (t_exp * total / done if done else 0.0)
        desc = (f"routing of all {s.T} tokens {t_route:.2f} s; {n_exp} of {len(rows_of)} "
                f"active experts ({done} of {total} kept rows) {t_exp:.2f} s, scaled by rows")
        if s.n_shared:
            Ws1, Ws3, Ws2 = _h64(self.inp.Ws1), _h64(self.inp.Ws3), _h64(self.inp.Ws2)
            t_sh, n_sh = 0.0, 0
            while t_sh < 0.2 * seconds and n_sh < s.T:
                m = min(s.T - n_sh, max(1, n_sh or 64))
                t0 = time.perf_counter()
                O.expert_ffn_rows(self.x[n_sh:n_sh + m], Ws1, Ws2, O.ACT_SWIGLU, Ws3)
                t_sh += time.perf_counter() - t0
                n_sh += m
            est += t_sh * s.T / n_sh
            desc += f"; shared expert on {n_sh} tokens {t_sh:.2f} s, scaled by tokens"
        return est, desc


def cpu_baseline(inp, seconds):
    """The float64 oracle on the host cores: all BLAS threads, then one."""
    ol = OracleLayer(inp)
    T = inp.shape.T
    cores = blas_threads()
    est, desc = ol.estimate(seconds)
    out = {"value": round(T / est, 2), "unit": "tokens/s", "cores": cores,
           "kind": "oracle", "cpu_model": cpu_model(), "host_cores": host_cores(),
           "sample": f"float64 numpy oracle, whole-layer time estimated from: {desc}"}
    with blas_limit(1) as limited:
        if limited:
            est1, desc1 = ol.estimate(seconds)
            out["one_core"] = {"value": round(T / est1, 2), "unit": "tokens/s", "cores": 1,
                               "sample": desc1}
        else:
            out["one_core"] = {"value": None, "unavailable": "no BLAS thread control found"}
    return out


def routing_parity(inp, topk_idx):
    """Near-tie and flipped tokens of the GPU's routing against the oracle on
    the whole batch (flips are excused only inside the near-tie band)."""
    import numpy as np
    import oracle.moe_oracle as O
    s = inp.shape
    sel = O.selection_scores(O.router_logits(_h64(inp.x), _h64(inp.W_r), _h64(inp.logit_offset)),
                             s.gate, _h64(inp.sel_bias))
    ref = O.topk_indices(sel, s.k)
    gpu = topk_idx.cpu().numpy().astype(np.int64)
    near = O.near_tie_tokens(sel, s.k, 1e-5)
    flip = np.any(gpu != ref, axis=1)
    return {"tokens": s.T, "near_tie_tokens": int(near.sum()), "flipped_tokens": int(flip.sum()),
            "flipped_outside_band": int((flip & ~near).sum()), "band": 1e-5}


# ----------------------------------------------------------------- arms
def workload_config(shape, extra=None):
    c = {"workload": f"{shape.name} MoE layer", "T": shape.T, "d": shape.d, "E": shape.E,
         "k": shape.k, "f": shape.f, "act": shape.act, "gate": shape.gate,
         "capacity_factor": shape.capacity_factor or None, "n_shared": shape.n_shared,
         "f_shared": shape.f_shared or None, "alpha": shape.alpha}
    if getattr(shape, "w2_fp8", False):
        c["expert_weights"] = "gate/up/down e4m3 + float32 channel scales"
    elif getattr(shape, "w_fp8", False):
        c["expert_weights"] = "gate/up e4m3 + float32 channel scales, down bf16"
    if extra:
        c.update(extra)
    return c


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch
    from sparse_mixture_experts_65_b300 import workloads as W

    shape = W.get(args.workload)
    dev = "cuda" if torch.cuda.is_available() else "cpu"   # input generation only
    inp = W.make_inputs(shape, dev)
    ol = OracleLayer(inp)
    steps, warm = args.steps, args.warmup
    budget = 150.0                                # whole run, seconds
    per = max(1.0, budget / (steps + warm))
    for _ in range(warm):
        ol.estimate(per)
    ests, desc = [], ""
    t0 = time.perf_counter()
    for i in range(steps):
        est, desc = ol.estimate(per, seed=i)
        ests.append(est)
    wall = time.perf_counter() - t0
    value = steps * shape.T / sum(ests)
    sample = (f"each step: the float64 oracle's whole-layer time estimated from {desc} "
              f"({wall:.0f} s of CPU time for all steps)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": round(sum(ests) / steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(shape),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "kind": "oracle",
                             "cores": blas_threads(), "cpu_model": cpu_model(),
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_layer(shape, K, Wm, stream, dist=None, sample_clocks=True):
    """Times K forward calls of one workload (inputs resident in HBM) and, in
    a separate shorter pass, each stage with CUDA events between the stages."""
    import torch
    from sparse_mixture_experts_65_b300 import layer as L
    from sparse_mixture_experts_65_b300 import workloads as W

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    inp = W.make_inputs(shape, "cuda")
    cfg = L.config_for(shape)
    fwd = L.bound_forward(cfg, inp, stream=stream)
    fp8 = inp.W1q is not None
    for _ in range(Wm):
        fwd()
    torch.cuda.synchronize()
    assert L.check_status(fwd.workspace) == 0, "device status after warm-up"
    kept = fwd.out.expert_counts.cpu().tolist()
    flags = L.plan_flags(cfg, fp8)
    combine_in_down = "combine_in_down" in flags
    fused = "fused_projections" in flags
    acc, layer = accounting(shape, kept, combine_in_down, fused)

    # The timed region runs the plain forward call, exactly as a user issues
    # it (no per-stage events: an event between two kernels would stop the
    # next one from starting its prologue early).
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device()) if sample_clocks else None
    if clocks:
        clocks.start()
    for _ in range(Wm):
        fwd()
    barrier()
    w0 = time.time()
    start.record(stream)
    for _ in range(K):
        fwd()
    end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    if clocks:
        clocks.mark(w0, w1)
        clocks.stop()
    barrier()
    ms_total = max_over_ranks(start.elapsed_time(end), dist, "cuda")
    assert L.check_status(fwd.workspace) == 0, "device status after the timed region"
    K_st = min(K, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)]
           for _ in range(K_st)]
    arrs = [L.BoundForward.event_array(e, stream) for e in evs]
    for i in range(K_st):
        fwd(arrs[i])
    torch.cuda.synchronize()
    stage_ms = {s: statistics.fmean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K_st))
                for j, s in enumerate(STAGES)}
    return {"inp": inp, "cfg": cfg, "fwd": fwd, "fp8": fp8, "acc": acc, "layer": layer,
            "fused": fused,
            "ms_total": ms_total, "ms_step": ms_total / K, "stage_ms": stage_ms,
            "clocks": clocks.summary() if clocks else None,
            "launches_per_step": L.launch_count(cfg, fp8)}


def layer_roofline(layer, ms_step, peaks):
    sec = ms_step / 1e3
    return {"hbm_frac": round(layer["bytes"] / sec / 1e9 / peaks["hbm_gbs"], 4),
            "hbm_frac_of_nominal": round(layer["bytes"] / sec / 1e9 / NOMINAL_HBM_GBS, 4),
            "tensor_frac_sustained": round(layer["flops"] / sec / 1e12 /
                                           peaks["bf16_tflops_sustained"], 4),
            "bytes_per_step": layer["bytes"], "flops_per_step": layer["flops"],
            "active_experts": layer["active_experts"], "kept_rows": layer["kept_rows"]}


# Two performance targets of the layer, measured in the default run beside the
# headline: the prefill-shaped layer's grouped GEMM against the bf16 tensor
# peak, and the decode-shaped layer's active-expert weight streaming against
# HBM, over the decode sweep.
TARGETS = (("mixtral", 100, "up", ">= 0.60 of bf16 dense tensor peak in the grouped GEMM"),
           ("gptoss1", 1000, "up", ">= 0.70 of HBM for active-expert weight reads"),
           ("gptoss16", 300, "up", ">= 0.70 of HBM for active-expert weight reads"),
           ("gptoss64", 300, "up", ">= 0.70 of HBM for active-expert weight reads"),
           ("gptoss256", 300, "up", ">= 0.70 of HBM for active-expert weight reads"))


def measure_targets(stream, peaks, peak_kind):
    import gc

    import torch
    from sparse_mixture_experts_65_b300 import workloads as W
    out = {}
    for name, K, stage, target in TARGETS:
        shape = W.get(name)
        m = measure_layer(shape, K, 5, stream)
        acc = m["acc"]
        roof = roofline_for(stage, acc, m["stage_ms"][stage], peaks, peak_kind, m["fp8"])
        if m["fused"] and stage == "up":
            roof["kernel"] = "up+down (one launch)"
        ent = {"target": target, "steps": K, "ms_per_step": round(m["ms_step"], 5),
               "tokens_per_s": round(shape.T / (m["ms_step"] / 1e3), 1),
               "stage_ms": {s: round(v, 5) for s, v in m["stage_ms"].items()},
               "kernel": roof, "layer_roofline": layer_roofline(m["layer"], m["ms_step"], peaks),
               "clocks": m["clocks"]}
        if shape.T <= 256:
            # decode: the active experts' gate/up weights streamed by the up
            # projection, over its duration (with both projections in one
            # launch: all their weights, over that launch)
            w = m["layer"]["w_up"] + (m["layer"]["w_dn"] if m["fused"] else 0)
            gbs = w / (m["stage_ms"][stage] / 1e3) / 1e9
            ent["weight_stream_gbs"] = round(gbs, 1)
            ent["weight_stream_frac"] = round(gbs / peaks["hbm_gbs"], 4)
        out[name] = ent
        del m
        gc.collect()
        torch.cuda.empty_cache()
    return out


def run_b300(args):
    import gc

    import torch
    from sparse_mixture_experts_65_b300 import layer as L
    from sparse_mixture_experts_65_b300 import workloads as W

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    shape = W.get(args.workload)
    stream = torch.cuda.current_stream()
    K, Wm = args.steps, args.warmup
    m = measure_layer(shape, K, Wm, stream, dist)
    inp, cfg, fwd, fp8, acc, layer = m["inp"], m["cfg"], m["fwd"], m["fp8"], m["acc"], m["layer"]
    stage_ms, ms_total, ms_step = m["stage_ms"], m["ms_total"], m["ms_step"]
    value = world * shape.T * K / (ms_total / 1e3)

    peaks, peak_kind = load_peaks()
    dominant = max(STAGES, key=lambda s: stage_ms[s])
    roof = roofline_for(dominant, acc, stage_ms[dominant], peaks, peak_kind, fp8)
    roof["traffic"] = ncu_traffic(dominant, shape.name)
    roof["share_of_step"] = round(stage_ms[dominant] / sum(stage_ms.values()), 4)
    if m["fused"] and dominant == "up":
        roof["kernel"] = "up+down (one launch)"
    layer_roof = layer_roofline(layer, ms_step, peaks)

    e2e = None
    if not args.no_e2e:
        # The user's call for a stream of batches in host memory: each step is
        # one batch, its x copied in from pinned host memory and its y and loss
        # copied back, the copies overlapping the layer of the neighbouring
        # batches (moe_forward_host_io_batches).  A ring of 4 pinned buffers
        # holds the batches (every step copies its full batch both ways).
        ring = 4
        x_h = [inp.x.cpu().pin_memory() for _ in range(ring)]
        y_h = [torch.empty_like(x_h[0]).pin_memory() for _ in range(ring)]
        aux_h = torch.empty(max(K, Wm), dtype=torch.float32).pin_memory()
        cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
        warm = L.BoundHostIOBatches(cfg, [x_h[i % ring] for i in range(Wm)],
                                    [y_h[i % ring] for i in range(Wm)], aux_h, inp,
                                    stream=stream, copy_in_stream=cin, copy_out_stream=cout)
        hio = L.BoundHostIOBatches(cfg, [x_h[i % ring] for i in range(K)],
                                   [y_h[i % ring] for i in range(K)], aux_h, inp, stream=stream,
                                   copy_in_stream=cin, copy_out_stream=cout,
                                   workspace=warm.workspace)
        warm()
        barrier()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        hio()
        e2.record(stream)
        torch.cuda.synchronize()
        barrier()
        assert L.check_status(hio.workspace) == 0, "device status after the host-memory batches"
        ms_e2e = max_over_ranks(s2.elapsed_time(e2), dist, "cuda")
        io = shape.T * shape.d * x_h[0].element_size()
        e2e = {"value": round(world * shape.T * K / (ms_e2e / 1e3), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": io, "d2h_bytes_per_step": io + 4,
               "ms_per_step": round(ms_e2e / K, 5),
               "api": hio._fn.__name__}
        del hio, warm, x_h, y_h

    cpu = routing = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        routing = routing_parity(inp, fwd.out.topk_idx)
        cpu = cpu_baseline(inp, args.cpu_seconds)

    launches = m["launches_per_step"]
    clocks = m["clocks"]
    targets = None
    if rank == 0 and world == 1 and args.targets:
        del m, inp, fwd
        gc.collect()
        torch.cuda.empty_cache()
        targets = measure_targets(stream, peaks, peak_kind)

    active_w = layer["active_weight_bytes"]
    l2_note = (f"inputs larger than L2: {active_w / 1e6:.0f} MB of active expert weights "
               f"stream every step (L2 {L2_BYTES / 1e6:.0f} MB)") if active_w > L2_BYTES else \
        f"working set {active_w / 1e6:.0f} MB fits L2: numbers include L2 reuse across steps"
    line = {"impl": "b300", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("bf16+e4m3" if fp8 else "bf16") if shape.dtype == "bf16" else "f32",
            "data": "synthetic (seeded; the layer shape and input distributions of the workload)",
            "config": workload_config(shape, {"l2": l2_note,
                                              "parallelism": f"replicas x{world}"}),
            "roofline": roof, "layer_roofline": layer_roof,
            "stages_ms": {s: round(v, 5) for s, v in stage_ms.items()},
            "routing": routing, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": K * launches, "clocks": clocks,
            "targets": targets, "source_sha": source_sha()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_b300(args)


if __name__ == "__main__":
    main()
