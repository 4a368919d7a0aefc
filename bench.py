#!/usr/bin/env python
"""Benchmark of the fused EXL3 routed-expert MoE layer on GB300.

Headline: the decode-shaped layer (hidden 5120, inter 1536, 192 experts, top-8,
K=3 mcg, bf16) at M=1 token: routed tokens/s of one layer call, with the L2
flushed (256 MB write) before every timed step so the trellis words come from
HBM.  The same line carries the M = 8 / 32 / 128 sweep, the other layers of
the five workloads (the 16-token tiny layer, the mixed-width 288-expert layer
at M=64, the M=3072 prefill layer with Zipf-skewed routing, the additive
residual layer at M=512), the HBM roofline of the dominant kernel, the
prompt-sized linear, an end-to-end figure through the C ABI with host buffers
and the float64 CPU oracle timed on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --case decode|prefill|linear --M ROWS   # one layer (profiling target)

With --gpus N > 1 (under torchrun) every rank runs an independent replica
(the layer has no exchange step on one GPU); value = tokens of all ranks /
max over ranks of the timed-region time.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "routed tokens/s and HBM GB/s (% roofline) per EXL3 MoE layer at M=1 and M=3072"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# Sources the decode-regime gate/up kernel is compiled from: its DRAM traffic
# in profiles/traffic.json is valid while these are unchanged.
GATE_UP_SOURCES = ("expert_gemm.cuh", "gemm_gateup.cu", "common.cuh", "epilogue.cuh",
                   "rotate_block.cuh", "kernels.h", "plan.h")


def _src_hash(files=GATE_UP_SOURCES):
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "trellis_quantized_moe_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(kernel):
    """DRAM bytes per launch from a committed ncu summary, if the sources match."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d.get(kernel)
        if e and e.get("src_hash") == _src_hash():
            return e["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


class Clocks:
    """nvidia-smi samples (200 ms) during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                for n, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
            os.unlink(self.path)
        except Exception:
            pass
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        return dist, dist.get_rank(), int(os.environ.get("LOCAL_RANK", "0")), ws
    return None, 0, 0, 1


def _max_over_ranks(dist, v):
    """The slowest rank's time: every rank gets the maximum of v."""
    if dist is None:
        return v
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _layer_bytes(w, ids):
    """Algorithmic HBM bytes of one layer call: trellis words of the touched
    experts, their fp16 rotation/scale vectors, activations in and out."""
    s = w.spec
    act = 2
    active = np.unique(ids)
    trellis = sum(3 * s.hidden * s.inter * int(s.K[e]) // 8 for e in active)
    vectors = len(active) * (4 * s.hidden + 5 * s.inter) * 2
    io = s.M * s.hidden * act * 2 + ids.size * (4 if s.ids_dtype == "i32" else 8) + ids.size * 2
    return trellis + vectors + io


# The trellis decode of one weight takes 4 integer operations: 2 on the ALU
# pipe (the state's right shift; the codebook's mask/xor as one LOP3) and 2 on
# the FMA pipe (the state's left shift as a multiply; the codebook multiply).
# Each pipe issues 64 lane-operations per cycle per SM (16 per sub-partition),
# so the decode peak is 2 x 64 / 4 = 32 weights per cycle per SM.
ALU_OPS_PER_WEIGHT = 4
ALU_LANES_PER_SM = 128


def _alu_peak_weights(dev):
    """Decode peak in weights/s: SMs x integer lanes x max SM clock / ops per weight."""
    import torch
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", 2070.0))
    except Exception:
        mhz = 2070.0
    return nsm * ALU_LANES_PER_SM * mhz * 1e6 / ALU_OPS_PER_WEIGHT, nsm, mhz


def _gateup_weights(w, ids):
    """Weights the gate/up kernel decodes: both projections of every touched
    expert, once per row group (one group per expert at M=1)."""
    s = w.spec
    return len(np.unique(ids)) * 2 * s.hidden * s.inter


def _gateup_bytes(w, ids):
    """Algorithmic bytes of the gate/up kernel: gate+up trellis of the touched
    experts, their vectors, rotated fp16 inputs in, fp16 down inputs out."""
    s = w.spec
    active = np.unique(ids)
    R = ids.size
    trellis = sum(2 * s.hidden * s.inter * int(s.K[e]) // 8 for e in active)
    vectors = len(active) * (2 * (s.hidden + 2 * s.inter) + s.inter) * 2
    return trellis + vectors + R * 2 * s.hidden * 2 + R * s.inter * 2


def _residual_bytes(w, ids):
    """Trellis bytes of the residual stages with a nonzero scale, over the
    experts the routes touch (the additive layer reads nothing else)."""
    s = w.spec
    total = 0
    for st in range(1, s.num_stages):
        K = int(s.residual_K[st - 1])
        for e in np.unique(ids):
            for p in range(3):
                if w.alpha[st - 1, e, p] != 0.0:
                    i, o = s.proj_shape(p)
                    total += i * o * K // 8
    return total


def _fp16_peak(dev, n=8192, reps=10):
    """Dense fp16 torch.matmul n^3 throughput (best of reps, CUDA events): the
    tensor-core denominator of the prefill and linear fractions."""
    import torch
    a = torch.randn(n, n, dtype=torch.float16, device=dev)
    b = torch.randn(n, n, dtype=torch.float16, device=dev)
    for _ in range(2):
        torch.matmul(a, b)
    best = float("inf")
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a, b)
        e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del a, b
    torch.cuda.empty_cache()
    return 2.0 * n ** 3 / (best * 1e-3) / 1e12


def run_reference(args):
    """The float64 oracle on the host cores, each step one bounded sample."""
    from oracle import exl3_oracle as O
    from workloads import MoEWorkload, act_to_f64, config, rw_to_f64
    w = MoEWorkload(config(1, M=1))
    s = w.spec
    x, rw = act_to_f64(w.x, s.act), rw_to_f64(w.rw, s.rw_dtype)

    def step():
        O.moe_forward(x, w.ids, rw, w.projection)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = args.steps * s.M / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded uniform trellis words, N(0,1) activations, softmax top-8 routing)",
        "config": {"workload": "decode-shaped EXL3 MoE layer, hidden 5120, inter 1536, 192 experts,"
                               " top-8, K=3 mcg, M=1", "M": 1},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": O.oracle_threads(), "kind": "oracle",
                         "sample": "one M=1 layer call (8 experts decoded) per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def cpu_baseline(budget_s=12.0):
    """Oracle tokens/s on the host cores: repeated M=1 decode-layer calls."""
    from oracle import exl3_oracle as O
    from workloads import MoEWorkload, act_to_f64, config, rw_to_f64
    n, t_used = 0, 0.0
    t_start = time.perf_counter()
    while t_used < budget_s and n < 6:
        w = MoEWorkload(config(1, M=1))
        s = w.spec
        x, rw = act_to_f64(w.x, s.act), rw_to_f64(w.rw, s.rw_dtype)
        t0 = time.perf_counter()
        O.moe_forward(x, w.ids, rw, w.projection)
        t_used += time.perf_counter() - t0
        n += 1
        if time.perf_counter() - t_start > 3 * budget_s:
            break
    return {"value": n / t_used, "unit": UNIT, "cores": O.oracle_threads(), "kind": "oracle",
            "sample": f"{n} M=1 decode-layer calls (8 experts each, float64, C decode + numpy)"}


def run_ours(args):
    import torch
    dist, rank, local_rank, world = _dist()
    torch.cuda.set_device(local_rank)
    import trellis_quantized_moe_gb300 as X
    from workloads import MoEWorkload, config

    hbm_peak, bf16_peak, bf16_sust, peak_src = _peaks()
    dev = torch.device("cuda", local_rank)

    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}

    def to_dev(a, dt):
        if dt == "bf16":
            return torch.from_numpy(a.view(np.int16).copy()).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def dev_inputs(w):
        s = w.spec
        x = to_dev(w.x, s.act)
        ids = torch.from_numpy(w.ids.astype(np.int64 if s.ids_dtype == "i64" else np.int32)).to(dev)
        rw = to_dev(w.rw, s.rw_dtype)
        out = torch.empty((s.M, s.hidden), dtype=tdt[s.act], device=dev)
        return x, ids, rw, out

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def timed(call, steps, warmup, profile=False):
        """Per-step device time (ms) with an L2 flush before each step."""
        for _ in range(warmup):
            flush.fill_(1)
            call()
        torch.cuda.synchronize()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        profs = [X.binding.ProfileEvents() for _ in range(steps)] if profile else None
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            flush.fill_(i & 0xFF)
            starts[i].record()
            if profile:
                with profs[i]:
                    call()
            else:
                call()
            ends[i].record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        if dist is not None:
            dist.barrier()
        ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        kern = np.array([p.times_ms() for p in profs]) if profile else None
        return ms, kern, wall

    if args.case in ("decode", "prefill"):
        # one case at args.M (profiling target); short JSON
        w = MoEWorkload(config(1 if args.case == "decode" else 3, M=args.M))
        ex = X.DeviceExperts.from_workload(w)
        s = w.spec
        ws = torch.empty(X.exl3_moe_workspace_bytes(s.M, s.topk, s.E, s.hidden, s.inter,
                                                    s.capacity), dtype=torch.uint8, device=dev)
        x, ids, rw, out = dev_inputs(w)
        ms, kern, _ = timed(lambda: X.exl3_moe_forward(x, ids, rw, ex, s.capacity, ws, out),
                            args.steps, args.warmup, profile=True)
        assert X.exl3_workspace_error(ws) == 0
        t = float(np.mean(ms))
        print(json.dumps({"case": f"{args.case} M={args.M}", "us": 1e3 * t,
                          "tokens_per_s": args.M / (t * 1e-3),
                          "layer_gbs": _layer_bytes(w, w.ids) / (t * 1e-3) / 1e9,
                          "kernel_us": [1e3 * float(v) for v in kern.mean(axis=0)]}))
        return

    if args.case == "linear":
        # the prompt-sized linear (5120 -> 1536, K=3 mcg, bf16) at args.M rows
        from workloads import CB_MCG, LinearWorkload
        lw = LinearWorkload(M=args.M, in_f=5120, out_f=1536, K=3, cb=CB_MCG, act="bf16", seed=41)
        ldp = X.DeviceProjection(lw.proj)
        lx = torch.from_numpy(lw.x.view(np.int16).copy()).to(dev).view(torch.bfloat16)
        ly = torch.empty((lw.M, 1536), dtype=torch.bfloat16, device=dev)
        lws = torch.empty(X.exl3_linear_workspace_bytes(lw.M, 5120, 1536), dtype=torch.uint8, device=dev)
        ms, _, _ = timed(lambda: X.exl3_linear(lx, ldp, ly, lws), args.steps, args.warmup)
        t = float(np.mean(ms))
        print(json.dumps({"case": f"linear M={args.M}", "us": 1e3 * t,
                          "tflops_dense_equiv": 2.0 * args.M * 5120 * 1536 / (t * 1e-3) / 1e12}))
        return

    def layer_case(cfg, name, steps, warmup, M=None):
        """One workload's layer: mean step time without events between the
        kernels, the per-kernel split from a separate profiled run, routed
        tokens and routes per second, and the HBM view (algorithmic bytes of
        the touched experts' trellis words, vectors and activations)."""
        w = MoEWorkload(config(cfg, M=M))
        s = w.spec
        ex = X.DeviceExperts.from_workload(w)
        st = (X.DeviceStages(w.residual, w.alpha, s.residual_K, s.E, device=dev)
              if s.num_stages > 1 else None)
        ws = torch.empty(X.exl3_moe_workspace_bytes(s.M, s.topk, s.E, s.hidden, s.inter, s.capacity),
                         dtype=torch.uint8, device=dev)
        x, ids, rw, out = dev_inputs(w)
        if st is None:
            call = lambda: X.exl3_moe_forward(x, ids, rw, ex, s.capacity, ws, out)  # noqa: E731
        else:
            call = lambda: X.exl3_moe_additive(x, ids, rw, ex, st, s.capacity, ws, out)  # noqa: E731
        c_ms, _, _ = timed(call, steps, warmup)
        _, c_kern, _ = timed(call, max(3, steps // 2), 1, profile=True)
        assert X.exl3_workspace_error(ws) == 0
        t = float(np.mean(c_ms))
        b = _layer_bytes(w, w.ids) + (_residual_bytes(w, w.ids) if st is not None else 0)
        res = {"workload": name, "M": s.M, "us": 1e3 * t, "tokens_per_s": s.M / (t * 1e-3),
               "routes_per_s": s.M * s.topk / (t * 1e-3), "algorithmic_bytes": b,
               "layer_gbs": b / (t * 1e-3) / 1e9, "layer_frac_hbm": b / (t * 1e-3) / 1e9 / hbm_peak,
               "regime": "prefill (tcgen05)" if int(ws[:64 * 4].view(torch.int32)[8].item()) else "decode",
               "kernel_us": [1e3 * float(v) for v in c_kern.mean(axis=0)]}
        del ex, st, ws
        torch.cuda.empty_cache()
        return res

    # ---------------- decode-shaped layer (headline M=1 and the M sweep)
    base = MoEWorkload(config(1, M=1))
    ex = X.DeviceExperts.from_workload(base)
    spec = base.spec
    Ms = [1, 8, 32, 128]
    wls = {M: MoEWorkload(config(1, M=M)) for M in Ms}
    ws = torch.empty(X.exl3_moe_workspace_bytes(128, 8, spec.E, spec.hidden, spec.inter,
                                                spec.capacity), dtype=torch.uint8, device=dev)
    inputs = {M: dev_inputs(wls[M]) for M in Ms}

    def layer(M):
        x, ids, rw, out = inputs[M]
        return lambda: X.exl3_moe_forward(x, ids, rw, ex, spec.capacity, ws, out)

    with Clocks(local_rank) as clk:
        ms, _, wall = timed(layer(1), args.steps, args.warmup)
    clocks = clk.summary()
    # per-kernel split from a separate run with events between the kernels
    # (events in the stream also serialise the programmatically dependent
    # launches, so the headline steps above run without them)
    _, kern, _ = timed(layer(1), max(5, args.steps // 4), 2, profile=True)
    assert X.exl3_workspace_error(ws) == 0
    t_step = float(np.mean(ms))
    t_step_max = _max_over_ranks(dist, t_step)
    value = world * 1 / (t_step_max * 1e-3)
    kmean = kern.mean(axis=0)
    w1 = wls[1]
    layer_bytes = _layer_bytes(w1, w1.ids)
    gu_bytes = _gateup_bytes(w1, w1.ids)
    gu_ms = float(kmean[2])
    achieved = gu_bytes / (gu_ms * 1e-3) / 1e9
    alu_peak, nsm, mhz = _alu_peak_weights(dev)
    gu_weights = _gateup_weights(w1, w1.ids)
    achieved_w = gu_weights / (gu_ms * 1e-3)

    sweep = {}
    for M in Ms[1:]:
        m_ms, _, _ = timed(layer(M), max(5, args.steps // 4), 2)
        _, m_kern, _ = timed(layer(M), 5, 1, profile=True)
        tm = float(np.mean(m_ms))
        b = _layer_bytes(wls[M], wls[M].ids)
        sweep[f"M={M}"] = {"us": 1e3 * tm, "tokens_per_s": M / (tm * 1e-3),
                           "routes_per_s": M * spec.topk / (tm * 1e-3),
                           "layer_gbs": b / (tm * 1e-3) / 1e9,
                           "layer_frac_hbm": b / (tm * 1e-3) / 1e9 / hbm_peak,
                           "kernel_us": [1e3 * float(v) for v in m_kern.mean(axis=0)]}

    # ---------------- the M=1 layer captured once in a CUDA graph and replayed
    def graph_timing():
        try:
            g = torch.cuda.CUDAGraph()
            cs = torch.cuda.Stream()
            cs.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(cs):
                layer(1)()                       # warm-up outside the capture
                cs.synchronize()
                with torch.cuda.graph(g, stream=cs):
                    layer(1)()
            torch.cuda.synchronize()
            g_ms, _, _ = timed(g.replay, args.steps, args.warmup)
            t = _max_over_ranks(dist, float(np.mean(g_ms)))
            return {"us": 1e3 * t, "tokens_per_s": world / (t * 1e-3)}
        except Exception as exc:                 # reported, not fatal
            return {"error": str(exc).splitlines()[0][:200]}

    graph = graph_timing()
    assert X.exl3_workspace_error(ws) == 0

    # ---------------- end to end through the C ABI with host buffers (M=1)
    # The step's inputs (activations, route ids, route weights) sit in one
    # pinned host buffer and one device buffer, each 16-byte aligned inside,
    # so a step is one host-to-device copy, the layer, one device-to-host copy.
    x0, ids0, rw0, out_d = inputs[1]
    parts = [x0, ids0, rw0]
    offs, nbytes = [], 0
    for t in parts:
        offs.append(nbytes)
        nbytes += (t.numel() * t.element_size() + 15) // 16 * 16
    stage_d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stage_h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()

    def view(buf, t, off):
        return buf[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    x_d, ids_d, rw_d = (view(stage_d, t, o) for t, o in zip(parts, offs))
    for t, o in zip(parts, offs):
        view(stage_h, t, o).copy_(t.cpu())
    out_h = torch.empty_like(out_d, device="cpu").pin_memory()

    def e2e_call():
        stage_d.copy_(stage_h, non_blocking=True)
        X.exl3_moe_forward(x_d, ids_d, rw_d, ex, spec.capacity, ws, out_d)
        out_h.copy_(out_d, non_blocking=True)

    e_ms, _, _ = timed(e2e_call, args.steps, args.warmup)
    e_t = _max_over_ranks(dist, float(np.mean(e_ms)))
    h2d = stage_h.numel()                       # the one staging copy, padding included
    d2h = out_h.numel() * out_h.element_size()

    # ---------------- the other workloads
    del ex
    torch.cuda.empty_cache()
    fp16_peak = _fp16_peak(dev)
    n_cfg = max(5, min(20, args.steps // 2))
    configs = {
        "tiny_m16": layer_case(0, "hidden 512, inter 256, 8 experts, top-2, 16 tokens, K=4 mcg, f16",
                               n_cfg, 3),
        "mixed_width_m64": layer_case(2, "hidden 4096, inter 1408, 288 experts, top-8, M=64, K in 4..8 "
                                         "per expert, 3inst (even) / mul1 (odd), f16, int64 ids",
                                      n_cfg, 3),
        "additive_m512": layer_case(4, "hidden 4096, inter 1408, 288 experts, top-8, M=512, base K=3 mcg "
                                       "+ one K=2 mcg residual stage (50% of projections at scale 0), "
                                       "bf16, int64 ids, f32 route weights",
                                    max(3, n_cfg // 2), 2),
    }

    # ---------------- prefill layer, M = 3072
    pw = MoEWorkload(config(3))
    ps = pw.spec
    pex = X.DeviceExperts.from_workload(pw)
    pws = torch.empty(X.exl3_moe_workspace_bytes(ps.M, ps.topk, ps.E, ps.hidden, ps.inter,
                                                 ps.capacity), dtype=torch.uint8, device=dev)
    px, pids, prw, pout = dev_inputs(pw)
    p_ms, p_kern, _ = timed(lambda: X.exl3_moe_forward(px, pids, prw, pex, ps.capacity, pws, pout),
                            max(3, min(10, args.steps // 5)), 1, profile=True)
    assert X.exl3_workspace_error(pws) == 0
    pt = float(np.mean(p_ms))
    flops = 2.0 * ps.M * ps.topk * 3 * ps.hidden * ps.inter
    prefill = {"workload": "hidden 5120, inter 1536, 192 experts, top-8, M=3072, K in {3,4} mcg, "
                           "Zipf(1.2) expert bias, capacity 512, bf16",
               "us": 1e3 * pt, "tokens_per_s": ps.M / (pt * 1e-3),
               "routes_per_s": ps.M * ps.topk / (pt * 1e-3),
               "tflops_dense_equiv": flops / (pt * 1e-3) / 1e12,
               "frac_of_fp16_peak": flops / (pt * 1e-3) / 1e12 / fp16_peak,
               "peak_tflops": fp16_peak,
               "peak_note": "dense fp16 torch.matmul 8192^3, best of 10, measured in this run",
               "frac_of_bf16_peak": flops / (pt * 1e-3) / 1e12 / bf16_peak,
               "layer_gbs": _layer_bytes(pw, pw.ids) / (pt * 1e-3) / 1e9,
               "kernel_us": [1e3 * float(v) for v in p_kern.mean(axis=0)]}
    del pex, pws
    torch.cuda.empty_cache()

    # ---------------- prompt-sized linear (one projection, no routing)
    from workloads import CB_MCG, LinearWorkload
    lw = LinearWorkload(M=4096, in_f=5120, out_f=1536, K=3, cb=CB_MCG, act="bf16", seed=41)
    ldp = X.DeviceProjection(lw.proj)
    lx = torch.from_numpy(lw.x.view(np.int16).copy()).to(dev).view(torch.bfloat16)
    ly = torch.empty((lw.M, 1536), dtype=torch.bfloat16, device=dev)
    lws = torch.empty(X.exl3_linear_workspace_bytes(lw.M, 5120, 1536), dtype=torch.uint8, device=dev)
    l_ms, _, _ = timed(lambda: X.exl3_linear(lx, ldp, ly, lws), max(3, min(10, args.steps // 5)), 2)
    lt = float(np.mean(l_ms))
    lflops = 2.0 * lw.M * 5120 * 1536
    linear = {"workload": "EXL3 linear 5120 -> 1536, K=3 mcg, bf16, M=4096 rows",
              "us": 1e3 * lt, "rows_per_s": lw.M / (lt * 1e-3),
              "tflops_dense_equiv": lflops / (lt * 1e-3) / 1e12,
              "frac_of_fp16_peak": lflops / (lt * 1e-3) / 1e12 / fp16_peak}
    del ldp, lws
    torch.cuda.empty_cache()

    if rank != 0:
        return
    cpu = cpu_baseline()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded uniform trellis words, N(0,1) activations, softmax top-8 routing)",
        "config": {"workload": "decode-shaped EXL3 MoE layer: hidden 5120, inter 1536, 192 experts,"
                               " top-8, M=1, K=3 mcg, bf16 in/out, f16 MMA operands, f32 accumulate",
                   "M": 1, "l2": "flushed before every timed step (256 MB write)",
                   "parallelism": f"replicas x{world}"},
        "routes_per_s": world * spec.topk / (t_step_max * 1e-3),
        "layer_gbs": layer_bytes / (t_step_max * 1e-3) / 1e9,
        "layer_frac_hbm": layer_bytes / (t_step_max * 1e-3) / 1e9 / hbm_peak,
        "kernel_us": dict(zip(["route_pack", "rotate", "gate_up", "down_combine"],
                              [1e3 * float(v) for v in kmean])),
        # the dominant kernel against HBM on its algorithmic bytes (the
        # metric's roofline); the integer-decode ceiling alongside
        "roofline": {"kernel": "k_expert_gemm<gate/up> (decode regime, M=1)", "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": _traffic("gate_up_m1"),
                     "algorithmic_bytes": gu_bytes, "peak_source": peak_src,
                     "alu_view": {"achieved": achieved_w / 1e9, "peak": alu_peak / 1e9,
                                  "unit": "Gweight/s", "frac": achieved_w / alu_peak,
                                  "algorithmic_weights": gu_weights,
                                  "peak_source": f"derived: {nsm} SMs x {ALU_LANES_PER_SM} integer "
                                                 f"lanes/clk (ALU + FMA pipes) x {mhz:.0f} MHz / "
                                                 f"{ALU_OPS_PER_WEIGHT} integer ops per decoded weight"}},
        "sweep": sweep,
        "graph_replay_m1": graph,
        "prefill_m3072": prefill,
        "configs": configs,
        "linear_m4096": linear,
        "fp16_dense_peak_tflops": fp16_peak,
        "e2e": {"value": world * 1 / (e_t * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "cpu_baseline": cpu,
        "clocks": clocks,
        # route pack, (rotate,) gate/up, down: layers of up to 32 routes rotate
        # inside the gate/up kernel
        "gpu_launches": (3 if 1 * spec.topk <= 32 else 4) * args.steps,
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--case", default="all", choices=["all", "decode", "prefill", "linear"],
                    help="decode / prefill / linear: only that layer at --M (profiling target)")
    ap.add_argument("--M", type=int, default=1)
    args = ap.parse_args()
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        run_reference(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
