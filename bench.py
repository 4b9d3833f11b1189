"""Benchmark of the grouped MXFP8 expert-FFN layer step on GB300.

One step = weight quantization of the bf16 masters (both orientations) +
route/permute/quantize + grouped gate_up GEMM with fused ScaledSwiGLU +
grouped down GEMM + combine + the full backward (dY quantization, down dgrad
with fused SwiGLU backward, down wgrad, gate_up dgrad, gate_up wgrad, dprob)
+ combine of dX.  Workload: Mixtral-8x7B-shaped expert MLP forward+backward
(T=16384, H=4096, I=14336, E=8, top-2), synthetic seeded inputs.

Metric: algorithmic TFLOP/s of the grouped expert MLP (18*R*H*I per step,
R = T*k) over the whole step time; also tokens/s and the fraction of the
dense MXFP8 tensor-core peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 (torchrun): every rank runs its own replica of the workload (the path
has no exchange step), timing is the max over ranks, value = all ranks' FLOPs
/ that time.  ``--impl reference`` times the CPU oracle on a bounded sample of
the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "mixtral_fwdbwd_T16384_H4096_I14336_E8_k2"
METRIC = "grouped expert-MLP fwd+bwd TFLOP/s (MXFP8, algorithmic 18*R*H*I per step)"
# dram__bytes_read.sum + dram__bytes_write.sum of the six grouped-GEMM launches of
# one step of the default workload, like `achieved` (which is over the same six
# launches): 5.558 GB from an ncu capture at T=4096, E=2 (every expert with the
# full workload's 4096 rows), times 4 for E=8 (profiles/ holds the summary).
# Set to None when the GEMM kernel changes, until it is captured again.
GEMM_TRAFFIC_BYTES = 22_233_000_000


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [s for s, p in zip(sm, power) if p > 200.0] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if gpus > 0 else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """The slowest rank's time: every replica's timed region ends with the barrier."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_replica: float, ms_max: float, world: int) -> float:
    """Whole-job rate of `world` independent replicas (weak scaling): all ranks' units / slowest time."""
    return world * units_per_replica / (ms_max * 1e-3)


# ------------------------------------------------------------------------------------
def run_cuda(args):
    import torch

    from moe_expert_ffn_03_gb300 import build, configs, synth
    from moe_expert_ffn_03_gb300.layer import ExpertFFN, launches_per_step
    from moe_expert_ffn_03_gb300.pipeline import HostPipeline

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    build.build()
    wl = pick_workload(args)
    train = wl.backward
    dev = torch.device("cuda", local)
    inp = synth.make_inputs(wl, seed=0, device=dev)
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=train, device=dev, bf16_training=train)
    stream = torch.cuda.current_stream()

    ev = {}
    # record: None (no events), "gemm" (only around the two grouped-MLP calls: the timed region,
    # where each event costs about 2 us of step time), "all" (every phase: a separate pass)
    GEMM_MARKS = ("route", "fwd", "comb", "bwd") if train else ("route", "fwd")

    def step(record=None):
        def mark(name):
            if record == "all" or (record == "gemm" and name in GEMM_MARKS):
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                ev.setdefault(name, []).append(e)
        mark("start")
        L.quantize_weights(inp["w_gu"], inp["w_d"])
        mark("wquant")
        L.route(inp["logits"], inp["x"])
        mark("route")
        L.ffn_forward()
        mark("fwd")
        L.combine_out()
        mark("comb")
        if train:
            L.ffn_backward(inp["dout"])
        mark("bwd")
        if train:
            L.combine_dx()
        mark("end")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    code, site = L.device_error()
    if code != 0:
        raise RuntimeError(f"device error {code} at site {site}")

    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step(record="gemm")
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    ms_total = t0.elapsed_time(t1)
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps

    def seg(a, b):
        return sum(x.elapsed_time(y) for x, y in zip(ev[a], ev[b])) / len(ev[a])

    # the grouped-MLP calls (the roofline's kernels) from the timed region itself
    gemm_parts = {"grouped_mlp_fwd_ms": seg("route", "fwd"),
                  "grouped_mlp_bwd_ms": seg("comb", "bwd") if train else 0.0}
    # every phase from a separate pass of the same steps, after the timed region
    ev.clear()
    for _ in range(args.steps):
        step(record="all")
    torch.cuda.synchronize()
    parts = {"weight_quant_ms": seg("start", "wquant"), "route_permute_ms": seg("wquant", "route"),
             "grouped_mlp_fwd_ms": gemm_parts["grouped_mlp_fwd_ms"], "combine_ms": seg("fwd", "comb"),
             "grouped_mlp_bwd_ms": gemm_parts["grouped_mlp_bwd_ms"], "combine_dx_ms": seg("bwd", "end")}
    code, site = L.device_error()
    if code != 0:
        raise RuntimeError(f"device error {code} at site {site}")

    flops = wl.flops_total()
    value = replica_throughput(flops, ms_step, world) / 1e12
    peaks, src = read_peaks()
    # the timed region is a fraction of a second: the burst bf16 figure is the one that applies
    # (x2: the nominal MXFP8/bf16 dense ratio 4.5/2.25); the sustained one is reported beside it
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    fp8_peak_sustained = 2.0 * peaks["bf16_tflops_sustained"]
    gemm_ms = parts["grouped_mlp_fwd_ms"] + parts["grouped_mlp_bwd_ms"]
    gemm_tflops = flops / (gemm_ms * 1e-3) / 1e12
    n_gemm = 6 if train else 2

    # ---- the tensor pipe's MXFP8 issue ceiling for the GEMM's instruction mix ----
    mma = mma_issue_ceiling(stream)

    # ---- end to end through the public API with pinned host buffers ----
    # HostPipeline: every step copies its inputs from pinned host memory and its results back;
    # the copies of step i+1's inputs and step i's results overlap the kernels on a copy stream.
    names = ("x", "logits", "dout") if train else ("x", "logits")
    host_sets = [{k: inp[k].cpu().pin_memory() for k in names} for _ in range(2)]
    out_sets = [{"out": torch.empty(L.out.shape, dtype=L.out.dtype).pin_memory(),
                 "dx": torch.empty(L.dx.shape, dtype=L.dx.dtype).pin_memory() if train else None}
                for _ in range(2)]
    bi = sum(t.numel() * t.element_size() for t in host_sets[0].values())
    bo = out_sets[0]["out"].numel() * 2 + (out_sets[0]["dx"].numel() * 2 if train else 0)
    pipe = HostPipeline(L, inp["w_gu"], inp["w_d"], stream)

    def host_steps(n):
        return [host_sets[i % 2] for i in range(n)], [out_sets[i % 2] for i in range(n)]

    pipe.run(*host_steps(max(1, args.warmup)))
    pipe.join()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipe.run(*host_steps(args.steps), after=e0)
    pipe.join()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    e2e_value = replica_throughput(flops, e2e_ms, world) / 1e12

    # the same steps with every copy in line on one stream, for comparison
    dev_in = {k: torch.empty_like(inp[k]) for k in names}

    def serial_step():
        for k in names:
            dev_in[k].copy_(host_sets[0][k], non_blocking=True)
        L.quantize_weights(inp["w_gu"], inp["w_d"])
        L.forward(dev_in["logits"], dev_in["x"])
        out_sets[0]["out"].copy_(L.out, non_blocking=True)
        if train:
            L.backward(dev_in["dout"])
            out_sets[0]["dx"].copy_(L.dx, non_blocking=True)

    serial_step()
    torch.cuda.synchronize()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(args.steps):
        serial_step()
    s1.record(stream)
    torch.cuda.synchronize()
    serial_ms = max_over_ranks(s0.elapsed_time(s1), world) / args.steps

    # ---- the same step replayed as one CUDA graph (launch gaps removed) ----
    graph = L.capture_step(inp["w_gu"], inp["w_d"], inp["logits"], inp["x"], inp.get("dout"))
    for _ in range(max(1, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(g0.elapsed_time(g1), world) / args.steps
    code, site = L.device_error()
    if code != 0:
        raise RuntimeError(f"device error {code} at site {site} (graph replay)")

    # ---- router on both sides (timed on its own; the step above starts from logits) ----
    router = None
    if train:
        w_r = synth.make_router_weight(wl, seed=0, device=dev)
        L.router_forward(inp["x"], w_r)
        L.router_backward(inp["x"], w_r)
        torch.cuda.synchronize()
        r0, r1, r2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        n_r = 10
        r0.record(stream)
        for _ in range(n_r):
            L.router_forward(inp["x"], w_r)
        r1.record(stream)
        for _ in range(n_r):
            L.router_backward(inp["x"], w_r)
        r2.record(stream)
        torch.cuda.synchronize()
        fwd_ms, bwd_ms = r0.elapsed_time(r1) / n_r, r1.elapsed_time(r2) / n_r
        xb = wl.T * wl.H * 2
        router = {"fwd_ms": round(fwd_ms, 4), "bwd_ms": round(bwd_ms, 4),
                  "fwd_gbs": round((xb + wl.E * wl.H * 2 + wl.T * wl.E * 4) / fwd_ms / 1e6, 1),
                  "bwd_gbs": round((3 * xb + 2 * wl.T * wl.E * 4) / bwd_ms / 1e6, 1),
                  "bytes": "fwd: x + W_r + logits; bwd: x (dW_r) + dx read and written + dlogits"}

    # ---- the same forward with bf16 operands (no quantization), for comparison ----
    L.forward_bf16(inp["x"], inp["w_gu"], inp["w_d"])
    torch.cuda.synchronize()
    from moe_expert_ffn_03_gb300 import binding as Bn
    b0, b1, b2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    n_b = 5
    gat = gem = 0.0
    for _ in range(n_b):
        b0.record(stream)
        Bn.moe_gather_rows(L.d, inp["x"], L.row_of, L.split_sizes, L.x_perm, L.ws)
        b1.record(stream)
        Bn.grouped_mlp_fwd_bf16(L.d, L.x_perm, L.split_sizes, L.prob_perm, inp["w_gu"], inp["w_d"], L.a_perm,
                                L.y_b16, L.ws)
        b2.record(stream)
        torch.cuda.synchronize()
        gat += b0.elapsed_time(b1)
        gem += b1.elapsed_time(b2)
    fwd_flops = 6.0 * wl.R * wl.H * wl.I
    bf16_fwd = {"gather_ms": round(gat / n_b, 4), "grouped_mlp_fwd_bf16_ms": round(gem / n_b, 4),
                "gemm_tflops": round(fwd_flops / (gem / n_b * 1e-3) / 1e12, 1),
                "frac_of_bf16_peak": round(fwd_flops / (gem / n_b * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"], 4),
                "mxfp8_grouped_mlp_fwd_ms": round(parts["grouped_mlp_fwd_ms"], 4)}

    # ---- the whole training step with bf16 operands (no quantization), for comparison ----
    bf16_train = None
    if train:
        def bf16_step():
            L.transpose_weights_bf16(inp["w_gu"], inp["w_d"])
            L.forward_bf16(inp["x"], inp["w_gu"], inp["w_d"])
            L.backward_bf16(inp["dout"])

        bf16_step()
        torch.cuda.synchronize()
        t0b = torch.cuda.Event(enable_timing=True)
        t1b = torch.cuda.Event(enable_timing=True)
        t0b.record(stream)
        for _ in range(n_b):
            bf16_step()
        t1b.record(stream)
        torch.cuda.synchronize()
        b_ms = t0b.elapsed_time(t1b) / n_b
        code, site = L.device_error()
        if code != 0:
            raise RuntimeError(f"device error {code} at site {site} (bf16 step)")
        bf16_train = {"ms_per_step": round(b_ms, 4), "tflops": round(flops / (b_ms * 1e-3) / 1e12, 1),
                      "frac_of_bf16_peak": round(flops / (b_ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"], 4),
                      "timed": "weight transposes + gather + bf16 forward + bf16 backward + both combines "
                               "(routing shared with the MXFP8 step, not timed here)",
                      "mxfp8_ms_per_step": round(ms_step, 4)}

    # ---- the same forward with per-tensor FP8 operands (one dynamic scale per expert tensor) ----
    L.quantize_weights_fp8_tensor(inp["w_gu"], inp["w_d"])
    L.forward_fp8_tensor(inp["x"])
    torch.cuda.synchronize()
    t0_, t1_, t2_, t3_ = (torch.cuda.Event(enable_timing=True) for _ in range(4))
    wq_t = qx_t = gm_t = 0.0
    for _ in range(n_b):
        t0_.record(stream)
        L.quantize_weights_fp8_tensor(inp["w_gu"], inp["w_d"])
        t1_.record(stream)
        Bn.moe_fp8_tensor_quantize_tokens(L.d, inp["x"], L.idx, L.row_of, L.split_sizes, L.t8_xq, L.t8_amax_x, L.ws)
        t2_.record(stream)
        Bn.grouped_mlp_fwd_fp8_tensor(L.d, L.t8_xq, L.t8_amax_x, L.split_sizes, L.prob_perm, L.t8_wgu,
                                      L.t8_amax_gu, L.t8_wd, L.t8_amax_d, L.t8_a, L.t8_aq, L.t8_amax_a, L.t8_y, L.ws)
        t3_.record(stream)
        torch.cuda.synchronize()
        wq_t += t0_.elapsed_time(t1_)
        qx_t += t1_.elapsed_time(t2_)
        gm_t += t2_.elapsed_time(t3_)
    t8_fwd = {"weight_quant_ms": round(wq_t / n_b, 4), "x_quant_ms": round(qx_t / n_b, 4),
              "grouped_mlp_fwd_fp8_tensor_ms": round(gm_t / n_b, 4),
              "tflops": round(fwd_flops / (gm_t / n_b * 1e-3) / 1e12, 1),
              "frac_of_fp8_peak": round(fwd_flops / (gm_t / n_b * 1e-3) / 1e12 / fp8_peak, 4),
              "timed": "gate_up GEMM (bf16 a + amax) + per-tensor quantize of a + down GEMM",
              "mxfp8_grouped_mlp_fwd_ms": round(parts["grouped_mlp_fwd_ms"], 4)}

    # ---- the whole training step with per-tensor FP8 operands, for comparison ----
    t8_train = None
    if train:
        def t8_step():
            L.quantize_weights_fp8_tensor(inp["w_gu"], inp["w_d"])
            L.forward_fp8_tensor(inp["x"])
            L.backward_fp8_tensor(inp["dout"])

        t8_step()
        torch.cuda.synchronize()
        t0t = torch.cuda.Event(enable_timing=True)
        t1t = torch.cuda.Event(enable_timing=True)
        t0t.record(stream)
        for _ in range(n_b):
            t8_step()
        t1t.record(stream)
        torch.cuda.synchronize()
        tt_ms = t0t.elapsed_time(t1t) / n_b
        code, site = L.device_error()
        if code != 0:
            raise RuntimeError(f"device error {code} at site {site} (per-tensor FP8 step)")
        t8_train = {"ms_per_step": round(tt_ms, 4), "tflops": round(flops / (tt_ms * 1e-3) / 1e12, 1),
                    "frac_of_fp8_peak": round(flops / (tt_ms * 1e-3) / 1e12 / fp8_peak, 4),
                    "timed": "weight amax + codes, x amax + codes, forward (bf16 a + its codes), backward "
                             "(dY and dH amax + codes, code transposes), both combines (routing shared)",
                    "mxfp8_ms_per_step": round(ms_step, 4)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_tokens, wl)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "mxfp8-e4m3 (ue8m0 block-32 scales, fp32 accumulate)",
        "data": "synthetic (seeded SplitMix64/Box-Muller: x~N(0,1), W~N(0,0.02^2), dout~N(0,0.01^2), logits~N(0,1))",
        "config": arm_config(wl, world),
        "tokens_per_s": round(replica_throughput(wl.T, ms_step, world), 1),
        "frac_of_mxfp8_peak": round(value / world / fp8_peak, 4),
        "frac_of_mxfp8_peak_sustained": round(value / world / fp8_peak_sustained, 4),
        "frac_of_mma_issue_ceiling": round(value / world / mma["tflops"], 4),
        "breakdown_ms": {k: round(v, 4) for k, v in parts.items()},
        "breakdown_how": "grouped_mlp_fwd/bwd from events around those calls inside the timed region; "
                         "the other phases from a separate pass of the same steps after it",
        "roofline": {"bound": "tensor", "kernel": f"grouped_gemm_kernel ({n_gemm} launches per step)",
                     "achieved": round(gemm_tflops, 2), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / fp8_peak, 4),
                     "traffic": GEMM_TRAFFIC_BYTES if wl.name == WORKLOAD else None,
                     "traffic_unit": "bytes per step over the six GEMM launches",
                     "peak_source": f"{src}: 2 x bf16_tflops (burst; the timed region is under a second; "
                                    f"fp8/bf16 nominal ratio 4.5/2.25)",
                     "frac_of_sustained_peak": round(gemm_tflops / fp8_peak_sustained, 4),
                     "mma_issue_ceiling": mma["tflops"],
                     "frac_of_mma_issue_ceiling": round(gemm_tflops / mma["tflops"], 4),
                     "timed": "grouped_mlp_fwd + grouped_mlp_bwd calls (the backward call also holds "
                              "4 small quantize/reduce launches)",
                     "launches_per_step": n_gemm},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "api": "HostPipeline.run (copies overlapped on a copy stream)",
                "serial_copies_ms_per_step": round(serial_ms, 4)},
        "gpu_launches": launches_per_step(wl.T, wl.E, wl.k, train) * args.steps,
        "clocks": clocks,
    }
    line["graph"] = {"ms_per_step": round(graph_ms, 4),
                     "value": round(replica_throughput(flops, graph_ms, world) / 1e12, 2), "unit": "TFLOP/s",
                     "how": "ExpertFFN.capture_step: the whole step as one CUDA graph, replayed"}
    line["mma_issue_ceiling"] = dict(mma, how="moe_selftest_mma_issue: per 128-deep K step 3 scale copies + "
                                               "4 tcgen05.mma.cta_group::2 mxf8f6f4 block_scale M=256 N=256 K=32, "
                                               "resident operands, no loads, no epilogue; best of 3")
    line["bf16_forward"] = bf16_fwd
    line["fp8_tensor_forward"] = t8_fwd
    if bf16_train is not None:
        line["bf16_training_step"] = bf16_train
    if t8_train is not None:
        line["fp8_tensor_training_step"] = t8_train
    if router is not None:
        line["router"] = router
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line))


def mma_issue_ceiling(stream, k_steps: int = 16384, reps: int = 3):
    """The library's MMA issue self-test: CTA pairs issuing the GEMM's MXFP8 MMAs (and scale
    copies) back to back on resident operands, no loads, no epilogue; best of `reps`."""
    import torch

    from moe_expert_ffn_03_gb300 import binding as Bn
    scratch = torch.zeros(256, dtype=torch.uint8, device=stream.device)
    Bn.moe_selftest_mma_issue(256, scratch, stream)
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pairs = Bn.moe_selftest_mma_issue(k_steps, scratch, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    code, site = Bn.moe_get_device_error(scratch, stream)
    if code != 0:
        raise RuntimeError(f"device error {code} at site {site} (MMA issue self-test)")
    tflops = pairs * k_steps * 2.0 * 256 * 256 * 128 / (best * 1e-3) / 1e12
    return {"tflops": round(tflops, 1), "ms": round(best, 4), "pairs": pairs, "k_steps": k_steps}


# ------------------------------------------------------------------------------------
_SAMPLE_INPUTS: dict = {}


def cpu_baseline(tokens: int, wl=None):
    """The oracle (numpy, float64) on a bounded sample: `tokens` tokens routed to the
    workload's first expert, full H and the first half of that expert's intermediate
    features (I/2 rows of the gate and of the up projection, I/2 columns of the down
    projection), forward and (when the workload trains) backward, weight quantization
    included (that quantization is most of the sample's time)."""
    import numpy as np
    import torch

    from moe_expert_ffn_03_gb300 import configs, synth
    from oracle import expert_ffn as ef
    from oracle import routing as rt

    wl = wl or configs.get(WORKLOAD)
    E_s = 1
    I_s = max(128, (wl.I // 2) // 128 * 128)
    key = (tokens, wl.name, I_s)
    if key not in _SAMPLE_INPUTS:
        # the first `tokens` tokens and expert 0's weights: the first values of each tensor's
        # counter-based stream, equal to the same slices of the full workload's tensors
        f64 = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
        sub = configs.small(tokens, wl.H, wl.I, wl.E, wl.k, routing=wl.routing, backward=True)
        x = synth.normal_bf16(synth.stream_key(0, synth.TID_X), (tokens, wl.H), 1.0, "cpu")
        dout = synth.normal_bf16(synth.stream_key(0, synth.TID_DOUT), (tokens, wl.H), sub.g_std, "cpu")
        w_gu0 = synth.normal_bf16(synth.stream_key(0, synth.TID_WGU), (1, 2 * wl.I, wl.H), sub.w_std, "cpu")
        w_d0 = synth.normal_bf16(synth.stream_key(0, synth.TID_WD), (1, wl.H, wl.I), sub.w_std, "cpu")
        logits = synth.make_logits(sub, 0, "cpu").numpy().copy()
        logits[:, E_s:] = -1e30                               # route over the sampled experts only
        w_gu = f64(torch.cat([w_gu0[:, :I_s], w_gu0[:, wl.I:wl.I + I_s]], dim=1))
        _SAMPLE_INPUTS.clear()
        _SAMPLE_INPUTS[key] = (f64(x), f64(dout), logits, w_gu, f64(w_d0[:, :, :I_s]))
    x, dout, logits, w_gu, w_d = _SAMPLE_INPUTS[key]
    t0 = time.perf_counter()
    k = min(wl.k, E_s)
    idx, prob = rt.route_topk(logits[:, :E_s], k)
    fwd = ef.forward(x, idx, prob.astype(np.float64), w_gu, w_d)
    if wl.backward:
        ef.backward(fwd, dout)
    dt = time.perf_counter() - t0
    flops = (18.0 if wl.backward else 6.0) * tokens * k * wl.H * I_s
    return {"value": round(flops / dt / 1e12, 5), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"{tokens} tokens x top-{k} over {E_s} of the {wl.E} experts, H={wl.H}, "
                      f"{I_s} of its I={wl.I} intermediate features, "
                      f"{'fwd+bwd' if wl.backward else 'fwd'} incl. weight quantization "
                      f"(numpy float64, BLAS threads = all host cores)"}


def arm_config(wl, world: int) -> dict:
    """The workload's config block, the same for both arms."""
    return {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
            "pass": "fwd+bwd" if wl.backward else "fwd", "global_batch_tokens": wl.T * world,
            "l2": "inputs larger than L2 (the bf16 weights are re-read every step); no flush",
            "parallelism": f"replicas x{world} (no exchange step)"}


def run_reference(args):
    world, rank, _ = dist_setup(0)
    if rank != 0:
        return
    wl = pick_workload(args)
    for _ in range(args.warmup):
        cpu_baseline(max(32, args.cpu_tokens // 4), wl)
    vals, secs = [], []
    for _ in range(args.steps):
        r = cpu_baseline(args.cpu_tokens, wl)
        vals.append(r["value"])
        secs.append(r["seconds"])
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * statistics.median(secs), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic", "config": arm_config(wl, max(1, args.gpus)),
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def pick_workload(args):
    from moe_expert_ffn_03_gb300 import configs
    wl = configs.get(args.workload)
    if args.tokens or args.experts:
        T = args.tokens or wl.T
        E = args.experts or wl.E
        wl = configs.small(T, wl.H, wl.I, E, min(wl.k, E), routing=wl.routing, backward=wl.backward,
                           name=f"{wl.name}_T{T}_E{E}")
    return wl


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=WORKLOAD, help="a workload name from moe_expert_ffn_03_gb300.configs")
    ap.add_argument("--tokens", type=int, default=0, help="override T (smaller cases for profiling)")
    ap.add_argument("--experts", type=int, default=0, help="override E (smaller cases for profiling)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=128)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "cuda":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
