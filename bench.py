#!/usr/bin/env python
"""Benchmark: fused QKV context-encoding projection on GB300, one JSON line.

A step is one pass of the whole path through the C ABI (scale-factor prep, the
tcgen05 MXFP8 GEMM with its fused epilogue, the norm + RoPE pass) over the Wan2.2
480p self-attention shape: T = 32760 tokens (21x30x52 latent grid), H = 5120,
40 Q + 40 KV heads of 128 (I = 15360), synthetic seeded inputs. The metric is the
projection's algorithmic FP8 TFLOP/s (2*T*H*I per step).

Timing: W untimed warm-up steps, then exactly K timed steps, each bracketed by CUDA
events on the launching stream; L2 is flushed (a 256 MB write) between timed steps,
outside the events. A barrier and a device synchronise bracket the timed region and
the step time is the maximum over ranks. Under torchrun each rank runs its own
replica of the workload (the path has no exchange step on one GPU), so `value` is
the work of all ranks divided by that time.

`--impl reference` times the float64 CPU oracle, as it stands, on this host's cores
(rank 0 only), on a bounded row sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused QKV-CTE FP8 TFLOP/s and % of dense FP8 peak at Wan 480p self-attn shape"
# GB300 dense FP8 tensor peak per GPU: NVIDIA's GB300 NVL72 specifications give 720 PFLOPS
# of FP8 for the 72-GPU rack with 2:4 sparsity, i.e. 10 PFLOPS sparse and 5 PFLOPS dense per
# GPU. The HGX B300 board's figure (72 PFLOPS sparse for 8 GPUs: 4.5 dense per GPU) belongs
# to the lower-power air-cooled part and is reported beside it for comparison only.
NOMINAL_FP8_TFLOPS = 5000.0
HGX_B300_FP8_TFLOPS = 4500.0
FP8_PER_BF16 = 2.0                  # nominal dense FP8 / BF16 tensor rate ratio
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="wan480p")
    p.add_argument("--call", type=int, default=0,
                   help="which call of a multi-call workload to time (cross: 0 = Q, 1 = K, 2 = V)")
    p.add_argument("--tile-n", type=int, default=0)
    p.add_argument("--gemm", choices=["auto", "pair", "single"], default="auto",
                   help="GEMM form: 256-row tiles on SM pairs, 128-row tiles on one SM, or the library's choice")
    p.add_argument("--norm-in-gemm", action="store_true",
                   help="run the norm/RoPE work inside the GEMM's epilogue warps instead of its own kernel")
    p.add_argument("--layout", choices=["bsd", "nbsd"], default="bsd",
                   help="output layout: BSD [T, I] or NBSd [heads, T, d_head]")
    p.add_argument("--input", choices=["fp8", "packed", "bf16"], default="fp8",
                   help="what the step is fed: e4m3 rows + scales, packed [T, H+4] rows, or bf16 activations")
    p.add_argument("--norm", choices=["across", "head_rms", "head_layer"], default="across",
                   help="qk-norm: across heads (Wan), or the per-head RMS / LayerNorm finished in the GEMM epilogue")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--e2e-chunk", type=int, default=0, help="row chunk of the host-streaming e2e leg (0: the library's 2048)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-flush", action="store_true", help="keep L2 warm between steps")
    p.add_argument("--cpu-rows", type=int, default=20480, help="oracle row sample for cpu_baseline")
    p.add_argument("--ref-rows", type=int, default=256, help="oracle row sample per reference step")
    p.add_argument("--sustained-s", type=float, default=1.2,
                   help="seconds of back-to-back steps for the sustained leg (0: skip)")
    return p.parse_args()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), float(m.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 0.0, "fallback"


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n)), "threadpoolctl"
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var]), var
    return os.cpu_count(), "cpu_count (BLAS default: all cores)"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 20 ms, kept only when their
    timestamp falls inside the timed region (mark_start / mark_end)."""

    FIELDS = ["timestamp", "index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    PERIOD_MS = 20

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)], stdout=self.out,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    @staticmethod
    def _epoch(stamp):
        import datetime

        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()  # nvidia-smi prints local time
            except ValueError:
                pass
        return None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    rows.append(parts)
        os.unlink(self.path)
        return self.summarise(rows, self.t0, self.t1)

    @classmethod
    def summarise(cls, rows, t0=None, t1=None):
        """Median SM clock, max clock and the throttle reasons seen, over the samples
        taken between t0 and t1 (epoch seconds); all samples if none fall inside."""
        if not rows:
            return None
        inside = rows
        if t0 is not None and t1 is not None:
            stamped = [(cls._epoch(r[0]), r) for r in rows]
            inside = [r for t, r in stamped if t is not None and t0 <= t <= t1]
        used = inside if inside else rows
        sm = [float(r[2]) for r in used if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in used if r[3].replace(".", "").isdigit()]
        reasons = set()
        for r in used:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 r[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        pw = []
        for r in used:
            try:
                pw.append(float(r[4]))
            except ValueError:
                pass
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_min_mhz": min(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "power_w_median": statistics.median(pw) if pw else None,
               "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons), "samples": len(used),
               "window": "timed region" if inside else "no sample fell inside the timed region: all samples"}
        if t0 is not None and t1 is not None:
            out["timed_region_s"] = round(t1 - t0, 3)
        return out


def _spread(step_ms):
    """Per-step device times: min, median, max, and the means of the first and last
    quarter of the timed steps (a drift between them shows clocks settling)."""
    if not step_ms:
        return None
    q = max(1, len(step_ms) // 4)
    return {"min": min(step_ms), "median": statistics.median(step_ms), "max": max(step_ms),
            "first_quarter_mean": statistics.mean(step_ms[:q]), "last_quarter_mean": statistics.mean(step_ms[-q:])}


def _k1_traffic(workload, tile_n, pair):
    """DRAM bytes per GEMM launch from the committed ncu summary of that GEMM form
    (profiles/qkv_gemm_mxf8{,_pair}_<workload>.md), if it was taken on the current
    kernel source and this workload/tile; else None."""
    name = "qkv_gemm_mxf8_pair" if pair else "qkv_gemm_mxf8"
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (name, workload))
    if not os.path.exists(path):
        return None
    try:
        rec = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith(("|", " ", "#", "-")):
                    k, v = line.split(":", 1)
                    rec[k.strip()] = v.strip()
        h = hashlib.sha256()
        for fn in rec["sources"].split():
            with open(os.path.join(ROOT, fn), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["source_sha256"]:
            return None
        if rec.get("workload") != workload or int(rec.get("tile_n", -1)) != tile_n:
            return None
        return int(rec["dram_bytes_per_launch"])
    except Exception:
        return None


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def replica_throughput(local_ms_total, units_per_rank, world, device=None):
    """Whole-job throughput of `world` replicas that each processed `units_per_rank`
    units in `local_ms_total` milliseconds: all ranks' units over the slowest rank's
    time. With world > 1 the time is max-reduced over the default process group.
    Returns (units per second, the max time in ms)."""
    total_ms = float(local_ms_total)
    if world > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return world * units_per_rank / (total_ms * 1e-3), total_ms


def run_reference(args):
    """The oracle, as it stands, on the host cores: a bounded row sample per step."""
    import numpy as np

    import workloads as wl
    from oracle import qkv_cte_oracle as O

    world, rank, _ = _dist()
    if rank != 0:
        return 0
    call = wl.workload(args.workload)[args.call]
    inp = wl.make_inputs(call)
    rows = wl.sample_rows(call, args.ref_rows).numpy()
    flops = 2.0 * len(rows) * call.hidden * call.width
    for _ in range(args.warmup):
        O.qkv_cte_from_inputs(call, inp, rows=rows)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        O.qkv_cte_from_inputs(call, inp, rows=rows)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = flops * args.steps / total / 1e12
    cores, how = _blas_threads()
    sample = (f"{len(rows)} seeded rows of {call.tokens} per step (rows are independent); "
              f"float64 numpy oracle, BLAS threads via {how}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(call),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


_INPUT_NOTE = {
    "fp8": "e4m3 codes [T, H] + fp32 row scales [T]",
    "packed": "packed [T, H+4] rows (codes + fp32 scale tail), unpacked inside the step",
    "bf16": "bf16 activations [T, H], row-quantised to e4m3 inside the step",
}


def _describe(call):
    """What the timed call computes, with its sizes."""
    if call.n_kv_heads == 0:
        kind = "Wan2.2-style cross-attention single-segment projection (separate Q, K or V call)"
    elif call.n_q_heads == 0:
        kind = "Wan2.2-style cross-attention K|V projection of the context tokens in one call"
    else:
        kind = "Wan2.2-style fused QKV self-attention projection"
    norm = {0: "no qk-norm", 1: "across-heads RMSNorm", 2: "per-head RMSNorm", 3: "per-head LayerNorm"}[call.norm]
    rope = ("3D-grid rotate-half RoPE" if call.rope_grid else "1D rotate-half RoPE") if call.rope else "no RoPE"
    return (f"{call.name}: {kind}, T={call.tokens} H={call.hidden} n_q={call.n_q_heads} n_kv={call.n_kv_heads} "
            f"d_head={call.d_head} I={call.width}, {norm}, {rope}")


def _config(call, layout="bsd", input_kind="fp8"):
    """The workload: what is computed, on which shapes and data layouts. The same for
    both arms (how our arm runs it, e.g. the GEMM form and the L2 flushing, is reported
    beside it, under "implementation")."""
    return {
        "workload": _describe(call),
        "tokens": call.tokens, "hidden": call.hidden, "width": call.width,
        "n_q_heads": call.n_q_heads, "n_kv_heads": call.n_kv_heads, "d_head": call.d_head,
        "output_layout": "NBSd [heads, T, d_head]" if layout == "nbsd" else "BSD [T, I]",
        "qk_norm": {0: "none", 1: "across heads (RMS)", 2: "per head RMS", 3: "per head LayerNorm"}[call.norm],
        "input": _INPUT_NOTE[input_kind],
    }


def _implementation(tile_n, flushed=True, op_norm_in_gemm=False, gemm_form=None, head_norm_in_epilogue=False):
    return {
        "tile_n": tile_n,
        "gemm_form": gemm_form,
        "norm_rope_work": ("inside the GEMM's epilogue" if head_norm_in_epilogue else
                           "inside the GEMM's epilogue warps" if op_norm_in_gemm else
                           "its own kernel, overlapped with the GEMM"),
        "l2": "flushed between timed steps (256 MB write, outside the step events)" if flushed else "not flushed",
    }


def run_ours(args):
    import numpy as np
    import torch

    import workloads as wl
    from rope_tcgen05_mxfp8_gb300 import (QKV_CTE_FLAG_GEMM_CTA_PAIR, QKV_CTE_FLAG_GEMM_SINGLE_CTA,
                                          QKV_CTE_FLAG_PROFILE, QKV_CTE_FLAG_SERIAL_PASSES, QKV_CTE_INPUT_BF16,
                                          QKV_CTE_INPUT_PACKED, QKV_CTE_INPUT_ROW_FP8, QKV_CTE_LAYOUT_BSD,
                                          QKV_CTE_LAYOUT_NBSD, QkvCte)
    from rope_tcgen05_mxfp8_gb300 import build as b

    world, rank, local = _dist()
    b.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize(dev)

    call = wl.workload(args.workload)[args.call]
    if args.norm != "across":
        call = dataclasses.replace(call, norm={"head_rms": 2, "head_layer": 3}[args.norm])
    inp = wl.make_inputs(call)
    g = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    gq = g["gamma_q"] if call.norm else None  # gammas only where a segment is normalised
    gk = g["gamma_k"] if call.norm else None
    gemm_flag = {"auto": 0, "pair": QKV_CTE_FLAG_GEMM_CTA_PAIR, "single": QKV_CTE_FLAG_GEMM_SINGLE_CTA}[args.gemm]
    if args.norm_in_gemm:
        from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_NORM_IN_GEMM

        gemm_flag |= QKV_CTE_FLAG_NORM_IN_GEMM
    layout = QKV_CTE_LAYOUT_NBSD if args.layout == "nbsd" else QKV_CTE_LAYOUT_BSD
    input_layout = {"fp8": QKV_CTE_INPUT_ROW_FP8, "packed": QKV_CTE_INPUT_PACKED, "bf16": QKV_CTE_INPUT_BF16}[args.input]
    # The step's activation input, resident on the device (and its host copy for e2e).
    if args.input == "bf16":
        a_host = wl.make_activations(call)
    elif args.input == "packed":
        a_host = torch.cat([inp["A"], inp["a_scale"].view(torch.uint8).reshape(call.tokens, 4)], dim=1)
    else:
        a_host = inp["A"]
    a_in = a_host.to(dev)
    a_scale_in = g["a_scale"] if args.input == "fp8" else None
    op = QkvCte(call.tokens, call.hidden, call.n_q_heads, call.n_kv_heads, call.d_head, norm=call.norm,
                rope=call.rope, eps=call.eps, tile_n=args.tile_n, flags=QKV_CTE_FLAG_PROFILE | gemm_flag, device=dev,
                output_layout=layout, input_layout=input_layout)
    tile_n = op.info.tile_n
    out = torch.empty(call.tokens, call.width, dtype=torch.bfloat16, device=dev)
    sumsq = torch.empty(call.tokens, 2, dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        op(a_in, a_scale_in, g["W"], g["w_sf"], g["bias"], gq, gk, g["cos"], g["sin"],
           out=out, sumsq=sumsq, stream=stream)

    for _ in range(max(args.warmup, 0)):
        if not args.no_flush:
            flush.zero_()
        step()
    op.status(stream)

    gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gpu_uuid)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    passes = []
    barrier()
    sampler.start()
    time.sleep(0.3)  # nvidia-smi's first sample
    sampler.mark_start()
    for i in range(args.steps):
        if not args.no_flush:
            flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
        passes.append(op.pass_times())
    torch.cuda.synchronize(dev)
    sampler.mark_end()
    barrier()
    clocks = sampler.stop()
    op.status(stream)
    step_ms = [s.elapsed_time(e) for s, e in ev]
    flops = call.flops
    per_s, total_ms = replica_throughput(sum(step_ms), flops * args.steps, world, device=dev)
    ms_per_step = total_ms / args.steps
    value = per_s / 1e12

    # Side measurement (outside the timed region, before the sustained leg so that both
    # forms see the clocks of a short run): the same step with the two passes serialised,
    # alternating with the overlapped step. The serialised runs time the norm/RoPE pass on
    # its own (its bandwidth roofline) and the GEMM alone; the pairs give the overlapped
    # step's cost against the GEMM alone under the same conditions.
    serial = QkvCte(call.tokens, call.hidden, call.n_q_heads, call.n_kv_heads, call.d_head, norm=call.norm,
                    rope=call.rope, eps=call.eps, tile_n=args.tile_n,
                    flags=QKV_CTE_FLAG_PROFILE | QKV_CTE_FLAG_SERIAL_PASSES | gemm_flag, device=dev,
                    output_layout=layout, input_layout=input_layout)
    ser, ovl = [], []
    for i in range(max(3, min(args.steps, 10))):
        if not args.no_flush:
            flush.zero_()
        serial(a_in, a_scale_in, g["W"], g["w_sf"], g["bias"], gq, gk, g["cos"],
               g["sin"], out=out, sumsq=sumsq, stream=stream)
        ser.append(serial.pass_times())
        if not args.no_flush:
            flush.zero_()
        step()
        ovl.append(op.pass_times())
    serial.status(stream)
    op.status(stream)
    serial.close()
    norm_ms = statistics.mean(p[2] for p in ser[1:])
    serial_gemm_ms = statistics.mean(p[1] for p in ser[1:])
    serial_run_ms = statistics.mean(p[3] for p in ser[1:])
    ovl_gemm_ms = statistics.mean(p[1] for p in ovl[1:])
    ovl_run_ms = statistics.mean(p[3] for p in ovl[1:])
    drag = {"gemm_alone_ms": serial_gemm_ms, "gemm_in_step_ms": ovl_gemm_ms, "step_ms": ovl_run_ms,
            "step_over_gemm_alone": ovl_run_ms / serial_gemm_ms,
            "gemm_in_step_over_alone": ovl_gemm_ms / serial_gemm_ms, "pairs": len(ser) - 1,
            "how": "alternating serialised and overlapped steps (L2 flushed before each); GEMM spans from the "
                   "kernels' %globaltimer stamps, the step from CUDA events around prep + GEMM + norm/RoPE"}

    # Sustained leg: back-to-back steps for at least --sustained-s seconds (L2 flushed
    # between steps as above), with their own clock record, so that the power cap the
    # short timed region may not reach is in the number.
    sustained = None
    if args.sustained_s > 0:
        n_sus = max(1, int(args.sustained_s / max(1e-4, statistics.median(step_ms) * 1e-3)) + 1)
        sus_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_sus)]
        sus_sampler = ClockSampler(gpu_uuid)
        barrier()
        sus_sampler.start()
        time.sleep(0.3)
        sus_sampler.mark_start()
        for i in range(n_sus):
            if not args.no_flush:
                flush.zero_()
            sus_ev[i][0].record(stream)
            step()
            sus_ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        sus_sampler.mark_end()
        barrier()
        sus_clocks = sus_sampler.stop()
        op.status(stream)
        sus_ms = [a.elapsed_time(b2) for a, b2 in sus_ev]
        sus_per_s, sus_total = replica_throughput(sum(sus_ms), call.flops * n_sus, world, device=dev)
        sus_value = sus_per_s / 1e12
        _, bf16_b, bf16_s, _ = _peaks()
        sus_peak = (bf16_s if bf16_s > 0 else bf16_b) * FP8_PER_BF16
        sustained = {"value": sus_value, "unit": "TFLOP/s", "steps": n_sus, "seconds_of_steps": sus_total * 1e-3,
                     "ms_per_step": sus_total / n_sus, "step_ms_spread": _spread(sus_ms),
                     "pct_nominal_dense_fp8_peak": 100.0 * sus_value / (world * NOMINAL_FP8_TFLOPS),
                     "frac_of_measured_sustained_fp8": sus_value / (world * sus_peak),
                     "measured_sustained_fp8_peak": sus_peak,
                     "clocks": sus_clocks,
                     "how": "back-to-back steps (L2 flushed between them, outside the per-step events), "
                            "per-step CUDA events, nvidia-smi clocks sampled every 20 ms inside the run; "
                            "peak = measured sustained bf16 x nominal fp8/bf16 ratio"}

    prep_ms = statistics.mean(p[0] for p in passes)
    gemm_ms = statistics.mean(p[1] for p in passes)
    norm_span_ms = statistics.mean(p[2] for p in passes)
    run_ms = statistics.mean(p[3] for p in passes)

    hbm_gbs, bf16, bf16_sus, peak_src = _peaks()
    # The tensor-peak denominator: the burst figure, or the sustained one when the power
    # cap was active during the timed steps (the kernel then ran at the clocks a long
    # run settles at)
    capped = bool(clocks) and "sw_power_cap" in (clocks.get("reasons") or [])
    bf16_used = bf16_sus if (capped and bf16_sus > 0) else bf16
    fp8_peak = bf16_used * FP8_PER_BF16
    peak_kind = "sustained (sw_power_cap was active in the timed steps)" if bf16_used != bf16 else "burst"
    k1_achieved = flops / (gemm_ms * 1e-3) / 1e12
    # norm + RoPE bytes this design must move: read the Q/K hand-off (2 bytes per
    # value plus one exponent byte per 16), write the bf16 Q/K columns of O, read the
    # fp32 cos/sin rows and the fp32 [T, 2] sums
    qk_cols = (call.n_q_heads + call.n_kv_heads) * call.d_head
    k2_bytes = (2 + 2) * call.tokens * qk_cols + call.tokens * qk_cols // 16 \
        + 2 * 4 * call.tokens * call.d_head + 8 * call.tokens
    k2_gbs = k2_bytes / (norm_ms * 1e-3) / 1e9 if norm_ms > 0 else None

    e2e = None
    if not args.no_e2e:
        # End to end through the host-streaming entry point: the step's activations
        # come from pinned host memory and all of O goes back to pinned host memory,
        # in row chunks with the copies overlapped with the computation.
        A_h = a_host.pin_memory()
        s_h = inp["a_scale"].pin_memory() if args.input == "fp8" else None
        O_h = torch.empty(call.tokens, call.width, dtype=torch.bfloat16).pin_memory()
        e2e_ev = []
        for i in range(args.warmup + args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if not args.no_flush:
                flush.zero_()
            e0.record(stream)
            op.run_host(A_h, s_h, g["W"], g["w_sf"], g["bias"], gq, gk, g["cos"], g["sin"], O_h,
                        w_col_scale=g["w_col_scale"], sumsq=sumsq, chunk_rows=args.e2e_chunk, stream=stream)
            e1.record(stream)
            if i >= args.warmup:
                e2e_ev.append((e0, e1))
        torch.cuda.synchronize(dev)
        e2e_per_s, e2e_ms = replica_throughput(sum(a.elapsed_time(b2) for a, b2 in e2e_ev), flops * args.steps,
                                               world, device=dev)
        e2e = {"value": e2e_per_s / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(A_h.numel() * A_h.element_size()
                                         + (s_h.numel() * s_h.element_size() if s_h is not None else 0)),
               "d2h_bytes_per_step": int(O_h.numel() * O_h.element_size()),
               "ms_per_step": e2e_ms / args.steps,
               "chunk_rows": args.e2e_chunk or 2048,
               "note": (f"qkv_cte_run_host: pinned host input ({_INPUT_NOTE[args.input]}) in, full bf16 O out, "
                        "row chunks with upload / compute / readback overlapped")}
        op.host_status(stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import qkv_cte_oracle as O

        rows = wl.sample_rows(call, args.cpu_rows).numpy()
        t0 = time.perf_counter()
        O.qkv_cte_from_inputs(call, inp, rows=rows)
        dt = time.perf_counter() - t0
        cores, how = _blas_threads()
        cpu = {"value": 2.0 * len(rows) * call.hidden * call.width / dt / 1e12, "unit": "TFLOP/s",
               "cores": cores, "kind": "oracle",
               "sample": (f"{len(rows)} seeded rows of the {call.tokens}-token workload in one oracle call "
                          f"({dt:.2f} s; float64 numpy, BLAS threads via {how})"),
               "rows_per_s": len(rows) / dt,
               # rows are independent: a whole step is the sample's time scaled by the row count
               # (an extrapolation unless the sample is every row)
               "full_step_s": dt * call.tokens / len(rows),
               "full_step_s_is": "measured" if len(rows) == call.tokens else "extrapolated linearly in rows"}

    gemm_form = "CTA pairs (M = 256 MMAs)" if op.info.cta_pair else "single CTAs (M = 128 MMAs)"
    traffic = _k1_traffic(args.workload, tile_n, bool(op.info.cta_pair))
    producer = None
    if args.input != "fp8":
        # bytes the producer step must move: read the input rows, write e4m3 codes + scales
        in_row = 2 * call.hidden if args.input == "bf16" else call.hidden + 4
        p_bytes = call.tokens * (in_row + call.hidden + 4)
        producer = {"kernel": "row_quantize_kernel" if args.input == "bf16" else "unpack_rows_kernel",
                    "bytes": p_bytes, "prep_ms": prep_ms,
                    "GB/s": p_bytes / (prep_ms * 1e-3) / 1e9,
                    "frac_of_hbm": p_bytes / (prep_ms * 1e-3) / 1e9 / hbm_gbs,
                    "how": "prep_ms (CUDA events) covers the producer launch plus the small scale-repack/"
                           "clear launch, so the rate is a lower bound for the producer alone"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic (seeded; Wan2.2 480p shapes and distributions)",
        "config": _config(call, layout=args.layout, input_kind=args.input),
        "implementation": _implementation(tile_n, flushed=not args.no_flush, op_norm_in_gemm=bool(op.info.norm_in_gemm),
                                          gemm_form=gemm_form),
        "pct_nominal_dense_fp8_peak": 100.0 * value / (world * NOMINAL_FP8_TFLOPS),
        "nominal_dense_fp8_peak": {"TFLOP/s": NOMINAL_FP8_TFLOPS,
                                   "source": "NVIDIA GB300 NVL72 specifications: FP8 720 PFLOPS per 72 GPUs with "
                                             "2:4 sparsity = 5 PFLOPS dense per GPU",
                                   "pct_of_hgx_b300_4500": 100.0 * value / (world * HGX_B300_FP8_TFLOPS)},
        "pct_measured_fp8_peak": 100.0 * value / (world * fp8_peak),
        "passes_ms": {"prep": prep_ms, "gemm_epilogue": gemm_ms, "norm_rope_span": norm_span_ms,
                      "run": run_ms, "exposed_after_gemm": run_ms - prep_ms - gemm_ms,
                      "serial": {"gemm_epilogue": serial_gemm_ms, "norm_rope": norm_ms, "run": serial_run_ms},
                      "overlap_vs_gemm_alone": drag,
                      "how": "prep and run: CUDA events on the launching stream; gemm_epilogue and "
                             "norm_rope: first-block start to last-block end from %globaltimer stamps "
                             "written by the kernels. In the timed steps the norm/RoPE pass overlaps the "
                             "GEMM; 'serial' is a side run with the passes serialised"},
        "norm_rope": {"GB/s": k2_gbs, "bytes": k2_bytes, "measured_on": "serial side run",
                      "frac_of_hbm": (k2_gbs / hbm_gbs) if k2_gbs else None, "peak_GB/s": hbm_gbs},
        "roofline": {"bound": "tensor",
                     "kernel": ("qkv_gemm_mxf8_pair_kernel<%d>" if op.info.cta_pair else "qkv_gemm_mxf8_kernel<%d>")
                     % tile_n, "achieved": k1_achieved,
                     "peak": fp8_peak, "unit": "TFLOP/s", "frac": k1_achieved / fp8_peak,
                     "traffic": traffic,
                     "peak_source": (f"{peak_src} bf16 {peak_kind} {bf16_used:.1f} TFLOP/s x nominal fp8/bf16 "
                                     f"ratio {FP8_PER_BF16:g}"),
                     "kernel_alone": {"achieved": flops / (serial_gemm_ms * 1e-3) / 1e12,
                                      "frac": flops / (serial_gemm_ms * 1e-3) / 1e12 / fp8_peak,
                                      "how": "the same kernel in the side run's serialised steps (the norm/RoPE "
                                             "pass after it instead of beside it)"}},
        "step_ms_spread": _spread(step_ms),
        "sustained": sustained,
        "clocks": clocks,
        "e2e": e2e,
        # prep + GEMM, the producer for a bf16 / packed input, and the norm/RoPE pass when
        # it is a kernel of its own (not per head, not run by the GEMM's epilogue warps)
        "gpu_launches": (2 + (args.input != "fp8")
                         + ((call.norm == 1 or (call.norm == 0 and call.rope == 1)) and not op.info.norm_in_gemm))
        * args.steps,
        "producer": producer,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main():
    args = _args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
