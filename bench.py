#!/usr/bin/env python
"""Benchmark of the W4A8 GEMM hot path on one GB300 (or N replicas).

Workload: the Llama-3-8B decode GEMMs with g128 progressive group
quantization -- M in {1, 8, 32, 64, 128, 256} tokens x the four linear layers
(qkv 6144x4096, o 4096x4096, gate_up 28672x4096, down 4096x14336).  One step
runs, for each of the 24 (M, layer) points, the per-token activation
quantization followed by the W4A8 GEMM with its fp16 epilogue; weights are
quantized and packed once at load time, outside the timed region.  Inputs are
seeded synthetic data (random-init weights with outlier input channels,
N(0,1) activations with outlier channels).

Reported: TOPS = sum 2*M*N*K / step time (whole job over all ranks), the
per-point roofline fractions, the dominant kernel's roofline against the
measured HBM peak, an end-to-end figure through the public API with
host<->device copies, SM clocks sampled during the timed region, and the CPU
oracle timed on a bounded sample (``cpu_baseline``).
``--impl reference`` times the CPU oracle alone as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W4A8-g128 GEMM TOPS & % of roofline (HBM / INT8 tensor) on 8B shapes, m=1–4096"
WORKLOAD = ("Llama-3-8B decode GEMMs g128: M in {1,8,32,64,128,256} x "
            "{qkv 6144x4096, o 4096x4096, gate_up 28672x4096, down 4096x14336}")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--copies", type=int, default=0,
                    help="packed-weight copies per layer rotated to defeat L2 (0: enough that one layer's "
                         "copies exceed twice the L2 size, at least 5)")
    ap.add_argument("--point-reps", type=int, default=24,
                    help="launches per CUDA graph when timing each point's kernels alone")
    ap.add_argument("--cpu-rows", type=int, default=192, help="weight rows in the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", default="qkv,o,gate_up,down")
    ap.add_argument("--ms", default="1,8,32,64,128,256")
    return ap.parse_args()


ROOT = os.path.dirname(os.path.abspath(__file__))
GEMM_SOURCES = ("qoq_gemm.cu", "qoq_gemm_f8.cu", "qoq_gemm_common.cuh", "qoq_device.cuh", "qoq_internal.h")
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "w4a8_gemm_traffic_llama3_8b_decode_step.md")


def gemm_traffic():
    """DRAM bytes of one step's GEMM launches from the committed ncu summary,
    or None when the GEMM kernel sources changed since that capture."""
    try:
        vals = {}
        for line in open(TRAFFIC_SUMMARY):
            if ":" in line and not line.startswith(("|", "#", " ")):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        h = hashlib.sha256()
        for f in GEMM_SOURCES:
            with open(os.path.join(ROOT, "w4a8_quantized_serving_qoq_gb300", "csrc", f), "rb") as fh:
                h.update(fh.read())
        if h.hexdigest()[:16] != vals.get("gemm_source_digest"):
            return None
        return int(vals["dram_bytes_per_step"]), int(vals["algorithmic_bytes_per_step"])
    except (OSError, KeyError, ValueError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------- clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest of every rank's value (replicas are timed by the slowest
    one); the value itself when there is no process group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tops(ops_per_replica_step: float, world: int, ms_step: float) -> float:
    """Whole-job throughput: each of the `world` replicas runs the whole step,
    so the job does world x its operations in the slowest replica's time."""
    return world * ops_per_replica_step / (ms_step * 1e-3) / 1e12


def gpu_pci_id(torch, dev: int) -> str | None:
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ----------------------------------------------------------- CPU oracle --
def oracle_sample(layers, Ms, rows: int, seed_base: int = 1):
    """Inputs of the bounded oracle sample: the first `rows` weight rows of
    every layer, quantized by the oracle, and the activations of every point."""
    import oracle
    from w4a8_quantized_serving_qoq_gb300 import synthetic
    sample = []
    for layer in layers:
        s = synthetic.layer_seed(1, layer)
        W = synthetic.weights(layer.N, layer.K, s, 0.02, 2)[:rows]
        wq = oracle.quantize_weights_group(np.ascontiguousarray(W), 128)
        for M in Ms:
            X = synthetic.activations(M, layer.K, s, 4)
            sample.append((layer, M, wq, X))
    return sample


def oracle_pass(sample):
    """One pass of the oracle over the sample; returns (seconds, ops)."""
    import oracle
    ops = 0
    t0 = time.perf_counter()
    for layer, M, wq, X in sample:
        Qx, sx, _ = oracle.quant_act(X)
        acc = oracle.gemm_i32_group(Qx, wq["q4"], wq["s_g"], wq["z"])
        oracle.epilogue_f64(acc, sx, wq["s_w"])
        ops += 2 * M * wq["q4"].shape[0] * layer.K
    return time.perf_counter() - t0, ops


def run_reference(args, layers, Ms):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    rows = 32
    sample = oracle_sample(layers, Ms, rows)
    for _ in range(args.warmup):
        oracle_pass(sample)
    tot_t, tot_ops = 0.0, 0
    for _ in range(args.steps):
        dt, ops = oracle_pass(sample)
        tot_t += dt
        tot_ops += ops
    tops = tot_ops / tot_t / 1e12
    desc = (f"oracle (plain single-threaded C) on the first {rows} weight rows of each layer, "
            f"all 24 (M, layer) points: quant_act + int32 GEMM + fp64 epilogue")
    line = {
        "impl": "reference", "metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "i32",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": desc},
        "cpu_baseline": {"value": tops, "unit": "TOPS", "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": tops, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ GPU path --
def main():
    args = parse_args()
    from w4a8_quantized_serving_qoq_gb300 import synthetic
    layer_by_name = {l.name: l for l in synthetic.LLAMA3_8B}
    layers = [layer_by_name[n] for n in args.layers.split(",")]
    Ms = [int(m) for m in args.ms.split(",")]
    if args.impl == "reference":
        run_reference(args, layers, Ms)
        return

    import torch
    import w4a8_quantized_serving_qoq_gb300 as qoq
    from w4a8_quantized_serving_qoq_gb300 import roofline

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    qoq.load()
    peaks, peaks_src = load_peaks()
    bw = peaks["hbm_gbs"] * 1e9
    p16 = peaks["bf16_tflops"] * 1e12  # fp16 dense tensor rate = bf16 rate
    stream = torch.cuda.current_stream()

    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2**20)
    # ---- load time: quantize + pack weights on the device, make copies ----
    weights = {}
    for layer in layers:
        s = synthetic.layer_seed(1, layer)
        W = torch.from_numpy(synthetic.weights(layer.N, layer.K, s, 0.02, 2)).to(dev)
        wq = qoq.qoq_quantize_weights(W, 128)
        packed = qoq.qoq_pack_weights(wq["q4"], wq["s_g"], wq["z"], 128)
        ncopy = args.copies or max(5, -(-2 * l2_bytes // packed.numel()) + 1)
        copies = [packed] + [packed.clone() for _ in range(ncopy - 1)]
        weights[layer.name] = (copies, wq["s_w"])
        del W, wq
    points = []
    ws_max = 256
    for M in Ms:
        for layer in layers:
            s = synthetic.layer_seed(1, layer)
            X = torch.from_numpy(synthetic.activations(M, layer.K, s, 4)).to(dev)
            Qx = torch.empty((M, layer.K), dtype=torch.int8, device=dev)
            sx = torch.empty((M,), dtype=torch.float16, device=dev)
            O = torch.empty((M, layer.N), dtype=torch.float16, device=dev)
            ws_max = max(ws_max, qoq.qoq_gemm_workspace_bytes(M, layer.N, layer.K, 128))
            # the quantizer also writes the activation operand the GEMM's path
            # reads (fp8 planes for decode sizes, an fp16 copy above)
            kind = qoq.qoq_gemm_path(M, layer.N, layer.K, 128)
            act = torch.empty((qoq.qoq_act_operand_bytes(M, layer.K, kind),), dtype=torch.uint8, device=dev)
            points.append(dict(layer=layer, M=M, X=X, Qx=Qx, sx=sx, O=O, act=act, kind=kind,
                               opt=qoq.gemm_options(act_operand=act, flags=qoq.QOQ_LAUNCH_OVERLAP)))
    ws = qoq.new_workspace(ws_max, dev)
    torch.cuda.synchronize()

    def quant_point(pt):
        qoq.qoq_quant_act_ex(pt["X"], pt["Qx"], pt["sx"], None, pt["act"], kind=pt["kind"], with_t=False,
                             flags=qoq.QOQ_LAUNCH_OVERLAP)

    def gemm_point(pt, copy_idx):
        layer = pt["layer"]
        copies, s_w = weights[layer.name]
        qoq.qoq_w4a8_gemm_ex(pt["Qx"], pt["sx"], None, copies[copy_idx % len(copies)], s_w, layer.N,
                             layer.K, 128, O=pt["O"], workspace=ws, options=pt["opt"])

    def run_point(i, pt, copy_idx):
        quant_point(pt)
        gemm_point(pt, copy_idx)

    def step():
        for i, pt in enumerate(points):
            run_point(i, pt, i)

    # eager warm-up (sets kernel attributes before capture), then capture one step
    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(gpu_pci_id(torch, local_rank))
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms_step = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dist, dev)
    ops_step = sum(roofline.gemm_ops(p["M"], p["layer"].N, p["layer"].K) for p in points)
    tops = whole_job_tops(ops_step, world, ms_step)

    # ---- per-point kernel times: each point's quantizer and GEMM alone, each
    # launched R times back to back in a CUDA graph (launch overlap as in the
    # step); the GEMMs rotate over the layer's weight copies, which together
    # exceed twice the L2 size, so every launch reads its weights from HBM ----
    def graph_us(fn, reps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for r in range(reps):
                fn(r)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3 / reps)
        del g
        return statistics.median(ts)

    pt_rows = []
    gemm_ms_total, bytes_total = 0.0, 0
    for i, pt in enumerate(points):
        layer, M = pt["layer"], pt["M"]
        copies, s_w = weights[layer.name]
        reps = max(args.point_reps, len(copies))
        t_q = 1e-3 * graph_us(lambda r: quant_point(pt), reps)
        t_g = 1e-3 * graph_us(lambda r: gemm_point(pt, r), reps)
        nbytes = roofline.w4a8_bytes(M, layer.N, layer.K)
        nops = roofline.gemm_ops(M, layer.N, layer.K)
        troof = roofline.roof_time(M, layer.N, layer.K, bw, p16)
        gemm_ms_total += t_g
        bytes_total += nbytes
        pt_rows.append({
            "layer": layer.name, "M": M, "gemm_us": round(1e3 * t_g, 2), "quant_us": round(1e3 * t_q, 2),
            "TOPS": round(nops / (t_g * 1e-3) / 1e12, 2), "GBs": round(nbytes / (t_g * 1e-3) / 1e9, 1),
            "bound": roofline.bound(M, layer.N, layer.K, bw, p16),
            "roof_frac": round(troof / (t_g * 1e-3), 3),
        })
    achieved_gbs = bytes_total / (gemm_ms_total * 1e-3) / 1e9
    traffic = gemm_traffic()
    troof_sum = sum(roofline.roof_time(p["M"], p["layer"].N, p["layer"].K, bw, p16) for p in points)

    # ---- end to end through the public API: host buffers, copies timed ----
    e2e = None
    if not args.no_e2e:
        hostX = [p["X"].cpu().pin_memory() for p in points]
        hostO = [torch.empty(p["O"].shape, dtype=torch.float16).pin_memory() for p in points]
        h2d = sum(h.numel() * 2 for h in hostX)
        d2h = sum(h.numel() * 2 for h in hostO)
        e2e_steps = max(3, min(args.steps, 10))

        # Transfers overlap the compute, as in a serving loop: the inputs go
        # up on a copy-in stream and the outputs come down on a copy-out
        # stream, in groups of consecutive points (up to about 2 MB of output
        # each, so large outputs go down while later points compute): a
        # group's compute waits for its inputs' event, its outputs are copied
        # once its last GEMM is done, and the step ends when all outputs are
        # on the host.  A step overwrites inputs and outputs only after the
        # previous step's readers of them have finished.
        copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        groups, cur, cur_bytes = [], [], 0
        for i, pt in enumerate(points):
            cur.append(i)
            cur_bytes += pt["O"].numel() * 2
            if cur_bytes >= 2 << 20:
                groups.append(cur)
                cur, cur_bytes = [], 0
        if cur:
            groups.append(cur)
        ev_in = [torch.cuda.Event() for _ in groups]
        ev_done = [torch.cuda.Event() for _ in groups]

        def e2e_step():
            copy_in.wait_stream(stream)
            with torch.cuda.stream(copy_in):
                for gi, grp in enumerate(groups):
                    for i in grp:
                        points[i]["X"].copy_(hostX[i], non_blocking=True)
                    ev_in[gi].record(copy_in)
            stream.wait_stream(copy_out)
            for gi, grp in enumerate(groups):
                stream.wait_event(ev_in[gi])
                for i in grp:
                    run_point(i, points[i], i)
                ev_done[gi].record(stream)
                copy_out.wait_event(ev_done[gi])
                with torch.cuda.stream(copy_out):
                    for i in grp:
                        hostO[i].copy_(points[i]["O"], non_blocking=True)
            stream.wait_stream(copy_out)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / e2e_steps, dist, dev)
        e2e = {"value": whole_job_tops(ops_step, world, e2e_ms), "unit": "TOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "path": "Python binding -> C ABI per call (no CUDA graph), pinned host buffers, host<->device copies on two side streams overlapping the compute"}

    # ---- CPU oracle on a bounded sample ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = oracle_sample(layers, Ms, args.cpu_rows)
        dt, ops = oracle_pass(sample)
        cpu = {"value": ops / dt / 1e12, "unit": "TOPS", "cores": 1, "kind": "oracle",
               "seconds": round(dt, 2),
               "sample": (f"first {args.cpu_rows} weight rows of each layer at all 24 (M, layer) points; "
                          f"quant_act + int32 GEMM + fp64 epilogue, plain single-threaded C "
                          f"({os.cpu_count()} host cores present)")}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "s8 x u4 -> exact i32 (e4m3 / fp16 tensor-core MMA), fp16 out", "data": "synthetic",
        "config": {"workload": WORKLOAD, "group": 128, "parallelism": f"replicas{world}",
                   "cuda_graph": True, "l2": "inputs larger than L2: packed-weight copies rotated, "
                   + ", ".join(f"{k} x{len(c)}" for k, (c, _) in weights.items())
                   + f" ({sum(len(c) * c[0].numel() for c, _ in weights.values()) / 1e6:.0f} MB)"},
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved_gbs / peaks["hbm_gbs"],
                     "traffic": traffic[0] if traffic else None,
                     "traffic_scope": "DRAM read+write bytes of the step's 24 GEMM launches (ncu, cold cache)",
                     "algorithmic_bytes_per_step": traffic[1] if traffic else None,
                     "peak_source": peaks_src, "kernel": "w4a8_gemm (fp8-operand kernel for M <= 32, fp16-operand kernel above)",
                     "time_weighted_roofline_frac": troof_sum / (gemm_ms_total * 1e-3),
                     "tensor_peak_tflops": peaks["bf16_tflops"]},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * len(points) * args.steps,
        "clocks": clk,
        "points": pt_rows,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
