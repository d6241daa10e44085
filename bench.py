#!/usr/bin/env python
"""Benchmark of the W4A8 GEMM hot path on one GB300 (or N replicas).

Headline workload: the Llama-3-8B linear layers with g128 progressive group
quantization over the whole token range of the metric -- the decode batches
M in {1, 8, 32, 64, 128, 256} and the prefill batch M = 4096 (4 sequences x
1024 tokens), each x the four layers (qkv 6144x4096, o 4096x4096, gate_up
28672x4096, down 4096x14336): 28 points.  One step runs, for every point,
the per-token activation quantization followed by the W4A8 GEMM with its
fp16 epilogue; weights are quantized and packed once at load time, outside
the timed region.  Inputs are seeded synthetic data (random-init weights
with outlier input channels, N(0,1) activations with outlier channels), one
seed per (workload, layer) as the input recipe states.

Two further workloads are timed point by point as separate blocks (they are
not part of the headline step): the Qwen1.5-72B-shaped FFN GEMMs (gate_up
59136x8192, down 8192x29568 at M in {64, 1024}) and the per-channel W4A8
variant on Llama-3-8B gate_up over M = 1 .. 4096.

Reported: TOPS = sum 2*M*N*K / step time (whole job over all ranks); per
point the GEMM's time alone (a CUDA graph of back-to-back launches rotating
over weight copies larger than L2), its bound (max of the HBM time of the
4-bit weight + 8-bit activation bytes and the tensor time of the MACs at the
fp16/bf16 dense peak) and its roofline fraction; the dominant kernel's
roofline; an end-to-end figure through the public API with host<->device
copies; SM clocks sampled over a loaded window that ends with the timed
region; and the CPU oracle timed on a bounded sample (``cpu_baseline``).
``--impl reference`` times the CPU oracle alone as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
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
WORKLOAD = ("Llama-3-8B GEMMs g128, decode M in {1,8,32,64,128,256} + prefill M=4096 x "
            "{qkv 6144x4096, o 4096x4096, gate_up 28672x4096, down 4096x14336}")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
BLOCKS = {
    "fused_quant": (1, "Llama-3-8B: RMS norm + per-token INT8 quant (K=4096, the qkv / gate_up input) and "
                       "SiLU-mul + quant (F=14336, the down input), M in {1,8,32,64,128,256,4096}"),
    "kv4_attention": (1, "Llama-3-8B decode attention over the KV4 cache (32 query / 8 KV heads, head dim 128): "
                         "batch 64 x lengths 512..1536 and batch 8 x 8192"),
    "qwen72b": (3, "Qwen1.5-72B-shaped FFN GEMMs g128: {gate_up 59136x8192, down 8192x29568} x M in {64,1024}"),
    "per_channel": (4, "Llama-3-8B gate_up 28672x4096, per-channel W4A8 (zero folded via t_x), M = 1..4096"),
}
GEMM_SOURCES = ("qoq_gemm.cu", "qoq_gemm_f8.cu", "qoq_gemv.cu", "qoq_gemm_common.cuh", "qoq_device.cuh",
                "qoq_internal.h", "qoq_dispatch_table.inc")
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "w4a8_gemm_traffic_llama3_8b_step.md")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--copies", type=int, default=0,
                    help="packed-weight copies per layer rotated to defeat L2 (0: enough that one layer's "
                         "copies exceed twice the L2 size, at least 3)")
    ap.add_argument("--point-reps", type=int, default=24,
                    help="launches per CUDA graph when timing each point's kernels alone")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="seconds of untimed step replays right before the timed region, with the clock "
                         "sampler running (the timed region itself is shorter than one sampling interval)")
    ap.add_argument("--cpu-rows", type=int, default=64, help="weight rows per layer in the oracle sample")
    ap.add_argument("--cpu-prefill-tokens", type=int, default=1024,
                    help="tokens of the prefill batch in the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-points", action="store_true", help="skip the per-point timings (and the blocks)")
    ap.add_argument("--blocks", default="fused_quant,kv4_attention,qwen72b,per_channel",
                    help="comma list of extra workloads timed point by point ('' for none)")
    ap.add_argument("--tune", action="store_true",
                    help="time the GEMM's candidate launch choices for every shape and token count of the "
                         "workloads on this GPU, write the planner's dispatch table (csrc/qoq_dispatch_table.inc) "
                         "and print a summary instead of the benchmark line")
    ap.add_argument("--block-ms", default="",
                    help="comma list: time only these token counts in the qwen72b and per_channel blocks")
    ap.add_argument("--layers", default="qkv,o,gate_up,down")
    ap.add_argument("--ms", default="1,8,32,64,128,256,4096",
                    help="token counts of the headline step (4096 = the prefill workload)")
    return ap.parse_args(argv)


# ----------------------------------------------------------- workloads --
def headline_points(layer_names, Ms):
    """(workload id, layer, M) of the headline step, M-major like a serving
    loop that runs every layer at one batch size before the next."""
    from w4a8_quantized_serving_qoq_gb300 import synthetic
    by = {l.name: l for l in synthetic.LLAMA3_8B}
    pts = []
    for M in Ms:
        wid = 2 if M == synthetic.PREFILL_M else 1
        for n in layer_names:
            pts.append((wid, by[n], M))
    return pts


def block_points(name):
    from w4a8_quantized_serving_qoq_gb300 import synthetic
    wid, _ = BLOCKS[name]
    _, layers, Ms, _, _, _, _ = synthetic.WORKLOADS[wid]
    return [(wid, layer, M) for layer in layers for M in Ms]


def group_of(wid):
    from w4a8_quantized_serving_qoq_gb300 import synthetic
    return synthetic.WORKLOADS[wid][6]


def gemm_source_digest():
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "w4a8_quantized_serving_qoq_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def gemm_traffic():
    """DRAM bytes per GEMM launch of the headline step from the committed ncu
    summary, keyed (workload, layer, M), or None when the GEMM kernel sources
    changed since that capture."""
    try:
        vals, per = {}, {}
        for line in open(TRAFFIC_SUMMARY):
            if line.startswith("traffic:"):
                _, key, dram = line.split()
                w, l, m = key.split("/")
                per[(int(w), l, int(m))] = int(dram)
            elif ":" in line and not line.startswith(("|", "#", " ")):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        if gemm_source_digest() != vals.get("gemm_source_digest"):
            return None
        return per or None
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
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[tuple[float, str]] = []
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
            self.lines.append((time.time(), line.strip()))

    def stop(self, window=None):
        """Summary of the samples taken while the GPU was loaded (host times
        within `window` = (t0, t1), when given)."""
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
        return summarize_clocks(self.lines, window)


def summarize_clocks(lines, window=None):
    sm, smax, power, reasons = [], [], [], set()
    for t, ln in lines:
        if window and not (window[0] <= t <= window[1] + 0.25):
            continue
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 10:
            continue
        try:
            sm.append(float(parts[2]))
            smax.append(float(parts[3]))
            power.append(float(parts[4]))
        except ValueError:
            continue
        for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                             parts[6:10]):
            if val.lower().startswith("active"):
                reasons.add(name)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
            "power_w_max": max(power), "reasons": sorted(reasons)}


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


def roofline_summary(rows, bw, p16):
    """Roofline of a set of per-point GEMM timings (rows carry layer N, K, M
    and gemm_us): per bound class the achieved rate against its peak, the
    dominant class (most GEMM time) and the time-weighted fraction
    sum(roof time) / sum(measured time)."""
    from w4a8_quantized_serving_qoq_gb300 import roofline
    cls = {}
    troof = tsum = 0.0
    for r in rows:
        t = r["gemm_us"] * 1e-6
        M, N, K = r["M"], r["N"], r["K"]
        c = cls.setdefault(r["bound"], {"time_s": 0.0, "bytes": 0, "flops": 0, "roof_s": 0.0, "points": 0})
        c["time_s"] += t
        c["bytes"] += roofline.w4a8_bytes(M, N, K)
        c["flops"] += roofline.gemm_ops(M, N, K)
        c["roof_s"] += roofline.roof_time(M, N, K, bw, p16)
        c["points"] += 1
        troof += roofline.roof_time(M, N, K, bw, p16)
        tsum += t
    out = {}
    for b, c in cls.items():
        if b == "hbm":
            ach, peak, unit = c["bytes"] / c["time_s"] / 1e9, bw / 1e9, "GB/s"
        else:
            ach, peak, unit = c["flops"] / c["time_s"] / 1e12, p16 / 1e12, "TFLOP/s"
        out[b] = {"achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak, "points": c["points"],
                  "gemm_time_us": 1e6 * c["time_s"], "time_weighted_roofline_frac": c["roof_s"] / c["time_s"]}
    dom = max(cls, key=lambda b: cls[b]["time_s"]) if cls else None
    return out, dom, (troof / tsum if tsum else None)


# ----------------------------------------------------------- CPU oracle --
def oracle_sample(points, rows: int, max_tokens: int):
    """Inputs of a bounded oracle sample: the first `rows` weight rows of each
    point's layer, quantized by the oracle, and the first min(M, max_tokens)
    tokens of each point's activations."""
    import oracle
    from w4a8_quantized_serving_qoq_gb300 import synthetic
    wcache, sample = {}, []
    for wid, layer, M in points:
        _, _, _, sigma, wo, xo, group = synthetic.WORKLOADS[wid]
        s = synthetic.layer_seed(wid, layer)
        if (wid, layer.name) not in wcache:
            W = synthetic.weights(layer.N, layer.K, s, sigma, wo, rows=rows)
            wcache[(wid, layer.name)] = (oracle.quantize_weights_group(W, 128) if group
                                         else oracle.quantize_weights_channel(W))
        m = min(M, max_tokens)
        X = synthetic.activations(M, layer.K, s, xo)[:m]
        sample.append((layer, m, group, wcache[(wid, layer.name)], np.ascontiguousarray(X)))
    return sample


def oracle_pass(sample):
    """One pass of the oracle over the sample; returns (seconds, ops)."""
    import oracle
    ops = 0
    t0 = time.perf_counter()
    for layer, M, group, wq, X in sample:
        Qx, sx, tx = oracle.quant_act(X)
        if group:
            acc = oracle.gemm_i32_group(Qx, wq["q4"], wq["s_g"], wq["z"])
        else:
            acc = oracle.gemm_i32_channel(Qx, tx, wq["q4"], wq["z"])
        oracle.epilogue_f64(acc, sx, wq["s_w"])
        ops += 2 * M * wq["q4"].shape[0] * layer.K
    return time.perf_counter() - t0, ops


def sample_desc(rows, tokens, npts):
    return (f"first {rows} weight rows of each layer and the first {tokens} tokens of the prefill batch "
            f"(all tokens of the decode batches), all {npts} (M, layer) points: quant_act + int32 GEMM + "
            f"fp64 epilogue, plain single-threaded C")


def run_reference(args, points):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    rows, tokens = 8, 256
    sample = oracle_sample(points, rows, tokens)
    for _ in range(args.warmup):
        oracle_pass(sample)
    tot_t, tot_ops = 0.0, 0
    for _ in range(args.steps):
        dt, ops = oracle_pass(sample)
        tot_t += dt
        tot_ops += ops
    tops = tot_ops / tot_t / 1e12
    desc = sample_desc(rows, tokens, len(points))
    line = {
        "impl": "reference", "metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "i32",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": desc},
        "cpu_baseline": {"value": tops, "unit": "TOPS", "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": tops, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- dispatch table --
DISPATCH_TABLE = os.path.join(ROOT, "w4a8_quantized_serving_qoq_gb300", "csrc", "qoq_dispatch_table.inc")


def gemm_candidates(M, N, K, group, sms):
    """(path, tokens_per_tile, ctas, schedule) launch choices timed by --tune;
    (0, 0, 0, 0) is the planner's current automatic choice.  ctas is the CTA
    count (paths 1 and 2) or the cluster size (path 3); schedules 1..4 are
    tried where there are at least two waves of tiles."""
    tiles = N // 128
    cands = [(0, 0, 0)]  # expanded to (path, bt, ctas, schedule) below
    if M <= 8:
        cands += [(3, 0, c) for c in (1, 2, 4, 8)]
    if group == 128 and M <= 64:
        for bt in (16, 32):
            if bt == 16 and M > 32:
                continue
            t = -(-M // bt) * tiles
            # whole-tile multiples below a wave too: fewer CTAs with longer
            # ranges can beat every SM at these latency-bound sizes
            cands += [(2, bt, c) for c in sorted({sms, sms - 8} | {t * f for f in (1, 2, 3, 4) if t * f <= sms})]
    cap = 128 if M > 64 else max(16, 1 << (max(M, 1) - 1).bit_length())
    for bt in (16, 32, 64, 128):
        if bt > cap or (M >= 256 and bt < 64):
            continue
        t = -(-M // bt) * tiles
        cands += [(1, bt, c) for c in sorted({sms} | {t * f for f in (1, 2, 3, 4) if t * f <= sms})]
    out = []
    for p_, b_, c_ in cands:
        t = -(-M // max(b_, 1)) * tiles if b_ else 0
        if p_ in (1, 2) and t >= 2 * c_:
            out += [(p_, b_, c_, sch) for sch in (1, 2, 3, 4)]
        else:
            out.append((p_, b_, c_, 0))
    return out


def write_dispatch_table(entries, sms):
    lines = ["// Measured launch choices of the W4A8 GEMM planner, written by",
             "// `python bench.py --tune` on a GPU (the entries apply only to GPUs with the",
             "// same SM count).  One entry per line:",
             "//   {N, K, group, M, num_sms, path, tokens_per_tile, ctas (path 3: cluster size), schedule},",
             "// with the measured time of the choice and of the planner's rules."]
    for e in sorted(entries, key=lambda e: (e["N"], e["K"], e["group"], e["M"])):
        lines.append(f"{{{e['N']}, {e['K']}, {e['group']}, {e['M']}, {sms}, {e['path']}, {e['bt']}, {e['ctas']}, "
                     f"{e['sched']}}},"
                     f"  // {e['us']:.2f} us (rules {e['rule_us']:.2f} us)")
    with open(DISPATCH_TABLE, "w") as f:
        f.write("\n".join(lines) + "\n")


def read_dispatch_table():
    """The launch choices the current dispatch table holds, keyed by (N, K,
    group, M): (path, tokens_per_tile, ctas, schedule)."""
    table = {}
    if not os.path.exists(DISPATCH_TABLE):
        return table
    pat = re.compile(r"^\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+)\},")
    with open(DISPATCH_TABLE) as f:
        for line in f:
            m = pat.match(line.strip())
            if m:
                v = [int(x) for x in m.groups()]
                table[tuple(v[:4])] = tuple(v[5:])
    return table


# A tabled choice stays while it times within this fraction of the fastest
# candidate: schedules that differ by less than the run-to-run noise would
# otherwise swap at every tuning run (and with them the DRAM traffic).
TUNE_KEEP_FRAC = 0.005


def pick_choice(times, prev):
    """The fastest candidate, unless the previously tabled choice `prev` is
    within TUNE_KEEP_FRAC of it."""
    best = min(times, key=times.get)
    if prev is not None and prev in times and times[prev] <= times[best] * (1.0 + TUNE_KEEP_FRAC):
        return prev
    return best


def run_tune(args):
    """Times every candidate launch choice of every GEMM point of the four
    full-size workloads (weights rotated past L2, graphs of back-to-back
    launches as in the per-point timings), keeps the fastest per (N, K,
    group, M) and writes the dispatch table the planner reads."""
    import torch
    import w4a8_quantized_serving_qoq_gb300 as qoq
    from w4a8_quantized_serving_qoq_gb300 import synthetic
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    l2_bytes = int(getattr(props, "L2_cache_size", 0) or 129 * 2**20)
    stream = torch.cuda.current_stream()
    tabled = read_dispatch_table()
    points = []
    for wid in (1, 2, 3, 4):
        _, layers, Ms, _, _, _, _ = synthetic.WORKLOADS[wid]
        points += [(wid, layer, M) for layer in layers for M in Ms]
    seen, entries, report = set(), [], []
    loaded = [None, None]
    for wid, layer, M in points:
        _, _, _, sigma, wo, xo, group = synthetic.WORKLOADS[wid]
        key = (layer.N, layer.K, group, M)
        if key in seen:
            continue
        seen.add(key)
        s_ = synthetic.layer_seed(wid, layer)
        if loaded[0] != (wid, layer.name):  # points come layer by layer: load each layer's weights once
            loaded[1] = None
            torch.cuda.empty_cache()
            W = torch.from_numpy(synthetic.weights(layer.N, layer.K, s_, sigma, wo)).to(dev)
            wq = qoq.qoq_quantize_weights(W, group)
            packed = qoq.qoq_pack_weights(wq["q4"], wq["s_g"], wq["z"], group)
            ncopy = max(3, -(-2 * l2_bytes // packed.numel()) + 1)
            loaded[:] = [(wid, layer.name), ([packed] + [packed.clone() for _ in range(ncopy - 1)], wq["s_w"])]
            del W, wq, packed
        copies, s_w = loaded[1]
        X = torch.from_numpy(synthetic.activations(M, layer.K, s_, xo)).to(dev)
        acts = {}
        Qx = sx = tx = None
        for kind in (1, 2, 3):
            if kind == 2 and group != 128:
                continue
            Qx, sx, tx, act = qoq.qoq_quant_act_ex(X, kind=kind, with_t=True)
            acts[kind] = act
        O = torch.empty((M, layer.N), dtype=torch.float16, device=dev)
        ws = qoq.new_workspace(1 << 20, dev)
        times = {}
        for cand in gemm_candidates(M, layer.N, layer.K, group, sms):
            path, bt, ctas, sched = cand
            try:
                kind = qoq.qoq_gemm_path(M, layer.N, layer.K, group, qoq.gemm_options(
                    kernel=path, tokens_per_tile=bt, num_ctas=ctas, schedule=sched))
            except qoq.QoqError:
                continue
            opt = qoq.gemm_options(kernel=path, tokens_per_tile=bt, num_ctas=ctas, act_operand=acts.get(kind),
                                   flags=qoq.QOQ_LAUNCH_OVERLAP, schedule=sched)
            need = qoq.qoq_gemm_workspace_bytes(M, layer.N, layer.K, group, opt)
            if need > ws.numel():
                ws = qoq.new_workspace(need, dev)

            def fn(r):
                qoq.qoq_w4a8_gemm_ex(Qx, sx, tx, copies[r % len(copies)], s_w, layer.N, layer.K, group, O=O,
                                     workspace=ws, options=opt)
            fn(0)
            torch.cuda.synchronize()
            reps = max(8 if M * layer.N * layer.K >= 2 ** 36 else args.point_reps, len(copies))
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
            times[cand] = statistics.median(ts)
        status = qoq.qoq_workspace_status(ws)[0]
        best = pick_choice(times, tabled.get((layer.N, layer.K, group, M)))
        rule_us = times[(0, 0, 0, 0)]
        if best == (0, 0, 0, 0):  # record what the automatic plan chose, so the table pins it
            info = qoq.qoq_gemm_plan(M, layer.N, layer.K, group, sms)
            best_entry = (info["path"], info["tokens_per_tile"] if info["path"] != 3 else 0,
                          info["num_ctas"] // (layer.N // 128) if info["path"] == 3 else info["num_ctas"], 0)
        else:
            best_entry = best
        entries.append(dict(N=layer.N, K=layer.K, group=group, M=M, path=best_entry[0], bt=best_entry[1],
                            ctas=best_entry[2], sched=best_entry[3], us=times[best], rule_us=rule_us))
        report.append({"workload": wid, "layer": layer.name, "M": M, "best": list(best_entry),
                       "best_us": round(times[best], 2), "rule_us": round(rule_us, 2), "status": status,
                       "candidates": {"/".join(map(str, c)): round(t, 2) for c, t in times.items()}})
        print(json.dumps(report[-1]), file=sys.stderr, flush=True)
        del copies, X, acts, O
    write_dispatch_table(entries, sms)
    print(json.dumps({"tuned": len(entries), "num_sms": sms, "table": DISPATCH_TABLE,
                      "rules_us": sum(e["rule_us"] for e in entries), "table_us": sum(e["us"] for e in entries),
                      "points": report}), flush=True)


# ------------------------------------------------------------ GPU path --
def main(argv=None):
    args = parse_args(argv)
    from w4a8_quantized_serving_qoq_gb300 import synthetic
    Ms = [int(m) for m in args.ms.split(",") if m]
    points = headline_points(args.layers.split(","), Ms)
    if args.impl == "reference":
        run_reference(args, points)
        return
    import w4a8_quantized_serving_qoq_gb300 as qoq
    if qoq.debug_build_requested():
        # The bounds-check library tests its accesses: its times are not the product's.
        raise SystemExit("bench.py times the release library: unset QOQ_DEBUG (QOQ_DEBUG=1 selects the "
                         "bounds-check build)")
    if args.tune:
        run_tune(args)
        return

    import torch
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
    blocks = [b for b in args.blocks.split(",") if b] if not args.no_points else []
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2**20)

    # ---- load time: quantize + pack weights on the device, make copies ----
    weights = {}

    def load_weights(wid, layer):
        key = (wid, layer.name)
        if key in weights:
            return weights[key]
        _, _, _, sigma, wo, _, group = synthetic.WORKLOADS[wid]
        W = torch.from_numpy(synthetic.weights(layer.N, layer.K, synthetic.layer_seed(wid, layer), sigma, wo)).to(dev)
        wq = qoq.qoq_quantize_weights(W, group)
        packed = qoq.qoq_pack_weights(wq["q4"], wq["s_g"], wq["z"], group)
        ncopy = args.copies or max(3, -(-2 * l2_bytes // packed.numel()) + 1)
        copies = [packed] + [packed.clone() for _ in range(ncopy - 1)]
        weights[key] = (copies, wq["s_w"])
        del W, wq
        return weights[key]

    def make_point(wid, layer, M):
        group = group_of(wid)
        _, _, _, _, _, xo, _ = synthetic.WORKLOADS[wid]
        load_weights(wid, layer)
        X = torch.from_numpy(synthetic.activations(M, layer.K, synthetic.layer_seed(wid, layer), xo)).to(dev)
        kind = qoq.qoq_gemm_path(M, layer.N, layer.K, group)
        plan = qoq.qoq_gemm_plan(M, layer.N, layer.K, group, torch.cuda.get_device_properties(dev).multi_processor_count)
        pt = dict(wid=wid, layer=layer, M=M, group=group, X=X, kind=kind, plan=plan,
                  Qx=torch.empty((M, layer.K), dtype=torch.int8, device=dev),
                  sx=torch.empty((M,), dtype=torch.float16, device=dev),
                  tx=torch.empty((M,), dtype=torch.int32, device=dev) if group == 0 else None,
                  O=torch.empty((M, layer.N), dtype=torch.float16, device=dev),
                  # the quantizer also writes the activation operand the GEMM's
                  # path reads (fp8 planes for decode sizes, an fp16 copy above)
                  act=torch.empty((qoq.qoq_act_operand_bytes(M, layer.K, kind),), dtype=torch.uint8, device=dev))
        pt["opt"] = qoq.gemm_options(act_operand=pt["act"], flags=qoq.QOQ_LAUNCH_OVERLAP)
        return pt

    pts = [make_point(*p) for p in points]
    ws_max = max([256] + [qoq.qoq_gemm_workspace_bytes(p["M"], p["layer"].N, p["layer"].K, p["group"]) for p in pts])
    ws = qoq.new_workspace(ws_max, dev)
    torch.cuda.synchronize()

    def quant_point(pt):
        qoq.qoq_quant_act_ex(pt["X"], pt["Qx"], pt["sx"], pt["tx"], pt["act"], kind=pt["kind"],
                             with_t=pt["group"] == 0, flags=qoq.QOQ_LAUNCH_OVERLAP)

    def gemm_point(pt, copy_idx):
        layer = pt["layer"]
        copies, s_w = weights[(pt["wid"], layer.name)]
        qoq.qoq_w4a8_gemm_ex(pt["Qx"], pt["sx"], pt["tx"], copies[copy_idx % len(copies)], s_w, layer.N,
                             layer.K, pt["group"], O=pt["O"], workspace=ws, options=pt["opt"])

    def run_point(pt, copy_idx):
        quant_point(pt)
        gemm_point(pt, copy_idx)

    def step():
        for i, pt in enumerate(pts):
            run_point(pt, i)

    # eager warm-up (sets kernel attributes before capture), then capture one step
    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    est_ms = 1e3 * (time.perf_counter() - t0) / max(3, args.warmup)

    # Clocks: the timed region (K steps) is shorter than one 200 ms sampling
    # interval, so the sampler runs over a loaded window of untimed replays
    # of the same step that ends with the timed region.
    clocks = ClockSampler(gpu_pci_id(torch, local_rank))
    clocks.start()
    time.sleep(0.3)
    w0 = time.time()
    for _ in range(int(args.soak_s * 1e3 / max(est_ms, 1e-3))):
        graph.replay()
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
    w1 = time.time()
    if dist:
        dist.barrier()
    clk = clocks.stop(window=(w0, w1))
    if clk:
        clk["window_s"] = round(w1 - w0, 2)
        clk["window"] = "untimed replays of the step, then the timed region"
    ms_step = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dist, dev)
    ops_step = sum(roofline.gemm_ops(p["M"], p["layer"].N, p["layer"].K) for p in pts)
    tops = whole_job_tops(ops_step, world, ms_step)
    del graph

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

    def time_points(plist):
        rows = []
        for pt in plist:
            layer, M = pt["layer"], pt["M"]
            copies, _ = weights[(pt["wid"], layer.name)]
            reps = max(args.point_reps, len(copies))
            if M * layer.N * layer.K >= 2 ** 36:  # long launches: fewer per graph
                reps = max(8, len(copies))
            run_point(pt, 0)  # eager once (kernel attributes) before capture
            torch.cuda.synchronize()
            t_q = graph_us(lambda r: quant_point(pt), reps)
            t_g = graph_us(lambda r: gemm_point(pt, r), reps)
            nbytes = roofline.w4a8_bytes(M, layer.N, layer.K)
            nops = roofline.gemm_ops(M, layer.N, layer.K)
            troof = roofline.roof_time(M, layer.N, layer.K, bw, p16)
            rows.append({
                "workload": pt["wid"], "layer": layer.name, "N": layer.N, "K": layer.K, "M": M,
                "group": pt["group"], "path": pt["plan"]["path"], "tokens_per_tile": pt["plan"]["tokens_per_tile"],
                "ctas": pt["plan"]["num_ctas"], "gemm_us": round(t_g, 2), "quant_us": round(t_q, 2),
                "TOPS": round(nops / (t_g * 1e-6) / 1e12, 2), "GBs": round(nbytes / (t_g * 1e-6) / 1e9, 1),
                "GBs_full": round(roofline.w4a8_bytes_full(M, layer.N, layer.K, pt["group"]) / (t_g * 1e-6) / 1e9, 1),
                "bound": roofline.bound(M, layer.N, layer.K, bw, p16),
                "roof_frac": round(troof / (t_g * 1e-6), 3),
            })
        return rows

    pt_rows, by_bound, dom, twf = [], {}, None, None
    if not args.no_points:
        pt_rows = time_points(pts)
        by_bound, dom, twf = roofline_summary(pt_rows, bw, p16)

    # ---- end to end through the public API: host buffers, copies timed ----
    e2e = None
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 10))

        # Transfers overlap the compute, as in a serving loop: the inputs go
        # up on a copy-in stream and the outputs come down on a copy-out
        # stream, in groups of points (up to about 2 MB of output each, so
        # large outputs go down while later points compute): a group's
        # compute waits for its inputs' event, its outputs are copied once its
        # last GEMM is done.  A group's inputs (and its outputs) are adjacent
        # in one pinned host buffer and one device buffer, so each group moves
        # in one copy per direction.  Device inputs and outputs are
        # double-buffered across steps, so step n + 1's inputs go up while
        # step n computes and its outputs come down; a buffer set is rewritten
        # only after step n - 1's readers of it (its compute for the inputs,
        # its device-to-host copies for the outputs) have finished, and the
        # timed region ends when the last step's outputs are on the host.  The
        # points run in another order than in the device-timed step (the same
        # work): most output bytes per unit of compute first (K ascending;
        # then more tokens first, smaller outputs first), so the
        # device-to-host copies, which take about as long as the compute,
        # start early in the step.
        copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        order = sorted(range(len(pts)), key=lambda i: (pts[i]["layer"].K, -pts[i]["M"], pts[i]["O"].numel()))
        groups, cur, cur_bytes = [], [], 0
        for i in order:
            pt = pts[i]
            cur.append(i)
            cur_bytes += pt["O"].numel() * 2
            if cur_bytes >= 2 << 20:
                groups.append(cur)
                cur, cur_bytes = [], 0
        if cur:
            groups.append(cur)

        def layout(key):
            """Element offsets (256-byte aligned) of each point's tensor in the
            processing order, and the total."""
            offs, at = {}, 0
            for i in order:
                offs[i] = at
                at += (pts[i][key].numel() + 127) // 128 * 128
            return offs, at

        x_off, x_tot = layout("X")
        o_off, o_tot = layout("O")

        def views(flat, offs, key):
            return {i: flat[offs[i]:offs[i] + pts[i][key].numel()].view(pts[i][key].shape) for i in order}

        hostX_flat = torch.empty((x_tot,), dtype=torch.float16).pin_memory()
        hostO_flat = torch.empty((o_tot,), dtype=torch.float16).pin_memory()
        hostX, hostO = views(hostX_flat, x_off, "X"), views(hostO_flat, o_off, "O")
        for i in order:
            hostX[i].copy_(pts[i]["X"].cpu())
        h2d = sum(pts[i]["X"].numel() * 2 for i in order)
        d2h = sum(pts[i]["O"].numel() * 2 for i in order)
        dX = [torch.empty((x_tot,), dtype=torch.float16, device=dev) for _ in range(2)]
        dO = [torch.empty((o_tot,), dtype=torch.float16, device=dev) for _ in range(2)]
        bufs = [{i: (views(dX[s_], x_off, "X")[i], views(dO[s_], o_off, "O")[i]) for i in order} for s_ in range(2)]
        orig = [(p["X"], p["O"]) for p in pts]

        def span(offs, key, grp):
            """The group's element range in the flat buffers."""
            a = offs[grp[0]]
            return a, offs[grp[-1]] + pts[grp[-1]][key].numel()

        x_span = [span(x_off, "X", g) for g in groups]
        o_span = [span(o_off, "O", g) for g in groups]
        ev_in = [[torch.cuda.Event() for _ in groups] for _ in range(2)]
        ev_done = [[torch.cuda.Event() for _ in groups] for _ in range(2)]
        ev_comp_end = [torch.cuda.Event() for _ in range(2)]
        ev_out_end = [torch.cuda.Event() for _ in range(2)]
        for e in ev_comp_end + ev_out_end:
            e.record(stream)

        def e2e_step(n):
            bs = n % 2
            copy_in.wait_event(ev_comp_end[bs])  # step n - 2 has read these inputs
            with torch.cuda.stream(copy_in):
                for gi in range(len(groups)):
                    a, b_ = x_span[gi]
                    dX[bs][a:b_].copy_(hostX_flat[a:b_], non_blocking=True)
                    ev_in[bs][gi].record(copy_in)
            stream.wait_event(ev_out_end[bs])  # step n - 2's outputs are on the host
            for gi, grp in enumerate(groups):
                stream.wait_event(ev_in[bs][gi])
                for i in grp:
                    pts[i]["X"], pts[i]["O"] = bufs[bs][i]
                    run_point(pts[i], i)
                ev_done[bs][gi].record(stream)
                copy_out.wait_event(ev_done[bs][gi])
                with torch.cuda.stream(copy_out):
                    a, b_ = o_span[gi]
                    hostO_flat[a:b_].copy_(dO[bs][a:b_], non_blocking=True)
            ev_comp_end[bs].record(stream)
            ev_out_end[bs].record(copy_out)

        for n in range(2):
            e2e_step(n)
        stream.wait_stream(copy_out)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        copy_in.wait_stream(stream)
        copy_out.wait_stream(stream)
        for n in range(e2e_steps):
            e2e_step(n)
        stream.wait_stream(copy_out)
        b.record(stream)
        torch.cuda.synchronize()
        for i, p in enumerate(pts):
            p["X"], p["O"] = orig[i]
        if dist:
            dist.barrier()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / e2e_steps, dist, dev)
        e2e = {"value": whole_job_tops(ops_step, world, e2e_ms), "unit": "TOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "path": "Python binding -> C ABI per call (no CUDA graph), pinned host buffers, host<->device copies on two side streams overlapping the compute (one copy per group of points and direction), device inputs and outputs double-buffered across steps"}
        del hostX, hostO, bufs, dX, dO, hostX_flat, hostO_flat

    # ---- further workloads, point by point ----
    block_out = {}

    def fused_quant_block():
        """The fused norm / activation + quantization kernels alone (graphs of
        back-to-back launches, inputs > L2 rotated), against the HBM roof of
        their bytes, and the unfused chain (torch's fp16 norm / SiLU-mul, then
        qoq_quant_act_ex) for comparison."""
        F_ = torch.nn.functional
        rows = []
        for M in [m for m in synthetic.DECODE_MS] + [synthetic.PREFILL_M]:
            for op, K in (("rmsnorm_quant", 4096), ("silu_mul_quant", 14336)):
                kind = qoq.qoq_gemm_path(M, 28672 if op == "rmsnorm_quant" else 4096, K, 128)
                kin = K if op == "rmsnorm_quant" else 2 * K
                nin = max(3, -(-2 * l2_bytes // (2 * M * kin)) + 1)
                gen = torch.Generator(device=dev)
                gen.manual_seed(M + K)
                Xs = [torch.randn((M, kin), generator=gen, device=dev).to(torch.float16) for _ in range(min(nin, 64))]
                gamma = (1 + 0.1 * torch.randn((K,), generator=gen, device=dev)).to(torch.float16)
                Qx = torch.empty((M, K), dtype=torch.int8, device=dev)
                sx = torch.empty((M,), dtype=torch.float16, device=dev)
                act = torch.empty((qoq.qoq_act_operand_bytes(M, K, kind),), dtype=torch.uint8, device=dev)

                def fused(r):
                    if op == "rmsnorm_quant":
                        qoq.qoq_rmsnorm_quant_act(Xs[r % len(Xs)], gamma, 1e-5, Qx, sx, None, act, kind=kind,
                                                  with_t=False, flags=qoq.QOQ_LAUNCH_OVERLAP)
                    else:
                        qoq.qoq_silu_mul_quant_act(Xs[r % len(Xs)], Qx, sx, None, act, kind=kind, with_t=False,
                                                   flags=qoq.QOQ_LAUNCH_OVERLAP)

                Ybuf = torch.empty((M, K), dtype=torch.float16, device=dev)

                def unfused(r):
                    Xr = Xs[r % len(Xs)]
                    if op == "rmsnorm_quant":
                        torch.mul(F_.rms_norm(Xr, (K,), eps=1e-5), gamma, out=Ybuf)
                    else:
                        torch.mul(F_.silu(Xr[:, :K]), Xr[:, K:], out=Ybuf)
                    qoq.qoq_quant_act_ex(Ybuf, Qx, sx, None, act, kind=kind, with_t=False)

                fused(0)
                unfused(0)
                torch.cuda.synchronize()
                reps = max(args.point_reps, len(Xs))
                t_f = graph_us(fused, reps)
                t_u = graph_us(unfused, reps)
                nbytes = 2 * M * kin + (2 * K if op == "rmsnorm_quant" else 0) + M * K + act.numel() + 2 * M
                rows.append({"op": op, "M": M, "K": K, "act_kind": kind, "us": round(t_f, 2),
                             "unfused_us": round(t_u, 2), "bytes": nbytes,
                             "GBs": round(nbytes / (t_f * 1e-6) / 1e9, 1),
                             "hbm_frac": round(nbytes / (t_f * 1e-6) / bw, 3)})
                del Xs
        tb = sum(r["bytes"] for r in rows)
        tt = sum(r["us"] for r in rows) * 1e-6
        return {"workload": BLOCKS["fused_quant"][1], "bound": "hbm",
                "bytes_weighted_hbm_frac": tb / tt / bw,
                "fused_vs_unfused_time": sum(r["us"] for r in rows) / sum(r["unfused_us"] for r in rows),
                "points": rows}

    def kv4_block():
        """Decode attention over the KV4 cache alone (graphs of back-to-back
        launches rotating over KV pools that together exceed twice the L2),
        against the HBM roof of its bytes: the 4-bit K and V codes with their
        fp16 scale and zero per token and head, Q and O."""
        rows = []
        hq, hkv, D = 32, 8, 128
        for name, B, lo, hi in (("batch64_len512-1536", 64, 512, 1536), ("batch8_len8192", 8, 8192, 8192)):
            rng = np.random.default_rng(B + lo)
            lens = rng.integers(lo, hi + 1, B).astype(np.int32)
            npg = (lens + 63) // 64
            max_pages = int(npg.max())
            num_pages = int(npg.sum())
            page_b = qoq.qoq_kv4_page_bytes(hkv)
            pool_bytes = num_pages * page_b
            npools = max(3, -(-2 * l2_bytes // pool_bytes) + 1)
            tab = np.full((B, max_pages), -1, np.int32)
            k = 0
            for b, n in enumerate(npg):
                tab[b, :n] = np.arange(k, k + n)
                k += n
            table = torch.from_numpy(tab).to(dev)
            seq = torch.from_numpy(np.concatenate([np.full(L, b, np.int32) for b, L in enumerate(lens)])).to(dev)
            pos = torch.from_numpy(np.concatenate([np.arange(L, dtype=np.int32) for L in lens])).to(dev)
            T = int(lens.sum())
            gen = torch.Generator(device=dev)
            gen.manual_seed(B)
            pools = []
            for _ in range(npools):
                Kt = torch.randn((T, hkv, D), generator=gen, device=dev)
                Kt[:, :, :3] *= 10.0
                Kt = Kt.to(torch.float16)
                Vt = torch.randn((T, hkv, D), generator=gen, device=dev).to(torch.float16)
                pool = torch.zeros((num_pages, page_b), dtype=torch.uint8, device=dev)
                qoq.qoq_kv4_append(Kt, Vt, seq, pos, table, pool)
                pools.append(pool)
                del Kt, Vt
            Q = torch.randn((B, hq, D), generator=gen, device=dev).to(torch.float16)
            O = torch.empty_like(Q)
            lens_d = torch.from_numpy(lens).to(dev)
            wsk = qoq.new_workspace(qoq.qoq_kv4_attention_workspace_bytes(B, hq, hkv, max_pages), dev)

            def attn(r):
                qoq.qoq_kv4_decode_attention(Q, pools[r % len(pools)], table, lens_d, hkv, D ** -0.5, O=O, workspace=wsk)

            attn(0)
            torch.cuda.synchronize()
            t = graph_us(attn, max(args.point_reps, npools))
            nbytes = T * hkv * 2 * (64 + 4) + 2 * 2 * B * hq * D + 4 * B * (max_pages + 1)
            rows.append({"config": name, "B": B, "tokens": T, "us": round(t, 2), "bytes": nbytes,
                         "GBs": round(nbytes / (t * 1e-6) / 1e9, 1), "hbm_frac": round(nbytes / (t * 1e-6) / bw, 3),
                         "status": qoq.qoq_workspace_status(wsk)[0]})
            del pools
        return {"workload": BLOCKS["kv4_attention"][1], "bound": "hbm",
                "bytes_weighted_hbm_frac": sum(r["bytes"] for r in rows) / (sum(r["us"] for r in rows) * 1e-6) / bw,
                "points": rows}

    for bname in blocks:
        if bname == "fused_quant":
            block_out[bname] = fused_quant_block()
            continue
        if bname == "kv4_attention":
            block_out[bname] = kv4_block()
            continue
        wid, desc = BLOCKS[bname]
        keep = {int(m) for m in args.block_ms.split(",") if m}
        bpts = [make_point(*p) for p in block_points(bname) if not keep or p[2] in keep]
        need = max(qoq.qoq_gemm_workspace_bytes(p["M"], p["layer"].N, p["layer"].K, p["group"]) for p in bpts)
        if need > ws.numel():
            ws = qoq.new_workspace(need, dev)
        torch.cuda.synchronize()
        rows = time_points(bpts)
        bb, bdom, btwf = roofline_summary(rows, bw, p16)
        block_out[bname] = {"workload": desc, "tops_gemm_only": sum(roofline.gemm_ops(r["M"], r["N"], r["K"]) for r in rows)
                            / (sum(r["gemm_us"] for r in rows) * 1e-6) / 1e12,
                            "time_weighted_roofline_frac": btwf, "by_bound": bb, "dominant_bound": bdom,
                            "points": rows}
        for p in bpts:
            del p["X"], p["Qx"], p["O"], p["act"]
        for k in [k for k in weights if k[0] == wid]:
            del weights[k]
        torch.cuda.empty_cache()

    # ---- CPU oracle on a bounded sample ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = oracle_sample(points, args.cpu_rows, args.cpu_prefill_tokens)
        dt, ops = oracle_pass(sample)
        cpu = {"value": ops / dt / 1e12, "unit": "TOPS", "cores": 1, "kind": "oracle",
               "seconds": round(dt, 2),
               "sample": sample_desc(args.cpu_rows, args.cpu_prefill_tokens, len(points))
               + f" ({os.cpu_count()} host cores present)"}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    # the dominant kernel's roofline: the bound class with the most GEMM time
    roof = None
    if dom:
        d = by_bound[dom]
        traffic = gemm_traffic()
        dom_rows = [r for r in pt_rows if r["bound"] == dom]
        tr = None
        if traffic and all((r["workload"], r["layer"], r["M"]) in traffic for r in dom_rows):
            tr = sum(traffic[(r["workload"], r["layer"], r["M"])] for r in dom_rows) / len(dom_rows)
        kern = sorted({("fp8-operand" if r["path"] == 2 else "fp16-operand") for r in dom_rows})
        roof = {"bound": "hbm" if dom == "hbm" else "tensor", "achieved": d["achieved"], "peak": d["peak"],
                "unit": d["unit"], "frac": d["frac"], "traffic": tr,
                "traffic_scope": "mean DRAM read+write bytes per GEMM launch of this bound class (ncu, cold cache)",
                "algorithmic_bytes_per_launch": sum(roofline.w4a8_bytes(r["M"], r["N"], r["K"]) for r in dom_rows)
                / len(dom_rows),
                "kernel": " + ".join(f"w4a8_gemm {k} kernel" for k in kern)
                + f" on the {d['points']} {dom}-bound points ({', '.join(sorted({str(r['M']) for r in dom_rows}, key=int))} tokens)",
                "peak_source": f"{peaks_src} ({'HBM copy' if dom == 'hbm' else 'cuBLAS bf16 dense, burst; fp16 rate = bf16 rate'})",
                "time_weighted_roofline_frac": twf,
                "by_bound": by_bound,
                "tensor_peak_tflops": peaks["bf16_tflops"], "tensor_peak_sustained_tflops": peaks["bf16_tflops_sustained"]}
    line = {
        "metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "s8 x u4 -> exact i32 (e4m3 / fp16 tensor-core MMA), fp16 out", "data": "synthetic",
        "config": {"workload": WORKLOAD, "group": 128, "parallelism": f"replicas{world}",
                   "cuda_graph": True, "l2": "inputs larger than L2: packed-weight copies rotated, "
                   + ", ".join(f"{k[1]}@w{k[0]} x{len(c)}" for k, (c, _) in weights.items())
                   + f" ({sum(len(c) * c[0].numel() for c, _ in weights.values()) / 1e6:.0f} MB)"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * len(pts) * args.steps,
        "clocks": clk,
        "points": pt_rows,
        "blocks": block_out,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
