"""Benchmark: weight-streaming Q8_0 decode projections on GB300.

One step = one decode token through the whole projection path of a synthetic
36-layer decoder (hidden 4096; q 4096x4096, k and v 1024x4096, o 4096x4096,
fused gate/up 24576x4096, down 4096x12288, lm-head 151936x4096; RMSNorm ->
quantize before q/k/v and gate/up; lm-head with the argmax epilogue and the
argmax reduce), about 8.04 GB of Q8_0 weights per token, batch 1 (or
--batch 8: 8 activations share each weight read), Int8Act by default.

  value           effective weight GB/s = weight bytes per token / device
                  time per token, inputs resident in HBM, one CUDA graph per
                  token (8 GB of weights per step: every step streams from
                  HBM, nothing fits the 129 MB L2)
  e2e             the same metric with the token input copied from pinned
                  host memory and the argmax read back to the host every step
  roofline        the gate/up GEMV launches (the largest share of a layer's
                  bytes), timed with CUDA events around each launch
  cpu_baseline    the CPU oracle on a bounded sample of the same sequence

``--impl reference`` times the CPU oracle (the reference arm of this
method, which has no other implementation) on the host cores.
Multi-GPU: replicas only (each rank runs its own copy of the sequence).
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

METRIC = "Q8_0 GEMV effective weight GB/s (36-layer decode projection sequence, per token)"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="int8act", choices=["dequant", "int8act", "twopass"])
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--layers", type=int, default=36)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration GEMV table and the other sequence forms")
    ap.add_argument("--workload", default="sequence", choices=["sequence", "gemv"],
                    help="sequence: the per-token decode projections (default); gemv: one "
                         "GEMV shape, launched back to back over rotated weight copies")
    ap.add_argument("--N", type=int, default=24576)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--S", type=int, default=1, help="split-K chunks (gemv workload)")
    ap.add_argument("--argmax", action="store_true", help="argmax epilogue + reduce (gemv workload)")
    ap.add_argument("--format", default=None, choices=["q4_0", "q4_1", "q5_0", "q5_1", "iq4_nl", "mxfp4", "q2_k",
                                                       "q3_k", "q4_k", "q5_k", "q6_k", "iq4_xs"],
                    help="gemv workload: a GGUF block format other than Q8_0 (lk_gemv_blk)")
    ap.add_argument("--glu", action="store_true",
                    help="gemv workload: the gate/up pair (two N/2-row matrices) with the SwiGLU + quantize epilogue")
    ap.add_argument("--path", default="auto", choices=["auto", "direct", "ring", "mma"])
    ap.add_argument("--chain", action="store_true",
                    help="sequence: the whole token as one cooperative chain launch (lk_gemv_chain; fused "
                         "prologues)")
    ap.add_argument("--fused-prologue", action="store_true",
                    help="sequence: every GEMV computes RMSNorm/quantize itself (one launch per projection) "
                         "instead of a separate norm/quantize launch before it (the default, faster on GB300)")
    ap.add_argument("--unfused", action="store_true", help=argparse.SUPPRESS)  # the default; kept for scripts
    ap.add_argument("--fuse", default="", help="sequence: comma-separated projections (q,k,v,o,gu,down,lm) "
                                               "that compute their own norm/quantize prologue")
    ap.add_argument("--prefill", action="append", default=[], help=argparse.SUPPRESS)  # name=warps
    ap.add_argument("--decoder", action="store_true",
                    help="sequence: the decoder-layer dataflow (residual add + norm + quantize launches, the gate/up "
                         "pair with its SwiGLU epilogue feeding down) instead of the projections alone")
    ap.add_argument("--no-pdl", action="store_true",
                    help="no programmatic dependent launches between the fused GEMVs")
    ap.add_argument("--fused", action="store_true", help="gemv workload: RMSNorm->quantize->GEMV in one launch")
    ap.add_argument("--norm", action="store_true",
                    help="gemv workload: an RMSNorm->quantize launch before every GEMV (the separate form)")
    ap.add_argument("--table", default=None,
                    help="write the per-config single-GEMV table (markdown) to this path")
    ap.add_argument("--cfg", action="append", default=[],
                    help="a launch setting name=value (a field of lk_launch_cfg, e.g. mma_tk=1024) for every "
                         "call; repeatable")
    return ap.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0}, "fallback"


def workload_name(a):
    flow = ("decoder layers: residual add + RMSNorm + quantize, SwiGLU + quantize in the gate/up launch"
            if getattr(a, "decoder", False) else "projections alone")
    return (f"decode projections: {a.layers} layers, hidden 4096, q 4096x4096, k/v 1024x4096, "
            f"o 4096x4096, gate/up 24576x4096 (a 2 x 12288x4096 pair), down 4096x12288, lm-head 151936x4096 + "
            f"argmax, batch {a.batch}, {a.mode}; {flow}")


# ---- clocks ------------------------------------------------------------------------

class Clocks:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [r for (t, r) in self.rows if t0 <= t <= t1] or [r for (_, r) in self.rows]
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                smax = max(smax, float(r[3]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- CPU oracle sample ---------------------------------------------------------------

def oracle_layer(oracle, w, mode, x, eps=1e-6):
    """One layer of the sequence on the CPU oracle; returns (the next layer's
    input, weight bytes).  With gate/up as a pair ("gate", "up": the decoder
    dataflow) x is the residual stream entering the layer; otherwise the
    projections-alone dataflow (down's input a fixed vector)."""
    def acts(v):
        if mode == oracle.DEQUANT:
            return dict(x=v)
        hi, lo, s = oracle.quantize(v, mode)
        return dict(hi=hi, lo=lo, s=s)

    nbytes = 0
    a = acts(oracle.rmsnorm(x, w["g_attn"], mode, eps))
    for n in ("q", "k", "v"):
        oracle.gemv(w[n][0], w[n][1], mode, **a)
        nbytes += w[n][0].size * 17 // 16
    o = oracle.gemv(w["o"][0], w["o"][1], mode, **acts(w["o_in"]))
    nbytes += w["o"][0].size * 17 // 16
    if "gate" in w:
        h_mid, y = oracle.add_rmsnorm(o, x, w["g_mlp"], mode, eps)
        _, _, hg, _ = oracle.glu(w["gate"][0], w["gate"][1], w["up"][0], w["up"][1], mode, **acts(y))
        nbytes += 2 * w["gate"][0].size * 17 // 16
        d = oracle.gemv(w["down"][0], w["down"][1], mode, **acts(hg))
        nbytes += w["down"][0].size * 17 // 16
        return (h_mid + d).astype("float32"), nbytes
    a = acts(oracle.rmsnorm(o, w["g_mlp"], mode, eps))
    oracle.gemv(w["gu"][0], w["gu"][1], mode, **a)
    nbytes += w["gu"][0].size * 17 // 16
    h = oracle.gemv(w["down"][0], w["down"][1], mode, **acts(w["d_in"]))
    nbytes += w["down"][0].size * 17 // 16
    return h, nbytes


def host_layer(stack_or_none, l, B, mode_seed=0):
    """Host (numpy) copy of layer l's inputs, from the device stack when given,
    else freshly drawn with the same recipe."""
    import numpy as np

    from q8_quantized_gemv_gb300 import synth
    if stack_or_none is not None:
        w = stack_or_none.layers[l]
        out = {}
        for n in ("q", "k", "v", "o", "gu", "gate", "up", "down"):
            if n in w:
                out[n] = (w[n][0].cpu().numpy(), w[n][1].cpu().numpy().view(np.uint16))
        for n in ("g_attn", "g_mlp", "o_in", "d_in"):
            out[n] = w[n].cpu().numpy()
        return out
    shapes = {"q": (4096, 4096), "k": (1024, 4096), "v": (1024, 4096), "o": (4096, 4096),
              "gate": (12288, 4096), "up": (12288, 4096), "down": (4096, 12288)}
    s = synth.SEED_BASE + 4 + 1000 * l + mode_seed
    out = {n: synth.q8_matrix(N, K, s + i) for i, (n, (N, K)) in enumerate(shapes.items())}
    out["g_attn"] = synth.norm_gain(4096, s + 10)
    out["g_mlp"] = synth.norm_gain(4096, s + 11)
    out["o_in"] = synth.activation(B, 4096, s + 12, outliers=True)
    out["d_in"] = synth.activation(B, 12288, s + 13, outliers=True)
    return out


def host_info():
    """The host the CPU timings ran on: logical CPUs, architecture, model."""
    import platform
    info = {"nproc": os.cpu_count(), "machine": platform.machine()}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip() in ("model name", "Model", "Hardware", "CPU part") and v.strip():
                    info["model"] = v.strip()
                    break
    except OSError:
        pass
    return info


def _time_oracle_layers(oracle, stack, a, mode, budget_s, first_layer=0):
    """Oracle layers of the sequence, in order from `first_layer`, until
    `budget_s` seconds of oracle time; returns (bytes, seconds, layers)."""
    import numpy as np
    x = stack.x0.cpu().numpy() if stack is not None else np.ones((a.batch, 4096), np.float32)
    tot_b, tot_t, n = 0, 0.0, 0
    for l in range(first_layer, a.layers):
        w = host_layer(stack, l, a.batch)
        t0 = time.perf_counter()
        x, nb = oracle_layer(oracle, w, mode, x)
        tot_t += time.perf_counter() - t0
        tot_b += nb
        n += 1
        if tot_t >= budget_s:
            break
    return tot_b, tot_t, n


def cpu_baseline(stack, a, budget_s):
    """The oracle on the host cores: all of them (its GEMV row loops over
    every logical CPU, bit-identical to one thread) for the reported value,
    and one thread beside it, each on a bounded sample of the sequence."""
    import oracle

    mode = {"dequant": 0, "int8act": 1, "twopass": 2}[a.mode]
    cores = os.cpu_count() or 1
    oracle.set_threads(1)
    b1, t1, n1 = _time_oracle_layers(oracle, stack, a, mode, budget_s / 3)
    used = oracle.set_threads(cores)
    try:
        bn, tn, nn = _time_oracle_layers(oracle, stack, a, mode, 2 * budget_s / 3)
    finally:
        oracle.set_threads(1)
    what = f"(full matrices, norm + quantize + 6 GEMVs each, batch {a.batch}, {a.mode}), C oracle"
    return {"value": bn / tn / 1e9, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"layers 0..{nn - 1} of the sequence {what}, GEMV rows over {used} threads",
            "seconds": tn, "host": host_info(),
            "single_thread": {"value": b1 / t1 / 1e9, "unit": UNIT, "cores": 1,
                              "sample": f"layers 0..{n1 - 1} of the sequence {what}, one thread",
                              "seconds": t1}}


# ---- reference arm: the CPU oracle -----------------------------------------------------

def run_reference(a, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    mode = {"dequant": 0, "int8act": 1, "twopass": 2}[a.mode]
    import numpy as np
    cores = oracle.set_threads(os.cpu_count() or 1)
    layers = [host_layer(None, l, a.batch) for l in range(2)]
    x0 = np.ones((a.batch, 4096), np.float32)

    def step():
        x, nb = x0, 0
        for w in layers:
            x, b = oracle_layer(oracle, w, mode, x)
            nb += b
        return nb

    for _ in range(a.warmup):
        step()
    t0 = time.perf_counter()
    nb = 0
    for _ in range(a.steps):
        nb += step()
    dt = time.perf_counter() - t0
    value = nb / dt / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": a.gpus,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": dt / a.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": _dtype(a.mode),
        "data": "synthetic", "config": {"workload": workload_name(a),
                                        "sample": "2 of the layers per step, on the host"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: layers 0-1 of the sequence (full matrices) in the C oracle, "
                                   f"GEMV rows over {cores} threads", "host": host_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def _dtype(mode):
    return {"dequant": "f32 x int8 -> f64", "int8act": "int8 x int8 -> int32, f32 combine",
            "twopass": "2x int8 x int8 -> int32, f32 combine"}[mode]


# ---- our arm ---------------------------------------------------------------------------------

def run_ours(a, rank, world):
    import torch

    from q8_quantized_gemv_gb300 import build, lk
    from q8_quantized_gemv_gb300.decode import DecodeStack

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    fused = (a.fused_prologue or a.chain) and not a.unfused
    if a.fuse and not fused:
        fused = [n for n in a.fuse.split(",") if n]
    prefill = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in a.prefill}
    stack = DecodeStack(layers=a.layers, batch=a.batch, mode=a.mode, device=dev, fused=fused, chain=a.chain and fused,
                        prefill=prefill, glu=a.decoder, pdl=not a.no_pdl, tune=_tune(a))
    tok_bytes = stack.weight_bytes()
    stream = torch.cuda.Stream(device=dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    # eager warm-up (also sets any per-kernel attributes before capture)
    with torch.cuda.stream(stream):
        for _ in range(2):
            stack.run_token()
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0

    # one CUDA graph per token
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        stack.run_token()
    x_in = stack.x_buf  # the token input buffer the launches read
    graph_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_e2e, stream=stream):
        stack.run_token(x_in=x_in)

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.5)
    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K tokens, inputs resident -------------------------------------
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    tw0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(a.steps):
            graph.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    tw1 = time.time()
    barrier()
    ms = ev0.elapsed_time(ev1) / a.steps
    clk = clocks.summary(tw0, tw1)
    clocks.stop()
    ms_max = _max_over_ranks(ms, dist, dev)
    value = replica_value(tok_bytes, world, ms_max)

    # ---- e2e: pinned host input -> device, graph, argmax -> pinned host, every step ------
    x_host = stack.x0.cpu().pin_memory()
    idx_host = torch.empty_like(stack.idx, device="cpu").pin_memory()
    with torch.cuda.stream(stream):
        for _ in range(3):
            x_in.copy_(x_host, non_blocking=True)
            graph_e2e.replay()
            idx_host.copy_(stack.idx, non_blocking=True)
            stream.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(1, min(a.steps, 200))
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_e2e):
            x_in.copy_(x_host, non_blocking=True)
            graph_e2e.replay()
            idx_host.copy_(stack.idx, non_blocking=True)
            stream.synchronize()
        e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = _max_over_ranks(e0.elapsed_time(e1) / n_e2e, dist, dev)
    e2e = {"value": tok_bytes * world / (ms_e2e * 1e-3) / 1e9, "unit": UNIT,
           "h2d_bytes_per_step": x_host.numel() * 4, "d2h_bytes_per_step": idx_host.numel() * 4,
           "ms_per_step": ms_e2e, "steps": n_e2e}

    # ---- roofline: CUDA events around every launch of the dominant kernel ---------------
    if stack.chain is not None:
        roof, per_name = roofline_chain(stack, stream, a, torch)
    else:
        roof, per_name = roofline(stack, stream, a, torch)

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": _dtype(a.mode), "data": "synthetic (seeded: int8 levels uniform on [-127, 127], f16 scales |N(0, 0.02)| + 1e-4, N(0, 1) activations with 1 % x20 outliers)",
        "config": {"workload": workload_name(a), "weight_bytes_per_step": tok_bytes,
                   "l2": "inputs larger than L2 (8.04 GB of weights per step)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "path": "auto", "fused_prologue": {k: v for k, v in stack.fused.items()},
                   "gemv_kernel": {k: "ring" if stack.fused[k] else {1: "direct", 2: "ring", 3: "mma"}.get(v, "none")
                                   for k, v in stack.kernel.items()},
                   "chain": stack.chain is not None,
                   "prefill": stack.prefill or "half of the warps",
                   "dataflow": "decoder (glu)" if stack.glu else "projections alone",
                   "pdl": not a.no_pdl, "launch_cfg": a.cfg,
                   "splitk": stack.splitk or "none (one activation row)"},
        "us_per_token": ms_max * 1e3,
        "pct_of_nominal_8TBs": value / world / NOMINAL_HBM_GBS,
        "roofline": roof,
        "gemv_by_projection": per_name,
        "e2e": e2e,
        "clocks": clk,
        "gpu_launches": stack.launches_per_token() * a.steps,
    }
    if rank == 0 and not a.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(stack, a, a.cpu_seconds)
    if rank == 0 and not a.no_configs:
        # after every timed region of the headline: the other configurations
        del graph, graph_e2e
        forms = [(1, "int8act"), (1, "twopass"), (1, "dequant"), (8, "int8act"), (8, "twopass"),
                 (16, "int8act"), (64, "int8act")]
        forms = [(b, m, False) for b, m in forms if (b, m) != (a.batch, a.mode) or a.decoder] + \
                [(b, m, True) for b, m in ((1, "int8act"), (1, "twopass"), (8, "int8act"))
                 if (b, m) != (a.batch, a.mode) or not a.decoder]
        out["sequences"] = measure_sequences(a, forms, dev)
        out["configs"] = measure_configs(a)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_blk_sequence(a, rank, world):
    """The 36-layer projection sequence with every matrix in block format
    `a.format` (BlkDecodeStack): one CUDA graph per token, timed like the
    Q8_0 sequence; the line carries the same keys (roofline: the gate/up
    launches of a token back to back; cpu_baseline: the oracle on one
    layer's projections)."""
    import numpy as np
    import torch

    import oracle
    from q8_quantized_gemv_gb300 import build, lk
    from q8_quantized_gemv_gb300.decode import BlkDecodeStack

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stack = BlkDecodeStack(a.format, layers=a.layers, batch=a.batch, mode=a.mode, device=dev, pdl=not a.no_pdl)
    tok_bytes = stack.weight_bytes()
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(2):
            stack.run_token()
    torch.cuda.synchronize()
    assert lk.lk_device_error(reset=True) == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        stack.run_token()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.5)
    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            graph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    tw0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(a.steps):
            graph.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    tw1 = time.time()
    if dist is not None:
        dist.barrier()
    clk = clocks.summary(tw0, tw1)
    clocks.stop()
    ms_max = _max_over_ranks(ev0.elapsed_time(ev1) / a.steps, dist, dev)
    value = replica_value(tok_bytes, world, ms_max)
    # e2e: the token input from pinned host memory, the argmax back, every step
    x_host = stack.x0.cpu().pin_memory()
    idx_host = torch.empty_like(stack.idx, device="cpu").pin_memory()
    n_e2e = max(1, min(a.steps, 200))
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            stack.x_buf.copy_(x_host, non_blocking=True)
            graph.replay()
            idx_host.copy_(stack.idx, non_blocking=True)
            stream.synchronize()
        e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = _max_over_ranks(e0.elapsed_time(e1) / n_e2e, dist, dev)
    # roofline: the token's gate/up launches back to back in one graph
    got = []

    def hook(name, launch):
        if name == "gu":
            got.append(launch)
        return launch()

    with torch.cuda.stream(stream):
        stack.run_token(hook=hook)
    torch.cuda.synchronize()
    g_gu = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_gu, stream=stream):
        for launch in got:
            launch()
    with torch.cuda.stream(stream):
        g_gu.replay()
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        reps = 5
        for _ in range(reps):
            g_gu.replay()
        r1.record(stream)
    torch.cuda.synchronize()
    gu_us = r0.elapsed_time(r1) * 1e3 / (reps * len(got))
    peaks, src = measured_peaks()
    gu_bytes = stack.weight_bytes("gu")
    act_b = a.batch * 4096 * (4 if stack.mode == lk.LK_DEQUANT else 2 if stack.mode == lk.LK_TWOPASS else 1)
    alg = gu_bytes + act_b + a.batch * stack.shapes["gu"][0] * 4
    roof = {"bound": "hbm", "achieved": alg / (gu_us * 1e-6) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": alg / (gu_us * 1e-6) / 1e9 / peaks["hbm_gbs"], "traffic": None, "peak_source": src,
            "kernel": f"gate/up {a.format.upper()} GEMV 24576x4096 (lk_gemv_blk)",
            "algorithmic_bytes_per_launch": alg, "avg_launch_us": gu_us, "launches_timed": reps * len(got)}
    out = {
        "metric": f"{a.format.upper()} GEMV effective weight GB/s (36-layer decode projection sequence, per token)",
        "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": _dtype(a.mode),
        "data": f"synthetic (seeded {a.format.upper()} blocks: random levels, scales and offsets; N(0, 1) activations "
                "with 1 % x20 outliers)",
        "config": {"workload": workload_name(a) + f", weights {a.format.upper()}", "weight_bytes_per_step": tok_bytes,
                   "l2": "inputs larger than L2", "parallelism": "replicas" if world > 1 else "single GPU"},
        "us_per_token": ms_max * 1e3,
        "roofline": roof,
        "e2e": {"value": tok_bytes * world / (ms_e2e * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": x_host.numel() * 4, "d2h_bytes_per_step": idx_host.numel() * 4,
                "ms_per_step": ms_e2e, "steps": n_e2e},
        "clocks": clk,
        "gpu_launches": stack.launches_per_token() * a.steps,
    }
    if rank == 0 and not a.no_cpu_baseline:
        # the oracle on layer 0's four projections (host copies), one thread
        F = oracle.FORMATS[a.format]
        w0 = stack.layers[0]
        host = {n: w0[n].cpu().numpy() for n in stack.shapes}
        t0 = time.perf_counter()
        nbytes = 0
        for n, (N, K) in stack.shapes.items():
            x = np.random.default_rng(0).standard_normal((a.batch, K)).astype(np.float32)
            if stack.mode == lk.LK_DEQUANT:
                oracle.gemv_blk(F, host[n], K, 0, x=x)
            else:
                hi, lo, sc = oracle.quantize(x, stack.mode)
                oracle.gemv_blk(F, host[n], K, stack.mode, hi=hi, lo=lo, s=sc)
            nbytes += stack.weight_bytes(n)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": nbytes / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
                               "sample": f"layer 0's q|k|v, o, gate/up and down ({a.format.upper()}), C oracle, "
                                         "one thread", "seconds": dt}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def _tune(a):
    """The --cfg launch settings as a dict of lk_launch_cfg fields."""
    return {kv.split("=")[0]: int(kv.split("=")[1]) for kv in a.cfg}


def _timing_event(torch, external):
    if external:
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return None
    return torch.cuda.Event(enable_timing=True)


def run_gemv(a, rank, world, quiet=False, sample_clocks=True):
    """One GEMV shape: per-launch CUDA-event durations over weight copies
    rotated so that every launch streams from HBM (copies x bytes >= 4 x L2)."""
    import torch

    from q8_quantized_gemv_gb300 import build, lk, synth

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    cfg = lk.launch_cfg(**dict(_tune(a), path=a.path, pdl=0 if a.no_pdl else 1))
    mode = lk.MODES[a.mode]
    N, K, B, S = a.N, a.K, a.batch, a.S
    wbytes = N * lk.lk_format_row_bytes(a.format, K) if a.format else N * K + N * K // 16
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, -(-4 * l2 // wbytes))
    if a.format:
        mats = [(synth.blk_matrix_torch(a.format, N, K, synth.SEED_BASE + 50 + r, dev), None) for r in range(R)]
    else:
        mats = [synth.q8_matrix_torch(N, K, synth.SEED_BASE + 50 + r, dev) for r in range(R)]
    x = synth.activation_torch(B, K, synth.SEED_BASE + 49, dev, outliers=True)
    acts = {"x": x}
    if mode != lk.LK_DEQUANT:
        xq = torch.empty((B, K), dtype=torch.int8, device=dev)
        xl = torch.empty((B, K), dtype=torch.int8, device=dev) if mode == lk.LK_TWOPASS else None
        xs = torch.empty((B, K // 32), dtype=torch.float32, device=dev)
        lk.lk_quantize_act(x, mode, xq, xl, xs)
        acts = {"xq": xq, "xl": xl, "xs": xs}
    y = torch.empty((B, N), dtype=torch.float32, device=dev)
    parts = torch.zeros((B * lk.lk_argmax_parts_max(N),), dtype=torch.int64, device=dev) if a.argmax else None
    idx = torch.empty((B,), dtype=torch.int32, device=dev)
    part = None
    if S > 1:
        part = torch.empty((lk.lk_splitk_workspace_bytes(mode, S, B, N),), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    gain = synth.norm_gain_torch(K, synth.SEED_BASE + 48, dev)

    xn = torch.empty((B, K), dtype=torch.float32, device=dev) if mode == lk.LK_DEQUANT else None

    F = N // 2
    gu_buf = torch.empty((2, B, F), dtype=torch.float32, device=dev) if a.glu else None
    h_glu = torch.empty((B, F), dtype=torch.float32, device=dev) if a.glu else None
    hact = ({"hq": torch.empty((B, F), dtype=torch.int8, device=dev),
             "hl": torch.empty((B, F), dtype=torch.int8, device=dev) if mode == lk.LK_TWOPASS else None,
             "hs": torch.empty((B, F // 32), dtype=torch.float32, device=dev)} if a.glu and mode else {})
    cnt = torch.zeros((F // 32,), dtype=torch.int32, device=dev) if a.glu else None

    def launch(r):
        wq, ws = mats[r % R]
        if a.format:
            lk.lk_gemv_blk(a.format, wq, K, mode, y, M=B, cfg=cfg, **acts)
            return
        if a.glu:
            # the two halves of the copy as the gate and the up matrix
            lk.lk_gemv_q8_glu(wq[:F], ws[:F], wq[F:], ws[F:], mode, gu_buf, h=h_glu, cnt=cnt, M=B, cfg=cfg, **hact,
                              **({"x": xn if xn is not None and a.norm else x} if mode == lk.LK_DEQUANT else acts))
            return
        if a.norm and not a.fused:
            if mode == lk.LK_DEQUANT:
                lk.lk_rmsnorm_quant(x, gain, mode, 1e-6, xn, cfg=cfg)
            else:
                lk.lk_rmsnorm_quant(x, gain, mode, 1e-6, None, acts["xq"], acts["xl"], acts["xs"], cfg=cfg)
        if a.fused:
            n = lk.lk_rmsnorm_quant_gemv_q8(wq, ws, mode, x, y, gain=gain, argmax_parts=parts, cfg=cfg)
            if a.argmax:
                lk.lk_argmax(idx, B, N, parts=parts, n_parts=n)
        elif S > 1:
            lk.lk_gemv_q8_splitk(wq, ws, mode, S, part, M=B, cfg=cfg, **acts)
            lk.lk_splitk_combine(mode, part, S, B, N, y, cfg=cfg)
        else:
            n = lk.lk_gemv_q8(wq, ws, mode, y, M=B, argmax_parts=parts, cfg=cfg,
                              **({"x": xn} if xn is not None and a.norm else acts))
            if a.argmax:
                lk.lk_argmax(idx, B, N, parts=parts, n_parts=n)

    with torch.cuda.stream(stream):
        for r in range(max(a.warmup, 3)):
            launch(r)
    torch.cuda.synchronize()
    # R back-to-back launches over the rotated copies, captured once, replayed
    # `steps` times: the per-launch time carries no host launch gaps
    Rg = max(R, 8)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for r in range(Rg):
            launch(r)
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    if sample_clocks:
        clocks.start()
        time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tw0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(a.steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    tw1 = time.time()
    clk = clocks.summary(tw0, tw1)
    clocks.stop()
    us = e0.elapsed_time(e1) * 1e3 / (a.steps * Rg)
    act_b = B * K * 4 if mode == lk.LK_DEQUANT else B * K * (2 if mode == lk.LK_TWOPASS else 1) + B * (K // 32) * 4
    alg = wbytes + act_b + B * N * 4 + (2 * S * B * N * (8 if mode == lk.LK_DEQUANT else 4) if S > 1 else 0)
    peaks, src = measured_peaks()
    gbs = wbytes / (us * 1e-6) / 1e9
    out = {"metric": ("block-format" if a.format else "Q8_0") + " GEMV effective weight GB/s", "value": gbs, "unit": UNIT, "n_gpus": world,
           "steps": a.steps, "warmup": a.warmup, "ms_per_step": us * 1e-3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": _dtype(a.mode), "data": "synthetic",
           "config": {"workload": (f"{a.format.upper()} GEMV" if a.format else "Q8_0 GEMV")
                                  + f" N={N} K={K} batch {B} {a.mode} S={S}"
                                  + (" gate/up pair + SwiGLU + quantize" if a.glu else "")
                                  + (" + argmax" if a.argmax else "") + (" fused norm+quant" if a.fused else "")
                                  + (" after a norm+quant launch" if a.norm and not a.fused else ""),
                      "rotation": f"{R} weight copies ({R * wbytes} bytes >= 4x L2), {max(R, 8)} launches per graph",
                      "path": a.path},
           "us_per_gemv": us, "pct_of_nominal_8TBs": gbs / NOMINAL_HBM_GBS,
           "roofline": {"bound": "hbm", "achieved": alg / (us * 1e-6) / 1e9, "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": alg / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], "traffic": None,
                        "peak_source": src, "algorithmic_bytes_per_launch": alg},
           "clocks": clk,
           "gpu_launches": a.steps * Rg * (1 + (1 if (S > 1 or a.argmax) else 0) + (1 if a.norm and not a.fused else 0)),
           "kernel": "blk" if a.format else
                     {1: "direct", 2: "ring", 3: "mma", 0: "none"}[lk.lk_gemv_kernel_for(N, K, mode, B,
                                                                                          S if S > 1 else 0,
                                                                                          cfg=cfg)]}
    del mats
    torch.cuda.empty_cache()
    if rank == 0 and not quiet:
        print(json.dumps(out), flush=True)
    return out


# The single-GEMV configurations of the workload: (label, keyword settings
# of run_gemv).  C1 and C3 in both forms: an RMSNorm -> quantize launch
# before the GEMV (the sequence's form) and the one-launch fused prologue.
def gemv_configs():
    out = []
    for m in ("dequant", "int8act", "twopass"):
        out.append(("C0 1024x1024", dict(N=1024, K=1024, mode=m)))
    for m in ("dequant", "int8act", "twopass"):
        out.append(("C1 q 4096x4096 (norm+quant launch, then GEMV)", dict(N=4096, K=4096, mode=m, norm=True)))
        out.append(("C1 gate/up 24576x4096 (norm+quant launch, then GEMV)", dict(N=24576, K=4096, mode=m, norm=True)))
        out.append(("C1 q 4096x4096 (norm+quant fused)", dict(N=4096, K=4096, mode=m, fused=True)))
        out.append(("C1 gate/up 24576x4096 (norm+quant fused)", dict(N=24576, K=4096, mode=m, fused=True)))
    for m in ("twopass", "dequant"):
        for S in (1, 2, 4, 8):
            out.append(("C2 o 5120x5120 split-K", dict(N=5120, K=5120, mode=m, S=S)))
            out.append(("C2 down 5120x25600 split-K", dict(N=5120, K=25600, mode=m, S=S)))
    for m in ("dequant", "int8act", "twopass"):
        out.append(("C3 lm-head 151936x4096 + argmax (norm launch, then GEMV)",
                    dict(N=151936, K=4096, mode=m, norm=True, argmax=True)))
        out.append(("C3 lm-head 151936x4096 + argmax (norm+quant fused)",
                    dict(N=151936, K=4096, mode=m, fused=True, argmax=True)))
    return out


def measure_configs(a):
    """Every single-GEMV configuration, timed as --workload gemv (back-to-back
    launches in a graph over rotated weight copies, CUDA events), at 1 GPU.
    Returns one dict per configuration."""
    import copy

    peaks, src = measured_peaks()
    rows = []
    for label, kw in gemv_configs():
        b = copy.copy(a)
        b.workload, b.steps, b.warmup = "gemv", 20, 3
        b.S, b.argmax, b.fused, b.norm, b.batch, b.path, b.no_pdl = 1, False, False, False, 1, "auto", False
        for k, v in kw.items():
            setattr(b, k, v)
        d = run_gemv(b, 0, 1, quiet=True, sample_clocks=False)
        rows.append({"config": label, "mode": b.mode, "M": b.batch, "S": b.S, "kernel": d["kernel"],
                     "us_per_gemv": d["us_per_gemv"], "weight_GBs": d["value"],
                     "frac_of_measured_hbm": d["value"] / peaks["hbm_gbs"],
                     "pct_of_nominal_8TBs": 100 * d["value"] / NOMINAL_HBM_GBS,
                     "roofline_frac": d["roofline"]["frac"]})
    return rows


def measure_sequences(a, forms, dev):
    """The per-token sequence in other forms (batch, mode, decoder dataflow):
    us per token and weight GB/s, one CUDA graph per token, `a.steps` tokens
    after warm-up."""
    import torch

    from q8_quantized_gemv_gb300.decode import DecodeStack
    peaks, _ = measured_peaks()
    out = []
    for batch, mode, glu in forms:
        st = DecodeStack(layers=a.layers, batch=batch, mode=mode, device=dev, glu=glu, pdl=True)
        s = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(s):
            st.run_token()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            st.run_token()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        steps = max(1, min(a.steps, 50))
        with torch.cuda.stream(s):
            for _ in range(max(3, a.warmup)):
                g.replay()
            e0.record(s)
            for _ in range(steps):
                g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / steps
        gbs = st.weight_bytes() / (us * 1e-6) / 1e9
        out.append({"batch": batch, "mode": mode, "dataflow": "decoder" if glu else "projections alone",
                    "us_per_token": us, "weight_GBs": gbs,
                    "frac_of_measured_hbm": gbs / peaks["hbm_gbs"], "pct_of_nominal_8TBs": 100 * gbs / NOMINAL_HBM_GBS,
                    "launches_per_token": st.launches_per_token()})
        del g, st
        torch.cuda.empty_cache()
    return out


def run_table(a, path):
    """The per-config table (measure_configs) as markdown rows in `path`, one
    JSON line per row to stdout."""
    peaks, _ = measured_peaks()
    rows = measure_configs(a)
    for r in rows:
        print(json.dumps(r), flush=True)
    with open(path, "w") as f:
        f.write("| Config | Mode | M | S | kernel | us/GEMV | weight GB/s | %% of 8 TB/s | %% of measured %.0f GB/s |\n"
                % peaks["hbm_gbs"])
        f.write("|---|---|---|---|---|---|---|---|---|\n")
        for r in rows:
            f.write(f"| {r['config']} | {r['mode']} | {r['M']} | {r['S']} | {r['kernel']} | {r['us_per_gemv']:.2f} "
                    f"| {r['weight_GBs']:.0f} | {r['pct_of_nominal_8TBs']:.1f} "
                    f"| {100 * r['frac_of_measured_hbm']:.1f} |\n")


def replica_value(bytes_per_step, world, ms_max):
    """Whole-job weight GB/s of `world` replicas: every rank streams its own
    copy of the weights each step, the slowest rank sets the time."""
    return bytes_per_step * world / (ms_max * 1e-3) / 1e9


def _max_over_ranks(v, dist, dev):
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def roofline_chain(stack, stream, a, torch):
    """The whole-token chain kernel is the only launch per token: time each
    launch with CUDA events (after the headline region)."""
    peaks, src = measured_peaks()
    steps = max(3, min(a.steps, 100))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        stack.run_token()
        for e0, e1 in evs:
            e0.record(stream)
            stack.run_token()
            e1.record(stream)
    torch.cuda.synchronize()
    us = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3
    B, mode = stack.B, stack.mode
    act = (lambda K: B * K * 4) if mode == 0 else (lambda K: B * K * (2 if mode == 2 else 1) + B * (K // 32) * 4)
    alg = stack.weight_bytes()
    for N, K in list(stack.shapes.values()) * stack.L + [(stack.V, stack.H)]:
        alg += B * K * 4 + B * N * 4  # raw f32 input read by the prologue, f32 output written
    achieved = alg / (us * 1e-6) / 1e9
    return ({"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
             "frac": achieved / peaks["hbm_gbs"], "traffic": chain_traffic(alg), "peak_source": src,
             "kernel": "gemv_chain_kernel (one cooperative launch per token)",
             "algorithmic_bytes_per_launch": alg, "avg_launch_us": us, "launches_timed": steps},
            {"chain": {"us": us, "GB/s": achieved, "launches": steps}})


def profile_traffic(key, kind, path=None):
    """A DRAM-traffic figure (bytes per launch) from profiles/traffic.txt (one
    ncu capture), if it was taken on the current sources of that kernel
    family (else None).  Lines: "<key>: <bytes> <family>=<sha256>"."""
    try:
        from q8_quantized_gemv_gb300 import build
        with open(path or os.path.join(ROOT, "profiles", "traffic.txt")) as f:
            for line in f:
                if line.startswith("#") or ":" not in line:
                    continue
                k, v = line.split(":", 1)
                if k.strip() != key:
                    continue
                val, tag = v.split()
                fam, sha = tag.split("=")
                if fam != kind or sha != build.sources_digest(kind):
                    return None
                return float(val)
    except (OSError, KeyError, ValueError, AttributeError):
        return None
    return None


def chain_traffic(alg):
    r = profile_traffic("gemv_chain_2layers_int8act_per_algorithmic_byte", "chain")
    return None if r is None else r * alg


def roofline(stack, stream, a, torch):
    peaks, src = measured_peaks()
    steps = max(1, min(a.steps, 50))
    graphs, marks = [], []
    for _ in range(steps):
        evs = []

        def hook(name, launch, evs=evs):
            e0 = _timing_event(torch, True)
            e1 = _timing_event(torch, True)
            if e0 is None:
                raise RuntimeError("this torch has no external CUDA events")
            e0.record(stream)
            r = launch()
            e1.record(stream)
            evs.append((name, e0, e1))
            return r

        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            stack.run_token(hook=hook)
        graphs.append(g)
        marks.append(evs)
    with torch.cuda.stream(stream):
        graphs[0].replay()
        torch.cuda.synchronize()
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()
    # the evs of each graph hold that replay's times
    times = {}
    for evs in marks:
        for name, e0, e1 in evs:
            times.setdefault(name, []).append(e0.elapsed_time(e1))
    B = stack.B
    act_b = B * (1 if stack.mode != 2 else 2)

    def alg_bytes(name):
        """weights + the activation read once + the outputs; "qkv" is the
        grouped q/k/v launch (one activation, three matrices)"""
        mats = [stack.shapes[n] for n in ("q", "k", "v")] if name == "qkv" else \
            [(stack.V, stack.H)] if name == "lm" else [stack.shapes[name]]
        K = mats[0][1]
        act = act_b * K + B * (K // 32) * 4 if stack.mode else B * K * 4
        return act + sum(N * K + N * K // 16 + B * N * 4 for N, K in mats)

    per = {}
    for name, ts in times.items():
        avg = sum(ts) / len(ts)
        per[name] = {"us": avg * 1e3, "GB/s": alg_bytes(name) / (avg * 1e-3) / 1e9, "launches": len(ts)}
    gu = per["gu"]
    peak = peaks["hbm_gbs"]
    kname = "ring_fused" if stack.fused["gu"] else {1: "direct", 2: "ring", 3: "mma"}.get(stack.kernel["gu"], "none")
    mname = {0: "dequant", 1: "int8act", 2: "twopass"}[stack.mode]
    # DRAM bytes per launch from one ncu capture of this kernel and shape, if
    # taken on the current sources (profiles/traffic.txt), else null
    traffic = profile_traffic(f"gemv_{kname}_gateup_24576x4096_{mname}_b{stack.B}",
                              "mma" if kname == "mma" else "ring")
    b2b_us, n_b2b = gu_back_to_back(stack, stream, a, torch)
    alg = alg_bytes("gu")
    roof = {"bound": "hbm", "achieved": alg / (b2b_us * 1e-6) / 1e9, "peak": peak, "unit": "GB/s",
            "frac": alg / (b2b_us * 1e-6) / 1e9 / peak, "traffic": traffic, "peak_source": src,
            "kernel": f"gate/up GEMV 24576x4096 ({kname} kernel)", "algorithmic_bytes_per_launch": alg,
            "avg_launch_us": b2b_us, "launches_timed": n_b2b,
            "timing": "CUDA events around a graph of the token's gate/up launches back to back (every layer's "
                      "matrix, each launch a programmatic dependent of the one before, as in the token)",
            "event_bracketed_us": gu["us"],
            "in_sequence_us": gu_in_sequence(stack, stream, torch)}
    tot_b = sum(alg_bytes(n) * len(ts) for n, ts in times.items())
    tot_t = sum(sum(ts) for ts in times.values())
    roof["all_gemv_event_bracketed"] = tot_b / (tot_t * 1e-3) / 1e9
    return roof, per


def _gu_launches(stack):
    """The token's gate/up launch closures, in order (one token is run to
    collect them; each closure repeats its launch with the same arguments)."""
    got = []

    def hook(name, launch):
        if name == "gu":
            got.append(launch)
        return launch()

    stack.run_token(hook=hook)
    return got


def gu_back_to_back(stack, stream, a, torch):
    """Average duration of the dominant kernel launched back to back: one
    graph of the token's gate/up launches (one per layer, each over its own
    matrix, so nothing is reused through L2), replayed; CUDA events around
    the replays on the launching stream.  Returns (us per launch, launches)."""
    with torch.cuda.stream(stream):
        launches = _gu_launches(stack)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for f in launches:
                f()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = max(3, min(a.steps, 50))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    n = reps * len(launches)
    return e0.elapsed_time(e1) * 1e3 / n, n


def gu_in_sequence(stack, stream, torch):
    """The gate/up launches' share of one captured token, from the library's
    launch timeline (%globaltimer, option "trace" 3): from the previous
    launch's last block end to this launch's last block end, averaged over
    the layers (us); None where the timeline does not cover the token."""
    from q8_quantized_gemv_gb300 import lk
    n = stack.launches_per_token() - 1  # every launch but the argmax reduce is recorded
    if n > lk.LK_TRACE_MAX_RECORDS:
        return None
    lk.lk_set_option("trace", 3)
    try:
        with torch.cuda.stream(stream):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                stack.run_token()
            g.replay()
            torch.cuda.synchronize()
            lk.lk_set_option("trace", 3)  # restart the record count, then one timed replay
            g.replay()
        torch.cuda.synchronize()
        raw = lk.lk_trace_read(lk.LK_TRACE_REC * lk.LK_TRACE_MAX_RECORDS)
    finally:
        lk.lk_set_option("trace", 0)
    R = lk.LK_TRACE_REC
    rec = [raw[i * R:(i + 1) * R] for i in range(n)]
    rows = 2 * stack.F
    spans = [(rec[i][3] - rec[i - 1][3]) / 1e3 for i in range(1, n) if rec[i][6] == rows and rec[i][5] in (1, 3)]
    return sum(spans) / len(spans) if spans else None


def main():
    a = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if a.impl == "reference":
        run_reference(a, rank)
        return
    if a.table:
        run_table(a, a.table)
        return
    if a.workload == "gemv":
        run_gemv(a, rank, world)
        return
    if a.format:
        run_blk_sequence(a, rank, world)
        return
    run_ours(a, rank, world)


if __name__ == "__main__":
    main()
