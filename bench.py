"""Benchmark of the sm_103a attention forward (one JSON line on stdout).

A step is one attention forward pass (one launch of the fused kernel) over one
batch of the base-encoder workload: B=32, H=8, n=m=512, d_k=d_v=64, bf16,
heads from bias-free Xavier projections of X ~ N(0,1), key padding with valid
lengths uniform in [256, 512]. Inputs are synthetic and seeded.

Device timing: the inputs and outputs rotate over enough copies that one pass
over all of them (> 2x the 129 MB L2) never re-reads a warm copy; exactly
--steps launches are captured in one CUDA graph, which is replayed back to back
(at least 10 replays and 200 ms of device time) with CUDA events on the
launching stream around every replay; ms_per_step is the median over replays of
replay time / steps, with p10 and p90 beside it. End-to-end timing goes through
the same C entry point with pinned host buffers: host->device copy of Q, K, V and
the key lengths, the forward pass, device->host copy of O and LSE, every step.

The CPU baseline runs the fp64 oracle on all host cores over the whole workload
(a seeded row sample when the whole would exceed --cpu-seconds); its outputs
also give the error of the timed GPU outputs ("oracle_check").
--impl reference times that oracle, as it stands, step by step.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the forward pass has no exchange step); value = all ranks' FLOPs / the slowest
rank's time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from transformer_scaled_dot_03_gb300 import inputs  # noqa: E402

METRIC = "attention fwd TFLOP/s (bf16) at 1 GB300 and % of dense BF16 tensor peak"
METRIC_BWD = "attention bwd TFLOP/s (bf16; nominal 2.5x the forward's FLOPs) at 1 GB300"
METRIC_PROJ = {"proj": "QKV projection + head split TFLOP/s (bf16) at 1 GB300",
               "outproj": "head merge + output projection TFLOP/s (bf16) at 1 GB300"}
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "base_encoder_keypad"
L2_BYTES = 129 * 1024 * 1024
MIN_REPLAYS = 10          # replays of the timed graph, at least
MIN_TIMED_MS = 200.0      # device time of the timed region, at least
MAX_GRAPH_STEPS = 4096    # launches captured in the timed graph, at most


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, 6800.0, "fallback"


KERNEL_SOURCES = ["transformer_scaled_dot_03_gb300/csrc/attn_kernel_dp.cuh",
                  "transformer_scaled_dot_03_gb300/csrc/attn_softmax.cuh",
                  "transformer_scaled_dot_03_gb300/csrc/sm103a.cuh",
                  "transformer_scaled_dot_03_gb300/csrc/attn_internal.h"]


def measured_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this workload with the current kernel sources; else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.md")
    try:
        fields = {}
        for line in open(path, encoding="utf-8"):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
        h = hashlib.sha256()
        for f in KERNEL_SOURCES:
            h.update(open(os.path.join(ROOT, f), "rb").read())
        if fields.get("workload") == workload and \
                fields.get("kernel_source_sha256_16") == h.hexdigest()[:16]:
            return int(fields["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        pass
    return None


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def quantile(xs, q):
    """Linear-interpolation quantile of an ascending list."""
    if len(xs) == 1:
        return xs[0]
    t = q * (len(xs) - 1)
    i = min(int(t), len(xs) - 2)
    return xs[i] + (xs[i + 1] - xs[i]) * (t - i)


def reduce_over_ranks(ms, e2e_ms, world):
    """Slowest rank's device and end-to-end step times (replicas run independently;
    this host-side max is the only cross-rank operation)."""
    if world <= 1:
        return ms, e2e_ms
    import torch.distributed as dist
    t = torch.tensor([ms, e2e_ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0]), float(t[1])


def job_value(flops_per_rank, world, ms):
    """Whole-job TFLOP/s: every rank's FLOPs over the slowest rank's step time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def workload_slopes(w):
    """Distance-bias slopes [H] of a workload with the linear bias, else None."""
    return inputs.alibi_slopes(w.H) if w.alibi else None


def make_workload(name):
    w = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(w)
    return w, x


def run_ours(args):
    import torch.distributed as dist
    from transformer_scaled_dot_03_gb300 import attn, build

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(attn.LIB_PATH):
        build.build()
    if world > 1:
        dist.barrier()
    attn.load()

    w, x = make_workload(args.workload)
    bwd = args.pass_ == "bwd"
    proj = args.pass_ in ("proj", "outproj")
    decode = w.path == "decode" and not bwd and not proj
    d_model = w.H * w.d_k
    if proj and (w.n != w.m or w.d_k != w.d_v or w.n % 32 != 0):
        raise SystemExit(f"--pass {args.pass_} needs a self-attention workload with n % 32 == 0")
    if args.pass_ == "proj":
        # X [B, n, d_model] times the stacked W_Q, W_K, W_V [3 d_model, d_model]
        flops = eff_flops = 2.0 * w.B * w.n * 3 * d_model * d_model
    elif args.pass_ == "outproj":
        flops = eff_flops = 2.0 * w.B * w.n * d_model * d_model
    else:
        # the backward's five products against the forward's two: 2.5x the nominal FLOPs
        flops = w.flops() * (2.5 if bwd else 1.0)
        eff_flops = effective_flops(w, x) * (2.5 if bwd else 1.0)
    qkv_bytes = x.Q.numel() * 2 + x.K.numel() * 2 + x.V.numel() * 2
    o_bytes = w.B * w.H * w.n * (w.d_v * 2 + 4)
    if args.pass_ == "proj":
        in_bytes, out_bytes = w.B * w.n * d_model * 2, qkv_bytes
    elif args.pass_ == "outproj":
        in_bytes = out_bytes = w.B * w.n * d_model * 2
    elif bwd:
        # inputs Q, K, V, O, LSE, dO; outputs dQ, dK, dV
        in_bytes = qkv_bytes + o_bytes + w.B * w.H * w.n * w.d_v * 2
        out_bytes = qkv_bytes
    else:
        in_bytes, out_bytes = qkv_bytes, o_bytes
    copies = max(2, math.ceil(2 * L2_BYTES / (in_bytes + out_bytes)))
    stream = torch.cuda.Stream(device=dev)
    lens_d = x.key_lengths.to(dev) if x.key_lengths is not None else None
    slopes_d = workload_slopes(w).to(dev) if w.alibi else None
    if w.alibi and (proj or decode):
        raise SystemExit("the distance-bias workloads have a forward and a backward pass only")
    dO_h = inputs.make_grad_output(w.B, w.H, w.n, w.d_v, seed=100 + w.seed) if bwd else None
    sets = []
    if proj:
        Wp, bp = inputs.make_linear((3 if args.pass_ == "proj" else 1) * d_model, d_model, seed=200 + w.seed,
                                    bias=True)
        Wp, bp = Wp.to(dev), bp.to(dev)
        a_h = inputs.make_inputs(w.B, 1, w.n, 1, d_model, d_model, seed=300 + w.seed).Q[:, 0].contiguous() \
            if args.pass_ == "proj" else x.Q
    with torch.cuda.stream(stream):
        for _ in range(copies if proj else 0):
            if args.pass_ == "proj":
                sets.append((a_h.to(dev), torch.empty_like(x.Q, device=dev), torch.empty_like(x.K, device=dev),
                             torch.empty_like(x.V, device=dev)))
            else:
                sets.append((a_h.to(dev), torch.empty(w.B, w.n, d_model, dtype=torch.bfloat16, device=dev)))
        for _ in range(0 if proj else copies):
            st = [x.Q.to(dev), x.K.to(dev), x.V.to(dev),
                  torch.empty(w.B, w.H, w.n, w.d_v, dtype=torch.bfloat16, device=dev),
                  torch.empty(w.B, w.H, w.n, dtype=torch.float32, device=dev)]
            if bwd:
                if w.alibi:
                    attn.attn_fwd_alibi(st[0], st[1], st[2], slopes_d, w.mask, lens_d, x.scale, O=st[3], LSE=st[4],
                                        stream=stream)
                else:
                    attn.attn_fwd(st[0], st[1], st[2], w.mask, lens_d, x.scale, O=st[3], LSE=st[4], stream=stream)
                st += [dO_h.to(dev), torch.empty_like(st[0]), torch.empty_like(st[1]), torch.empty_like(st[2])]
            sets.append(tuple(st))
    if proj:
        ws_bytes, launches_per_step = 0, 1
    elif bwd:
        ws_bytes = attn.bwd_workspace_size(w.B, w.H, w.n, w.m, w.d_k, w.d_v)
        launches_per_step = 3                        # preparation, main kernel, dQ conversion
    elif decode:
        ws_bytes = attn.decode_workspace_size(w.B, w.H, w.n, w.m, w.d_k, w.d_v)
        launches_per_step = 2 if ws_bytes else 1    # the few-row pass merges its key chunks
    else:
        ws_bytes, launches_per_step = 0, 1
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
    torch.cuda.synchronize(dev)

    def run(st, lens, on=None, wsp=None):
        on = stream if on is None else on
        wsp = ws if wsp is None else wsp
        if args.pass_ == "proj":
            X, Q, K, V = st
            attn.proj_heads(X, Wp, w.H, bp, 3, outs=[Q, K, V], stream=on)
        elif args.pass_ == "outproj":
            O, Y = st
            attn.merge_proj(O, Wp, bp, Y=Y, stream=on)
        elif bwd:
            Q, K, V, O, L, dO, dQ, dK, dV = st
            attn.attn_bwd(Q, K, V, O, L, dO, w.mask, lens, x.scale, dQ, dK, dV, workspace=wsp, stream=on,
                          slopes=slopes_d)
        elif decode:
            Q, K, V, O, L = st
            attn.attn_decode(Q, K, V, w.mask, lens, x.scale, O=O, LSE=L, workspace=wsp, stream=on)
        elif w.alibi:
            Q, K, V, O, L = st
            attn.attn_fwd_alibi(Q, K, V, slopes_d, w.mask, lens, x.scale, O=O, LSE=L, stream=on)
        else:
            Q, K, V, O, L = st
            attn.attn_fwd(Q, K, V, w.mask, lens, x.scale, O=O, LSE=L, stream=on)

    def step(i):
        run(sets[i % copies], lens_d)

    # warm-up (also creates the status word before any graph capture)
    torch.cuda.nvtx.range_push("warm-up")
    for i in range(args.warmup):
        step(i)
    torch.cuda.nvtx.range_pop()
    rc, detail = attn.device_status(stream)
    if rc != attn.ATTN_OK:
        raise RuntimeError(f"device status {rc} ({detail}) after warm-up")

    # One CUDA graph of exactly K steps over the rotating copies, replayed R times
    # between events: R >= MIN_REPLAYS and R*K steps take at least MIN_TIMED_MS, so
    # the spread over replays and the clock samples cover a real timed region.
    G = args.steps
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for i in range(G):
                step(i)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):      # replay() launches on the current stream
        graph.replay()
        c0.record(stream)
        graph.replay()
        c1.record(stream)
    torch.cuda.synchronize(dev)
    replay_ms = max(c0.elapsed_time(c1), 1e-3)
    reps = max(MIN_REPLAYS, math.ceil(MIN_TIMED_MS / replay_ms))
    if world > 1:
        # every rank replays the same number of times
        t = torch.tensor([reps], dtype=torch.int64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        reps = int(t[0])

    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    torch.cuda.nvtx.range_push("timed region")
    with Clocks(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter()
        with torch.cuda.stream(stream):
            evs[0].record(stream)
            for r in range(reps):
                graph.replay()
                evs[r + 1].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
        if world > 1:
            dist.barrier()
    torch.cuda.nvtx.range_pop()
    dev_ms_total = evs[0].elapsed_time(evs[-1])
    per_step = sorted(evs[r].elapsed_time(evs[r + 1]) / G for r in range(reps))
    med = statistics.median(per_step)
    spread = {"median": round(med, 6), "p10": round(quantile(per_step, 0.1), 6),
              "p90": round(quantile(per_step, 0.9), 6), "mean": round(dev_ms_total / (reps * G), 6),
              "over": f"{reps} replays of a {G}-step graph"}
    rc, detail = attn.device_status(stream)
    if rc != attn.ATTN_OK:
        raise RuntimeError(f"device status {rc} ({detail}) after the timed region")

    # end to end through the C entry point with pinned host buffers: every input of
    # the pass host -> device, the pass, every output device -> host. Steps alternate
    # between two streams, each with its own device buffers (and workspace), so one
    # step's copies overlap the next step's copies and pass, as a caller streaming
    # batches through the library would run them.
    n_in = 1 if proj else (6 if bwd else 3)  # X or O; Q, K, V (+ O, LSE, dO for the backward)
    host_in = [t.cpu().pin_memory() for t in sets[0][:n_in]]
    hlens = x.key_lengths.pin_memory() if x.key_lengths is not None else None
    lanes = []
    for k in range(2):
        dev_set = sets[k % copies]
        lanes.append({
            "stream": stream if k == 0 else torch.cuda.Stream(device=dev),
            "set": dev_set,
            "host_out": [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_set[n_in:]],
            "lens": torch.empty_like(lens_d) if lens_d is not None else None,
            "ws": ws if k == 0 or ws is None else torch.empty_like(ws),
        })
    e2e_steps = max(4, args.e2e_steps)

    def e2e_step(i):
        ln = lanes[i % 2]
        with torch.cuda.stream(ln["stream"]):
            for h, d in zip(host_in, ln["set"][:n_in]):
                d.copy_(h, non_blocking=True)
            if ln["lens"] is not None:
                ln["lens"].copy_(hlens, non_blocking=True)
            run(ln["set"], ln["lens"], on=ln["stream"], wsp=ln["ws"])
            for h, d in zip(ln["host_out"], ln["set"][n_in:]):
                h.copy_(d, non_blocking=True)

    torch.cuda.nvtx.range_push("end to end")
    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    joined = torch.cuda.Event()
    e0.record(stream)
    lanes[1]["stream"].wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    joined.record(lanes[1]["stream"])
    stream.wait_event(joined)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    torch.cuda.nvtx.range_pop()
    h2d = sum(t.numel() * t.element_size() for t in host_in) + (hlens.numel() * 4 if hlens is not None else 0)
    d2h = sum(t.numel() * t.element_size() for t in lanes[0]["host_out"])

    ms, e2e_ms = reduce_over_ranks(med, e2e_ms, world)
    value = job_value(flops, world, ms)
    e2e_value = job_value(flops, world, e2e_ms)
    peak, peak_sus, hbm, src = peaks()
    kernel_tflops = flops / (ms * 1e-3) / 1e12
    alg_bytes = w.decode_bytes(x.key_lengths) if decode else in_bytes + out_bytes
    hbm_gbs = alg_bytes / (ms * 1e-3) / 1e9
    if kernel_tflops > 1.25 * peak or hbm_gbs > 1.25 * hbm or dev_ms_total < 0.5 * t_wall * 1e3:
        raise RuntimeError(f"implausible timing: {kernel_tflops:.1f} TFLOP/s, device {dev_ms_total:.2f} ms "
                           f"vs wall {t_wall * 1e3:.2f} ms")

    # the committed traffic figure belongs to the forward tensor-core kernel
    traffic = args.traffic if args.traffic is not None else (
        None if (bwd or decode or proj) else measured_traffic(w.name))
    if decode:
        roofline = {"bound": "hbm", "achieved": round(hbm_gbs, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(hbm_gbs / hbm, 4), "traffic": traffic,
                    "traffic_unit": "bytes per launch (ncu dram read+write)",
                    "peak_source": f"{src} HBM copy",
                    "algorithmic_bytes": alg_bytes}
    else:
        # The binding roof is the resource whose lower bound on the time is larger:
        # FLOPs / tensor peak against algorithmic bytes / HBM bandwidth (the ridge
        # is peak / bandwidth flop/B; below it the pass is memory-bound).
        t_tensor = flops / (peak * 1e12)
        t_hbm = alg_bytes / (hbm * 1e9)
        if t_hbm > t_tensor:
            roofline = {"bound": "hbm", "achieved": round(hbm_gbs, 1), "peak": hbm, "unit": "GB/s",
                        "frac": round(hbm_gbs / hbm, 4), "traffic": traffic,
                        "traffic_unit": "bytes per launch (ncu dram read+write)",
                        "peak_source": f"{src} HBM copy", "algorithmic_bytes": alg_bytes,
                        "arithmetic_intensity": round(flops / alg_bytes, 1),
                        "ridge": round(peak * 1e12 / (hbm * 1e9), 1),
                        "tensor_tflops_achieved": round(kernel_tflops, 2),
                        "tensor_frac": round(kernel_tflops / peak, 4)}
        else:
            roofline = {"bound": "tensor", "achieved": round(kernel_tflops, 2),
                        "peak": peak, "unit": "TFLOP/s", "frac": round(kernel_tflops / peak, 4),
                        "traffic": traffic,
                        "traffic_unit": "bytes per launch (ncu dram read+write)",
                        "peak_source": f"{src} bf16 burst", "algorithmic_bytes": alg_bytes,
                        "arithmetic_intensity": round(flops / alg_bytes, 1),
                        "ridge": round(peak * 1e12 / (hbm * 1e9), 1),
                        "hbm_gbs_achieved": round(hbm_gbs, 1), "hbm_frac": round(hbm_gbs / hbm, 4)}

    result = None
    if rank == 0:
        cpu = check = None
        if world == 1 and not args.no_cpu_baseline and not bwd and not proj:
            O_gpu = sets[0][3].float().cpu()
            L_gpu = sets[0][4].cpu()
            cpu, check = cpu_baseline(w, x, args.cpu_seconds, O_gpu, L_gpu)
        clocks = clk.summary()
        result = {
            "metric": METRIC_BWD if bwd else (METRIC_PROJ[args.pass_] if proj else METRIC),
            "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": G, "warmup": args.warmup, "ms_per_step": round(ms, 6),
            "ms_per_step_spread": spread,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; bias-free Xavier projections of X~N(0,1))",
            "config": {"workload": w.name, "pass": args.pass_ if (bwd or proj) else ("decode" if decode else "fwd"),
                       "B": w.B, "H": w.H, "n": w.n, "m": w.m,
                       "d_k": w.d_k, "d_v": w.d_v, "mask": w.mask,
                       "distance_bias": "alibi slopes 2^(-8h/H)" if w.alibi else None,
                       "key_lengths": [w.len_lo, w.len_hi] if w.mask in inputs.LENGTH_MASKS else None,
                       "global_batch": w.B * world, "parallelism": f"replicas{world}",
                       "l2": f"rotating {copies} input/output sets "
                             f"({copies * (in_bytes + out_bytes) / 2**20:.0f} MiB > 2x L2)",
                       "timing": f"median over {reps} replays of a CUDA graph of exactly {G} steps, "
                                 f"events around every replay ({dev_ms_total:.1f} ms timed)"},
            "pct_of_peak": round(100.0 * value / world / peak, 2),
            "effective_tflops": round(world * eff_flops / (ms * 1e-3) / 1e12, 2),
            "roofline": roofline,
            "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                    "pipelining": "steps alternate over two streams with their own buffers"},
            "gpu_launches": reps * G * launches_per_step,
            "clocks": clocks,
            "wall_s_timed": round(t_wall, 3),
        }
        if cpu is not None:
            result["cpu_baseline"] = cpu
            result["oracle_check"] = check
    if world > 1:
        dist.destroy_process_group()
    return result


def effective_flops(w, x):
    """FLOPs of the (query, key) pairs the masks leave visible, counted exactly with
    the drawn key lengths: 2*(d_k + d_v) per pair."""
    i = torch.arange(w.n, dtype=torch.float64)
    if w.mask == inputs.MASK_CAUSAL_CACHE:
        # keys j < len_b with j <= i + len_b - n
        lens = x.key_lengths.to(torch.float64).clamp(0, w.m)
        pairs = float((i[None, :] + lens[:, None] - w.n + 1).clamp(min=0).minimum(lens[:, None]).sum()) * w.H
        return 2.0 * (w.d_k + w.d_v) * pairs
    if w.mask in (inputs.MASK_CAUSAL, inputs.MASK_CAUSAL_KEY_PADDING):
        per_row_cap = (i + (w.m - w.n) + 1).clamp(0, w.m)      # keys j <= i + m - n
    else:
        per_row_cap = torch.full((w.n,), float(w.m), dtype=torch.float64)
    if x.key_lengths is not None:
        lens = x.key_lengths.to(torch.float64).clamp(0, w.m)
        pairs = float(torch.minimum(per_row_cap[None, :], lens[:, None]).sum()) * w.H
    else:
        pairs = float(per_row_cap.sum()) * w.B * w.H
    return 2.0 * (w.d_k + w.d_v) * pairs


def oracle_rows_for(w, x, seconds, threads, seed):
    """The oracle's rows for a run of about `seconds`: every row when the whole
    workload fits, else a seeded sample. Two calibration runs (k and 2k rows)
    separate the per-row cost from the fixed cost of a call (widening the inputs
    to fp64). Returns the rows, or None for all of them."""
    from oracle import oracle
    total_rows = w.B * w.H * w.n
    k = min(total_rows, 16 * threads)
    times = []
    for count in (k, min(total_rows, 2 * k)):
        probe = inputs.sample_rows(w.B, w.H, w.n, count, seed=seed)
        t0 = time.perf_counter()
        oracle.attn_rows(x.Q, x.K, x.V, probe, w.mask, x.key_lengths, x.scale, slopes=workload_slopes(w),
                         threads=threads)
        times.append(time.perf_counter() - t0)
    per_row = max(times[1] - times[0], 1e-3 * times[0]) / max(k, 1)
    fixed = max(times[0] - k * per_row, 0.0)
    if fixed + per_row * total_rows <= seconds:
        return None
    count = int(max(seconds - fixed, 0.0) / per_row)
    return inputs.sample_rows(w.B, w.H, w.n, max(threads, min(count, total_rows)), seed=seed + 1)


def cpu_baseline(w, x, seconds, O_gpu, L_gpu):
    """The fp64 oracle as it stands, on all host cores, over the whole workload (or a
    seeded row sample when the whole would take longer than `seconds`); scaled to
    TFLOP/s of the nominal FLOP model. Its outputs also give the error of the GPU's
    timed outputs O_gpu, L_gpu (one rotating copy; every copy holds the same result)."""
    import numpy as np
    from oracle import oracle

    threads = oracle.default_threads()
    total_rows = w.B * w.H * w.n
    flops_per_row = w.flops() / total_rows
    rows = oracle_rows_for(w, x, seconds, threads, seed=11)
    t0 = time.perf_counter()
    if rows is None:
        Or, Lr = oracle.attn_fwd(x.Q, x.K, x.V, w.mask, x.key_lengths, x.scale, slopes=workload_slopes(w),
                                 threads=threads)
        Or, Lr = Or.reshape(-1, w.d_v), Lr.reshape(-1)
        count = total_rows
    else:
        Or, Lr = oracle.attn_rows(x.Q, x.K, x.V, rows, w.mask, x.key_lengths, x.scale, slopes=workload_slopes(w),
                                  threads=threads)
        count = rows.numel()
    dt = time.perf_counter() - t0
    O = O_gpu.reshape(-1, w.d_v).double().numpy()
    L = L_gpu.reshape(-1).double().numpy()
    if rows is not None:
        O, L = O[rows.numpy()], L[rows.numpy()]
    err = np.abs(O - Or)
    live = ~np.isneginf(Lr)
    sample = f"all {total_rows} query rows" if rows is None else f"{count} of {total_rows} query rows (seeded)"
    cpu = {"value": round(flops_per_row * count / dt / 1e12, 6), "unit": UNIT, "cores": threads,
           "kind": "oracle", "seconds": round(dt, 2), "sample": f"{sample} of {w.name}, fp64"}
    check = {"rows": sample, "o_max_abs": float(err.max()), "o_mean_abs": float(err.mean()),
             "lse_max_abs": float(np.abs(L[live] - Lr[live]).max()) if live.any() else 0.0,
             "lse_empty_rows_match": bool(np.array_equal(np.isneginf(L), ~live)),
             "tolerance": {"o_max_abs": 1e-2, "o_mean_abs": 1e-3, "lse_max_abs": 1e-3}}
    return cpu, check


def run_reference(args):
    """The oracle as it stands on the host cores, timed step by step: a step is the
    whole workload when it fits the time budget (--cpu-seconds over all steps), else
    the same seeded row sample every step; value = nominal FLOPs of the rows run /
    measured time, ms_per_step the measured time of one step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    w, x = make_workload(args.workload)
    from oracle import oracle
    oracle.build()
    threads = oracle.default_threads()
    total_rows = w.B * w.H * w.n
    flops_per_row = w.flops() / total_rows
    rows = oracle_rows_for(w, x, args.cpu_seconds / (args.steps + args.warmup), threads, seed=21)
    secs = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        if rows is None:
            oracle.attn_fwd(x.Q, x.K, x.V, w.mask, x.key_lengths, x.scale, slopes=workload_slopes(w),
                            threads=threads)
        else:
            oracle.attn_rows(x.Q, x.K, x.V, rows, w.mask, x.key_lengths, x.scale, slopes=workload_slopes(w),
                             threads=threads)
        if i >= args.warmup:
            secs.append(time.perf_counter() - t0)
    nrows = total_rows if rows is None else rows.numel()
    ms = statistics.median(secs) * 1e3
    v = flops_per_row * nrows / (ms * 1e-3) / 1e12
    sample = (f"all {total_rows} query rows of {w.name} per step, fp64" if rows is None else
              f"{nrows} of {total_rows} query rows of {w.name} per step (seeded, the same each step), fp64")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "ms_per_step_spread": {"median": round(ms, 3), "p10": round(quantile(sorted(secs), 0.1) * 1e3, 3),
                                   "p90": round(quantile(sorted(secs), 0.9) * 1e3, 3)},
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "n": w.n, "m": w.m, "d_k": w.d_k,
                       "d_v": w.d_v, "mask": w.mask, "parallelism": "host cores"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(sum(secs), 2)}


def run_launches(args):
    """Untimed launches of the pass on the workload's inputs, for a profiler to
    capture (no timing, no JSON line)."""
    from transformer_scaled_dot_03_gb300 import attn, build
    build.build()
    attn.load()
    w, x = make_workload(args.workload)
    dev = torch.device("cuda", 0)
    Q, K, V = x.Q.to(dev), x.K.to(dev), x.V.to(dev)
    lens = x.key_lengths.to(dev) if x.key_lengths is not None else None
    slopes = workload_slopes(w).to(dev) if w.alibi else None
    if args.pass_ == "bwd":
        # the forward once for O and LSE, then the backward launches
        if slopes is not None:
            O, L = attn.attn_fwd_alibi(Q, K, V, slopes, w.mask, lens, x.scale)
        else:
            O, L = attn.attn_fwd(Q, K, V, w.mask, lens, x.scale)
        dO = inputs.make_grad_output(w.B, w.H, w.n, w.d_v, seed=100 + w.seed).to(dev)
        for _ in range(args.launches):
            attn.attn_bwd(Q, K, V, O, L, dO, w.mask, lens, x.scale, slopes=slopes)
    for _ in range(args.launches if args.pass_ != "bwd" else 0):
        if w.path == "decode":
            attn.attn_decode(Q, K, V, w.mask, lens, x.scale)
        elif slopes is not None:
            attn.attn_fwd_alibi(Q, K, V, slopes, w.mask, lens, x.scale)
        else:
            attn.attn_fwd(Q, K, V, w.mask, lens, x.scale)
    rc, detail = attn.device_status()
    if rc != attn.ATTN_OK:
        raise RuntimeError(f"device status {rc} ({detail})")
    print(f"{args.launches} launches of {w.name}: ok", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100,
                    help="steps in the timed CUDA graph (replayed until >= 10 replays and >= 200 ms)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=inputs.WORKLOAD_ORDER + inputs.VARIANT_ORDER + inputs.DECODE_ORDER
                    + inputs.ALIBI_ORDER)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd", "proj", "outproj"], default="fwd",
                    help="fwd: the forward (the headline); bwd: the backward of the same workload; "
                         "proj / outproj: the projections around it (weights resident)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--launches", type=int, default=0,
                    help="only run this many untimed launches of the pass (fwd, or bwd after one forward) "
                         "on the workload (for profilers)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch from an ncu capture of the current kernel")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if not 1 <= args.steps <= MAX_GRAPH_STEPS:
        ap.error(f"--steps must be in [1, {MAX_GRAPH_STEPS}]")
    if args.launches > 0:
        run_launches(args)
        return
    res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
