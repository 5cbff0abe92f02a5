"""Benchmark of the fused MoE FFN layer on one GB300 (or N replicas).

Headline workload (the JSON line's ``value``): the decode bf16 MoE layer, T=1
token, H=2048, E=128, top_k=8, I=768, Is=512.  One step = one layer call on
one token batch.  Step s runs on layer copy s mod 16 (16 copies at distinct
addresses, 16 x 1.21 GB, far larger than the 129 MB L2) and token s mod 100
(100 distinct seeded tokens), so every step streams its weights from HBM.
Steps are captured in CUDA graphs and replayed; CUDA events on the launching
stream time them, after warm-up and a pre-roll that keeps the GPU busy while
the clocks are sampled.

At N=1 the same run also measures every other workload and reports each one
under ``configs``: decode bf16 T=8, decode 4-bit T=1/2/4/8, batched bf16 and
batched 4-bit T=64/256 (the grouped-GEMM path) and the 48-layer 4-bit decode
stack (pre-norm RMSNorm + residual per layer, each token's output feeding the
next token), each with its own roofline and oracle CPU baseline.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead (the reference arm).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W]
       [--config decode_bf16|decode_q4|decode_i8|batched_bf16|batched_q4|stack_q4] [--T T] [--no-extras] [--no-cpu-baseline]
"""

from __future__ import annotations

import argparse
import json
import math
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

import datagen  # noqa: E402

METRIC = "MoE-layer tokens/s & µs/layer at 1 GB300; % of HBM roofline (decode)"
UNIT = "tokens/s"
H, E, K_TOP, I, IS = 2048, 128, 8, 768, 512
N_LAYER_COPIES = 16
N_TOKENS = 100
SEED = 20261202
STACK_LAYERS = 48
PREROLL_S = 0.15  # GPU work enqueued right before each timed region (clock samples under load, full launch queue)
# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the dominant kernel from the committed ncu
# captures (profiles/), per (config, T); None until captured for the current kernel.
NCU_TRAFFIC_BYTES = {("batched_q4", 256): 238_398_464}
# Extra workloads measured in the default N=1 run: (config, T, steps, warm-up steps, oracle budget in s)
EXTRAS = [("decode_bf16", 8, 400, 20, 3.0), ("two_stream_bf16", 1, 400, 20, 0.0), ("two_stream_bf16", 8, 400, 20, 0.0),
          ("decode_q4", 1, 400, 20, 3.0), ("decode_q4", 2, 400, 20, 3.0),
          ("decode_q4", 4, 400, 20, 3.0), ("decode_q4", 8, 400, 20, 3.0), ("decode_i8", 1, 400, 20, 3.0),
          ("decode_i8", 2, 400, 20, 3.0), ("decode_i8", 4, 400, 20, 3.0), ("decode_i8", 8, 400, 20, 3.0),
          ("batched_bf16", 64, 64, 5, 3.0),
          ("batched_bf16", 256, 64, 5, 4.0), ("batched_q4", 64, 64, 5, 3.0), ("batched_q4", 256, 64, 5, 4.0),
          ("stack_q4", 1, 32, 3, 6.0)]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def init_ranks():
    """(dist or None, world, rank, local rank): one process per GPU under torchrun (NCCL), else one process."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    return dist, world, rank, local


def whole_job(ms_local: float, units_per_rank: int, world: int, dist=None, device="cpu"):
    """The job's timed-region duration (the slowest rank's, ms) and its throughput: every rank processed
    units_per_rank units (replicas, weak scaling), so the whole job did units_per_rank * world of them."""
    ms = ms_local
    if dist is not None:
        import torch

        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, units_per_rank * world / (ms / 1000.0)


def wfmt_of(cfg: str) -> int:
    if cfg == "decode_i8":
        return datagen.WFMT_I8
    return datagen.WFMT_Q4B32 if cfg in ("decode_q4", "batched_q4", "stack_q4") else datagen.WFMT_BF16


def dtype_of(wfmt: int) -> str:
    return {datagen.WFMT_BF16: "bf16", datagen.WFMT_Q4B32: "q4b32 weights, fp32 accumulate",
            datagen.WFMT_I8: "int8 weights and per-token int8 activation, int32 dot, fp32 epilogue"}[wfmt]


def workload(cfg: str, T: int):
    wfmt = wfmt_of(cfg)
    shapes = datagen.Shapes(T=T, H=H, E=E, top_k=K_TOP, I=I, Is=IS)
    name = {
        "decode_bf16": f"decode bf16 MoE FFN layer: T={T}, H={H}, E={E}, top_k={K_TOP}, I={I}, Is={IS}",
        "two_stream_bf16": f"decode bf16 MoE FFN layer as two branches on two CUDA streams (routed on the main stream, "
                           f"gated shared expert on a forked stream, event join, join add): T={T}, H={H}, E={E}, "
                           f"top_k={K_TOP}, I={I}, Is={IS}",
        "decode_q4": f"decode 4-bit MoE FFN layer (blocks of 32, fp16 scale): T={T}, H={H}, E={E}, top_k={K_TOP}, I={I}, Is={IS}",
        "decode_i8": f"decode int8 MoE FFN layer (int8 rows + fp32 row scale, int8 activation per token): T={T}, H={H}, "
                     f"E={E}, top_k={K_TOP}, I={I}, Is={IS}",
        "batched_bf16": f"batched bf16 MoE FFN layer (grouped GEMMs): T={T}, H={H}, E={E}, top_k={K_TOP}, I={I}, Is={IS}",
        "batched_q4": f"batched 4-bit MoE FFN layer (grouped GEMMs, fp16 operands): T={T}, H={H}, E={E}, top_k={K_TOP}, "
                      f"I={I}, Is={IS}",
        "stack_q4": f"{STACK_LAYERS}-layer 4-bit decode stack (pre-norm RMSNorm + residual per layer, independent seeded "
                    f"layers), T=1, sequential tokens; layer H={H}, E={E}, top_k={K_TOP}, I={I}, Is={IS}",
    }[cfg]
    return shapes, wfmt, name


def algorithmic_bytes(shapes, wfmt, U: float) -> float:
    """router + shared-gate vector + U unique experts + shared expert + x + out."""
    eb = datagen.expert_bytes(wfmt, shapes.H, shapes.I)
    sb = datagen.expert_bytes(wfmt, shapes.H, shapes.Is)
    return (shapes.E * shapes.H * 2 + shapes.H * 2 + U * eb + sb + shapes.T * shapes.H * 2 + shapes.T * shapes.H * 4)


def token_batch(step_token: int, T: int) -> np.ndarray:
    return np.stack([datagen.token_x(SEED, step_token * T + t, H, datagen.ACT_BF16) for t in range(T)])


def kernel_names(cfg: str, T: int) -> str:
    if cfg == "stack_q4":
        return "k_rows per layer, block form; duration = step time / layers"
    if cfg == "two_stream_bf16":
        return "k_rows routed part (main stream) + k_rows shared part (aux stream) + join add; duration = step time"
    if T > 8:
        return (("k_gemm_q4<0>, k_gemm_q4<1>" if cfg == "batched_q4" else "k_gemm<0>, k_gemm<1>")
                + " (+ routing, gather, combine); duration = step time")
    return "k_rows (one kernel per layer call, programmatic dependent launch); duration = step time"


def roofline(bytes_per_step: float, ms_per_step: float, cfg: str, T: int):
    peak, peak_kind = peaks()
    achieved = bytes_per_step / (ms_per_step / 1000.0) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "peak_kind": peak_kind, "traffic": NCU_TRAFFIC_BYTES.get((cfg, T)),
            "algorithmic_bytes_per_step": bytes_per_step, "kernel": kernel_names(cfg, T)}


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons, power = [], 0.0, set(), []
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower() in ("active", "0x1") or v == "1":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------- oracle (CPU baseline, reference arm)


def oracle_rate(shapes, wfmt, budget_s: float, max_calls: int, layer=None):
    """The oracle as it stands on the host cores: layer calls of T tokens until the budget is spent.
    Returns (tokens/s, calls, seconds, threads used, cores offered)."""
    import oracle

    if layer is None:
        layer = datagen.make_layer(SEED, datagen.Shapes(1, H, E, K_TOP, I, IS), wfmt)
    threads = oracle.nthreads()
    done = 0
    t0 = time.perf_counter()
    while done < max_calls:
        x = token_batch(done % N_TOKENS, shapes.T)
        oracle.moe_ffn(shapes, datagen.ACT_BF16, wfmt, x, layer.router_w, layer.expert_w, layer.shexp_w,
                       layer.shexp_gate_w, threads=threads)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done * shapes.T / dt, done, dt, oracle.threads_used(shapes, threads), threads


def oracle_stack_rate(layers, budget_s: float, max_tokens: int):
    """Tokens/s of the oracle through all stack layers (block form), sequential tokens from the seeded x0."""
    import oracle

    s1 = datagen.Shapes(1, H, E, K_TOP, I, IS)
    threads = oracle.nthreads()
    x = datagen.normal_f32(SEED, 7, H, 1.0).reshape(1, H)
    done = 0
    t0 = time.perf_counter()
    while done < max_tokens:
        for lay in layers:
            x, _, _ = oracle.block_step(s1, datagen.WFMT_Q4B32, x, lay.router_w, lay.expert_w, lay.shexp_w,
                                        lay.shexp_gate_w, threads=threads)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done / dt, done, dt, oracle.threads_used(s1, threads), threads


def cpu_entry(rate, n, dt, used, offered, what):
    return {"value": rate, "unit": UNIT, "cores": used, "cores_available": offered, "kind": "oracle",
            "sample": f"{what} ({dt:.1f} s; oracle threads: {used} of the {offered} host cores offered by "
                      f"sched_getaffinity)"}


def stack_layers_host(wfmt=datagen.WFMT_Q4B32):
    from concurrent.futures import ThreadPoolExecutor

    s1 = datagen.Shapes(1, H, E, K_TOP, I, IS)
    with ThreadPoolExecutor(max_workers=3) as pool:
        return list(pool.map(lambda l: datagen.make_layer(SEED + 1000 + l, s1, wfmt), range(STACK_LAYERS)))


def run_reference(args, shapes, wfmt, name):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    budget = 60.0
    if args.config == "stack_q4":
        layers = stack_layers_host()
        oracle_stack_rate(layers, 0.0, 1)  # warm-up: one token
        rate, n, dt, used, offered = oracle_stack_rate(layers, budget, args.steps)
        what = f"{n} tokens through {STACK_LAYERS} layers (of {args.steps} requested; bounded to ~{budget:.0f} s)"
    else:
        layer = datagen.make_layer(SEED, datagen.Shapes(1, H, E, K_TOP, I, IS), wfmt)
        oracle_rate(shapes, wfmt, 0.0, 1, layer)  # warm-up: one call
        rate, n, dt, used, offered = oracle_rate(shapes, wfmt, budget, args.steps, layer)
        what = f"{n} layer calls of T={shapes.T} (of {args.steps} requested; bounded to ~{budget:.0f} s)"
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus, "steps": n,
        "warmup": args.warmup, "ms_per_step": dt / n * 1000.0, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "parallelism": "replicas only"},
        "cpu_baseline": cpu_entry(rate, n, dt, used, offered, what),
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU timing


class Resident:
    """N_LAYER_COPIES copies of one seeded layer on the device at distinct addresses, and the host layer."""

    def __init__(self, wfmt: int, dev, n_copies: int):
        import torch

        self.wfmt = wfmt
        self.host = datagen.make_layer(SEED, datagen.Shapes(1, H, E, K_TOP, I, IS), wfmt)
        lay = self.host
        router = torch.from_numpy(lay.router_w.view(np.int16)).to(dev)
        gvec = torch.from_numpy(lay.shexp_gate_w.view(np.int16)).to(dev)
        ew0 = torch.from_numpy(lay.expert_w).to(dev)
        sw0 = torch.from_numpy(lay.shexp_w).to(dev)
        self.copies = [(router.clone(), ew0.clone(), sw0.clone(), gvec.clone()) for _ in range(n_copies)]
        del ew0, sw0


def timed_replays(stream, graphs_and_reps, clocks, est_ms_per_replay):
    """Pre-roll (about PREROLL_S of the first graph, clocks sampled), then the timed replays between two
    events on the launching stream.  Returns the timed milliseconds and the clock record."""
    import torch

    g0 = graphs_and_reps[0][0]
    n_pre = max(1, int(math.ceil(PREROLL_S * 1000.0 / max(est_ms_per_replay, 1e-3))))
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
        time.sleep(0.1)
    with torch.cuda.stream(stream):
        for _ in range(n_pre):
            g0.replay()
        ev0.record(stream)
        for g, reps in graphs_and_reps:
            for _ in range(reps):
                g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks is not None else None
    return ev0.elapsed_time(ev1), clk


def time_layer(fb, res: Resident, cfg: str, T: int, steps: int, warmup: int, stream, dev, clocks=None,
               dist=None, world=1):
    """Steps of one layer call each (copy s mod n, token s mod N_TOKENS) in CUDA graphs.  Returns a dict."""
    import torch

    shapes, wfmt, name = workload(cfg, T)
    n_copies = len(res.copies)
    xs_host = np.stack([token_batch(t, T) for t in range(N_TOKENS)])  # [N_TOKENS, T, H] bf16 bits
    xs = torch.from_numpy(xs_host.view(np.int16)).to(dev)
    plan, ws_bytes = fb.moe_ffn_prepare(shapes, fb.ACT_BF16, wfmt)
    launches_per_step = fb.moe_ffn_query(plan, fb.QUERY_LAUNCHES_PER_EXECUTE)
    two = cfg == "two_stream_bf16"
    if two:
        launches_per_step = 3  # routed part, shared part, join add
        ws_two = torch.empty(fb.moe_ffn_query(plan, fb.QUERY_TWO_STREAM_WORKSPACE), dtype=torch.uint8, device=dev)
        aux = torch.cuda.Stream(device=dev)
        ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H), dtype=torch.float32, device=dev)

    def run_step(x, r, ew, sw, gv):
        if two:
            fb.moe_ffn_execute_two_stream(plan, ws_two, x, r, ew, sw, gv, out, aux_stream=aux, fork_event=ev_fork,
                                          join_event=ev_join, stream=stream)
        else:
            fb.moe_ffn_execute(plan, ws, x, r, ew, sw, gv, out, stream=stream)

    def step_args(s):
        r, ew, sw, gv = res.copies[s % n_copies]
        return xs[s % N_TOKENS], r, ew, sw, gv

    # unique experts of every token batch (for the byte count)
    ids = torch.empty((T, K_TOP), dtype=torch.int32, device=dev)
    uniq = []
    with torch.cuda.stream(stream):
        for t in range(N_TOKENS):
            x, r, ew, sw, gv = step_args(t)
            fb.moe_ffn_execute_ex(plan, ws, x, r, ew, sw, gv, out, ids, None, stream=stream)
            uniq.append(len(np.unique(ids.cpu().numpy())))
    torch.cuda.synchronize()
    if fb.moe_ffn_read_status(plan, ws, stream) != 0:
        raise RuntimeError(f"{cfg} T={T}: device status after the routing pass")
    U_mean = float(np.mean(uniq))
    bytes_per_step = algorithmic_bytes(shapes, wfmt, U_mean)

    graph_steps = min(steps, 400)  # 400 = lcm(16 copies, 100 tokens): every (copy, token) pair once

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in range(n):
                run_step(*step_args(s))
        return g

    with torch.cuda.stream(stream):
        for s in range(max(3, warmup)):
            run_step(*step_args(s))
    torch.cuda.synchronize()
    g_main = capture(graph_steps)
    reps, rem = divmod(steps, graph_steps)
    g_rem = capture(rem) if rem else None
    # one untimed replay, also the estimate for the pre-roll
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g_main.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    est = e0.elapsed_time(e1)
    if dist is not None:
        dist.barrier()
    plan_graphs = [(g_main, reps)] + ([(g_rem, 1)] if g_rem is not None else [])
    ms_local, clk = timed_replays(stream, plan_graphs, clocks, est)
    if dist is not None:
        dist.barrier()
    ms, value = whole_job(ms_local, steps * T, world, dist, dev)
    if fb.moe_ffn_read_status(plan, ws, stream) != 0:
        raise RuntimeError(f"{cfg} T={T}: device status after the timed region")
    ms_per_step = ms / steps
    result = {"workload": name, "config": cfg, "T": T, "steps": steps, "warmup": max(3, warmup),
              "ms_per_step": ms_per_step, "us_per_layer": ms_per_step * 1000.0, "tokens_per_s": value,
              "unique_experts_per_step": U_mean, "roofline": roofline(bytes_per_step, ms_per_step, cfg, T),
              "gpu_launches": steps * launches_per_step, "clocks": clk,
              "_plan": plan, "_ws": ws, "_xs_host": xs_host, "_out": out}
    return result


def e2e_layer(fb, res: Resident, r: dict, stream, dev, world: int, n_steps: int):
    """The same layer end to end through the public API, as a server streams independent token batches: every
    step copies its x from pinned host memory to the device, executes, and copies out back to pinned host
    memory.  The copies run on their own streams, double-buffered, so step s + 1's input copy and step s - 1's
    output copy overlap step s's layer; the whole sequence is captured in a CUDA graph and replayed once inside
    the timed region (the host launches nothing per step)."""
    import torch

    T = r["T"]
    plan, ws, xs_host = r["_plan"], r["_ws"], r["_xs_host"]
    n_copies = len(res.copies)
    x_pin = torch.from_numpy(xs_host.view(np.int16)).pin_memory()
    out_pin = torch.empty((n_steps, T, H), dtype=torch.float32).pin_memory()
    x_dev = [torch.empty((T, H), dtype=torch.int16, device=dev) for _ in range(2)]
    out_dev = [torch.empty((T, H), dtype=torch.float32, device=dev) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def steps():
        ev_k = [None, None]  # the layer of step s - 2 (buffer s % 2) has read x_dev and written out_dev
        ev_d = [None, None]  # out_dev of step s - 2 has been copied out
        h2d.wait_stream(stream)  # fork the copy streams from the layer's stream
        d2h.wait_stream(stream)
        for s in range(n_steps):
            b = s & 1
            rw, ew, sw, gv = res.copies[s % n_copies]
            with torch.cuda.stream(h2d):
                if ev_k[b] is not None:
                    h2d.wait_event(ev_k[b])
                x_dev[b].copy_(x_pin[s % N_TOKENS], non_blocking=True)
                ev_x = torch.cuda.Event()
                ev_x.record(h2d)
            stream.wait_event(ev_x)
            if ev_d[b] is not None:
                stream.wait_event(ev_d[b])
            fb.moe_ffn_execute(plan, ws, x_dev[b], rw, ew, sw, gv, out_dev[b], stream=stream)
            ev_k[b] = torch.cuda.Event()
            ev_k[b].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_k[b])
                out_pin[s].copy_(out_dev[b], non_blocking=True)
                ev_d[b] = torch.cuda.Event()
                ev_d[b].record(d2h)
        # join the side streams back
        stream.wait_stream(h2d)
        stream.wait_stream(d2h)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        steps()  # eager warm-up pass (same calls)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        steps()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    # the last step's output arrived in host memory
    assert np.isfinite(out_pin[n_steps - 1].numpy()).all()
    return {"value": n_steps * T * world / (e0.elapsed_time(e1) / 1000.0), "unit": UNIT,
            "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 4, "steps": n_steps,
            "how": "public-API calls captured in one CUDA graph: per step a pinned H2D of x, execute, a D2H of out "
                   "into pinned memory; copies on their own streams, double-buffered"}


def time_stack(fb, layers_host, steps: int, warmup: int, stream, dev, clocks=None, dist=None, world=1):
    """One step = one token through STACK_LAYERS layers in block form (x_res updated in place); the timed steps
    are consecutive tokens, each starting from the previous token's output."""
    import torch

    _, wfmt, name = workload("stack_q4", 1)
    s1 = datagen.Shapes(1, H, E, K_TOP, I, IS)
    layers = [(torch.from_numpy(l.router_w.view(np.int16)).to(dev), torch.from_numpy(l.expert_w).to(dev),
               torch.from_numpy(l.shexp_w).to(dev), torch.from_numpy(l.shexp_gate_w.view(np.int16)).to(dev))
              for l in layers_host]
    plan, ws_bytes = fb.moe_ffn_prepare(s1, fb.ACT_BF16, wfmt)
    launches = fb.moe_ffn_query(plan, fb.QUERY_LAUNCHES_PER_EXECUTE) * STACK_LAYERS
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    x0 = torch.from_numpy(datagen.normal_f32(SEED, 7, H, 1.0).reshape(1, H)).to(dev)
    x_res = x0.clone()

    def token_pass():
        for r, ew, sw, gv in layers:
            fb.moe_ffn_execute_block(plan, ws, x_res, r, ew, sw, gv, eps=1e-6, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            token_pass()
    torch.cuda.synchronize()
    if fb.moe_ffn_read_status(plan, ws, stream) != 0:
        raise RuntimeError("stack: device status after warm-up")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        token_pass()
    x_res.copy_(x0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    est = e0.elapsed_time(e1)
    if dist is not None:
        dist.barrier()
    ms_local, clk = timed_replays(stream, [(g, steps)], clocks, est)
    if dist is not None:
        dist.barrier()
    ms, value = whole_job(ms_local, steps, world, dist, dev)
    if fb.moe_ffn_read_status(plan, ws, stream) != 0:
        raise RuntimeError("stack: device status after the timed region")
    final = x_res.cpu().numpy()
    if not np.all(np.isfinite(final)):
        raise RuntimeError("stack: non-finite output")
    ms_per_step = ms / steps
    bytes_per_step = STACK_LAYERS * algorithmic_bytes(s1, wfmt, float(K_TOP))
    # end to end: each token's input from pinned host memory, its output back
    e2e_steps = min(steps, 64)
    x_pin = torch.from_numpy(final.copy()).pin_memory()
    out_pin = torch.empty((e2e_steps, 1, H), dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(e2e_steps):
            x_res.copy_(x_pin if i == 0 else out_pin[i - 1], non_blocking=True)
            token_pass()
            out_pin[i].copy_(x_res, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e = {"value": e2e_steps * world / (e0.elapsed_time(e1) / 1000.0), "unit": UNIT, "h2d_bytes_per_step": H * 4,
           "d2h_bytes_per_step": H * 4, "steps": e2e_steps,
           "how": f"eager public-API calls per token: pinned H2D of x, {STACK_LAYERS} layers, D2H"}
    fb.moe_ffn_destroy(plan)
    del layers
    return {"workload": name, "config": "stack_q4", "T": 1, "layers": STACK_LAYERS, "steps": steps,
            "warmup": max(3, warmup), "ms_per_step": ms_per_step, "us_per_layer": ms_per_step * 1000.0 / STACK_LAYERS,
            "tokens_per_s": value, "roofline": roofline(bytes_per_step, ms_per_step, "stack_q4", 1),
            "gpu_launches": steps * launches, "clocks": clk, "e2e": e2e}


def public(d: dict) -> dict:
    return {k: v for k, v in d.items() if not k.startswith("_")}


# ----------------------------------------------------------------------------- GPU arm


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="default: 4000 decode, 200 batched, 128 stack")
    ap.add_argument("--warmup", type=int, default=None, help="default: 200 decode, 20 batched, 8 stack")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="decode_bf16",
                    choices=["decode_bf16", "decode_q4", "decode_i8", "batched_bf16", "batched_q4", "stack_q4"])
    ap.add_argument("--T", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="measure the selected workload only")
    ap.add_argument("--copies", type=int, default=N_LAYER_COPIES, help="layer copies rotated (profiling: fewer)")
    args = ap.parse_args()
    if args.config == "stack_q4":
        args.T = 1
    kind = "stack" if args.config == "stack_q4" else ("batched" if args.T > 8 else "decode")
    if args.steps is None:
        args.steps = {"decode": 4000, "batched": 200, "stack": 128}[kind]
    if args.warmup is None:
        args.warmup = {"decode": 200, "batched": 20, "stack": 8}[kind]
    shapes, wfmt, name = workload(args.config, args.T)
    if args.impl == "reference":
        return run_reference(args, shapes, wfmt, name)

    import torch

    import fusion_backend_gb300 as fb

    dist, world, rank, local = init_ranks()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    want_cpu = rank == 0 and not args.no_cpu_baseline
    resident = {}

    def res_for(w):
        if w not in resident:
            resident[w] = Resident(w, dev, max(1, args.copies))
        return resident[w]

    # ---- the headline line
    stack_host = None
    if args.config == "stack_q4":
        stack_host = stack_layers_host()
        main_r = time_stack(fb, stack_host, args.steps, args.warmup, stream, dev, ClockSampler(local), dist, world)
        e2e = main_r.pop("e2e")
        cpu = None
        if want_cpu:
            cpu = cpu_entry(*oracle_stack_rate(stack_host, 15.0, 1000),
                            what=f"tokens through {STACK_LAYERS} layers, sequential")
    else:
        main_r = time_layer(fb, res_for(wfmt), args.config, args.T, args.steps, args.warmup, stream, dev,
                            ClockSampler(local), dist, world)
        e2e = e2e_layer(fb, res_for(wfmt), main_r, stream, dev, world, min(args.steps, 2000))
        cpu = None
        if want_cpu:
            rate, n, dt, used, offered = oracle_rate(shapes, wfmt, 15.0, 100000, res_for(wfmt).host)
            cpu = cpu_entry(rate, n, dt, used, offered, f"{n} layer calls of T={args.T} on layer seed {SEED}")
        fb.moe_ffn_destroy(main_r["_plan"])

    # ---- every other workload (one GPU only)
    extras = []
    if world == 1 and not args.no_extras:
        for cfg, T, steps, warm, budget in EXTRAS:
            if (cfg, T) == (args.config, args.T):
                continue
            try:
                sh, w, _ = workload(cfg, T)
                if cfg == "stack_q4":
                    if stack_host is None:
                        stack_host = stack_layers_host()
                    r = time_stack(fb, stack_host, steps, warm, stream, dev, ClockSampler(local))
                    r.pop("e2e")
                    if want_cpu:
                        r["cpu_baseline"] = cpu_entry(*oracle_stack_rate(stack_host, budget, 1000),
                                                      what=f"tokens through {STACK_LAYERS} layers, sequential")
                else:
                    r = time_layer(fb, res_for(w), cfg, T, steps, warm, stream, dev, ClockSampler(local))
                    fb.moe_ffn_destroy(r["_plan"])
                    if want_cpu and budget > 0:
                        rate, n, dt, used, offered = oracle_rate(sh, w, budget, 100000, res_for(w).host)
                        r["cpu_baseline"] = cpu_entry(rate, n, dt, used, offered, f"{n} layer calls of T={T}")
                extras.append(public(r))
            except Exception as exc:  # a failed extra is reported, the headline line stands
                extras.append({"config": cfg, "T": T, "error": f"{type(exc).__name__}: {exc}"})
            torch.cuda.synchronize()

    if rank == 0:
        cfg_block = {"workload": name, "parallelism": "replicas only" if world == 1 else f"{world} replicas"}
        if args.config == "stack_q4":
            cfg_block.update({"layers": STACK_LAYERS, "tokens": args.steps,
                              "l2": f"inputs larger than L2: {STACK_LAYERS} layers of "
                                    f"{datagen.expert_bytes(wfmt, H, I) * E / 1e9:.2f} GB"})
        else:
            cfg_block.update({"layers_rotated": max(1, args.copies), "distinct_tokens": N_TOKENS,
                              "rotation": "step s: layer copy s mod copies, token s mod distinct_tokens",
                              "unique_experts_per_step": main_r["unique_experts_per_step"],
                              "l2": f"inputs larger than L2: {max(1, args.copies)} layer copies of "
                                    f"{datagen.expert_bytes(wfmt, H, I) * E / 1e9:.2f} GB rotated"})
        line = {
            "metric": METRIC, "value": main_r["tokens_per_s"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": main_r["warmup"], "ms_per_step": main_r["ms_per_step"], "us_per_layer": main_r["us_per_layer"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dtype_of(wfmt), "data": "synthetic",
            "config": cfg_block, "roofline": main_r["roofline"], "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": main_r["gpu_launches"], "clocks": main_r["clocks"],
        }
        if extras:
            line["configs"] = extras
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
