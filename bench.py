"""Benchmark of the fused MoE FFN layer on one GB300 (or N replicas).

Default workload: the decode bf16 MoE layer, T=1 token, H=2048, E=128,
top_k=8, I=768, Is=512.  One step = one layer call on one token batch.  The
timed steps rotate through 16 copies of the layer at distinct addresses
(16 x 1.21 GB, far larger than the 129 MB L2) and 100 distinct seeded
tokens, so every step streams its weights from HBM.  Steps are captured in a
CUDA graph and replayed; CUDA events on the launching stream time them.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead (the reference arm).

With ``--config batched_bf16 --T 64`` (or 256) the same layer runs on the
batched path (routing, expert-sorted gather, grouped GEMMs on the tensor
cores, combine); ``--config batched_q4`` does the same with 4-bit weights.  ``--config stack_q4`` runs the 48-layer 4-bit decode stack
(pre-norm RMSNorm and residual add per layer, independent seeded layers);
a step is one token through all 48 layers, and each token's output feeds the
next token's input (128 sequential tokens by default).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode_bf16|decode_q4|batched_bf16|batched_q4|stack_q4] [--T T]
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
# dram__bytes_read.sum + dram__bytes_write.sum of one k_rows launch from the
# committed ncu capture (profiles/), per config; None until captured for the
# current kernel.
NCU_TRAFFIC_BYTES = {"decode_bf16": 83_209_216, "decode_q4": 23_105_792, "batched_bf16": 823_113_984,
                     "batched_q4": 238_398_464, "stack_q4": None}
STACK_LAYERS = 48


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


def workload(cfg: str, T: int):
    wfmt = datagen.WFMT_Q4B32 if cfg in ("decode_q4", "batched_q4", "stack_q4") else datagen.WFMT_BF16
    shapes = datagen.Shapes(T=T, H=H, E=E, top_k=K_TOP, I=I, Is=IS)
    name = {
        "decode_bf16": f"decode bf16 MoE FFN layer: T={T}, H={H}, E={E}, top_k={K_TOP}, I={I}, Is={IS}",
        "decode_q4": f"decode 4-bit MoE FFN layer (blocks of 32, fp16 scale): T={T}, H={H}, E={E}, top_k={K_TOP}, I={I}, Is={IS}",
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
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower() in ("active", "0x1") or v == "1":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- reference arm (oracle on CPU)


def oracle_rate(shapes, wfmt, budget_s: float, max_tokens: int):
    import oracle

    layer = datagen.make_layer(SEED, datagen.Shapes(1, H, E, K_TOP, I, IS), wfmt)
    s1 = datagen.Shapes(shapes.T, H, E, K_TOP, I, IS)
    threads = oracle.nthreads()
    done = 0
    t0 = time.perf_counter()
    while done < max_tokens:
        x = token_batch(done, shapes.T)
        oracle.moe_ffn(s1, datagen.ACT_BF16, wfmt, x, layer.router_w, layer.expert_w, layer.shexp_w,
                       layer.shexp_gate_w, threads=threads)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    used = min(threads, shapes.T * K_TOP + shapes.T)
    return done * shapes.T / dt, done, dt, used


def run_reference(args, shapes, wfmt, name):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    # warm-up: one call
    oracle_rate(shapes, wfmt, 0.0, max(1, min(args.warmup, 1)))
    budget = 60.0
    rate, n, dt, used = oracle_rate(shapes, wfmt, budget, args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus, "steps": n,
        "warmup": args.warmup, "ms_per_step": dt / n * 1000.0, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "parallelism": "replicas only"},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": f"{n} layer calls of T={shapes.T} (of {args.steps} requested; bounded to ~{budget:.0f} s)"},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- 48-layer stack (config 4)


def run_stack(args, shapes, wfmt, name):
    """One step = one token through STACK_LAYERS layers in block form (x_res updated in place); the timed
    steps are consecutive tokens, each starting from the previous token's output."""
    from concurrent.futures import ThreadPoolExecutor

    import torch

    import fusion_backend_gb300 as fb

    dist, world, rank, local = init_ranks()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    s1 = datagen.Shapes(1, H, E, K_TOP, I, IS)

    def gen(l):
        lay = datagen.make_layer(SEED + 1000 + l, s1, wfmt)
        return (torch.from_numpy(lay.router_w.view(np.int16)).to(dev), torch.from_numpy(lay.expert_w).to(dev),
                torch.from_numpy(lay.shexp_w).to(dev), torch.from_numpy(lay.shexp_gate_w.view(np.int16)).to(dev))

    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as pool:
        layers = list(pool.map(gen, range(STACK_LAYERS)))
    plan, ws_bytes = fb.moe_ffn_prepare(s1, fb.ACT_BF16, wfmt)
    launches = fb.moe_ffn_query(plan, fb.QUERY_LAUNCHES_PER_EXECUTE) * STACK_LAYERS
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    x0 = torch.from_numpy(datagen.normal_f32(SEED, 7, H, 1.0).reshape(1, H)).to(dev)
    x_res = x0.clone()
    stream = torch.cuda.Stream(device=dev)

    def token_pass():
        for r, ew, sw, gv in layers:
            fb.moe_ffn_execute_block(plan, ws, x_res, r, ew, sw, gv, eps=1e-6, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            token_pass()
    torch.cuda.synchronize()
    if fb.moe_ffn_read_status(plan, ws, stream) != 0:
        raise RuntimeError("device status after warm-up")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        token_pass()
    x_res.copy_(x0)
    torch.cuda.synchronize()
    steps = args.steps
    clocks = ClockSampler(local)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    ms, value = whole_job(ev0.elapsed_time(ev1), steps, world, dist, dev)
    if fb.moe_ffn_read_status(plan, ws, stream) != 0:
        raise RuntimeError("device status after the timed region")
    final = x_res.cpu().numpy()
    if not np.all(np.isfinite(final)):
        raise RuntimeError("non-finite stack output")
    ms_per_step = ms / steps
    bytes_per_step = STACK_LAYERS * algorithmic_bytes(s1, wfmt, float(K_TOP))
    peak, peak_kind = peaks()
    achieved = bytes_per_step / (ms_per_step / 1000.0) / 1e9
    # end to end: each token's input from pinned host memory, its output back
    e2e_steps = min(steps, 64)
    x_pin = torch.from_numpy(final.copy()).pin_memory()
    out_pin = torch.empty((e2e_steps, 1, H), dtype=torch.float32).pin_memory()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(e2e_steps):
            x_res.copy_(x_pin if i == 0 else out_pin[i - 1], non_blocking=True)
            token_pass()
            out_pin[i].copy_(x_res, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_value = e2e_steps * world / (e0.elapsed_time(e1) / 1000.0)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "us_per_layer": ms_per_step * 1000.0 / STACK_LAYERS, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "q4b32 weights, fp32 accumulate", "data": "synthetic",
            "config": {"workload": name, "layers": STACK_LAYERS, "tokens": steps,
                       "l2": f"inputs larger than L2: {STACK_LAYERS} layers of {datagen.expert_bytes(wfmt, H, I) * E / 1e9:.2f} GB",
                       "parallelism": "replicas only" if world == 1 else f"{world} replicas"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind, "traffic": NCU_TRAFFIC_BYTES.get(args.config),
                         "algorithmic_bytes_per_step": bytes_per_step,
                         "kernel": "k_rows (+ k_route) per layer; duration = step time / layers"},
            "cpu_baseline": None,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": H * 4, "d2h_bytes_per_step": H * 4,
                    "steps": e2e_steps, "how": "eager public-API calls per token: pinned H2D of x, 48 layers, D2H"},
            "gpu_launches": steps * launches,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    fb.moe_ffn_destroy(plan)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- GPU arm


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="default: 64000 decode, 2000 batched, 128 stack")
    ap.add_argument("--warmup", type=int, default=None, help="default: 1600 decode, 20 batched, 8 stack")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="decode_bf16", choices=["decode_bf16", "decode_q4", "batched_bf16", "batched_q4", "stack_q4"])
    ap.add_argument("--T", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--copies", type=int, default=N_LAYER_COPIES, help="layer copies rotated (profiling: fewer)")
    args = ap.parse_args()
    if args.config == "stack_q4":
        args.T = 1
    kind = "stack" if args.config == "stack_q4" else ("batched" if args.T > 8 else "decode")
    if args.steps is None:
        args.steps = {"decode": 64000, "batched": 2000, "stack": 128}[kind]
    if args.warmup is None:
        args.warmup = {"decode": 1600, "batched": 20, "stack": 8}[kind]
    shapes, wfmt, name = workload(args.config, args.T)
    if args.impl == "reference":
        return run_reference(args, shapes, wfmt, name)
    if args.config == "stack_q4":
        return run_stack(args, shapes, wfmt, name)

    import torch

    import fusion_backend_gb300 as fb

    dist, world, rank, local = init_ranks()
    torch.cuda.set_device(local)

    def barrier():
        if dist is not None:
            dist.barrier()

    T = shapes.T
    dev = torch.device("cuda", local)
    layer = datagen.make_layer(SEED, datagen.Shapes(1, H, E, K_TOP, I, IS), wfmt)
    router = torch.from_numpy(layer.router_w.view(np.int16)).to(dev)
    gvec = torch.from_numpy(layer.shexp_gate_w.view(np.int16)).to(dev)
    ew0 = torch.from_numpy(layer.expert_w).to(dev)
    sw0 = torch.from_numpy(layer.shexp_w).to(dev)
    copies = []
    n_copies = max(1, args.copies)
    for _ in range(n_copies):  # distinct addresses, same values: no L2 reuse across steps
        copies.append((router.clone(), ew0.clone(), sw0.clone(), gvec.clone()))
    del ew0, sw0
    xs_host = np.stack([token_batch(t, T) for t in range(N_TOKENS)])  # [N_TOKENS, T, H] bf16 bits
    xs = torch.from_numpy(xs_host.view(np.int16)).to(dev)
    plan, ws_bytes = fb.moe_ffn_prepare(shapes, fb.ACT_BF16, wfmt)
    launches_per_step = fb.moe_ffn_query(plan, fb.QUERY_LAUNCHES_PER_EXECUTE)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step_args(s):
        r, ew, sw, gv = copies[s % n_copies]
        return xs[(s // n_copies) % N_TOKENS], r, ew, sw, gv

    # Unique experts per step (for the byte count): routing of each (token) once.
    ids = torch.empty((T, K_TOP), dtype=torch.int32, device=dev)
    uniq = []
    with torch.cuda.stream(stream):
        for t in range(N_TOKENS):
            x, r, ew, sw, gv = step_args(t * n_copies)
            fb.moe_ffn_execute_ex(plan, ws, x, r, ew, sw, gv, out, ids, None, stream=stream)
            uniq.append(len(np.unique(ids.cpu().numpy())))
    torch.cuda.synchronize()
    status = fb.moe_ffn_read_status(plan, ws, stream)
    if status != 0:
        raise RuntimeError(f"device status {status}")
    U_mean = float(np.mean(uniq))
    bytes_per_step = algorithmic_bytes(shapes, wfmt, U_mean)

    graph_steps = min(args.steps, n_copies * N_TOKENS)

    def capture(n, first):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in range(first, first + n):
                x, r, ew, sw, gv = step_args(s)
                fb.moe_ffn_execute(plan, ws, x, r, ew, sw, gv, out, stream=stream)
        return g

    # warm-up (eager, then one capture replay)
    with torch.cuda.stream(stream):
        for s in range(max(3, min(args.warmup, graph_steps))):
            x, r, ew, sw, gv = step_args(s)
            fb.moe_ffn_execute(plan, ws, x, r, ew, sw, gv, out, stream=stream)
    torch.cuda.synchronize()
    g_main = capture(graph_steps, 0)
    reps, rem = divmod(args.steps, graph_steps)
    g_rem = capture(rem, 0) if rem else None
    g_main.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    steps = args.steps
    ms, value = whole_job(ev0.elapsed_time(ev1), steps * T, world, dist, dev)
    status = fb.moe_ffn_read_status(plan, ws, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    ms_per_step = ms / steps
    peak, peak_kind = peaks()
    achieved_gbs = bytes_per_step / (ms_per_step / 1000.0) / 1e9

    # ---- end to end through the public API with host buffers (eager calls)
    e2e_steps = min(steps, 2000)
    x_pin = torch.from_numpy(xs_host.view(np.int16)).pin_memory()
    out_pin = torch.empty((e2e_steps, T, H), dtype=torch.float32).pin_memory()
    x_dev = torch.empty((T, H), dtype=torch.int16, device=dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for s in range(e2e_steps):
            r, ew, sw, gv = copies[s % n_copies]
            x_dev.copy_(x_pin[(s // n_copies) % N_TOKENS], non_blocking=True)
            fb.moe_ffn_execute(plan, ws, x_dev, r, ew, sw, gv, out, stream=stream)
            out_pin[s].copy_(out, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_value = e2e_steps * T * world / (e2e_ms / 1000.0)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, n, dt, used = oracle_rate(shapes, wfmt, 15.0, 100000)
        cpu = {"value": rate, "unit": UNIT, "cores": used, "kind": "oracle",
               "sample": f"{n} layer calls of T={T} on layer seed {SEED} ({dt:.1f} s, all host threads offered)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "us_per_layer": ms_per_step * 1000.0, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wfmt == 0 else "q4b32 weights, fp32 accumulate",
            "data": "synthetic",
            "config": {"workload": name, "layers_rotated": n_copies, "distinct_tokens": N_TOKENS,
                       "unique_experts_per_step": U_mean,
                       "l2": f"inputs larger than L2: {n_copies} layer copies of {datagen.expert_bytes(wfmt, H, I) * E / 1e9:.2f} GB rotated",
                       "parallelism": "replicas only" if world == 1 else f"{world} replicas"},
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                         "frac": achieved_gbs / peak, "peak_kind": peak_kind,
                         "traffic": NCU_TRAFFIC_BYTES.get(args.config),
                         "algorithmic_bytes_per_step": bytes_per_step,
                         "kernel": (("k_gemm_q4<0>, k_gemm_q4<1>" if wfmt else "k_gemm<0>, k_gemm<1>")
                                    + " (+ routing, gather, combine); duration = step time"
                                    if T > 8 else "k_rows (+ k_route, programmatic dependent launch); duration = step time")},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 4,
                    "steps": e2e_steps, "how": "eager public-API calls: pinned H2D of x, execute, D2H of out"},
            "gpu_launches": steps * launches_per_step,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    fb.moe_ffn_destroy(plan)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
