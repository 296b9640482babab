"""Benchmark: one MoE FFN layer forward on B300, through the library's C ABI.

A step is one pass of the whole layer (router Linear, softmax/top-K, histogram + scan +
capacity, dispatch permutation, grouped expert FFN, combine, aux statistics) over one
batch of seeded synthetic input of the Mixtral-shaped layer (T=4096, d=4096, E=8, K=2,
F=16384, bf16, capacity factor 1.25) unless ``--workload`` picks another shape.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  ``value`` is tokens/s of the whole job (all ranks; each
rank runs an independent replica, no collective on the data path).  L2 is flushed (a
512 MiB device write) before every timed step, outside the step's CUDA events.
``--impl reference`` times the fp64 CPU oracle on this host instead, on a bounded sample
of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from routing_dispatch_expert_04_b300.workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "MoE-layer fwd tokens/s; grouped-GEMM % bf16 peak; dispatch/combine HBM GB/s"
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (identity for one process)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank_step: int, steps: int, world: int,
                           seconds_local: float, device=None) -> float:
    """Tokens of all ranks divided by the slowest rank's time (replicas, weak scaling)."""
    return world * tokens_per_rank_step * steps / max_over_ranks(seconds_local, world, device)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_digest(*rel):
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key: str, digest: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source; None otherwise."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(kernel_key)
    if not ent or ent.get("source_digest") != digest:
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------- CPU oracle
def oracle_sample(wl, host, budget_s: float, rows_budget: int):
    """Time the fp64 oracle on a bounded sample: routing, dispatch plan, combine and aux
    in full, the expert FFN on up to ``rows_budget`` kept rows, scaled linearly to all R
    kept rows.  Returns (seconds for the whole layer, description)."""
    from oracle import moe_oracle as O
    t0 = time.perf_counter()
    _, L32 = O.router_logits(host["x"], host["w_r"], host["b_r"])
    p = O.softmax(L32)
    ids = O.top_k(L32, wl.K)
    w = O.routing_weights(p, ids)
    C = O.capacity(wl.T, wl.E, wl.capacity_factor)
    plan = O.dispatch_plan(ids, wl.E, C)
    O.aux_stats(ids, p, wl.E, wl.alpha)
    t_route = time.perf_counter() - t0
    R = plan["R"]
    offs = plan["offsets"]
    done = 0
    t_ffn = 0.0
    for e in range(wl.E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        n = min(hi - lo, rows_budget - done)
        if n <= 0:
            continue
        rows = plan["src"][lo:lo + n] // wl.K
        t1 = time.perf_counter()
        O.expert_ffn(host["x"][rows], host["w1"](e), host["w2"](e))
        t_ffn += time.perf_counter() - t1
        done += n
        if done >= rows_budget or t_ffn > budget_s:
            break
    t1 = time.perf_counter()
    O.combine(np.zeros((R, wl.d)), plan["slot"], w, wl.T)
    t_comb = time.perf_counter() - t1
    scale = R / max(done, 1)
    total = t_route + t_ffn * scale + t_comb
    desc = (f"routing, dispatch plan, combine and aux over all {wl.T} tokens; expert FFN "
            f"on {done} of {R} kept rows, its time scaled by {scale:.1f}")
    return total, desc


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("internal_api") == "openblas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count()


def host_views(wl, inp):
    """Host fp32 views of the inputs; expert weights fetched per expert on demand."""
    def f32(t):
        return None if t is None else t.float().cpu().numpy()
    return {"x": f32(inp["x"]), "w_r": f32(inp["w_r"]), "b_r": f32(inp["b_r"]),
            "w1": lambda e: f32(inp["w1"][e]), "w2": lambda e: f32(inp["w2"][e])}


# ---------------------------------------------------------------------------- our arm
def run_ours(args, wl):
    from routing_dispatch_expert_04_b300 import native as N
    from routing_dispatch_expert_04_b300.layer import MoELayer

    world, rank, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk = peaks()

    N.set_gemm_pairing({"auto": N.GEMM_AUTO, "single": N.GEMM_SINGLE, "pair": N.GEMM_PAIR,
                        "split": N.GEMM_SPLIT, "pair_t": N.GEMM_PAIR_T}[args.gemm])
    inp = make_inputs(wl, dev, seed=0)
    layer = MoELayer.from_workload(wl, inp, device=dev, fused_dispatch=args.dispatch == "fused",
                                   experts=args.experts, shared_sms=args.shared_sms)
    x = inp["x"]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    stage_names = layer.stage_names()
    n_ev = len(stage_names) + 1
    # one CUDA graph per step, with timing events recorded as graph nodes before every stage
    marks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n_ev)]
    kernels_per_step = layer.capture(x, marks=marks)

    for _ in range(args.warmup):
        flush.zero_()
        layer.replay()
    torch.cuda.synchronize()
    layer.check_device_status()

    stage_ms = {n: [] for n in stage_names}
    step_ms = []
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush.zero_()
        layer.replay()
        torch.cuda.synchronize()   # the graph's events are re-recorded by the next replay
        for i, n in enumerate(stage_names):
            stage_ms[n].append(marks[i].elapsed_time(marks[i + 1]))
        step_ms.append(marks[0].elapsed_time(marks[-1]))
    torch.cuda.synchronize()
    launches = kernels_per_step * args.steps
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    layer.check_device_status()

    local_s = sum(step_ms) / 1e3
    value = whole_job_tokens_per_s(wl.T, args.steps, world, local_s, dev)
    total_s = world * wl.T * args.steps / value

    # ---- algorithmic work of this batch (see the per-stage byte/flop model)
    R = int(layer.offsets[-1].item())
    b = 2 if wl.dtype == "bf16" else 4
    slot = layer.slot
    t_active = int((slot >= 0).any(dim=1).sum().item())
    A = wl.T * wl.K
    flops_up = 2.0 * R * wl.d * wl.F
    flops_down = 2.0 * R * wl.F * wl.d
    # dispatch: the routing plan (ids read, positions, slot and src written) and, when
    # not fused into the first expert GEMM, each token row read once and written to its
    # kept packed rows
    bytes_dispatch = A * 12 + R * 4
    if args.dispatch == "copy":
        bytes_dispatch += t_active * wl.d * b + R * wl.d * b
    yb = 2 if wl.dtype == "bf16" else 4  # expert outputs: fp16 for bf16 layers
    bytes_combine = R * wl.d * yb + wl.T * wl.d * b + A * 8 + (wl.T * wl.d * yb if layer.shared else 0)
    bytes_route = wl.T * wl.d * b + wl.E * wl.d * b + wl.T * wl.E * 4 * 2 + A * 8
    med = {n: statistics.median(v) for n, v in stage_ms.items()}
    avg = {n: sum(v) / len(v) for n, v in stage_ms.items()}

    dom = "expert_up" if avg["expert_up"] >= avg["expert_down"] else "expert_down"
    dom_flops = flops_up if dom == "expert_up" else flops_down
    achieved_tf = dom_flops / (avg[dom] * 1e-3) / 1e12
    kernel_srcs = ["routing_dispatch_expert_04_b300/csrc/" + f
                   for f in ("gemm_tc.cu", "gemm_tc2.cu", "gemm_tc2t.cu", "tc_common.cuh",
                             "tc_ptx.cuh")]
    traffic = recorded_traffic(f"{dom}:{wl.name}:{args.experts}:{args.gemm}",
                               source_digest(*kernel_srcs))
    if args.experts == "e4m3":
        # FP8 contraction: the measured bf16 peak times the nominal fp8/bf16 ratio (2)
        peak_tf, peak_src = 2.0 * pk["bf16_tflops"], f"{pk['source']} bf16 dense (burst) x 2 (nominal e4m3/bf16)"
    else:
        peak_tf, peak_src = pk["bf16_tflops"], f"{pk['source']} bf16 dense (burst)"
    roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved_tf, 2),
                "peak": peak_tf, "unit": "TFLOP/s",
                "frac": round(achieved_tf / peak_tf, 4), "traffic": traffic,
                "peak_source": peak_src,
                "algorithmic_flops_per_launch": dom_flops}
    hbm = pk["hbm_gbs"]

    def gbs(nbytes, ms):
        return nbytes / (ms * 1e-3) / 1e9

    stages = {
        "ms_median": {n: round(v, 4) for n, v in med.items()},
        "expert_up_tflops": round(flops_up / (avg["expert_up"] * 1e-3) / 1e12, 2),
        "expert_down_tflops": round(flops_down / (avg["expert_down"] * 1e-3) / 1e12, 2),
        "grouped_gemm_frac_of_peak": round(
            (flops_up + flops_down) / ((avg["expert_up"] + avg["expert_down"]) * 1e-3) / 1e12
            / peak_tf, 4),
        "dispatch_gbs": round(gbs(bytes_dispatch, avg["dispatch"]), 1),
        "dispatch_frac_of_hbm": round(gbs(bytes_dispatch, avg["dispatch"]) / hbm, 4),
        "combine_gbs": round(gbs(bytes_combine, avg["combine"]), 1),
        "combine_frac_of_hbm": round(gbs(bytes_combine, avg["combine"]) / hbm, 4),
        "route_gbs": round(gbs(bytes_route, avg["route"]), 1),
        "rows_kept": R, "tokens_with_kept_rows": t_active,
        "bytes": {"dispatch": bytes_dispatch, "combine": bytes_combine, "route": bytes_route},
        "flops": {"expert_up": flops_up, "expert_down": flops_down},
    }

    # ---- end to end through the public API with host buffers: every step uploads its
    # input from pinned host memory and downloads its output and aux statistics; the
    # steps are pipelined (upload of step i+1 and download of step i-1 overlap step i)
    from routing_dispatch_expert_04_b300.layer import HostStream
    hs = HostStream(layer, x)
    x_host = x.cpu().pin_memory()
    y_hosts = [torch.empty((wl.T, wl.d), dtype=layer.dtype).pin_memory() for _ in range(2)]
    st_hosts = [torch.empty(2 * wl.E + 1, dtype=torch.float32).pin_memory() for _ in range(2)]
    for i in range(max(1, args.warmup)):
        hs.run(x_host, y_hosts[i & 1], st_hosts[i & 1])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    hs.h2d.wait_event(a)
    for i in range(args.steps):
        hs.run(x_host, y_hosts[i & 1], st_hosts[i & 1])
    stream.wait_stream(hs.d2h)
    z.record(stream)
    z.synchronize()
    e2e_s = max_over_ranks(a.elapsed_time(z) / 1e3, world, dev)
    e2e = {"value": round(world * wl.T * args.steps / e2e_s, 1), "unit": "tokens/s",
           "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
           "d2h_bytes_per_step": y_hosts[0].numel() * y_hosts[0].element_size() + st_hosts[0].numel() * 4,
           "ms_per_step": round(e2e_s * 1e3 / args.steps, 4),
           "pipelining": "two device slots; upload i+1 and download i-1 overlap step i"}
    layer.check_device_status()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        host = host_views(wl, inp)
        secs, desc = oracle_sample(wl, host, budget_s=args.cpu_budget, rows_budget=args.cpu_rows)
        cpu = {"value": round(wl.T / secs, 3), "unit": "tokens/s", "cores": blas_threads(),
               "kind": "oracle", "sample": desc}

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_s * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype if args.experts == "bf16" else f"{wl.dtype} layer, e4m3 expert GEMMs",
        "data": "synthetic",
        "config": {"workload": f"{wl.name}: T={wl.T} d={wl.d} E={wl.E} K={wl.K} F={wl.F} "
                               f"{wl.dtype} capacity_factor={wl.capacity_factor}",
                   "capacity": layer.cfg.capacity, "parallelism": f"replicas x{world}",
                   "expert_gemm": args.gemm, "dispatch": args.dispatch, "experts": args.experts,
                   "shared_expert_sms": args.shared_sms if layer.shared else None,
                   "l2": "flushed before each step (512 MiB device write, outside the events)"},
        "roofline": roofline, "stages": stages, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches, "gpu_launches_per_step": kernels_per_step,
        "launch_mode": "one CUDA graph per step (library kernels + the scan's memset node)",
        "clocks": clk,
        "device": torch.cuda.get_device_name(dev),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------------------- reference
def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = make_inputs(wl, dev, seed=0)
    host = host_views(wl, inp)
    cores = blas_threads()
    for _ in range(args.warmup):
        oracle_sample(wl, host, budget_s=args.ref_budget, rows_budget=args.ref_rows)
    secs, descs = [], None
    for _ in range(args.steps):
        s, descs = oracle_sample(wl, host, budget_s=args.ref_budget, rows_budget=args.ref_rows)
        secs.append(s)
    total = sum(secs)
    value = wl.T * args.steps / total
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total * 1e3 / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name}: T={wl.T} d={wl.d} E={wl.E} K={wl.K} F={wl.F} "
                               f"{wl.dtype} capacity_factor={wl.capacity_factor}",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": descs},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral", choices=sorted(WORKLOADS))
    ap.add_argument("--gemm", choices=["auto", "single", "pair", "split", "pair_t"], default="auto",
                    help="expert GEMM kernels: one CTA per 128-row tile, CTA pairs per "
                         "256-row tile, pairs for whole 256-row tiles + one CTA for the "
                         "rest, pairs with the tokens on the MMA's N side, or the "
                         "library's choice")
    ap.add_argument("--shared-sms", type=int, default=0,
                    help="SMs for the shared expert beside the routed GEMMs (0: beside routing)")
    ap.add_argument("--dispatch", choices=["fused", "copy"], default="copy",
                    help="fused: the first expert GEMM gathers its rows from x while loading "
                         "them; copy: the dispatch step copies them into a packed buffer")
    ap.add_argument("--experts", choices=["bf16", "e4m3"], default="bf16",
                    help="expert Linears in bf16 (the layer's precision) or the FP8 variant "
                         "(per-row E4M3 operands); an e4m3 line is a different precision "
                         "and says so in its dtype")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--cpu-rows", type=int, default=512)
    ap.add_argument("--ref-budget", type=float, default=6.0)
    ap.add_argument("--ref-rows", type=int, default=128)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
