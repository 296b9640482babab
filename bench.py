"""Benchmark: one MoE FFN layer forward on B300, through the library's C ABI.

A step is one pass of the whole layer (router Linear, softmax/top-K, histogram + scan +
capacity, dispatch permutation, grouped expert FFN, combine, aux statistics) over one
batch of seeded synthetic input of the Mixtral-shaped layer (T=4096, d=4096, E=8, K=2,
F=16384, bf16, capacity factor 1.25) unless ``--workload`` picks another shape.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  ``value`` is tokens/s of the whole job (all ranks; each
rank runs an independent replica, no collective on the data path).  L2 is flushed (a
512 MiB device write) before every timed step, outside the step's CUDA events.  After
the headline workload the same measurement runs, one after the other with the device
memory freed in between, on the other bf16 layer shapes (DeepSeek-V3, Qwen3-30B-A3B,
64K tokens); their results go into the line's ``workloads`` record.

``cpu_baseline`` is the fp64 CPU oracle timed on this host: the whole layer for the
Mixtral- and Qwen3-shaped workloads, a labelled extrapolation from whole expert blocks
for the two largest.  ``--impl reference`` times the same oracle as the reference arm:
each step is half a layer (the routing and half of the experts, then the other half and
the combine), so two steps are exactly one layer forward.
"""

from __future__ import annotations

import argparse
import gc
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
L2_NOTE = "flushed before each timed GPU step (512 MiB device write, outside the events)"
EXTRA_WORKLOADS = ("dsv3", "qwen3", "long")


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


def workload_config(wl, capacity: int, world: int) -> dict:
    """The `config` record: the workload and how it is measured.  Both arms print exactly
    this record (implementation settings go elsewhere)."""
    return {"workload": f"{wl.name}: T={wl.T} d={wl.d} E={wl.E} K={wl.K} F={wl.F} "
                        f"{wl.dtype} capacity_factor={wl.capacity_factor}",
            "capacity": capacity, "parallelism": f"replicas x{world}", "l2": L2_NOTE}


def gpu_uuid(device) -> str:
    """nvidia-smi's identifier of a CUDA device: its UUID, which (unlike the CUDA ordinal)
    names the same physical GPU whatever CUDA_VISIBLE_DEVICES says."""
    u = str(torch.cuda.get_device_properties(device).uuid)
    return u if u.startswith("GPU-") else "GPU-" + u


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.gpu = gpu_uuid(device)
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
                "reasons": sorted(reasons), "samples": len(sm), "gpu": self.gpu}


def source_digest(*rel):
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


GEMM_SOURCES = ["routing_dispatch_expert_04_b300/csrc/" + f
                for f in ("gemm_tc.cu", "gemm_tc2.cu", "gemm_tc2t.cu", "gemm_tc2m.cu",
                          "tc_common.cuh", "tc_ptx.cuh")]


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
            "w1": lambda e: f32(inp["w1"][e]), "w2": lambda e: f32(inp["w2"][e]),
            "w1s": f32(inp["w1s"][0]) if wl.shared else None,
            "w2s": f32(inp["w2s"][0]) if wl.shared else None}


def oracle_full_layer(wl, inp):
    """The whole fp64 oracle layer forward (moe_forward) on the workload, timed once after
    a warm-up on one expert block (which touches buffers of the same sizes).  Returns
    (seconds, description)."""
    from oracle import moe_oracle as O
    h = host_views(wl, inp)
    w1 = inp["w1"].float().cpu().numpy()
    w2 = inp["w2"].float().cpu().numpy()
    C = O.capacity(wl.T, wl.E, wl.capacity_factor)
    n0 = min(wl.T * wl.K // wl.E, wl.T)
    O.expert_ffn(h["x"][:max(n0, 1)], w1[0], w2[0])
    shared = (h["w1s"], h["w2s"]) if wl.shared else None
    t0 = time.perf_counter()
    O.moe_forward(h["x"], h["w_r"], h["b_r"], w1, w2, wl.K, C, wl.alpha, shared=shared)
    secs = time.perf_counter() - t0
    return secs, (f"the whole layer (moe_forward: routing, dispatch plan, every expert's "
                  f"kept rows, combine, aux) over all {wl.T} tokens, timed once after a "
                  f"warm-up on one expert block")


def oracle_extrapolated(wl, inp, rows_budget: int, block_rows: int):
    """Routing, dispatch plan, aux and combine in full; the expert FFN on whole blocks of
    up to ``block_rows`` kept rows (the layer's own GEMM shapes), experts in order, until
    ``rows_budget`` rows; the FFN time scaled linearly to all R kept rows (and the shared
    expert, if any, timed on one block and scaled to T rows).  Returns (seconds, desc)."""
    from oracle import moe_oracle as O
    h = host_views(wl, inp)
    O.expert_ffn(h["x"][:min(block_rows, wl.T)], h["w1"](0), h["w2"](0))  # warm-up
    t0 = time.perf_counter()
    _, L32 = O.router_logits(h["x"], h["w_r"], h["b_r"])
    p = O.softmax(L32)
    ids = O.top_k(L32, wl.K)
    w = O.routing_weights(p, ids)
    C = O.capacity(wl.T, wl.E, wl.capacity_factor)
    plan = O.dispatch_plan(ids, wl.E, C)
    O.aux_stats(ids, p, wl.E, wl.alpha)
    t_route = time.perf_counter() - t0
    R, offs = plan["R"], plan["offsets"]
    done, t_ffn = 0, 0.0
    for e in range(wl.E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        n = min(hi - lo, block_rows)
        if n <= 0:
            continue
        rows = plan["src"][lo:lo + n] // wl.K
        w1e, w2e = h["w1"](e), h["w2"](e)
        t1 = time.perf_counter()
        O.expert_ffn(h["x"][rows], w1e, w2e)
        t_ffn += time.perf_counter() - t1
        done += n
        if done >= rows_budget:
            break
    t_shared, shared_note = 0.0, ""
    if wl.shared:
        n = min(block_rows, wl.T)
        t1 = time.perf_counter()
        O.dense_ffn(h["x"][:n], h["w1s"], h["w2s"])
        t_shared = (time.perf_counter() - t1) * wl.T / n
        shared_note = f"; shared expert on {n} of {wl.T} tokens, scaled by {wl.T / n:.1f}"
    t1 = time.perf_counter()
    O.combine(np.zeros((R, wl.d)), plan["slot"], w, wl.T)
    t_comb = time.perf_counter() - t1
    scale = R / max(done, 1)
    total = t_route + t_ffn * scale + t_shared + t_comb
    return total, (f"routing, dispatch plan, aux and combine over all {wl.T} tokens; expert FFN "
                   f"on {done} of {R} kept rows (blocks of up to {block_rows} rows of one "
                   f"expert), its time scaled by {scale:.1f}{shared_note}")


def cpu_baseline(wl, inp, full: bool) -> dict:
    if full:
        secs, desc = oracle_full_layer(wl, inp)
    else:
        secs, desc = oracle_extrapolated(wl, inp, rows_budget=4096,
                                         block_rows=1024 if wl.E <= 16 else 512)
    return {"value": round(wl.T / secs, 3), "unit": "tokens/s", "cores": blas_threads(),
            "kind": "oracle", "sample": desc, "extrapolated": not full,
            "seconds_per_layer": round(secs, 3)}


# ---------------------------------------------------------------------------- our arm
def measure(wl, args, dev, world, pk, with_traffic: bool):
    """One workload on this GPU: the CUDA-graph step timed with per-stage events, and the
    end-to-end rate through the host-buffer pipeline.  Returns a plain dict (no device
    tensors survive the call)."""
    from routing_dispatch_expert_04_b300.layer import HostStream, MoELayer

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
    # the library's clock telemetry (SM cycles and nanoseconds summed over the tensor-core
    # kernels' CTAs, at bytes 64..79 of each workspace) over the timed steps
    workspaces = [w for w in (layer.ws, layer.ws_s) if w is not None]
    for w in workspaces:
        w[64:80].zero_()
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for _ in range(args.steps):
        flush.zero_()
        layer.replay()
        torch.cuda.synchronize()   # the graph's events are re-recorded by the next replay
        for i, n in enumerate(stage_names):
            stage_ms[n].append(marks[i].elapsed_time(marks[i + 1]))
        step_ms.append(marks[0].elapsed_time(marks[-1]))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    layer.check_device_status()
    tele = sum(w[64:80].view(torch.int64) for w in workspaces).tolist()
    clk["tensor_kernels_sm_mhz"] = round(tele[0] / tele[1] * 1e3, 1) if tele[1] > 0 else None

    local_s = sum(step_ms) / 1e3
    value = whole_job_tokens_per_s(wl.T, args.steps, world, local_s, dev)
    total_s = world * wl.T * args.steps / value

    # ---- algorithmic work of this batch (the per-stage byte/flop model)
    R = int(layer.offsets[-1].item())
    b = 2 if wl.dtype == "bf16" else 4
    t_active = int((layer.slot >= 0).any(dim=1).sum().item())
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
    # expert GEMM bytes: the weights (W1 bf16, W2 fp16: 2 bytes each, or 1 for E4M3), the
    # A rows read and the output rows written (h and y_perm fp16)
    wbytes = wl.E * wl.F * wl.d * (1 if args.experts == "e4m3" else 2)
    bytes_up = wbytes + R * wl.d * b + R * wl.F * 2
    bytes_down = wbytes + R * wl.F * 2 + R * wl.d * 2
    med = {n: statistics.median(v) for n, v in stage_ms.items()}
    avg = {n: sum(v) / len(v) for n, v in stage_ms.items()}
    hbm = pk["hbm_gbs"]
    if args.experts == "e4m3":
        # FP8 contraction: the measured bf16 peak times the nominal fp8/bf16 ratio (2)
        peak_tf, peak_src = 2.0 * pk["bf16_tflops"], f"{pk['source']} bf16 dense (burst) x 2 (nominal e4m3/bf16)"
    else:
        peak_tf, peak_src = pk["bf16_tflops"], f"{pk['source']} bf16 dense (burst)"

    def gbs(nbytes, ms):
        return nbytes / (ms * 1e-3) / 1e9

    def gemm_rec(flops, nbytes, ms):
        tf = flops / (ms * 1e-3) / 1e12
        g = gbs(nbytes, ms)
        ft, fh = tf / peak_tf, g / hbm
        return {"ms": round(ms, 4), "tflops": round(tf, 2), "frac_of_tensor_peak": round(ft, 4),
                "gbs": round(g, 1), "frac_of_hbm": round(fh, 4),
                "binding": "tensor" if ft >= fh else "hbm"}

    stages = {
        "ms_median": {n: round(v, 4) for n, v in med.items()},
        "expert_up": gemm_rec(flops_up, bytes_up, avg["expert_up"]),
        "expert_down": gemm_rec(flops_down, bytes_down, avg["expert_down"]),
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
        "bytes": {"dispatch": bytes_dispatch, "combine": bytes_combine, "route": bytes_route,
                  "expert_up": bytes_up, "expert_down": bytes_down},
        "flops": {"expert_up": flops_up, "expert_down": flops_down},
        "peak": {"tensor_tflops": peak_tf, "tensor_source": peak_src, "hbm_gbs": hbm,
                 "hbm_source": f"{pk['source']} copy bandwidth"},
    }

    dom = "expert_up" if avg["expert_up"] >= avg["expert_down"] else "expert_down"
    dom_flops = flops_up if dom == "expert_up" else flops_down
    achieved_tf = dom_flops / (avg[dom] * 1e-3) / 1e12
    traffic = None
    if with_traffic:
        traffic = recorded_traffic(f"{dom}:{wl.name}:{args.experts}:{args.gemm}",
                                   source_digest(*GEMM_SOURCES))
    roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved_tf, 2),
                "peak": peak_tf, "unit": "TFLOP/s",
                "frac": round(achieved_tf / peak_tf, 4), "traffic": traffic,
                "peak_source": peak_src, "algorithmic_flops_per_launch": dom_flops}
    sus = pk.get("bf16_tflops_sustained")
    if sus and args.experts == "bf16":
        roofline["peak_sustained"] = sus
        roofline["frac_of_sustained"] = round(achieved_tf / sus, 4)
    mhz = clk.get("tensor_kernels_sm_mhz")
    if mhz:
        # dense bf16 rate of a B300 SM: 8192 flop per clock (M=128, N=256, K=16 per 128 clocks)
        per_clock_peak = 148 * 8192 * mhz * 1e6 / 1e12 * (2 if args.experts == "e4m3" else 1)
        roofline["sm_mhz_in_kernel"] = mhz
        roofline["frac_of_peak_at_that_clock"] = round(achieved_tf / per_clock_peak, 4)

    # ---- a layer with a shared expert overlaps it with routing and dispatch, so those
    # stages share the GPU; the same step on one stream (shared expert after the routed
    # experts) shows each stage on its own
    serial = None
    if layer.shared and layer.overlap:
        layer.overlap = False
        s_names = layer.stage_names()
        s_marks = [torch.cuda.Event(enable_timing=True, external=True)
                   for _ in range(len(s_names) + 1)]
        layer.capture(x, marks=s_marks)
        s_ms = {n: [] for n in s_names}
        for _ in range(max(args.warmup, 3)):
            flush.zero_()
            layer.replay()
        for _ in range(args.steps):
            flush.zero_()
            layer.replay()
            torch.cuda.synchronize()
            for i, n in enumerate(s_names):
                s_ms[n].append(s_marks[i].elapsed_time(s_marks[i + 1]))
        layer.check_device_status()
        s_avg = {n: sum(v) / len(v) for n, v in s_ms.items()}
        serial = {"ms_median": {n: round(statistics.median(v), 4) for n, v in s_ms.items()},
                  "ms_per_step": round(sum(s_avg.values()), 4),
                  "dispatch_frac_of_hbm": round(gbs(bytes_dispatch, s_avg["dispatch"]) / hbm, 4),
                  "combine_frac_of_hbm": round(gbs(bytes_combine, s_avg["combine"]) / hbm, 4),
                  "note": "one stream: route, dispatch, routed experts, shared expert, combine, "
                          "aux"}
        layer.overlap = True
        layer.capture(x)  # back to the overlapped graph for the end-to-end run
    stages["serial_schedule"] = serial

    # ---- end to end through the public API with host buffers: every step uploads its
    # input from pinned host memory and downloads its output and aux statistics; the
    # steps are pipelined (upload of step i+1 and download of step i-1 overlap step i)
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
    capacity = layer.cfg.capacity
    shared = layer.shared
    del hs, layer, flush, marks, x_host, y_hosts, st_hosts
    gc.collect()
    torch.cuda.synchronize()
    return {"value": value, "ms_per_step": total_s * 1e3 / args.steps, "stages": stages,
            "roofline": roofline, "e2e": e2e, "clocks": clk, "kernels_per_step": kernels_per_step,
            "capacity": capacity, "shared": shared, "inputs": inp}


def run_ours(args, wl):
    from routing_dispatch_expert_04_b300 import native as N

    world, rank, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk = peaks()
    N.set_gemm_pairing({"auto": N.GEMM_AUTO, "single": N.GEMM_SINGLE, "pair": N.GEMM_PAIR,
                        "split": N.GEMM_SPLIT, "pair_t": N.GEMM_PAIR_T,
                        "mixed": N.GEMM_MIXED}[args.gemm])
    do_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline

    m = measure(wl, args, dev, world, pk, with_traffic=True)
    cpu = cpu_baseline(wl, m["inputs"], full=True) if do_cpu else None
    launches = m["kernels_per_step"] * args.steps
    del m["inputs"]
    torch.cuda.empty_cache()

    extra = {}
    names = [] if args.extra_workloads in ("", "none") else args.extra_workloads.split(",")
    for name in names:
        if name == wl.name:
            continue
        xw = WORKLOADS[name]
        r = measure(xw, args, dev, world, pk, with_traffic=False)
        rec = {"config": workload_config(xw, r["capacity"], world),
               "tokens_per_s": round(r["value"], 1), "ms_per_step": round(r["ms_per_step"], 4),
               "e2e_tokens_per_s": r["e2e"]["value"], "e2e": r["e2e"],
               "stages": r["stages"], "clocks": r["clocks"],
               "gpu_launches_per_step": r["kernels_per_step"]}
        if do_cpu:
            rec["cpu_baseline"] = cpu_baseline(xw, r["inputs"], full=(name == "qwen3"))
        launches += r["kernels_per_step"] * args.steps
        del r
        gc.collect()
        torch.cuda.empty_cache()
        extra[name] = rec

    out = {
        "metric": METRIC, "value": round(m["value"], 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(m["ms_per_step"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype if args.experts == "bf16" else f"{wl.dtype} layer, e4m3 expert GEMMs",
        "data": "synthetic",
        "config": workload_config(wl, m["capacity"], world),
        "settings": {"expert_gemm": args.gemm, "dispatch": args.dispatch, "experts": args.experts,
                     "shared_expert_sms": args.shared_sms if m["shared"] else None},
        "roofline": m["roofline"], "stages": m["stages"], "cpu_baseline": cpu, "e2e": m["e2e"],
        "gpu_launches": launches, "gpu_launches_per_step": m["kernels_per_step"],
        "launch_mode": "one CUDA graph per step (library kernels + the scan's memset node)",
        "clocks": m["clocks"],
        "workloads": extra,
        "device": torch.cuda.get_device_name(dev),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------------------- reference
class HalfLayerOracle:
    """The fp64 oracle layer forward cut into two half-layer steps: an even step runs the
    routing, the dispatch plan and the aux statistics over all T tokens and the expert FFN
    of the first half of the experts; an odd step the FFN of the other half and the
    combine.  Every expert block is whole (all its kept rows), so two consecutive steps
    are exactly one moe_forward's work in the same library calls."""

    def __init__(self, wl, inp):
        from oracle import moe_oracle as O
        self.O, self.wl = O, wl
        h = host_views(wl, inp)
        self.x, self.w_r, self.b_r = h["x"], h["w_r"], h["b_r"]
        self.w1 = inp["w1"].float().cpu().numpy()
        self.w2 = inp["w2"].float().cpu().numpy()
        self.shared = (h["w1s"], h["w2s"]) if wl.shared else None
        self.C = O.capacity(wl.T, wl.E, wl.capacity_factor)
        self.half = (wl.E + 1) // 2
        self.i = 0

    def _experts(self, lo_e, hi_e):
        O, wl, p = self.O, self.wl, self.plan
        offs = p["offsets"]
        for e in range(lo_e, hi_e):
            lo, hi = int(offs[e]), int(offs[e + 1])
            if hi > lo:
                self.y_perm[lo:hi], _ = O.expert_ffn(self.x_perm[lo:hi], self.w1[e], self.w2[e])

    def step(self):
        O, wl = self.O, self.wl
        if self.i % 2 == 0:
            _, L32 = O.router_logits(self.x, self.w_r, self.b_r)
            prob = O.softmax(L32)
            ids = O.top_k(L32, wl.K)
            self.w = O.routing_weights(prob, ids)
            self.plan = O.dispatch_plan(ids, wl.E, self.C)
            O.aux_stats(ids, prob, wl.E, wl.alpha)
            src = self.plan["src"].astype(np.int64)
            self.x_perm = O.widen(self.x)[src // wl.K]
            self.y_perm = np.zeros((self.plan["R"], wl.d))
            self._experts(0, self.half)
        else:
            self._experts(self.half, wl.E)
            ys = O.expert_ffn(O.widen(self.x), *self.shared)[0] if self.shared else None
            self.y = O.combine(self.y_perm, self.plan["slot"], self.w, wl.T, ys)
        self.i += 1


def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from oracle import moe_oracle as O
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = make_inputs(wl, dev, seed=0)
    C = O.capacity(wl.T, wl.E, wl.capacity_factor)
    cores = blas_threads()
    orc = HalfLayerOracle(wl, inp)
    del inp
    for _ in range(args.warmup):
        orc.step()
    secs = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        orc.step()
        secs.append(time.perf_counter() - t0)
    total = sum(secs)
    # two half-layer steps are one layer forward of T tokens
    value = wl.T * (args.steps / 2) / total
    desc = (f"each step half a layer forward of the fp64 oracle (even steps: routing, dispatch "
            f"plan and aux over all {wl.T} tokens, then the whole kept blocks of experts "
            f"0..{orc.half - 1}; odd steps: experts {orc.half}..{wl.E - 1} and the combine), "
            f"so two steps are one moe_forward; rank 0 only")
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total * 1e3 / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, C, world),
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": desc, "extrapolated": False},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "step_seconds": {"min": round(min(secs), 3), "max": round(max(secs), 3)},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral", choices=sorted(WORKLOADS))
    ap.add_argument("--extra-workloads", default=",".join(EXTRA_WORKLOADS),
                    help="comma-separated workloads measured after the headline one and "
                         "reported in the line's `workloads` record ('none' to skip)")
    ap.add_argument("--gemm", choices=["auto", "single", "pair", "split", "pair_t", "mixed"],
                    default="auto",
                    help="expert GEMM kernels: one CTA per 128-row tile, CTA pairs per "
                         "256-row tile, pairs for whole 256-row tiles + one CTA for the "
                         "rest, pairs with the tokens on the MMA's N side, pairs for whole "
                         "tiles + transposed pair tiles for the rest in one launch, or the "
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
