"""Time one stage of the MoE layer forward on its own, with only that stage's buffers.

    python -m routing_dispatch_expert_04_b300.stage_bench --stage dispatch --workload long \
        [--tokens T] [--iters N] [--warmup W]

Stages: ``route`` (router Linear + softmax/top-K), ``route_plan`` (the same with the
dispatch plan in the routing kernel's tail), ``dispatch`` (histogram/scan/capacity + row
permutation), ``dispatch_planned`` (slot/src and the row copy after ``route_plan``),
``combine`` (weighted gather back to token order), ``expert_up`` and
``expert_down`` (the two grouped expert GEMMs, ``--experts bf16|e4m3``).  The routing that
feeds the later stages is computed by the library from the workload's seeded inputs; the
rows the GEMMs and the combine read are seeded values of the layer's scale (their cost
does not depend on them).  Only the stage's own weights are allocated (none for routing,
dispatch and combine), so most stages fit in a few GB of device memory -- the size a
profiler capture should use.

L2 is flushed (a 512 MiB device write) before every timed launch.  Prints one JSON line
with the median time, the stage's algorithmic bytes and the achieved GB/s (and TFLOP/s
for the GEMMs).  With ``--profile-range`` one more launch of the stage runs between
cudaProfilerStart and cudaProfilerStop, for a profiler's range replay: the counters then
cover the whole stage, for the split plan both of its GEMM kernels (launched concurrently
as in the layer; whether a profiler lets them overlap is the profiler's choice).  With
``--graph`` the stage is captured in a CUDA graph after the warm-up, and the timed and
profiled launches are replays of it, as in the layer's step.  ``--tokens`` and
``--num-experts`` shrink the workload (same d, F, K and routing recipe) for profiler
captures that must stay a few GB on the device.
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import statistics
import time

import torch

from . import native as N
from .workloads import WORKLOADS, make_inputs

L2_FLUSH_BYTES = 512 << 20


def stage_bytes(stage, wl, T, R, t_active, b, experts="bf16"):
    """Bytes the stage must move at least (inputs read once, outputs written once)."""
    A = T * wl.K
    if stage in ("expert_up", "expert_down"):
        wb = 1 if experts == "e4m3" else 2          # weight element bytes
        ab = 1 if experts == "e4m3" else (b if stage == "expert_up" else 2)
        n_in, n_out = (wl.d, wl.F) if stage == "expert_up" else (wl.F, wl.d)
        return wl.E * wl.F * wl.d * wb + R * n_in * ab + R * n_out * 2
    if stage == "route":
        return T * wl.d * b + wl.E * wl.d * b + T * wl.E * 4 * 2 + A * 8
    if stage == "route_plan":  # + the positions written
        return T * wl.d * b + wl.E * wl.d * b + T * wl.E * 4 * 2 + A * 12
    if stage == "dispatch_planned":  # ids and positions read, slot written, rows copied
        return t_active * wl.d * b + R * wl.d * b + A * 12 + R * 4
    if stage == "dispatch":
        return t_active * wl.d * b + R * wl.d * b + A * 12 + R * 4
    if stage == "combine":
        yb = 2 if wl.dtype == "bf16" else 4  # expert outputs: fp16 for bf16 layers
        return R * wl.d * yb + T * wl.d * b + A * 8
    raise ValueError(stage)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--stage", required=True,
                    choices=["route", "route_plan", "dispatch", "dispatch_planned", "combine",
                             "expert_up", "expert_down"])
    ap.add_argument("--experts", choices=["bf16", "e4m3"], default="bf16",
                    help="operand format of the expert GEMM stages")
    ap.add_argument("--gemm", choices=["auto", "single", "pair", "split", "pair_t", "mixed"],
                    default="auto",
                    help="expert-GEMM plan (moe_set_gemm_pairing) for the GEMM stages")
    ap.add_argument("--sustain", type=float, default=0.0,
                    help="also loop the stage back to back for this many seconds and report "
                         "its mean time and the memory controller's busy fraction (nvidia-smi)")
    ap.add_argument("--profile-range", action="store_true",
                    help="run one more launch between cudaProfilerStart/Stop")
    ap.add_argument("--library", action="store_true",
                    help="GEMM stages: time cuBLAS (torch.bmm) on the same expert GEMMs instead "
                         "of this library's kernels; needs equal rows in every expert")
    ap.add_argument("--graph", action="store_true",
                    help="capture the stage in a CUDA graph after the warm-up and time (and "
                         "profile) its replays, as the layer's step runs it")
    ap.add_argument("--workload", default="long", choices=sorted(WORKLOADS))
    ap.add_argument("--tokens", type=int, default=0, help="override the token count T")
    ap.add_argument("--num-experts", type=int, default=0,
                    help="override the routed expert count E (a smaller case of the same "
                         "layer, e.g. for a profiler capture that must stay a few GB)")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    args = ap.parse_args()

    N.set_gemm_pairing({"auto": N.GEMM_AUTO, "single": N.GEMM_SINGLE, "pair": N.GEMM_PAIR,
                        "split": N.GEMM_SPLIT, "pair_t": N.GEMM_PAIR_T,
                        "mixed": N.GEMM_MIXED}[args.gemm])
    wl = WORKLOADS[args.workload]
    if args.tokens > 0:
        wl = wl.scaled(args.tokens)
    if args.num_experts > 0:
        if args.num_experts < wl.K:
            raise SystemExit(f"--num-experts must be at least K = {wl.K}")
        wl = dataclasses.replace(wl, name=f"{wl.name}_E{args.num_experts}", E=args.num_experts)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = make_inputs(wl, dev, seed=0, weights=False)
    cfg = N.make_config(wl.T, wl.d, wl.E, wl.K, wl.F, wl.dtype,
                        N.capacity(wl.T, wl.E, wl.capacity_factor), False, wl.alpha)
    T, E, K, d = wl.T, wl.E, wl.K, wl.d
    rows_cap = max(N.rows_capacity(cfg), 1)
    i32, f32 = torch.int32, torch.float32
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device=dev)
    logits = torch.empty((T, E), dtype=f32, device=dev)
    ids = torch.empty((T, K), dtype=i32, device=dev)
    w = torch.empty((T, K), dtype=f32, device=dev)
    counts = torch.empty(E, dtype=i32, device=dev)
    offsets = torch.empty(E + 1, dtype=i32, device=dev)
    slot = torch.empty((T, K), dtype=i32, device=dev)
    src = torch.empty(rows_cap, dtype=i32, device=dev)
    x = inp["x"]
    N.route(cfg, x, inp["w_r"], inp["b_r"], logits, ids, w, ws)
    N.dispatch(cfg, None, ids, counts, offsets, slot, src, None, ws)
    st = N.sync_status(ws)
    if st != 0:
        raise N.MoeError("routing", st)
    R = int(offsets[-1].item())
    t_active = int((slot >= 0).any(dim=1).sum().item())

    if args.stage == "route":
        def run():
            N.route(cfg, x, inp["w_r"], inp["b_r"], logits, ids, w, ws)
    elif args.stage == "route_plan":
        def run():
            N.route_plan(cfg, x, inp["w_r"], inp["b_r"], None, logits, ids, w, counts, offsets, ws)
    elif args.stage == "dispatch_planned":
        x_perm = torch.empty((rows_cap, d), dtype=x.dtype, device=dev)
        N.route_plan(cfg, x, inp["w_r"], inp["b_r"], None, logits, ids, w, counts, offsets, ws)

        def run():
            N.dispatch_planned(cfg, x, ids, offsets, slot, src, x_perm, ws)
    elif args.stage == "dispatch":
        x_perm = torch.empty((rows_cap, d), dtype=x.dtype, device=dev)

        def run():
            N.dispatch(cfg, x, ids, counts, offsets, slot, src, x_perm, ws)
    elif args.stage == "combine":
        g = torch.Generator(device=dev)
        g.manual_seed(1)
        y_perm = torch.randn((rows_cap, d), generator=g, device=dev, dtype=f32)
        if wl.dtype == "bf16":
            y_perm = y_perm.half()  # expert outputs of bf16 layers are fp16
        y = torch.empty((T, d), dtype=x.dtype, device=dev)

        def run():
            N.combine(cfg, y_perm, slot, w, None, y)
    else:
        run = _gemm_stage(args.stage, args.experts, wl, cfg, x, ids, counts, offsets, slot,
                          src, ws, rows_cap, dev, args.library)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.zero_()
        run()
    torch.cuda.synchronize()
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run()
        run = graph.replay
        run()
        torch.cuda.synchronize()
    ms = []
    stream = torch.cuda.current_stream()
    for _ in range(args.iters):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        z.record(stream)
        z.synchronize()
        ms.append(a.elapsed_time(z))
    sustained = _sustain(run, args.sustain) if args.sustain > 0 else None
    if args.profile_range:
        flush.zero_()
        torch.cuda.synchronize()
        torch.cuda.cudart().cudaProfilerStart()
        run()
        torch.cuda.synchronize()
        torch.cuda.cudart().cudaProfilerStop()
    st = N.sync_status(ws)
    if st != 0:
        raise N.MoeError(args.stage, st)
    b = 2 if wl.dtype == "bf16" else 4
    nbytes = stage_bytes(args.stage, wl, T, R, t_active, b, args.experts)
    med = statistics.median(ms)
    line = {"stage": args.stage, "workload": wl.name, "T": T, "rows_kept": R,
            "tokens_with_kept_rows": t_active, "ms_median": round(med, 5),
            "bytes": nbytes, "gbs": round(nbytes / (med * 1e-3) / 1e9, 1), "iters": args.iters}
    if sustained is not None:
        line.update(sustained)
    if args.stage in ("expert_up", "expert_down"):
        flops = 2.0 * R * wl.d * wl.F
        line.update({"experts": args.experts, "gemm": "cublas bmm" if args.library else args.gemm,
                     "flops": flops,
                     "tflops": round(flops / (med * 1e-3) / 1e12, 1)})
    print(json.dumps(line), flush=True)


def _sustain(run, seconds):
    """Loop the stage back to back (no L2 flush) for `seconds` while nvidia-smi samples the
    memory controller's busy fraction every 100 ms: the fraction of time the device memory
    was being read or written, which scales with the DRAM bytes per second even where a
    profiler would serialise concurrent kernels."""
    import subprocess
    for _ in range(5):
        run()
    torch.cuda.synchronize()
    # nvidia-smi is given the device's UUID: its own indices need not follow the CUDA
    # ordinals (CUDA_VISIBLE_DEVICES, a leased GPU of a shared machine)
    uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    smi = subprocess.Popen(["nvidia-smi", f"--id={uuid}",
                            "--query-gpu=utilization.memory,clocks.sm,clocks.mem",
                            "--format=csv,noheader,nounits", "-lms", "100"],
                           stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    t0, n = time.time(), 0
    a.record()
    while time.time() - t0 < seconds:
        for _ in range(20):
            run()
        n += 20
        torch.cuda.synchronize()
    z.record()
    z.synchronize()
    smi.terminate()
    rows = []
    for line in smi.communicate()[0].splitlines()[3:-2]:  # drop the ramp at both ends
        parts = [p.strip() for p in line.split(",")]
        if len(parts) == 3 and all(p.isdigit() for p in parts):
            rows.append([int(p) for p in parts])

    def median(col):
        v = sorted(r[col] for r in rows)
        return v[len(v) // 2] if v else None
    # utilization.memory is the fraction of sample periods the memory controller was busy,
    # in whole percent: an indirect, time-based figure, not a byte count
    return {"sustained_ms": round(a.elapsed_time(z) / n, 5), "sustained_launches": n,
            "gpu": uuid, "mem_busy_pct_median": median(0), "sm_mhz_median": median(1),
            "mem_mhz_median": median(2), "mem_busy_samples": len(rows)}


def _gemm_stage(stage, experts, wl, cfg, x, ids, counts, offsets, slot, src, ws, rows_cap, dev,
                library=False):
    """Buffers and launch of one expert-GEMM stage over the workload's kept rows: A is the
    dispatched token rows (expert_up) or seeded fp16 rows of the scale of h (expert_down);
    the weights are seeded N(0, 1/fan_in) values (W2 in fp16, as the layer stores it for
    bf16 layers).  E4M3 stages quantise A and the weights once, outside the timed launch.
    ``library``: the same GEMMs (same operands, flops and bytes, no GELU) as one cuBLAS
    batched GEMM, torch.bmm over the experts, for comparison; every expert must hold the
    same number of rows."""
    E, d, F = wl.E, wl.d, wl.F
    g = torch.Generator(device=dev)
    g.manual_seed(2)
    if stage == "expert_up":
        a = torch.empty((rows_cap, d), dtype=x.dtype, device=dev)
        N.dispatch(cfg, x, ids, counts, offsets, slot, src, a, ws)
        w = (torch.randn((E, F, d), generator=g, device=dev) * d ** -0.5).to(x.dtype)
        out = torch.empty((rows_cap, F), dtype=torch.float16, device=dev)
        n_in, n_out = d, F
    else:
        a = (torch.randn((rows_cap, F), generator=g, device=dev) * 0.5).half()
        w = (torch.randn((E, d, F), generator=g, device=dev) * F ** -0.5).half()
        out = torch.empty((rows_cap, d), dtype=torch.float16, device=dev)
        n_in, n_out = F, d
    if library:
        cnt = torch.diff(offsets)
        per = int(cnt[0].item())
        if experts != "bf16" or not bool((cnt == per).all().item()) or per == 0:
            raise SystemExit("--library needs bf16 experts with equal rows per expert")
        a3 = a[:E * per].view(E, per, n_in)
        wt = w.transpose(1, 2)
        o3 = torch.empty((E, per, n_out), dtype=a.dtype, device=dev)

        def run():
            torch.bmm(a3, wt, out=o3)
        return run
    if experts == "bf16":
        fn = N.expert_up if stage == "expert_up" else N.expert_down

        def run():
            fn(cfg, a, offsets, E, rows_cap, w, out, ws)
        return run
    aq = torch.empty((rows_cap, n_in), dtype=torch.uint8, device=dev)
    sa = torch.empty(rows_cap, dtype=torch.float32, device=dev)
    wq = torch.empty((E * n_out, n_in), dtype=torch.uint8, device=dev)
    sw = torch.empty(E * n_out, dtype=torch.float32, device=dev)
    N.quantize_e4m3(a, aq, sa)
    N.quantize_e4m3(w.reshape(E * n_out, n_in), wq, sw)
    del w
    if stage == "expert_up":
        def run():
            N.expert_up_e4m3(cfg, aq, sa, None, offsets, E, rows_cap, wq, sw, out, ws)
    else:
        def run():
            N.expert_down_e4m3(cfg, aq, sa, offsets, E, rows_cap, wq, sw, out, ws)
    return run


if __name__ == "__main__":
    main()
