"""Time one stage of the MoE layer forward on its own, with only that stage's buffers.

    python -m routing_dispatch_expert_04_b300.stage_bench --stage dispatch --workload long \
        [--tokens T] [--iters N] [--warmup W]

Stages: ``route`` (router Linear + softmax/top-K), ``dispatch`` (histogram/scan/capacity
+ row permutation), ``combine`` (weighted gather back to token order).  The routing that
feeds dispatch and combine is computed by the library from the workload's seeded
inputs; the expert outputs that combine reads are seeded N(0, 1) values (combine's cost
does not depend on them).  No expert weights are allocated, so a stage of a large
workload fits in a few GB of device memory -- the size a profiler capture should use.

L2 is flushed (a 512 MiB device write) before every timed launch.  Prints one JSON line
with the median time, the stage's algorithmic bytes and the achieved GB/s.
"""

from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import native as N
from .workloads import WORKLOADS, make_inputs

L2_FLUSH_BYTES = 512 << 20


def stage_bytes(stage, wl, T, R, t_active, b):
    """Bytes the stage must move at least (inputs read once, outputs written once)."""
    A = T * wl.K
    if stage == "route":
        return T * wl.d * b + wl.E * wl.d * b + T * wl.E * 4 * 2 + A * 8
    if stage == "dispatch":
        return t_active * wl.d * b + R * wl.d * b + A * 12 + R * 4
    if stage == "combine":
        yb = 2 if wl.dtype == "bf16" else 4  # expert outputs: fp16 for bf16 layers
        return R * wl.d * yb + T * wl.d * b + A * 8
    raise ValueError(stage)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--stage", required=True, choices=["route", "dispatch", "combine"])
    ap.add_argument("--workload", default="long", choices=sorted(WORKLOADS))
    ap.add_argument("--tokens", type=int, default=0, help="override the token count T")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    args = ap.parse_args()

    wl = WORKLOADS[args.workload]
    if args.tokens > 0:
        wl = wl.scaled(args.tokens)
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
    elif args.stage == "dispatch":
        x_perm = torch.empty((rows_cap, d), dtype=x.dtype, device=dev)

        def run():
            N.dispatch(cfg, x, ids, counts, offsets, slot, src, x_perm, ws)
    else:
        g = torch.Generator(device=dev)
        g.manual_seed(1)
        y_perm = torch.randn((rows_cap, d), generator=g, device=dev, dtype=f32)
        if wl.dtype == "bf16":
            y_perm = y_perm.half()  # expert outputs of bf16 layers are fp16
        y = torch.empty((T, d), dtype=x.dtype, device=dev)

        def run():
            N.combine(cfg, y_perm, slot, w, None, y)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.zero_()
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
    st = N.sync_status(ws)
    if st != 0:
        raise N.MoeError(args.stage, st)
    b = 2 if wl.dtype == "bf16" else 4
    nbytes = stage_bytes(args.stage, wl, T, R, t_active, b)
    med = statistics.median(ms)
    print(json.dumps({"stage": args.stage, "workload": wl.name, "T": T, "rows_kept": R,
                      "tokens_with_kept_rows": t_active, "ms_median": round(med, 5),
                      "bytes": nbytes, "gbs": round(nbytes / (med * 1e-3) / 1e9, 1),
                      "iters": args.iters}), flush=True)


if __name__ == "__main__":
    main()
