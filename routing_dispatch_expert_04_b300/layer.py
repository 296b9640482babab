"""One MoE FFN layer forward on one GPU, driven through the C ABI.

:class:`MoELayer` owns the device buffers of one layer shape and issues, on one CUDA
stream and without any host synchronisation, the calls of the layer in the order the
expert-parallelism pages give it ("Expert Parallelism (EP)", "Key math / How it
works": route, dispatch, expert GEMMs, combine), followed by the aux statistics:

    moe_route -> moe_dispatch -> moe_expert_up -> moe_expert_down
      [-> shared expert: moe_expert_up / moe_expert_down over all tokens]
      -> moe_combine -> moe_aux_stats

With token-major drop order (the default) the first two calls are moe_route_plan (the
routing kernel ranks the assignments and counts them per block, a small scan turns the
counts into per-block bases, counts and offsets) and moe_dispatch_planned (slot/src and
the row copy).

Buffers are torch tensors (device memory only); every step runs in the library's
kernels.
"""

from __future__ import annotations

import torch

from . import native as N


class MoELayer:
    def __init__(self, T, d, E, K, F, dtype, capacity_factor, alpha, w_r, b_r, w1, w2,
                 w1s=None, w2s=None, renormalize=False, device="cuda", overlap=True,
                 drop_order="token", capacity_mode="tokens", sel_bias=None,
                 fused_dispatch=False, experts="bf16", shared_sms=0, plan_in_route=True):
        """``plan_in_route``: True (default): with token-major drop order (the default) the
        routing step also computes the dispatch plan -- counts, offsets and every
        assignment's rank and block base (moe_route_plan) -- and the dispatch step only
        builds slot/src and copies the rows (moe_dispatch_planned); False: the plan runs in
        the dispatch step (moe_route, then moe_dispatch's own scan), as slot-major order
        always does.  Routing plus dispatch on B300, planned vs not: Mixtral shape 45 vs
        49 us, Qwen3 78 vs 78, DeepSeek-V3 265 vs 266, 64K tokens 260 vs 262.
        ``shared_sms``: with a shared expert and ``overlap``, 0 (default) runs the shared
        expert beside routing and dispatch; n > 0 runs it on n SMs beside the routed expert
        GEMMs, which then get the other SMs (moe_set_gemm_sms).
        ``fused_dispatch``: the first expert Linear gathers its rows from x while loading
        them (moe_expert_up_gather), so the dispatch step writes only the routing plan;
        by default the dispatch copies the rows into x_perm first, which measures faster
        on B300 (TMA row gathers move 512 bytes per instruction).
        ``experts``: "bf16" (default) or "e4m3": the FP8 variant of the expert Linears
        (per-row E4M3 operands, moe_expert_up_e4m3 / moe_expert_down_e4m3); bf16 layers
        only.
        ``drop_order``: "token" (flat order) or "slot" (first choices first) decides which
        assignments a full expert drops.  ``capacity_mode``: "tokens" gives the capacity as
        printed, C = floor(T/E * cf); "assignments" counts top-K assignments,
        C = floor(T*K/E * cf).  ``sel_bias``: optional [E] fp32 device tensor, a
        selection-only expert bias (see :meth:`adjust_selection_bias`)."""
        if capacity_mode == "tokens":
            C = N.capacity(T, E, capacity_factor)
        elif capacity_mode == "assignments":
            C = N.capacity_assignments(T, E, K, capacity_factor)
        else:
            raise ValueError(capacity_mode)
        self.cfg = N.make_config(T, d, E, K, F, dtype, C, renormalize, alpha, drop_order)
        self.planned = bool(plan_in_route) and drop_order == "token"
        self.sel_bias = sel_bias
        self.T, self.d, self.E, self.K, self.F = T, d, E, K, F
        self.dtype = torch.float32 if dtype == "f32" else torch.bfloat16
        self.device = torch.device(device)
        self.w_r, self.b_r, self.w1 = w_r, b_r, w1
        self.w1s = w1s
        self.rows_cap = N.rows_capacity(self.cfg)
        R = max(self.rows_cap, 1)
        dev, dt = self.device, self.dtype
        i32, f32 = torch.int32, torch.float32
        self.ws = torch.zeros(N.workspace_size(self.cfg), dtype=torch.uint8, device=dev)
        # the shared expert runs beside routing and the routed experts on the side stream,
        # and calls that can run concurrently need separate workspaces
        self.ws_s = (torch.zeros(N.workspace_size(self.cfg), dtype=torch.uint8, device=dev)
                     if w1s is not None else None)
        self.logits = torch.empty((T, E), dtype=f32, device=dev)
        self.ids = torch.empty((T, K), dtype=i32, device=dev)
        self.w = torch.empty((T, K), dtype=f32, device=dev)
        self.counts = torch.empty(E, dtype=i32, device=dev)
        self.offsets = torch.empty(E + 1, dtype=i32, device=dev)
        self.slot = torch.empty((T, K), dtype=i32, device=dev)
        self.src = torch.empty(R, dtype=i32, device=dev)
        self.fused_dispatch = fused_dispatch
        self.x_perm = None if fused_dispatch else torch.empty((R, d), dtype=dt, device=dev)
        # the intermediate activation is fp16 for bf16 layers (see moe_expert_up)
        self.h_dtype = torch.float16 if dtype == "bf16" else torch.float32
        self.h = torch.empty((R, F), dtype=self.h_dtype, device=dev)
        # expert outputs: fp16 for bf16 layers (see moe_expert_down), fp32 otherwise
        self.y_perm = torch.empty((R, d), dtype=self.h_dtype, device=dev)
        self.y = torch.empty((T, d), dtype=dt, device=dev)
        self.f = torch.empty(E, dtype=f32, device=dev)
        self.P = torch.empty(E, dtype=f32, device=dev)
        self.l_aux = torch.empty(1, dtype=f32, device=dev)
        # independent work goes on a second stream: the shared expert (needs only x) runs
        # beside routing and the routed experts, the aux statistics (need only the routing
        # results) beside the expert GEMMs
        self.overlap = overlap
        self.shared_sms = int(shared_sms) if w1s is not None else 0
        self.side = torch.cuda.Stream(device=dev) if overlap else None
        self.graph = None
        if experts not in ("bf16", "e4m3") or (experts == "e4m3" and dtype != "bf16"):
            raise ValueError(f"experts={experts!r} with dtype={dtype!r}")
        self.experts = experts
        self.shared = w1s is not None
        if self.shared:
            self.shared_offsets = torch.tensor([0, T], dtype=i32, device=dev)
            self.h_s = torch.empty((max(T, 1), F), dtype=self.h_dtype, device=dev)
            self.y_s = torch.empty((max(T, 1), d), dtype=self.h_dtype, device=dev)
        if experts == "bf16":
            self.w2 = self._down_weights(w2)
            self.w2s = self._down_weights(w2s) if self.shared else None
            return
        # E4M3 experts: weights quantised once per output channel, activation buffers
        u8 = torch.uint8
        self.w1q, self.w1_sc = self._quantized(w1.reshape(E * F, d))
        self.w2q, self.w2_sc = self._quantized(w2.reshape(E * d, F))
        xrows = T if fused_dispatch else R
        self.xq = torch.empty((max(xrows, 1), d), dtype=u8, device=dev)
        self.x_sc = torch.empty(max(xrows, 1), dtype=f32, device=dev)
        self.hq = torch.empty((R, F), dtype=u8, device=dev)
        self.h_sc = torch.empty(R, dtype=f32, device=dev)
        if self.shared:
            self.w1sq, self.w1s_sc = self._quantized(w1s.reshape(F, d))
            self.w2sq, self.w2s_sc = self._quantized(w2s.reshape(d, F))
            self.xsq = torch.empty((max(T, 1), d), dtype=u8, device=dev)
            self.xs_sc = torch.empty(max(T, 1), dtype=f32, device=dev)
            self.hsq = torch.empty((max(T, 1), F), dtype=u8, device=dev)
            self.hs_sc = torch.empty(max(T, 1), dtype=f32, device=dev)

    def _quantized(self, w):
        codes = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
        scales = torch.empty(w.shape[0], dtype=torch.float32, device=w.device)
        N.quantize_e4m3(w, codes, scales)
        return codes, scales

    def _down_weights(self, w2):
        """Second-Linear weights in the operand type the kernels take: an fp16 copy of bf16
        weights (converted once by the library), fp32 weights as they are."""
        if w2.dtype != torch.bfloat16:
            return w2
        out = torch.empty(w2.shape, dtype=torch.float16, device=w2.device)
        N.bf16_to_f16(w2, out, self.ws)
        st = N.sync_status(self.ws)
        if st != 0:
            raise N.MoeError("moe_bf16_to_f16", st)
        return out

    @classmethod
    def from_workload(cls, wl, inputs, device="cuda", renormalize=False, overlap=True,
                      drop_order="token", capacity_mode="tokens", sel_bias=None,
                      fused_dispatch=False, experts="bf16", shared_sms=0, plan_in_route=True):
        return cls(wl.T, wl.d, wl.E, wl.K, wl.F, wl.dtype, wl.capacity_factor, wl.alpha,
                   inputs["w_r"], inputs["b_r"], inputs["w1"], inputs["w2"],
                   inputs.get("w1s"), inputs.get("w2s"), renormalize=renormalize, device=device,
                   overlap=overlap, drop_order=drop_order, capacity_mode=capacity_mode,
                   sel_bias=sel_bias, fused_dispatch=fused_dispatch, experts=experts,
                   shared_sms=shared_sms, plan_in_route=plan_in_route)

    # ---------------------------------------------------------------- stages
    def route(self, x, stream=None, logits_in=None):
        """Router + softmax + top-K (and, with ``planned``, the dispatch plan).  With
        ``logits_in`` (fp32 [T,E]) the router Linear is skipped and those logits drive the
        routing."""
        if logits_in is not None:
            self.logits.copy_(logits_in)
            x, w_r, b_r = None, None, None
        else:
            w_r, b_r = self.w_r, self.b_r
        if self.planned:
            N.route_plan(self.cfg, x, w_r, b_r, self.sel_bias, self.logits, self.ids, self.w,
                         self.counts, self.offsets, self.ws, stream)
        elif self.sel_bias is None:
            N.route(self.cfg, x, w_r, b_r, self.logits, self.ids, self.w, self.ws, stream)
        else:
            N.route_select_bias(self.cfg, x, w_r, b_r, self.sel_bias, self.logits, self.ids,
                                self.w, self.ws, stream)

    def adjust_selection_bias(self, gamma: float, stream=None):
        """After a forward: nudge the selection-only bias toward balance from this step's
        pre-drop counts (lower over-loaded experts, raise under-loaded ones by gamma)."""
        if self.sel_bias is None:
            raise ValueError("the layer has no selection bias")
        N.adjust_select_bias(self.cfg, self.counts, self.sel_bias, gamma, stream)

    def dispatch(self, x, stream=None):
        """Routing plan (counts, offsets, slot, src); with the unfused dispatch also the
        row copy into x_perm."""
        copy = x is not None and not self.fused_dispatch
        if self.planned:
            N.dispatch_planned(self.cfg, x if copy else None, self.ids, self.offsets, self.slot,
                               self.src, self.x_perm if copy else None, self.ws, stream)
            return
        N.dispatch(self.cfg, x if copy else None, self.ids, self.counts, self.offsets, self.slot,
                   self.src, self.x_perm if copy else None, self.ws, stream)

    def experts_up(self, x, stream=None):
        if self.experts == "e4m3":
            kept = self.offsets[self.E:]  # rows actually packed (device)
            if self.fused_dispatch:
                N.quantize_e4m3(x, self.xq, self.x_sc, None, stream)
                N.expert_up_e4m3(self.cfg, self.xq, self.x_sc, self.src, self.offsets, self.E,
                                 self.rows_cap, self.w1q, self.w1_sc, self.h, self.ws, stream)
            else:
                N.quantize_e4m3(self.x_perm, self.xq, self.x_sc, kept, stream)
                N.expert_up_e4m3(self.cfg, self.xq, self.x_sc, None, self.offsets, self.E,
                                 self.rows_cap, self.w1q, self.w1_sc, self.h, self.ws, stream)
            return
        if self.fused_dispatch:
            N.expert_up_gather(self.cfg, x, self.src, self.offsets, self.E, self.rows_cap,
                               self.w1, self.h, self.ws, stream)
        else:
            N.expert_up(self.cfg, self.x_perm, self.offsets, self.E, self.rows_cap, self.w1,
                        self.h, self.ws, stream)

    def experts_down(self, stream=None):
        if self.experts == "e4m3":
            N.quantize_e4m3(self.h, self.hq, self.h_sc, self.offsets[self.E:], stream)
            N.expert_down_e4m3(self.cfg, self.hq, self.h_sc, self.offsets, self.E, self.rows_cap,
                               self.w2q, self.w2_sc, self.y_perm, self.ws, stream)
            return
        N.expert_down(self.cfg, self.h, self.offsets, self.E, self.rows_cap, self.w2, self.y_perm,
                      self.ws, stream)

    def shared_expert(self, x, stream=None):
        if self.experts == "e4m3":
            N.quantize_e4m3(x, self.xsq, self.xs_sc, None, stream)
            N.expert_up_e4m3(self.cfg, self.xsq, self.xs_sc, None, self.shared_offsets, 1, self.T,
                             self.w1sq, self.w1s_sc, self.h_s, self.ws_s, stream)
            N.quantize_e4m3(self.h_s, self.hsq, self.hs_sc, None, stream)
            N.expert_down_e4m3(self.cfg, self.hsq, self.hs_sc, self.shared_offsets, 1, self.T,
                               self.w2sq, self.w2s_sc, self.y_s, self.ws_s, stream)
            return
        N.expert_up(self.cfg, x, self.shared_offsets, 1, self.T, self.w1s, self.h_s, self.ws_s,
                    stream)
        N.expert_down(self.cfg, self.h_s, self.shared_offsets, 1, self.T, self.w2s, self.y_s,
                      self.ws_s, stream)

    def combine(self, stream=None, y=None):
        N.combine(self.cfg, self.y_perm, self.slot, self.w, self.y_s if self.shared else None,
                  self.y if y is None else y, stream)

    def aux(self, stream=None, stats=None):
        """stats: optional (f, P, l_aux) output tensors instead of the layer's own."""
        f, P, l_aux = (self.f, self.P, self.l_aux) if stats is None else stats
        N.aux_stats(self.cfg, self.counts, self.ws, f, P, l_aux, stream)

    # ---------------------------------------------------------------- whole layer
    def stage_names(self):
        """Stages timed on the main stream, in order (with overlap the shared expert and
        the aux statistics run on the side stream and are not separate stages)."""
        names = ["route", "dispatch", "expert_up", "expert_down"]
        if self.overlap:
            return names + ["combine"]
        if self.shared:
            names.append("shared_expert")
        return names + ["combine", "aux"]

    def forward(self, x, stream=None, logits_in=None, marks=None, y=None, stats=None):
        """Enqueue the whole layer; returns the output buffer (``self.y`` unless ``y`` is
        given; ``stats`` = (f, P, l_aux) redirects the aux statistics the same way).

        With ``overlap`` the work goes on the current stream plus the layer's side stream,
        forked and joined with events (so it can be captured in a CUDA graph); otherwise
        everything goes on ``stream``.  ``marks``: optional len(stage_names()) + 1 CUDA
        events recorded on the main stream before each stage and after the last one."""
        def mark(i):
            if marks is not None:
                marks[i].record()
        if not self.overlap:
            mark(0)
            self.route(x, stream, logits_in)
            mark(1)
            self.dispatch(x, stream)
            mark(2)
            self.experts_up(x, stream)
            mark(3)
            self.experts_down(stream)
            i = 4
            if self.shared:
                mark(i)
                self.shared_expert(x, stream)
                i += 1
            mark(i)
            self.combine(stream, y)
            mark(i + 1)
            self.aux(stream, stats)
            mark(i + 2)
            return self.y if y is None else y
        main = torch.cuda.current_stream()
        side = self.side
        beside_gemms = self.shared and self.shared_sms > 0
        if self.shared and not beside_gemms:
            fork = torch.cuda.Event()
            fork.record(main)
            side.wait_event(fork)
            with torch.cuda.stream(side):
                self.shared_expert(x)
        mark(0)
        self.route(x, None, logits_in)
        mark(1)
        self.dispatch(x)
        routed = torch.cuda.Event()
        routed.record(main)
        side.wait_event(routed)
        try:
            with torch.cuda.stream(side):
                # the aux statistics share the workspace with the expert GEMMs running on
                # the main stream: moe_aux_stats may (it touches only its own region of
                # the workspace, the GEMMs only the status word)
                self.aux(None, stats)
                if beside_gemms:  # on its own SMs, beside the routed expert GEMMs
                    N.set_gemm_sms(self.shared_sms)
                    self.shared_expert(x)
            joined = torch.cuda.Event()
            joined.record(side)
            if beside_gemms:
                N.set_gemm_sms(max(N.num_sms(self.device) - self.shared_sms, 2))
            mark(2)
            self.experts_up(x)
            mark(3)
            self.experts_down()
            mark(4)
        finally:
            N.set_gemm_sms(0)
        main.wait_event(joined)
        self.combine(None, y)
        mark(5)
        return self.y if y is None else y

    def capture(self, x, marks=None):
        """Record the whole forward on the input buffer ``x`` as one CUDA graph, so a step
        costs one launch instead of one per kernel.  ``marks`` (events created with
        ``external=True``) become timing nodes inside the graph.  Returns the number of
        library kernels one replay launches."""
        self.forward(x)            # first use of every kernel happens outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        before = N.launch_count()
        with torch.cuda.graph(graph):
            self.forward(x, marks=marks)
        self.graph = graph
        self.graph_x = x
        self.graph_kernels = N.launch_count() - before
        return self.graph_kernels

    def replay(self):
        """Run the captured forward on the current stream."""
        self.graph.replay()
        return self.y

    def forward_host(self, x_host, y_host, x_dev=None, stream=None):
        """End-to-end call with host buffers: copy x (pinned host) in, run the layer (the
        captured graph when there is one, into its input buffer), copy y back into pinned
        host memory, all on the current stream."""
        if self.graph is not None:
            self.graph_x.copy_(x_host, non_blocking=True)
            self.replay()
        else:
            x_dev.copy_(x_host, non_blocking=True)
            self.forward(x_dev, stream)
        y_host.copy_(self.y, non_blocking=True)
        return y_host

    def check_device_status(self):
        for ws in (self.ws, self.ws_s):
            if ws is None:
                continue
            st = N.sync_status(ws)
            if st != 0:
                raise N.MoeError("moe_sync_status", st)


class HostStream:
    """Layer forwards on batches that live in pinned host memory, pipelined.

    Batch i is uploaded on a copy stream, run through the layer (one CUDA-graph replay)
    on the compute stream, and its output and aux statistics are downloaded on a second
    copy stream.  Two device input slots and two output slots alternate, so batch i+1's
    upload and batch i-1's download overlap batch i's compute; events order every reuse
    of a slot.  All work is enqueued; :meth:`run` returns without synchronising."""

    def __init__(self, layer: MoELayer, x_like):
        self.layer = layer
        dev = layer.device
        E = layer.E
        self.xb = [x_like.clone() for _ in range(2)]  # valid data for the warm-up forward
        self.yb = [torch.empty_like(layer.y) for _ in range(2)]
        self.sb = [(torch.empty(E, dtype=torch.float32, device=dev),
                    torch.empty(E, dtype=torch.float32, device=dev),
                    torch.empty(1, dtype=torch.float32, device=dev)) for _ in range(2)]
        self.h2d = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.uploaded = [torch.cuda.Event() for _ in range(2)]
        self.downloaded = [torch.cuda.Event() for _ in range(2)]
        self.graphs = []
        for s in range(2):
            layer.forward(self.xb[s], y=self.yb[s], stats=self.sb[s])  # outside capture first
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                layer.forward(self.xb[s], y=self.yb[s], stats=self.sb[s])
            self.graphs.append(g)
        self.i = 0

    def run(self, x_host, y_host, stats_host=None):
        """Enqueue one batch: x_host (pinned, like x) in, y_host (pinned, like y) and
        optionally stats_host (pinned fp32 [2E+1]: f, P, l_aux) out."""
        s = self.i & 1
        self.i += 1
        main = torch.cuda.current_stream()
        with torch.cuda.stream(self.h2d):
            self.h2d.wait_event(self.computed[s])        # the slot's previous batch is done
            self.xb[s].copy_(x_host, non_blocking=True)
            self.uploaded[s].record(self.h2d)
        main.wait_event(self.uploaded[s])
        main.wait_event(self.downloaded[s])              # the slot's previous output is out
        self.graphs[s].replay()
        self.computed[s].record(main)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.computed[s])
            y_host.copy_(self.yb[s], non_blocking=True)
            if stats_host is not None:
                E = self.layer.E
                f, P, l_aux = self.sb[s]
                stats_host[:E].copy_(f, non_blocking=True)
                stats_host[E:2 * E].copy_(P, non_blocking=True)
                stats_host[2 * E:].copy_(l_aux, non_blocking=True)
            self.downloaded[s].record(self.d2h)
        return y_host
