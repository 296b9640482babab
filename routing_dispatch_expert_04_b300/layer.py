"""One MoE FFN layer forward on one GPU, driven through the C ABI.

:class:`MoELayer` owns the device buffers of one layer shape and issues, on one CUDA
stream and without any host synchronisation, the calls of the layer in the order the
expert-parallelism pages give it ("Expert Parallelism (EP)", "Key math / How it
works": route, dispatch, expert GEMMs, combine), followed by the aux statistics:

    moe_route -> moe_dispatch -> moe_expert_up -> moe_expert_down
      [-> shared expert: moe_expert_up / moe_expert_down over all tokens]
      -> moe_combine -> moe_aux_stats

Buffers are torch tensors (device memory only); every step runs in the library's
kernels.
"""

from __future__ import annotations

import torch

from . import native as N


class MoELayer:
    def __init__(self, T, d, E, K, F, dtype, capacity_factor, alpha, w_r, b_r, w1, w2,
                 w1s=None, w2s=None, renormalize=False, device="cuda"):
        self.cfg = N.make_config(T, d, E, K, F, dtype, N.capacity(T, E, capacity_factor),
                                 renormalize, alpha)
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
        self.logits = torch.empty((T, E), dtype=f32, device=dev)
        self.ids = torch.empty((T, K), dtype=i32, device=dev)
        self.w = torch.empty((T, K), dtype=f32, device=dev)
        self.counts = torch.empty(E, dtype=i32, device=dev)
        self.offsets = torch.empty(E + 1, dtype=i32, device=dev)
        self.slot = torch.empty((T, K), dtype=i32, device=dev)
        self.src = torch.empty(R, dtype=i32, device=dev)
        self.x_perm = torch.empty((R, d), dtype=dt, device=dev)
        # the intermediate activation is fp16 for bf16 layers (see moe_expert_up)
        self.h_dtype = torch.float16 if dtype == "bf16" else torch.float32
        self.h = torch.empty((R, F), dtype=self.h_dtype, device=dev)
        self.y_perm = torch.empty((R, d), dtype=f32, device=dev)
        self.y = torch.empty((T, d), dtype=dt, device=dev)
        self.f = torch.empty(E, dtype=f32, device=dev)
        self.P = torch.empty(E, dtype=f32, device=dev)
        self.l_aux = torch.empty(1, dtype=f32, device=dev)
        self.w2 = self._down_weights(w2)
        self.shared = w1s is not None
        self.w2s = self._down_weights(w2s) if self.shared else None
        if self.shared:
            self.shared_offsets = torch.tensor([0, T], dtype=i32, device=dev)
            self.h_s = torch.empty((max(T, 1), F), dtype=self.h_dtype, device=dev)
            self.y_s = torch.empty((max(T, 1), d), dtype=f32, device=dev)

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
    def from_workload(cls, wl, inputs, device="cuda", renormalize=False):
        return cls(wl.T, wl.d, wl.E, wl.K, wl.F, wl.dtype, wl.capacity_factor, wl.alpha,
                   inputs["w_r"], inputs["b_r"], inputs["w1"], inputs["w2"],
                   inputs.get("w1s"), inputs.get("w2s"), renormalize=renormalize, device=device)

    # ---------------------------------------------------------------- stages
    def route(self, x, stream=None, logits_in=None):
        """Router + softmax + top-K.  With ``logits_in`` (fp32 [T,E]) the router Linear is
        skipped and those logits drive the routing."""
        if logits_in is not None:
            self.logits.copy_(logits_in)
            N.route(self.cfg, None, None, None, self.logits, self.ids, self.w, self.ws, stream)
        else:
            N.route(self.cfg, x, self.w_r, self.b_r, self.logits, self.ids, self.w, self.ws, stream)

    def dispatch(self, x, stream=None):
        N.dispatch(self.cfg, x, self.ids, self.counts, self.offsets, self.slot, self.src,
                   None if x is None else self.x_perm, self.ws, stream)

    def experts_up(self, stream=None):
        N.expert_up(self.cfg, self.x_perm, self.offsets, self.E, self.rows_cap, self.w1, self.h,
                    self.ws, stream)

    def experts_down(self, stream=None):
        N.expert_down(self.cfg, self.h, self.offsets, self.E, self.rows_cap, self.w2, self.y_perm,
                      self.ws, stream)

    def shared_expert(self, x, stream=None):
        N.expert_up(self.cfg, x, self.shared_offsets, 1, self.T, self.w1s, self.h_s, self.ws, stream)
        N.expert_down(self.cfg, self.h_s, self.shared_offsets, 1, self.T, self.w2s, self.y_s, self.ws,
                      stream)

    def combine(self, stream=None):
        N.combine(self.cfg, self.y_perm, self.slot, self.w, self.y_s if self.shared else None, self.y,
                  stream)

    def aux(self, stream=None):
        N.aux_stats(self.cfg, self.counts, self.ws, self.f, self.P, self.l_aux, stream)

    # ---------------------------------------------------------------- whole layer
    def forward(self, x, stream=None, logits_in=None):
        """Enqueue the whole layer on ``stream``; returns the output buffer ``self.y``."""
        self.route(x, stream, logits_in)
        self.dispatch(x, stream)
        self.experts_up(stream)
        self.experts_down(stream)
        if self.shared:
            self.shared_expert(x, stream)
        self.combine(stream)
        self.aux(stream)
        return self.y

    def forward_host(self, x_host, y_host, x_dev, stream=None):
        """End-to-end call with host buffers: copy x (pinned host) in, run the layer, copy
        y back into pinned host memory, all on one stream."""
        x_dev.copy_(x_host, non_blocking=True)
        self.forward(x_dev, stream)
        y_host.copy_(self.y, non_blocking=True)
        return y_host

    def check_device_status(self):
        st = N.sync_status(self.ws)
        if st != 0:
            raise N.MoeError("moe_sync_status", st)
