"""Seeded synthetic workloads shaped like the MoE layers the expert-parallelism pages name.

This module only draws random tensors.  It holds none of the layer's arithmetic (no
routing, capacity or FFN); the tests feed its tensors to both the CUDA library and the
CPU oracle.

Shapes (from the pages' model references: Mixtral 8x7B in "Expert Parallelism (MoE)",
DeepSeek-V3's 256 routed + 1 shared experts in "Expert Parallelism (EP)", Qwen3-30B-A3B
in the Hugging Face "Expert parallelism" page, and the 64K-token all-to-all case):

=========  ======  =====  ===  =  =====  =====  ======  ===========================
name       T       d      E    K  F      dtype  cf      router bias
=========  ======  =====  ===  =  =====  =====  ======  ===========================
tiny       256     128    8    2  512    f32    1.25    none
mixtral    4096    4096   8    2  16384  bf16   1.25    none
dsv3       8192    7168   256  8  2048   bf16   none    N(0, 0.5^2), + 1 shared exp.
qwen3      16384   2048   128  8  768    bf16   1.5     none
long       65536   4096   8    2  16384  bf16   1.0     Zipf(s=1.2)-ranked
=========  ======  =====  ===  =  =====  =====  ======  ===========================

Recipe (seed 0): one ``torch.Generator`` on the target device; tensors are drawn in
fp32 in the order X, W_r, b_r, W1, W2, (W1s, W2s) and cast to the storage dtype with
round-to-nearest-even.  X ~ N(0, 1); every weight ~ N(0, 1/fan_in) (W_r and W1:
fan_in = d; W2: fan_in = F).  W1 and W2 are drawn one expert at a time so that the
fp32 staging copy stays small.

The 64K-token workload's router bias is b[e] = -beta * s * ln(rank(e)) with s = 1.2,
rank a seed-0 permutation of 1..E, and beta = 1.0124.  beta was fitted once by
Monte Carlo with i.i.d. N(0, 1) logit noise (the distribution X . W_r^T has under this
recipe) so that, under top-2 routing, the rank-1 expert draws 40% of the assignments
before dropping; the realised share on the seed-0 tensors is measured, not assumed.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import torch

ZIPF_S = 1.2
ZIPF_BETA = 1.0124


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    K: int
    F: int
    dtype: str                      # "f32" or "bf16"
    capacity_factor: Optional[float]  # None: no dropping
    alpha: float = 0.01
    bias: Optional[str] = None      # None | "normal" | "zipf"
    shared: bool = False

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def scaled(self, T: int) -> "Workload":
        """Same layer with a different token count (for smaller parity cases)."""
        return Workload(self.name + f"_T{T}", T, self.d, self.E, self.K, self.F, self.dtype,
                        self.capacity_factor, self.alpha, self.bias, self.shared)


WORKLOADS = {
    "tiny": Workload("tiny", 256, 128, 8, 2, 512, "f32", 1.25),
    "mixtral": Workload("mixtral", 4096, 4096, 8, 2, 16384, "bf16", 1.25),
    "dsv3": Workload("dsv3", 8192, 7168, 256, 8, 2048, "bf16", None, bias="normal", shared=True),
    "qwen3": Workload("qwen3", 16384, 2048, 128, 8, 768, "bf16", 1.5),
    "long": Workload("long", 65536, 4096, 8, 2, 16384, "bf16", 1.0, bias="zipf"),
}


def _normal(shape, std, g, device, dtype):
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_inputs(wl: Workload, device="cpu", seed: int = 0, weights: bool = True) -> dict:
    """Draw the layer's inputs.  Returns a dict of tensors on ``device``:
    x [T,d], w_r [E,d], b_r [E] fp32 or None, w1 [E,F,d], w2 [E,d,F],
    and for the shared expert w1s [1,F,d], w2s [1,d,F].  ``weights=False`` skips the
    expert weights (routing-only cases)."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = wl.torch_dtype
    out = {}
    out["x"] = _normal((wl.T, wl.d), 1.0, g, device, dt)
    out["w_r"] = _normal((wl.E, wl.d), 1.0 / math.sqrt(wl.d), g, device, dt)
    if wl.bias == "normal":
        out["b_r"] = _normal((wl.E,), 0.5, g, device, torch.float32)
    elif wl.bias == "zipf":
        rank = torch.randperm(wl.E, generator=g, device=device).to(torch.float32) + 1.0
        out["b_r"] = (-ZIPF_BETA * ZIPF_S) * torch.log(rank)
    else:
        out["b_r"] = None
    if weights:
        w1 = torch.empty((wl.E, wl.F, wl.d), device=device, dtype=dt)
        for e in range(wl.E):
            w1[e] = _normal((wl.F, wl.d), 1.0 / math.sqrt(wl.d), g, device, dt)
        w2 = torch.empty((wl.E, wl.d, wl.F), device=device, dtype=dt)
        for e in range(wl.E):
            w2[e] = _normal((wl.d, wl.F), 1.0 / math.sqrt(wl.F), g, device, dt)
        out["w1"], out["w2"] = w1, w2
        if wl.shared:
            out["w1s"] = _normal((1, wl.F, wl.d), 1.0 / math.sqrt(wl.d), g, device, dt)
            out["w2s"] = _normal((1, wl.d, wl.F), 1.0 / math.sqrt(wl.F), g, device, dt)
    return out


def make_logits(T: int, E: int, device="cpu", seed: int = 0, ties: bool = False):
    """fp32 router logits for routing-only cases: N(0,1), optionally quantised to a
    coarse grid (multiples of 1/4 in [-2, 2]) so that exact ties are frequent."""
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    L = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    if ties:
        L = torch.clamp(torch.round(L * 4.0) / 4.0, -2.0, 2.0)
    return L
