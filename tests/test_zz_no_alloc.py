"""moe_dispatch_noalloc: the dispatch step for callers that cannot allocate device memory
when they run the layer (code inside a custom allocator or memory pool, plugins barred
from cudaMalloc).  Its scratch is a static device array inside the library, so the call
takes no workspace.  Its outputs must equal moe_dispatch's on the same inputs, call after
call, while the array keeps the previous call's contents.

This file is collected last so that a run stopping at its first failure has run every
other test before this one."""

import ctypes

import numpy as np
import pytest
import torch

from routing_dispatch_expert_04_b300 import build as B
from routing_dispatch_expert_04_b300 import native as N
from routing_dispatch_expert_04_b300.workloads import make_logits


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Host-side check: no CUDA call is made for a config whose scratch would not fit."""
    B.build()
    cfg = N.make_config(400000, 64, 256, 8, 64, "bf16", -1)   # 3.2M assignments
    fake = ctypes.c_void_p(1 << 20)
    st = N.lib().moe_dispatch_noalloc(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, fake,
                                      None)
    assert st == 2  # MOE_ERR_UNSUPPORTED


def _dispatch_both(T, d, E, K, C, seed, dtype):
    cfg = N.make_config(T, d, E, K, 64, dtype, C)
    dev = "cuda"
    R = max(N.rows_capacity(cfg), 1)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x = torch.randn(T, d, generator=g, device=dev).to(tdt)
    L = make_logits(T, E, device=dev, seed=seed, ties=(seed % 2 == 1))
    ids = torch.topk(L, K, dim=1).indices.to(torch.int32).contiguous()

    def bufs():
        return dict(counts=torch.full((E,), -9, dtype=torch.int32, device=dev),
                    offsets=torch.full((E + 1,), -9, dtype=torch.int32, device=dev),
                    slot=torch.full((T, K), -9, dtype=torch.int32, device=dev),
                    src=torch.full((R,), -9, dtype=torch.int32, device=dev),
                    x_perm=torch.zeros((R, d), dtype=tdt, device=dev))

    a, b = bufs(), bufs()
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device=dev)
    N.dispatch(cfg, x, ids, a["counts"], a["offsets"], a["slot"], a["src"], a["x_perm"], ws)
    N.dispatch_noalloc(cfg, x, ids, b["counts"], b["offsets"], b["slot"], b["src"], b["x_perm"])
    torch.cuda.synchronize()
    assert N.sync_status(ws) == 0
    return a, b


@pytest.mark.gpu
def test_noalloc_dispatch_matches_workspace_dispatch_two_calls():
    assert torch.cuda.is_available()
    B.build()
    # two calls in a row with different sizes: the second reuses the static scratch
    for (T, d, E, K, C, seed, dt) in [(6000, 256, 16, 4, 1600, 1, "bf16"),
                                      (4096, 128, 8, 2, 640, 2, "f32")]:
        a, b = _dispatch_both(T, d, E, K, C, seed, dt)
        for key in ("counts", "offsets", "slot", "src"):
            assert torch.equal(a[key], b[key]), key
        R = int(a["offsets"][-1].item())
        assert torch.equal(a["x_perm"][:R], b["x_perm"][:R])
