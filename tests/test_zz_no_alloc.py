"""moe_dispatch_noalloc: the dispatch step for callers that cannot allocate device memory
when they run the layer (code inside a custom allocator or memory pool, plugins barred
from cudaMalloc).  Its scratch is a static device array inside the library, so the call
takes no workspace.  Its outputs must equal moe_dispatch's on the same inputs, call after
call, while the array keeps the previous call's contents -- and the oracle's dispatch
plan; the errors its kernels record must reach the caller through
moe_dispatch_noalloc_status.

This file is collected last so that a run stopping at its first failure has run every
other test before this one."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
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


def test_noalloc_rejects_the_configs_moe_dispatch_rejects():
    """Host-side check: the two entry points validate the config identically (bad drop
    order, renormalize flag, vector width, K > E) before any CUDA call."""
    B.build()
    fake = ctypes.c_void_p(1 << 20)
    bad = [N.make_config(64, 64, 8, 2, 64, "bf16", 8, drop_order=2),
           N.make_config(64, 64, 8, 2, 64, "bf16", 8),
           N.make_config(64, 60, 8, 2, 64, "bf16", 8),
           N.make_config(64, 64, 4, 8, 64, "bf16", 8)]
    bad[1].renormalize = 3
    for cfg in bad:
        a = N.lib().moe_dispatch(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, fake,
                                 fake, None)
        b = N.lib().moe_dispatch_noalloc(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake,
                                         fake, None)
        assert a == b and a in (1, 2), (a, b)


def _ids(T, E, K, seed, dev="cuda"):
    L = make_logits(T, E, device=dev, seed=seed, ties=(seed % 2 == 1))
    # top-K by (logit desc, id asc), as the routing kernels order them
    order = torch.sort(-L, dim=1, stable=True).indices[:, :K]
    return order.to(torch.int32).contiguous()


def _dispatch_both(T, d, E, K, C, seed, dtype, order="token", with_x=True):
    cfg = N.make_config(T, d, E, K, 64, dtype, C, drop_order=order)
    dev = "cuda"
    R = max(N.rows_capacity(cfg), 1)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x = torch.randn(T, d, generator=g, device=dev).to(tdt) if with_x else None
    ids = _ids(T, E, K, seed)

    def bufs():
        return dict(counts=torch.full((E,), -9, dtype=torch.int32, device=dev),
                    offsets=torch.full((E + 1,), -9, dtype=torch.int32, device=dev),
                    slot=torch.full((T, K), -9, dtype=torch.int32, device=dev),
                    src=torch.full((R,), -9, dtype=torch.int32, device=dev),
                    x_perm=torch.zeros((R, d), dtype=tdt, device=dev) if with_x else None)

    a, b = bufs(), bufs()
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device=dev)
    N.dispatch(cfg, x, ids, a["counts"], a["offsets"], a["slot"], a["src"], a["x_perm"], ws)
    N.dispatch_noalloc(cfg, x, ids, b["counts"], b["offsets"], b["slot"], b["src"], b["x_perm"])
    torch.cuda.synchronize()
    assert N.sync_status(ws) == 0
    assert N.dispatch_noalloc_status() == 0
    return a, b, ids, x


def _check(a, b, ids, x, E, K, C, order):
    """Bit for bit against moe_dispatch, and against the oracle's dispatch plan."""
    for key in ("counts", "offsets", "slot", "src"):
        assert torch.equal(a[key], b[key]), key
    R = int(a["offsets"][-1].item())
    plan = O.dispatch_plan(ids.cpu().numpy(), E, C, order)
    assert np.array_equal(b["counts"].cpu().numpy(), plan["counts"])
    assert np.array_equal(b["offsets"].cpu().numpy(), plan["offsets"])
    assert np.array_equal(b["slot"].cpu().numpy().reshape(-1), plan["slot"])
    assert np.array_equal(b["src"].cpu().numpy()[:R], plan["src"])
    if x is not None:
        assert torch.equal(a["x_perm"][:R], b["x_perm"][:R])
        rows = torch.from_numpy(plan["src"].astype(np.int64) // K).cuda()
        assert torch.equal(b["x_perm"][:R], x[rows])


@pytest.mark.gpu
def test_noalloc_dispatch_matches_workspace_dispatch_two_calls():
    assert torch.cuda.is_available()
    B.build()
    assert N.dispatch_noalloc_status() == 0
    # calls in a row with different sizes: each reuses the static scratch the previous one
    # left; token- and slot-major drop order, finite and unbounded capacity, with and
    # without the row copy
    cases = [(6000, 256, 16, 4, 1600, 1, "bf16", "token", True),
             (4096, 128, 8, 2, 640, 2, "f32", "token", True),
             (5000, 64, 32, 4, 500, 3, "bf16", "slot", True),
             (3000, 128, 64, 8, -1, 4, "bf16", "token", True),
             (7000, 64, 8, 2, 1000, 5, "bf16", "slot", False)]
    for (T, d, E, K, C, seed, dt, order, with_x) in cases:
        a, b, ids, x = _dispatch_both(T, d, E, K, C, seed, dt, order, with_x)
        _check(a, b, ids, x, E, K, C, order)


@pytest.mark.gpu
def test_noalloc_errors_reach_the_caller():
    """Device-side errors stay in the static array's status word, across calls, until
    moe_dispatch_noalloc_status reads and clears them: a scan block that withholds its
    counts (the bounded look-back wait gives up; the kernel still terminates) and an
    expert id out of range.  The next call after each is clean and matches the oracle."""
    assert torch.cuda.is_available()
    B.build()
    assert N.dispatch_noalloc_status() == 0
    T, E, K, C = 6000, 8, 2, 1700          # 12000 assignments -> 3 scan blocks
    cfg = N.make_config(T, 64, E, K, 64, "bf16", C)
    dev = "cuda"
    ids = _ids(T, E, K, 7)
    out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               slot=torch.empty((T, K), dtype=torch.int32, device=dev),
               src=torch.empty(T * K, dtype=torch.int32, device=dev))

    def call(ids_):
        N.dispatch_noalloc(cfg, None, ids_, out["counts"], out["offsets"], out["slot"],
                           out["src"], None)

    N.arm_scan_timeout(0, 2000)
    call(ids)
    call(ids)  # a clean call in between does not clear the recorded error
    assert N.dispatch_noalloc_status() == 4   # MOE_ERR_TIMEOUT
    assert N.dispatch_noalloc_status() == 0   # cleared
    call(ids)
    assert N.dispatch_noalloc_status() == 0
    plan = O.dispatch_plan(ids.cpu().numpy(), E, C)
    assert np.array_equal(out["slot"].cpu().numpy().reshape(-1), plan["slot"])
    assert np.array_equal(out["offsets"].cpu().numpy(), plan["offsets"])

    bad = ids.clone()
    bad[5, 1] = E
    call(bad)
    assert N.dispatch_noalloc_status() == 5   # MOE_ERR_DEVICE
    assert int(out["slot"][5, 1].item()) == -1
    assert int(out["counts"].sum().item()) == T * K - 1
    assert N.dispatch_noalloc_status() == 0
