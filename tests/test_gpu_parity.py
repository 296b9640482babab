"""GPU parity: the CUDA library, called through its C ABI, against the fp64 oracle.

Tolerances: routing ids, counts, offsets, slot, src and the drop mask are compared bit
for bit when the routing kernels are fed the oracle's fp32 logits; routing weights, P_i
and L_aux within 1e-6 relative (fp32 softmax against fp64); layer output
max|GPU - oracle| / RMS(oracle) <= 1e-4 for fp32 layers; for bf16 layers the same bound
2e-2 applies to the error in excess of half an output ulp (bf16 rounding of the exact
result alone reaches 0.02-0.04 of RMS on these shapes), and the literal value is
reported.  Outputs are compared over the tokens a near-tie cannot flip (logit gap of
the K-th and (K+1)-th expert >= 1e-4, plus the capacity cascade those tokens can cause).
"""

import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from routing_dispatch_expert_04_b300 import build as B
from routing_dispatch_expert_04_b300 import native as N
from routing_dispatch_expert_04_b300.layer import MoELayer
from routing_dispatch_expert_04_b300.workloads import WORKLOADS, Workload, make_inputs, make_logits
from parity_helpers import (assert_rounded_to, comparable_tokens, layer_output_error,
                            rel_rms_err, to_np)

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    N.lib()


def _routing_only(T, E, K, C, L32, renorm=False, sel_bias=None, order="token"):
    """Drive moe_route (logits given) + moe_dispatch (no row copy) + moe_aux_stats."""
    cfg = N.make_config(T, 8, E, K, 8, "bf16", C, renorm, 0.01, order)
    dev = "cuda"
    R = max(N.rows_capacity(cfg), 1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device=dev)
    logits = torch.from_numpy(np.ascontiguousarray(L32)).to(dev)
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    src = torch.full((R,), -7, dtype=torch.int32, device=dev)
    f = torch.empty(E, dtype=torch.float32, device=dev)
    P = torch.empty(E, dtype=torch.float32, device=dev)
    l = torch.empty(1, dtype=torch.float32, device=dev)
    if sel_bias is None:
        N.route(cfg, None, None, None, logits, ids, w, ws)
    else:
        N.route_select_bias(cfg, None, None, None, torch.from_numpy(sel_bias).to(dev), logits,
                            ids, w, ws)
    N.dispatch(cfg, None, ids, counts, offsets, slot, src, None, ws)
    N.aux_stats(cfg, counts, ws, f, P, l)
    assert N.sync_status(ws) == 0
    out = dict(ids=to_np(ids), w=to_np(w), counts=to_np(counts), offsets=to_np(offsets),
               slot=to_np(slot), src=to_np(src), f=to_np(f), P=to_np(P), l_aux=float(l.item()))
    if order == "token":
        # the same routing with the dispatch plan computed in the routing step
        # (moe_route_plan + moe_dispatch_planned) on a fresh workspace: identical results
        ws2 = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device=dev)
        sel = None if sel_bias is None else torch.from_numpy(sel_bias).to(dev)
        ids2, w2, counts2, offsets2, slot2 = (torch.empty_like(t) for t in (ids, w, counts, offsets, slot))
        src2 = torch.full((R,), -7, dtype=torch.int32, device=dev)
        f2, P2, l2 = torch.empty_like(f), torch.empty_like(P), torch.empty_like(l)
        N.route_plan(cfg, None, None, None, sel, logits, ids2, w2, counts2, offsets2, ws2)
        N.dispatch_planned(cfg, None, ids2, offsets2, slot2, src2, None, ws2)
        N.aux_stats(cfg, counts2, ws2, f2, P2, l2)
        assert N.sync_status(ws2) == 0
        # both paths run the same routing grid, so even P's fixed-order sums agree
        for a, b in ((ids, ids2), (w, w2), (counts, counts2), (offsets, offsets2), (slot, slot2),
                     (f, f2), (P, P2), (l, l2)):
            assert torch.equal(a, b)
        Rk = int(offsets[-1].item())
        assert torch.equal(src[:Rk], src2[:Rk])
    return out


def _check_routing(g, L32, K, C, E, renorm=False, alpha=0.01, sel_bias=None, order="token"):
    ids = O.top_k(L32, K, sel_bias)
    p = O.softmax(L32)
    w = O.routing_weights(p, ids, renorm)
    plan = O.dispatch_plan(ids, E, C, order)
    assert np.array_equal(g["ids"], ids)
    assert np.max(np.abs(g["w"] - w) / np.abs(w)) <= 1e-6
    assert np.array_equal(g["counts"], plan["counts"])
    assert np.array_equal(g["offsets"], plan["offsets"])
    assert np.array_equal(g["slot"], plan["slot"].reshape(-1, K))
    R = plan["R"]
    assert np.array_equal(g["src"][:R], plan["src"])
    f, P, l_aux = O.aux_stats(ids, p, E, alpha)
    assert np.array_equal(g["f"], f.astype(np.float32))
    assert np.max(np.abs(g["P"] - P) / np.maximum(P, 1e-30)) <= 1e-6
    assert abs(g["l_aux"] - l_aux) <= 1e-6 * l_aux
    return plan


# ------------------------------------------------------------------ routing, bit-exact
@pytest.mark.parametrize("T,E,K,cf,ties,renorm", [
    (256, 8, 2, 1.25, False, False),
    (4096, 8, 2, 1.25, True, False),
    (8192, 256, 8, None, False, False),
    (16384, 128, 8, 1.5, True, False),
    (65536, 8, 2, 1.0, False, False),
    (5000, 64, 4, 0.9, True, True),
    (4097, 33, 5, 2.0, True, False),
    (1, 1, 1, 1.0, False, False),
    (37, 5, 5, 0.5, True, False),
    (300, 256, 32, 1.0, True, True),     # the largest supported top-K
    (77, 32, 32, 0.7, True, False),      # K = E = 32
])
def test_routing_bit_exact_random_logits(T, E, K, cf, ties, renorm):
    L32 = make_logits(T, E, seed=T + E, ties=ties).numpy()
    C = O.capacity(T, E, cf)
    g = _routing_only(T, E, K, C, L32, renorm)
    _check_routing(g, L32, K, C, E, renorm)


@pytest.mark.parametrize("name", ["tiny", "mixtral", "dsv3", "qwen3", "long"])
def test_routing_bit_exact_workload_logits(name):
    """Full-size workloads: the oracle computes the fp32 logits in fp64 from the seeded
    X, W_r and b_r; the GPU routing kernels are fed those logits."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl, "cuda", weights=False)
    _, L32 = O.router_logits(to_np(inp["x"]), to_np(inp["w_r"]),
                             None if inp["b_r"] is None else to_np(inp["b_r"]))
    C = O.capacity(wl.T, wl.E, wl.capacity_factor)
    g = _routing_only(wl.T, wl.E, wl.K, C, L32)
    plan = _check_routing(g, L32, wl.K, C, wl.E, alpha=wl.alpha)
    if C >= 0:
        assert (plan["kept"] <= C).all()
    if name == "long":
        share = float(plan["counts"].max()) / (wl.T * wl.K)
        assert 0.37 <= share <= 0.43, share


@pytest.mark.parametrize("T,E,K,cf,ties,bias,order,cap", [
    (4096, 8, 2, 1.25, True, True, "token", "tokens"),
    (4096, 8, 2, 1.25, False, False, "slot", "tokens"),
    (16384, 128, 8, 1.5, True, True, "slot", "assignments"),
    (8192, 256, 8, None, False, True, "token", "tokens"),
    (5000, 64, 4, 0.9, True, True, "slot", "tokens"),
    (65536, 8, 2, 1.0, False, False, "slot", "assignments"),
    (37, 5, 5, 0.5, True, True, "slot", "tokens"),
])
def test_routing_variants_bit_exact(T, E, K, cf, ties, bias, order, cap):
    """Selection-only bias, slot-major drop priority and capacity counting assignments:
    ids, counts, offsets, slot, src bit for bit; weights and P from the unbiased
    softmax."""
    L32 = make_logits(T, E, seed=T + 7 * E, ties=ties).numpy()
    rng = np.random.default_rng(T + E)
    b = (np.round(rng.standard_normal(E) * 4) / 8).astype(np.float32) if bias else None
    C = O.capacity(T, E, cf) if cap == "tokens" else O.capacity_assignments(T, E, K, cf)
    g = _routing_only(T, E, K, C, L32, sel_bias=b, order=order)
    _check_routing(g, L32, K, C, E, sel_bias=b, order=order)


def test_adjust_selection_bias_matches_oracle():
    T, E, K = 3000, 64, 4
    L32 = make_logits(T, E, seed=21).numpy()
    g = _routing_only(T, E, K, -1, L32)
    b = np.random.default_rng(3).standard_normal(E).astype(np.float32)
    cfg = N.make_config(T, 8, E, K, 8, "bf16", -1)
    counts = torch.from_numpy(g["counts"]).cuda()
    bias = torch.from_numpy(b).cuda()
    N.adjust_select_bias(cfg, counts, bias, 1e-3)
    torch.cuda.synchronize()
    want = O.adjust_selection_bias(b, g["counts"], T, K, 1e-3)
    assert np.array_equal(bias.cpu().numpy(), want)
    with pytest.raises(N.MoeError):
        N.adjust_select_bias(cfg, counts, bias, -1.0)


@pytest.mark.parametrize("T,E,K", [(4096, 8, 2), (8192, 256, 8), (16384, 128, 8), (37, 5, 5),
                                   (1, 1, 1)])
def test_aux_loss_grad(T, E, K):
    """Backward of the aux loss against the oracle's fp64 gradient.  Every entry is
    (alpha/T) p (f_j - sum_i f_i p_i) with p, f <= 1, computed in fp32: the bound is
    1e-5 of alpha/T (the gradient itself vanishes when every expert is chosen equally)."""
    L32 = make_logits(T, E, seed=T + 3 * E).numpy()
    g = _routing_only(T, E, K, -1, L32)
    cfg = N.make_config(T, 8, E, K, 8, "bf16", -1, False, 0.01)
    logits = torch.from_numpy(L32).cuda()
    f = torch.from_numpy(g["f"]).cuda()
    grad = torch.full((T, E), 7.0, dtype=torch.float32, device="cuda")
    N.aux_loss_grad(cfg, logits, f, grad)
    torch.cuda.synchronize()
    ref = O.aux_loss_grad_logits(L32, O.top_k(L32, K), 0.01)
    assert np.max(np.abs(grad.cpu().numpy() - ref)) <= 1e-5 * 0.01 / T


def test_scan_spans_many_blocks_all_one_expert():
    """Every assignment to one expert (collapsed router): the look-back carries one
    expert's running count across all scan blocks."""
    T, E, K = 20000, 16, 2
    L32 = np.zeros((T, E), dtype=np.float32)
    L32[:, 3] = 5.0
    L32[:, 7] = 4.0
    C = 1000
    g = _routing_only(T, E, K, C, L32)
    _check_routing(g, L32, K, C, E)
    assert g["offsets"].tolist()[-1] == 2 * C


def test_scan_timeout_is_reported_and_recovers():
    """A scan block withholds its published counts (test hook); its successor's bounded
    wait runs out, the kernel still terminates, and the status word says so.  The next
    call is unaffected."""
    T, E, K = 6000, 8, 2            # 12000 assignments -> 3 scan blocks
    L32 = make_logits(T, E, seed=3).numpy()
    N.arm_scan_timeout(0, 2000)
    cfg = N.make_config(T, 8, E, K, 8, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    logits = torch.from_numpy(L32).cuda()
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    slot = torch.empty((T, K), dtype=torch.int32, device="cuda")
    src = torch.empty(T * K, dtype=torch.int32, device="cuda")
    N.route(cfg, None, None, None, logits, ids, w, ws)
    N.dispatch(cfg, None, ids, counts, offsets, slot, src, None, ws)
    assert N.sync_status(ws) == 4  # MOE_ERR_TIMEOUT
    assert N.sync_status(ws) == 0  # cleared
    g = _routing_only(T, E, K, -1, L32)
    _check_routing(g, L32, K, -1, E)


@pytest.mark.parametrize("T,E,K,C", [(4000, 8, 2, 600), (20000, 8, 2, 3000), (3000, 128, 8, 150),
                                     (2500, 256, 8, -1)])
def test_route_plan_reuses_its_workspace(T, E, K, C):
    """The plan from the routing kernel, three calls on one workspace with different
    logits: each call's counts, offsets and slots match the oracle (the plan scan's
    finished counter is reset by its last block; 20000 tokens = 2500 routing blocks, more
    than one pass of the plan scan)."""
    cfg = N.make_config(T, 8, E, K, 8, "bf16", C)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    slot = torch.empty((T, K), dtype=torch.int32, device="cuda")
    src = torch.empty(T * K, dtype=torch.int32, device="cuda")
    for seed in (5, 6, 7):
        L32 = make_logits(T, E, seed=seed).numpy()
        logits = torch.from_numpy(L32).cuda()
        N.route_plan(cfg, None, None, None, None, logits, ids, w, counts, offsets, ws)
        N.dispatch_planned(cfg, None, ids, offsets, slot, src, None, ws)
        assert N.sync_status(ws) == 0
        plan = O.dispatch_plan(O.top_k(L32, K), E, C)
        assert np.array_equal(to_np(counts), plan["counts"])
        assert np.array_equal(to_np(offsets), plan["offsets"])
        assert np.array_equal(to_np(slot).reshape(-1), plan["slot"])
        assert np.array_equal(to_np(src)[:plan["R"]], plan["src"])


@pytest.mark.parametrize("idx", [2, 4, 5])
def test_layer_plan_in_route_matches_separate_scan(idx):
    """The layer with the dispatch plan from the routing step (default) and with the plan
    in the dispatch step's own scan give identical outputs and statistics."""
    wl = SMALL[idx]
    inp = make_inputs(wl, "cuda")
    a = MoELayer.from_workload(wl, inp, plan_in_route=True)
    b = MoELayer.from_workload(wl, inp, plan_in_route=False)
    assert a.planned and not b.planned
    for layer in (a, b):
        layer.forward(inp["x"])
        layer.check_device_status()
    torch.cuda.synchronize()
    for name in ("ids", "counts", "offsets", "slot", "y", "f", "P", "l_aux"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def test_out_of_range_expert_id_reported():
    T, E, K = 100, 8, 2
    cfg = N.make_config(T, 8, E, K, 8, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    ids = torch.randint(0, E, (T, K), dtype=torch.int32, device="cuda")
    ids[5, 1] = E
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    slot = torch.empty((T, K), dtype=torch.int32, device="cuda")
    src = torch.empty(T * K, dtype=torch.int32, device="cuda")
    N.dispatch(cfg, None, ids, counts, offsets, slot, src, None, ws)
    assert N.sync_status(ws) == 5  # MOE_ERR_DEVICE
    assert int(slot[5, 1].item()) == -1
    assert int(counts.sum().item()) == T * K - 1


# ------------------------------------------------------------------ whole layer
def _layer_case(wl: Workload, seed=0, logits_from_oracle=False, renorm=False, fused=True):
    inp = make_inputs(wl, "cuda", seed=seed)
    layer = MoELayer.from_workload(wl, inp, renormalize=renorm, fused_dispatch=fused)
    x_np = to_np(inp["x"])
    b_np = None if inp["b_r"] is None else to_np(inp["b_r"])
    _, L32 = O.router_logits(x_np, to_np(inp["w_r"]), b_np)
    layer.forward(inp["x"], logits_in=torch.from_numpy(L32).cuda() if logits_from_oracle else None)
    layer.check_device_status()
    torch.cuda.synchronize()
    shared = (to_np(inp["w1s"])[0], to_np(inp["w2s"])[0]) if wl.shared else None
    C = O.capacity(wl.T, wl.E, wl.capacity_factor)
    ref = O.moe_forward(x_np, to_np(inp["w_r"]), b_np, to_np(inp["w1"]), to_np(inp["w2"]),
                        wl.K, C, wl.alpha, renormalize=renorm, shared=shared,
                        logits32=L32 if logits_from_oracle else None)
    return layer, ref, L32, C


SMALL = [
    Workload("tiny", 256, 128, 8, 2, 512, "f32", 1.25),
    Workload("f32_ragged", 203, 36, 5, 3, 92, "f32", 1.1),
    Workload("bf16_small", 300, 256, 8, 2, 384, "bf16", 1.25),
    Workload("bf16_ragged", 517, 136, 16, 4, 200, "bf16", 0.8),
    Workload("bf16_bias_shared", 333, 128, 32, 8, 96, "bf16", None, bias="normal", shared=True),
    Workload("bf16_zipf", 1000, 192, 8, 2, 256, "bf16", 1.0, bias="zipf"),
    Workload("bf16_single_expert", 130, 64, 1, 1, 64, "bf16", None),
    Workload("bf16_k_eq_e", 90, 64, 4, 4, 128, "bf16", 1.0),
]


@pytest.mark.parametrize("fused", [True, False], ids=["fused_dispatch", "copy_dispatch"])
@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_layer_end_to_end_small(wl, fused):
    """The whole layer from x, the GPU computing its own router logits.  Outputs are
    compared over the tokens no near tie can flip; at least 90% of them.  When a near
    tie's capacity cascade leaves fewer, the case runs again with the GPU routing fed the
    oracle's fp32 logits, where every token is comparable."""
    layer, ref, L32, C = _layer_case(wl, fused=fused)
    # router logits themselves
    Lg = to_np(layer.logits)
    assert np.max(np.abs(Lg - L32) / (1 + np.abs(L32))) <= 1e-5
    keep = comparable_tokens(L32, ref["ids"], wl.K, C)
    if keep.mean() < 0.9:
        print(f"{wl.name}: {keep.mean():.2%} comparable from the GPU's own logits; "
              "rerun with the oracle's logits")
        layer, ref, L32, C = _layer_case(wl, fused=fused, logits_from_oracle=True)
        keep = np.ones(wl.T, dtype=bool)
    assert keep.mean() >= 0.9
    y = to_np(layer.y)
    err, literal = layer_output_error(y[keep], ref["y"][keep], wl.dtype)
    print(f"{wl.name}: output error {err:.4g} (literal max|err|/rms {literal:.4g})")
    assert err <= TOL[wl.dtype], (err, literal)
    assert np.array_equal(to_np(layer.ids)[keep], ref["ids"][keep])


@pytest.mark.parametrize("fused", [True, False], ids=["fused_dispatch", "copy_dispatch"])
@pytest.mark.parametrize("wl", SMALL[:6], ids=[w.name for w in SMALL[:6]])
def test_layer_stages_with_oracle_logits(wl, fused):
    """Fed the oracle's logits, every stage matches: routing bit-exact, packed rows
    exact (copied dispatch), h and y_perm within tolerance, combine within tolerance,
    aux stats."""
    layer, ref, L32, C = _layer_case(wl, logits_from_oracle=True, fused=fused)
    R = ref["R"]
    assert np.array_equal(to_np(layer.ids), ref["ids"])
    assert np.array_equal(to_np(layer.offsets), ref["offsets"])
    assert np.array_equal(to_np(layer.slot), ref["slot"].reshape(wl.T, wl.K))
    assert np.array_equal(to_np(layer.src)[:R], ref["src"])
    if not fused:
        assert np.array_equal(to_np(layer.x_perm)[:R], ref["x_perm"])
    tol = TOL[wl.dtype]
    hdt = "f16" if wl.dtype == "bf16" else "f32"
    assert_rounded_to(to_np(layer.h)[:R], ref["h"], hdt)
    assert rel_rms_err(to_np(layer.y_perm)[:R], ref["y_perm"]) <= tol
    err, literal = layer_output_error(to_np(layer.y), ref["y"], wl.dtype)
    assert err <= tol, (err, literal)
    assert np.max(np.abs(to_np(layer.P) - ref["P"]) / ref["P"]) <= 1e-6
    assert abs(layer.l_aux.item() - ref["l_aux"]) <= 1e-6 * ref["l_aux"]


@pytest.mark.parametrize("idx,order,cap", [(2, "slot", "assignments"), (3, "slot", "tokens"),
                                         (4, "token", "assignments")])
def test_layer_routing_variants_end_to_end(idx, order, cap):
    """Whole layer with a selection-only bias, slot-major drop priority and/or capacity
    counting assignments, fed the oracle's logits: routing bit for bit, output within
    tolerance; then one bias adjustment step matches the oracle's."""
    wl = SMALL[idx]
    inp = make_inputs(wl, "cuda")
    rng = np.random.default_rng(idx)
    b = (rng.standard_normal(wl.E) * 0.3).astype(np.float32)
    sel = torch.from_numpy(b).cuda()
    layer = MoELayer.from_workload(wl, inp, drop_order=order, capacity_mode=cap, sel_bias=sel)
    x_np = to_np(inp["x"])
    b_np = None if inp["b_r"] is None else to_np(inp["b_r"])
    _, L32 = O.router_logits(x_np, to_np(inp["w_r"]), b_np)
    layer.forward(inp["x"], logits_in=torch.from_numpy(L32).cuda())
    layer.check_device_status()
    C = (O.capacity(wl.T, wl.E, wl.capacity_factor) if cap == "tokens"
         else O.capacity_assignments(wl.T, wl.E, wl.K, wl.capacity_factor))
    assert layer.cfg.capacity == C
    shared = (to_np(inp["w1s"])[0], to_np(inp["w2s"])[0]) if wl.shared else None
    ref = O.moe_forward(x_np, to_np(inp["w_r"]), b_np, to_np(inp["w1"]), to_np(inp["w2"]),
                        wl.K, C, wl.alpha, shared=shared, logits32=L32, sel_bias=b, order=order)
    assert np.array_equal(to_np(layer.ids), ref["ids"])
    assert np.array_equal(to_np(layer.slot), ref["slot"].reshape(wl.T, wl.K))
    assert np.array_equal(to_np(layer.src)[:ref["R"]], ref["src"])
    err, literal = layer_output_error(to_np(layer.y), ref["y"], wl.dtype)
    assert err <= TOL[wl.dtype], (err, literal)
    layer.adjust_selection_bias(0.01)
    torch.cuda.synchronize()
    assert np.array_equal(sel.cpu().numpy(),
                          O.adjust_selection_bias(b, ref["counts"], wl.T, wl.K, 0.01))


def test_capacity_zero_drops_everything():
    wl = Workload("cap0", 64, 64, 8, 2, 64, "bf16", 0.1)  # C = floor(64*0.1/8) = 0
    layer, ref, L32, C = _layer_case(wl)
    assert C == 0
    assert int(layer.offsets[-1].item()) == 0
    assert (to_np(layer.slot) == -1).all()
    assert (to_np(layer.y) == 0).all()


def test_empty_batch():
    wl = Workload("empty", 0, 64, 8, 2, 64, "bf16", 1.0)
    inp = make_inputs(wl, "cuda")
    layer = MoELayer.from_workload(wl, inp)
    layer.forward(inp["x"])
    layer.check_device_status()
    assert (to_np(layer.counts) == 0).all() and (to_np(layer.offsets) == 0).all()
    assert (to_np(layer.f) == 0).all() and layer.l_aux.item() == 0.0


def test_determinism_two_runs():
    wl = SMALL[3]
    inp = make_inputs(wl, "cuda")
    layer = MoELayer.from_workload(wl, inp)
    layer.forward(inp["x"])
    y1 = layer.y.clone()
    p1 = layer.P.clone()
    layer.forward(inp["x"])
    assert torch.equal(y1, layer.y) and torch.equal(p1, layer.P)


# ------------------------------------------------------------------ full-size workloads
class _ExpertWeights:
    """Host fp32 copies of one expert's weights, fetched from the device once."""

    def __init__(self, inp):
        self.inp, self.cache = inp, {}

    def __call__(self, e):
        if e not in self.cache:
            self.cache[e] = (to_np(self.inp["w1"][e]), to_np(self.inp["w2"][e]))
        return self.cache[e]


def _check_expert_rows(wl, layer, x_np, weights, e, chunk=1024):
    """Every packed row of expert e as the GPU packed it: its x_perm rows are exactly the
    token rows src // K name, and its h and y_perm rows match the oracle's FFN of those
    token rows (h within its fp16 storage rounding, y_perm within the layer tolerance);
    the oracle runs in chunks of rows.  Returns the number of rows compared."""
    g_offs = to_np(layer.offsets)
    lo, hi = int(g_offs[e]), int(g_offs[e + 1])
    src = to_np(layer.src)[lo:hi].astype(np.int64)
    assert ((src >= 0) & (src < wl.T * wl.K)).all()
    toks = src // wl.K
    w1, w2 = weights(e)
    hdt = "f16" if wl.dtype == "bf16" else "f32"
    for c0 in range(lo, hi, chunk):
        c1 = min(hi, c0 + chunk)
        rows = toks[c0 - lo:c1 - lo]
        assert np.array_equal(to_np(layer.x_perm[c0:c1]), x_np[rows])
        y_ref, h_ref = O.expert_ffn(x_np[rows], w1, w2)
        assert_rounded_to(to_np(layer.h[c0:c1]), h_ref, hdt)
        assert rel_rms_err(to_np(layer.y_perm[c0:c1]), y_ref) <= TOL[wl.dtype]
    return hi - lo


def _sampled_full_check(name, n_tokens=512, seed=0):
    """Full-size workload in the bench's launch configuration (the default expert-GEMM
    plan, copied dispatch):
    - routing in full against the oracle's own logits (near ties and their capacity
      cascade excluded; bit for bit everywhere when nothing is excluded);
    - every packed row of two experts -- expert 0 and the most loaded other expert --
      against the oracle's FFN of the rows the GPU packed (on the Mixtral shape this
      includes each expert's rows 512-639, which the split plan's one-CTA kernel
      computes; on the 64K shape the whole 8192-row top expert);
    - the layer output on ``n_tokens`` sampled comparable tokens, each token's kept
      experts evaluated by the oracle (Y = sum of routing weight x expert output, plus
      the shared expert)."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl, "cuda")
    layer = MoELayer.from_workload(wl, inp)
    layer.forward(inp["x"])
    layer.check_device_status()
    torch.cuda.synchronize()
    x_np = to_np(inp["x"])
    b_np = None if inp["b_r"] is None else to_np(inp["b_r"])
    _, L32 = O.router_logits(x_np, to_np(inp["w_r"]), b_np)
    C = O.capacity(wl.T, wl.E, wl.capacity_factor)
    ids = O.top_k(L32, wl.K)
    plan = O.dispatch_plan(ids, wl.E, C)
    keep = comparable_tokens(L32, ids, wl.K, C)
    g_ids = to_np(layer.ids)
    assert np.array_equal(g_ids[keep], ids[keep])
    if keep.all():
        assert np.array_equal(to_np(layer.offsets), plan["offsets"])
        assert np.array_equal(to_np(layer.slot), plan["slot"].reshape(wl.T, wl.K))
    tol = TOL[wl.dtype]
    weights = _ExpertWeights(inp)
    kept = np.diff(to_np(layer.offsets))
    e_big = 1 + int(np.argmax(kept[1:])) if wl.E > 1 else 0
    n_rows = 0
    for e in sorted({0, e_big}):
        n_rows += _check_expert_rows(wl, layer, x_np, weights, e)
    print(f"{name}: {n_rows} packed rows of experts {sorted({0, e_big})} compared")
    # token sample: the oracle evaluates each sampled token's kept experts one by one
    rng = np.random.default_rng(seed)
    cand = np.nonzero(keep)[0]
    toks = rng.choice(cand, size=min(n_tokens, cand.size), replace=False)
    w = O.routing_weights(O.softmax(L32[toks]), ids[toks])
    keepmask = plan["keep"].reshape(wl.T, wl.K)[toks]
    need = sorted({int(e) for t_i in range(len(toks)) for k, e in enumerate(ids[toks[t_i]])
                   if keepmask[t_i, k]})
    Y = np.zeros((len(toks), wl.d))
    for e in need:
        sel = [(t_i, k) for t_i in range(len(toks)) for k in range(wl.K)
               if ids[toks[t_i], k] == e and keepmask[t_i, k]]
        rows = np.array([toks[t_i] for t_i, _ in sel])
        ye, _ = O.expert_ffn(x_np[rows], *weights(e))
        for j, (t_i, k) in enumerate(sel):
            Y[t_i] += w[t_i, k] * ye[j]
        if e not in (0, e_big):
            weights.cache.pop(e, None)
    if wl.shared:
        Y += O.dense_ffn(x_np[toks], to_np(inp["w1s"][0]), to_np(inp["w2s"][0]))
    err, literal = layer_output_error(to_np(layer.y)[toks], Y, wl.dtype)
    print(f"{name}: {len(toks)} sampled tokens, output error {err:.4g} (literal {literal:.4g})")
    assert len(toks) >= min(n_tokens, wl.T // 2)
    assert err <= tol, (err, literal)


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3", "long"])
def test_full_size_sampled(name):
    _sampled_full_check(name)


@pytest.mark.parametrize("idx,overlap", [(2, True), (4, True), (4, False)])
def test_graph_replay_matches_eager(idx, overlap):
    """The whole forward captured as one CUDA graph (timing events as graph nodes, with or
    without the side-stream overlap) reproduces the serial eager forward bit for bit,
    replay after replay."""
    wl = SMALL[idx]
    inp = make_inputs(wl, "cuda")
    serial = MoELayer.from_workload(wl, inp, overlap=False)
    serial.forward(inp["x"])
    torch.cuda.synchronize()
    y_ref = serial.y.clone()
    l_ref = serial.l_aux.clone()
    layer = MoELayer.from_workload(wl, inp, overlap=overlap)
    marks = [torch.cuda.Event(enable_timing=True, external=True)
             for _ in range(len(layer.stage_names()) + 1)]
    n = layer.capture(inp["x"], marks=marks)
    assert n >= 7
    for _ in range(2):
        layer.y.zero_()
        layer.l_aux.zero_()
        layer.replay()
        torch.cuda.synchronize()
        assert torch.equal(layer.y, y_ref) and torch.equal(layer.l_aux, l_ref)
        assert marks[0].elapsed_time(marks[-1]) > 0
    layer.check_device_status()


def test_shared_expert_beside_routed_gemms_matches():
    """The shared expert on a few SMs beside the routed expert GEMMs (SM budgets set per
    call with moe_set_gemm_sms) gives exactly the default schedule's output, eager and
    replayed from a CUDA graph; the budget is back at 0 afterwards."""
    wl = Workload("shared_beside", 2048, 256, 16, 4, 512, "bf16", None, bias="normal",
                  shared=True)
    inp = make_inputs(wl, "cuda")
    base = MoELayer.from_workload(wl, inp)
    base.forward(inp["x"])
    torch.cuda.synchronize()
    y_ref = base.y.clone()
    layer = MoELayer.from_workload(wl, inp, shared_sms=16)
    layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert torch.equal(layer.y, y_ref)
    layer.capture(inp["x"])
    layer.y.zero_()
    layer.replay()
    torch.cuda.synchronize()
    assert torch.equal(layer.y, y_ref)
    layer.check_device_status()


@pytest.mark.parametrize("mode", [N.GEMM_SINGLE, N.GEMM_PAIR, N.GEMM_SPLIT, N.GEMM_PAIR_T,
                                  N.GEMM_MIXED],
                         ids=["single", "pair", "split", "pair_t", "mixed"])
def test_gemm_sm_budget_gives_same_result(mode):
    """An expert GEMM limited to a few SMs computes the same values as on all of them."""
    offs = [0, 300, 812, 813, 1400]
    G, rows, Kd, Nn = 4, 1400, 512, 768
    cfg = N.make_config(rows, Kd, G, 1, Nn, "bf16", -1)
    ws = torch.zeros(N.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    a = torch.randn((rows, Kd), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((G, Nn, Kd), generator=g, device="cuda") * Kd ** -0.5).to(torch.bfloat16)
    off_t = torch.tensor(offs, dtype=torch.int32, device="cuda")
    outs = []
    N.set_gemm_pairing(mode)
    try:
        for budget in (0, 12):
            N.set_gemm_sms(budget)
            h = torch.zeros((rows, Nn), dtype=torch.float16, device="cuda")
            N.expert_up(cfg, a, off_t, G, rows, w, h, ws)
            outs.append(h)
    finally:
        N.set_gemm_sms(0)
        N.set_gemm_pairing(N.GEMM_AUTO)
    assert N.sync_status(ws) == 0
    assert torch.equal(outs[0], outs[1])


def test_host_stream_pipeline_matches_eager():
    """Pipelined host-buffer forwards (two device slots, uploads/downloads on their own
    streams) give, batch by batch, exactly the eager forward's output and statistics,
    with different inputs alternating so a slot mix-up would show."""
    from routing_dispatch_expert_04_b300.layer import HostStream
    wl = SMALL[4]                                   # bf16, bias, shared expert
    inp = make_inputs(wl, "cuda")
    x2 = make_inputs(wl, "cuda", seed=1, weights=False)["x"]
    layer = MoELayer.from_workload(wl, inp)
    refs = []
    for x in (inp["x"], x2):
        layer.forward(x)
        torch.cuda.synchronize()
        refs.append((layer.y.clone().cpu(), torch.cat([layer.f, layer.P, layer.l_aux]).cpu()))
    hs = HostStream(layer, inp["x"])
    xs = [inp["x"].cpu().pin_memory(), x2.cpu().pin_memory()]
    n = 6
    ys = [torch.empty((wl.T, wl.d), dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    sts = [torch.empty(2 * wl.E + 1, dtype=torch.float32).pin_memory() for _ in range(n)]
    for i in range(n):
        hs.run(xs[i & 1], ys[i], sts[i])
    torch.cuda.synchronize()
    layer.check_device_status()
    for i in range(n):
        assert torch.equal(ys[i], refs[i & 1][0]), i
        assert torch.equal(sts[i], refs[i & 1][1]), i


def test_split_plan_captured_matches_eager_and_oracle():
    """A layer whose experts hold whole 256-row tiles plus a remainder (C = 320 -> 256 +
    64) takes the split plan: the pair kernel and the one-CTA kernel run concurrently,
    the second on the library's side stream.  Captured in a CUDA graph, it reproduces the
    eager forward bit for bit, and the eager forward matches the oracle."""
    wl = Workload("split_case", 2048, 512, 8, 2, 1024, "bf16", 1.25)
    assert N.capacity(wl.T, wl.E, wl.capacity_factor) == 320
    inp = make_inputs(wl, "cuda")
    layer = MoELayer.from_workload(wl, inp)
    x_np = to_np(inp["x"])
    _, L32 = O.router_logits(x_np, to_np(inp["w_r"]), None)
    layer.forward(inp["x"], logits_in=torch.from_numpy(L32).cuda())
    layer.check_device_status()
    ref = O.moe_forward(x_np, to_np(inp["w_r"]), None, to_np(inp["w1"]), to_np(inp["w2"]),
                        wl.K, 320, wl.alpha, logits32=L32)
    assert np.array_equal(to_np(layer.offsets), ref["offsets"])
    err, literal = layer_output_error(to_np(layer.y), ref["y"], "bf16")
    assert err <= TOL["bf16"], (err, literal)
    layer.forward(inp["x"])
    torch.cuda.synchronize()
    y_eager = layer.y.clone()
    layer.capture(inp["x"])
    for _ in range(2):
        layer.y.zero_()
        layer.replay()
        torch.cuda.synchronize()
        assert torch.equal(layer.y, y_eager)
    layer.check_device_status()


def test_dispatch_reuses_its_workspace_across_calls_and_sizes():
    """Consecutive dispatch calls on one workspace, with the scan spanning different
    numbers of chunks (3, 1, 8, 3 chunks of 4096 assignments), each match the oracle's
    plan: the scan's ticket is reset and its look-back descriptors carry each call's epoch,
    so no stale descriptor of an earlier call is ever taken for a published one."""
    E, K = 16, 2
    cfg_big = N.make_config(16384, 8, E, K, 8, "bf16", 1500)
    ws = torch.zeros(N.workspace_size(cfg_big), dtype=torch.uint8, device="cuda")
    for i, T in enumerate((6000, 1000, 16384, 6000)):
        cfg = N.make_config(T, 8, E, K, 8, "bf16", T * 3 // E // 2)
        C = cfg.capacity
        L32 = make_logits(T, E, seed=40 + i, ties=(i % 2 == 1)).numpy()
        logits = torch.from_numpy(L32).cuda()
        ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, K), dtype=torch.float32, device="cuda")
        counts = torch.empty(E, dtype=torch.int32, device="cuda")
        offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        slot = torch.empty((T, K), dtype=torch.int32, device="cuda")
        src = torch.empty(T * K, dtype=torch.int32, device="cuda")
        N.route(cfg, None, None, None, logits, ids, w, ws)
        N.dispatch(cfg, None, ids, counts, offsets, slot, src, None, ws)
        assert N.sync_status(ws) == 0
        plan = O.dispatch_plan(O.top_k(L32, K), E, C)
        assert np.array_equal(to_np(counts), plan["counts"]), T
        assert np.array_equal(to_np(offsets), plan["offsets"]), T
        assert np.array_equal(to_np(slot).reshape(-1), plan["slot"]), T
