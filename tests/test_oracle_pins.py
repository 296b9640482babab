"""Pins for the fp64 oracle: values and properties fixed by the expert-parallelism pages
or by mathematics, each computed here by a route other than the oracle's own code.

CPU only.  Sources: "Expert Parallelism (MoE)" sections "MoE Layer Structure",
"The All-to-All Communication", "Load Balancing: The Auxiliary Loss", "Top-K Routing and
Capacity Factor"; "Expert Parallelism (EP)" section "Key math / How it works".
"""

import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- dispatch packing
def test_worked_dispatch_example():
    """The pages' example: T1, T3 -> expert 0; T2 -> expert 1; T4 -> expert 3."""
    g = _load("dispatch_worked_example.json")
    ids = np.array(g["topk_ids"], dtype=np.int32)
    plan = O.dispatch_plan(ids, g["E"], -1)
    ex = g["expected"]
    assert plan["counts"].tolist() == ex["counts"]
    assert plan["offsets"].tolist() == ex["offsets"]
    assert plan["src"].tolist() == ex["src"]
    assert plan["slot"].tolist() == ex["slot"]
    order = [g["tokens"][a // g["K"]] for a in plan["src"]]
    assert order == ex["packed_order"]


def test_worked_example_with_capacity_one():
    """Same routing with capacity 1: T3 arrives when expert 0 already holds T1, so T3 is
    the one dropped ("tokens that would push an expert over capacity are dropped")."""
    g = _load("dispatch_worked_example.json")
    ids = np.array(g["topk_ids"], dtype=np.int32)
    plan = O.dispatch_plan(ids, g["E"], 1)
    assert plan["counts"].tolist() == [2, 1, 0, 1]
    assert plan["kept"].tolist() == [1, 1, 0, 1]
    assert plan["offsets"].tolist() == [0, 1, 2, 2, 3]
    assert plan["slot"].tolist() == [0, 1, -1, 2]
    assert plan["src"].tolist() == [0, 1, 3]


# ---------------------------------------------------------------- capacity
@pytest.mark.parametrize("T,E,cf,C", [
    (256, 8, 1.25, 40), (4096, 8, 1.25, 640), (8192, 256, None, -1),
    (16384, 128, 1.5, 192), (65536, 8, 1.0, 8192), (10, 3, 1.0, 3), (7, 2, 1.5, 5),
])
def test_capacity_formula(T, E, cf, C):
    """capacity = (tokens_per_batch / N_experts) * capacity_factor, floored."""
    assert O.capacity(T, E, cf) == C


def _bruteforce_keep(ids_flat, E, C):
    """Capacity by a second route: one-hot cumulative sums give each assignment's
    1-based arrival number within its expert."""
    A = ids_flat.size
    onehot = np.zeros((A, E), dtype=np.int64)
    onehot[np.arange(A), ids_flat] = 1
    arrival = np.cumsum(onehot, axis=0)[np.arange(A), ids_flat]  # 1-based
    return (arrival <= C) if C >= 0 else np.ones(A, bool), arrival - 1


@pytest.mark.parametrize("seed,T,E,K,C", [
    (0, 64, 8, 2, 10), (1, 50, 4, 1, 7), (2, 33, 16, 4, 5), (3, 40, 8, 2, -1),
    (4, 1, 1, 1, 0), (5, 20, 3, 3, 100), (6, 100, 5, 2, 0),
])
def test_capacity_and_drop_invariants(seed, T, E, K, C):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    plan = O.dispatch_plan(ids, E, C)
    keep_bf, pos_bf = _bruteforce_keep(ids.reshape(-1).astype(np.int64), E, C)
    assert np.array_equal(plan["keep"], keep_bf)
    assert np.array_equal(plan["pos"], pos_bf)
    counts_bf = np.bincount(ids.reshape(-1), minlength=E)
    assert np.array_equal(plan["counts"], counts_bf)
    kept = plan["kept"]
    if C >= 0:
        assert (kept <= C).all()
    dropped = int((plan["slot"] < 0).sum())
    assert int(kept.sum()) == T * K - dropped == plan["R"]
    offs = plan["offsets"]
    assert offs[0] == 0 and (np.diff(offs) == kept).all()
    # slot and src are inverse permutations on the kept assignments
    src, slot = plan["src"], plan["slot"]
    assert np.array_equal(slot[src], np.arange(plan["R"]))
    # each expert's block holds only its own assignments, in ascending flat order
    flat = ids.reshape(-1)
    for e in range(E):
        blk = src[offs[e]:offs[e + 1]]
        assert (flat[blk] == e).all()
        assert (np.diff(blk) > 0).all()


# ---------------------------------------------------------------- top-K
def _bruteforce_topk(row, K):
    """Selection by repeated maximum of (value, -index): K passes over the row."""
    chosen = []
    for _ in range(K):
        best = None
        for e, v in enumerate(row):
            if e in chosen:
                continue
            if best is None or v > row[best]:
                best = e
        chosen.append(best)
    return chosen


@pytest.mark.parametrize("seed,E,K,ties", [(0, 8, 2, False), (1, 8, 2, True),
                                           (2, 16, 8, True), (3, 5, 5, True), (4, 33, 3, False)])
def test_topk_bruteforce(seed, E, K, ties):
    rng = np.random.default_rng(seed)
    L = rng.standard_normal((60, E)).astype(np.float32)
    if ties:
        L = (np.round(L * 2) / 2).astype(np.float32)
    ids = O.top_k(L, K)
    for t in range(L.shape[0]):
        assert ids[t].tolist() == _bruteforce_topk(L[t].tolist(), K)


def test_topk_hand_ties():
    L = np.array([[1.0, 3.0, 3.0, 2.0], [0.0, 0.0, 0.0, 0.0], [-1.0, -0.0, 0.0, -2.0]],
                 dtype=np.float32)
    assert O.top_k(L, 2).tolist() == [[1, 2], [0, 1], [1, 2]]
    assert O.top_k(L, 3).tolist() == [[1, 2, 3], [0, 1, 2], [1, 2, 0]]


# ---------------------------------------------------------------- softmax
def test_softmax_values():
    p = O.softmax(np.array([[0.0, math.log(3.0)], [5.0, 5.0], [7.0, -1e30]], dtype=np.float32))
    assert np.allclose(p, [[0.25, 0.75], [0.5, 0.5], [1.0, 0.0]], rtol=1e-7, atol=0)
    assert O.softmax(np.array([[123.0]], dtype=np.float32))[0, 0] == 1.0
    rng = np.random.default_rng(0)
    p = O.softmax(rng.standard_normal((100, 37)).astype(np.float32) * 10)
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-14)


# ---------------------------------------------------------------- GELU and the FFN
def test_gelu_normal_cdf_table():
    table = _load("normal_cdf_table.json")["phi"]
    for z, phi in table.items():
        z = float(z)
        assert abs(float(O.gelu(z)) - z * phi) <= 1e-15 * max(1.0, abs(z))
    assert O.gelu(0.0) == 0.0
    assert abs(float(O.gelu(10.0)) - 10.0) < 1e-20 + 1e-15
    assert abs(float(O.gelu(-10.0))) < 1e-20


def test_expert_ffn_hand_cases():
    """Linear(d->F) -> GELU -> Linear(F->d) with Linear weights stored [out, in]."""
    phi = {float(k): v for k, v in _load("normal_cdf_table.json")["phi"].items()}
    g1, gm1 = 1.0 * phi[1.0], -1.0 * phi[-1.0]
    # d=1, F=2
    y, h = O.expert_ffn(np.array([[1.0]]), np.array([[1.0], [-1.0]]), np.array([[2.0, 3.0]]))
    assert np.allclose(h, [[g1, gm1]], rtol=1e-15)
    assert np.allclose(y, [[2 * g1 + 3 * gm1]], rtol=1e-14)
    # d=2, F=1, asymmetric weights catch a transposed operand
    y, h = O.expert_ffn(np.array([[1.0, 0.0]]), np.array([[1.0, 2.0]]), np.array([[1.0], [5.0]]))
    assert np.allclose(h, [[g1]], rtol=1e-15)
    assert np.allclose(y, [[g1, 5 * g1]], rtol=1e-14)
    # two rows, second has x=[0.5, 0] -> z=0.5
    y, _ = O.expert_ffn(np.array([[1.0, 0.0], [0.5, 0.0]]), np.array([[1.0, 2.0]]),
                        np.array([[1.0], [5.0]]))
    assert np.allclose(y[1], [0.5 * phi[0.5], 2.5 * phi[0.5]], rtol=1e-14)


def _tiny_inputs(seed, T, d, E, F, bias=False):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d)).astype(np.float32)
    w_r = (rng.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
    b_r = rng.standard_normal(E).astype(np.float32) if bias else None
    w1 = (rng.standard_normal((E, F, d)) / math.sqrt(d)).astype(np.float32)
    w2 = (rng.standard_normal((E, d, F)) / math.sqrt(F)).astype(np.float32)
    return x, w_r, b_r, w1, w2


def test_single_expert_reduces_to_dense_ffn():
    """E=1, K=1, no drop: softmax over one expert is exactly 1 and every token goes to
    that expert, so the layer is the standard FFN of "MoE Layer Structure"."""
    x, w_r, b_r, w1, w2 = _tiny_inputs(0, 37, 16, 1, 24, bias=True)
    out = O.moe_forward(x, w_r, b_r, w1, w2, K=1, C=-1, alpha=0.01)
    assert (out["w"] == 1.0).all()
    dense = O.dense_ffn(x, w1[0], w2[0])
    assert np.array_equal(out["y"], dense)


@pytest.mark.parametrize("seed,T,E,K,cf,renorm,shared", [
    (0, 256, 8, 2, 1.25, False, False),
    (1, 64, 4, 2, 0.5, False, True),
    (2, 48, 6, 3, None, True, False),
    (3, 80, 8, 1, 1.0, False, False),
])
def test_bruteforce_dense_evaluation(seed, T, E, K, cf, renorm, shared):
    """Evaluate every expert on every token, mask to (top-K and kept), weight and sum;
    it must equal the routed, packed, combined output."""
    d, F = 12, 20
    x, w_r, b_r, w1, w2 = _tiny_inputs(seed, T, d, E, F, bias=True)
    sh = None
    if shared:
        rng = np.random.default_rng(100 + seed)
        sh = (rng.standard_normal((F, d)) / math.sqrt(d), rng.standard_normal((d, F)) / math.sqrt(F))
    C = O.capacity(T, E, cf)
    out = O.moe_forward(x, w_r, b_r, w1, w2, K=K, C=C, alpha=0.01, renormalize=renorm, shared=sh)
    L = (x.astype(np.float64) @ w_r.astype(np.float64).T + b_r.astype(np.float64)).astype(np.float32)
    ids = np.array([_bruteforce_topk(L[t].tolist(), K) for t in range(T)])
    keep, _ = _bruteforce_keep(ids.reshape(-1), E, C)
    keep = keep.reshape(T, K)
    Y = np.zeros((T, d))
    for t in range(T):
        z = L[t].astype(np.float64)
        p = np.exp(z - z.max()); p /= p.sum()
        wsel = p[ids[t]]
        if renorm:
            wsel = wsel / wsel.sum()
        for k in range(K):
            if keep[t, k]:
                e = ids[t, k]
                h = x[t].astype(np.float64) @ w1[e].astype(np.float64).T
                h = h * 0.5 * (1.0 + np.array([math.erf(v / math.sqrt(2)) for v in h]))
                Y[t] += wsel[k] * (h @ w2[e].astype(np.float64).T)
        if shared:
            h = x[t].astype(np.float64) @ sh[0].T
            h = h * 0.5 * (1.0 + np.array([math.erf(v / math.sqrt(2)) for v in h]))
            Y[t] += h @ sh[1].T
    scale = np.sqrt(np.mean(Y ** 2))
    assert np.max(np.abs(out["y"] - Y)) <= 1e-12 * scale


def test_dropped_assignment_contributes_zero():
    x, w_r, _, w1, w2 = _tiny_inputs(0, 3, 8, 2, 8)
    L = np.array([[5.0, 0.0]] * 3, dtype=np.float32)  # all three tokens pick expert 0
    out = O.moe_forward(x, w_r, None, w1, w2, K=1, C=1, alpha=0.01, logits32=L)
    assert out["slot"].tolist() == [0, -1, -1]
    assert (out["y"][1:] == 0.0).all()
    assert np.abs(out["y"][0]).max() > 0


# ---------------------------------------------------------------- aux statistics
def test_aux_balanced_closed_form():
    """Each expert receives exactly T*K/E assignments and P_i = 1/E: L = alpha/E."""
    E, K, m = 8, 2, 16
    T = E * m
    ids = np.array([[(t + k) % E for k in range(K)] for t in range(T)], dtype=np.int32)
    p = np.full((T, E), 1.0 / E)
    f, P, L = O.aux_stats(ids, p, E, 0.01)
    assert np.allclose(f, 1.0 / E, rtol=0, atol=1e-16) and abs(f.sum() - 1) < 1e-15
    assert abs(L - 0.01 / E) < 1e-17


@pytest.mark.parametrize("M", [0.5, 3.0, 20.0])
def test_aux_collapsed_top1_closed_form(M):
    """All tokens on expert 0 with logit +M above the rest: f=(1,0,...), and
    P_0 = e^M / (e^M + E - 1), so L = alpha * P_0 (-> alpha as M grows)."""
    E, T, alpha = 8, 50, 0.01
    L32 = np.zeros((T, E), dtype=np.float32)
    L32[:, 0] = M
    out = O.moe_forward(np.zeros((T, 4), np.float32), np.zeros((E, 4), np.float32), None,
                        np.zeros((E, 4, 4), np.float32), np.zeros((E, 4, 4), np.float32),
                        K=1, C=-1, alpha=alpha, logits32=L32)
    P0 = math.exp(M) / (math.exp(M) + E - 1)
    assert out["f"].tolist() == [1.0] + [0.0] * (E - 1)
    assert abs(out["l_aux"] - alpha * P0) < 1e-15
    assert abs(out["P"].sum() - 1.0) < 1e-14


def test_aux_collapsed_top2_closed_form():
    """Logits (M, M, 0, ...), K=2: both tokens' picks are {0, 1}; f = (1/2, 1/2, 0, ...),
    P_0 = P_1 = e^M / (2 e^M + E - 2), L = alpha (P_0 + P_1) / 2.  Experts chosen by
    no token contribute 0."""
    E, T, alpha, M = 6, 40, 0.01, 2.0
    L32 = np.zeros((T, E), dtype=np.float32)
    L32[:, :2] = M
    out = O.moe_forward(np.zeros((T, 4), np.float32), np.zeros((E, 4), np.float32), None,
                        np.zeros((E, 4, 4), np.float32), np.zeros((E, 4, 4), np.float32),
                        K=2, C=-1, alpha=alpha, logits32=L32)
    P0 = math.exp(np.float32(M)) / (2 * math.exp(np.float32(M)) + E - 2)
    assert out["ids"].tolist() == [[0, 1]] * T
    assert np.allclose(out["f"], [0.5, 0.5, 0, 0, 0, 0], atol=0)
    assert abs(out["l_aux"] - alpha * (P0 + P0) / 2) < 1e-15
    assert (out["f"][2:] * out["P"][2:] == 0).all()


def test_aux_fraction_sums_to_one():
    rng = np.random.default_rng(7)
    L32 = rng.standard_normal((300, 16)).astype(np.float32)
    ids = O.top_k(L32, 4)
    f, P, _ = O.aux_stats(ids, O.softmax(L32), 16, 0.01)
    assert abs(f.sum() - 1.0) < 1e-14 and abs(P.sum() - 1.0) < 1e-13


def test_renormalized_weights_sum_to_one():
    rng = np.random.default_rng(8)
    L32 = rng.standard_normal((50, 8)).astype(np.float32)
    ids = O.top_k(L32, 3)
    w = O.routing_weights(O.softmax(L32), ids, renormalize=True)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-15)
    assert (np.diff(w, axis=1) <= 0).all()   # sorted by logit => by weight


def test_combine_worked_example_weights():
    """Y = sum over selected experts of expert_output * routing_weight, by hand."""
    y_perm = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0]])
    slot = np.array([[0, 2], [1, -1]])
    w = np.array([[0.5, 0.25], [2.0, 7.0]])
    Y = O.combine(y_perm, slot, w, 2)
    assert Y.tolist() == [[0.5 + 25.0, 1.0 + 50.0], [20.0, 40.0]]


def test_all_subsets_topk_small():
    """Exhaustive: for every 0/1/2-valued row of length 4, the chosen set has the largest
    value sum among K-subsets, and among equal sums the lexicographically smallest ids."""
    for vals in itertools.product([0.0, 1.0, 2.0], repeat=4):
        L = np.array([vals], dtype=np.float32)
        for K in (1, 2, 3):
            got = O.top_k(L, K)[0].tolist()
            best = max(itertools.combinations(range(4), K),
                       key=lambda s: (sum(vals[i] for i in s), [-i for i in s]))
            assert sorted(got) == list(best)
            assert [vals[i] for i in got] == sorted([vals[i] for i in got], reverse=True)


def test_aux_empty_batch_is_zero():
    f, P, L = O.aux_stats(np.zeros((0, 2), np.int32), np.zeros((0, 4)), 4, 0.01)
    assert f.tolist() == [0.0] * 4 and P.tolist() == [0.0] * 4 and L == 0.0


# ---------------------------------------------------------------- routing variants
# "Expert Parallelism (EP)", "Load balancing" names DeepSeek-V3's auxiliary-loss-free
# bias-adjustment scheme and capacity-factor dropping without fixing their details; the
# variants below are readings.  These tests pin the oracle to those readings by routes
# other than its own code: reductions to the default path, brute force, hand cases.
def test_selection_bias_zero_is_plain_topk():
    rng = np.random.default_rng(11)
    L = rng.standard_normal((50, 9)).astype(np.float32)
    assert np.array_equal(O.top_k(L, 3, np.zeros(9, np.float32)), O.top_k(L, 3))


def test_selection_bias_moves_choice_not_weights():
    """A large bias on expert 4 makes it every token's first choice, while the routing
    weights and P_i remain those of the unbiased softmax."""
    rng = np.random.default_rng(12)
    T, E, K = 40, 6, 2
    L = rng.standard_normal((T, E)).astype(np.float32)
    b = np.zeros(E, np.float32)
    b[4] = 100.0
    ids = O.top_k(L, K, b)
    assert (ids[:, 0] == 4).all()
    p = O.softmax(L)
    w = O.routing_weights(p, ids)
    # weight of the forced expert = its unbiased probability, computed here directly
    z = L.astype(np.float64)
    direct = np.exp(z[:, 4] - z.max(axis=1)) / np.exp(z - z.max(axis=1, keepdims=True)).sum(axis=1)
    assert np.allclose(w[:, 0], direct, rtol=1e-13, atol=0)
    # second choice: the best of the others by the unbiased logits
    others = np.where(np.arange(E) == 4, -np.inf, z)
    assert np.array_equal(ids[:, 1], np.argmax(others, axis=1))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_selection_bias_bruteforce(seed):
    """Top-K by the fp32 score s = fl(L + b) with (s desc, id asc), checked by Python's
    sort of explicit (key, id) pairs on a coarse grid that makes ties frequent."""
    rng = np.random.default_rng(seed)
    T, E, K = 30, 7, 3
    L = (np.round(rng.standard_normal((T, E)) * 2) / 2).astype(np.float32)
    b = (np.round(rng.standard_normal(E) * 2) / 4).astype(np.float32)
    ids = O.top_k(L, K, b)
    for t in range(T):
        keys = [(-(float(np.float32(L[t, e]) + np.float32(b[e]))), e) for e in range(E)]
        want = [e for _, e in sorted(keys)[:K]]
        assert ids[t].tolist() == want


def test_adjust_selection_bias_hand_case():
    """counts [5, 3, 0, 8] with T*K = 16 over E = 4 (mean 4): expert 0 and 3 are over the
    mean (lowered), 1 and 2 under it (raised)."""
    b = np.array([0.5, -0.25, 0.0, 1.0], np.float32)
    nb = O.adjust_selection_bias(b, [5, 3, 0, 8], T=8, K=2, gamma=0.125)
    assert nb.tolist() == [0.375, -0.125, 0.125, 0.875]
    assert nb.dtype == np.float32


def test_adjust_selection_bias_at_mean_and_rounding():
    """An expert exactly at the mean keeps its bias; the update is one fp32 addition, so
    a step below half an ulp of the bias leaves it unchanged."""
    b = np.array([1.0, 1.0, 1.0], np.float32)
    assert O.adjust_selection_bias(b, [2, 2, 2], T=3, K=2, gamma=0.5).tolist() == [1.0, 1.0, 1.0]
    tiny = O.adjust_selection_bias(b, [3, 2, 1], T=3, K=2, gamma=2.0 ** -30)
    assert tiny.tolist() == [1.0, 1.0, 1.0]


def test_slot_major_hand_case():
    """T=3, K=2, E=2, C=2, choices [[0,1],[1,0],[0,1]].  Token-major arrival drops token
    2's first choice (expert 0 already holds tokens 0 and 1); slot-major arrival takes
    every first choice before any second choice, so token 2's first choice is kept and
    token 1's second choice is dropped instead."""
    ids = np.array([[0, 1], [1, 0], [0, 1]], np.int32)
    tok = O.dispatch_plan(ids, 2, 2, "token")
    slt = O.dispatch_plan(ids, 2, 2, "slot")
    assert tok["slot"].reshape(3, 2).tolist() == [[0, 2], [3, 1], [-1, -1]]
    # slot-major: expert 0 packs (t0,k0), (t2,k0); expert 1 packs (t1,k0), (t0,k1)
    assert slt["slot"].reshape(3, 2).tolist() == [[0, 3], [2, -1], [1, -1]]
    assert slt["src"].tolist() == [0, 4, 2, 1]
    assert slt["counts"].tolist() == tok["counts"].tolist() == [3, 3]


def test_slot_major_with_one_choice_is_token_major():
    rng = np.random.default_rng(5)
    ids = rng.integers(0, 6, size=(70, 1)).astype(np.int32)
    a, b = O.dispatch_plan(ids, 6, 9, "token"), O.dispatch_plan(ids, 6, 9, "slot")
    for key in ("counts", "offsets", "slot", "src"):
        assert np.array_equal(a[key], b[key])


@pytest.mark.parametrize("seed,T,E,K,C", [(0, 64, 8, 2, 10), (1, 33, 16, 4, 5), (2, 40, 5, 3, 0),
                                          (3, 25, 4, 4, 100)])
def test_slot_major_bruteforce(seed, T, E, K, C):
    """Arrival numbers by one-hot cumulative sums over the transposed stream."""
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, K)).astype(np.int32)
    plan = O.dispatch_plan(ids, E, C, "slot")
    stream = ids.T.reshape(-1)                      # k-major: (k=0, all t), (k=1, all t)...
    keep_s, pos_s = _bruteforce_keep(stream, E, C)
    keep = keep_s.reshape(K, T).T.reshape(-1)
    pos = pos_s.reshape(K, T).T.reshape(-1)
    assert np.array_equal(plan["keep"], keep)
    assert np.array_equal(plan["pos"], pos)
    # inside each expert's block, rows follow the transposed stream
    for e in range(E):
        lo, hi = plan["offsets"][e], plan["offsets"][e + 1]
        a = plan["src"][lo:hi].astype(np.int64)
        order_key = (a % K) * T + a // K
        assert (np.diff(order_key) > 0).all()


@pytest.mark.parametrize("T,E,K,cf,C", [(256, 8, 2, 1.25, 80), (4096, 8, 2, 1.25, 1280),
                                        (16384, 128, 8, 1.5, 1536), (65536, 8, 2, 1.0, 16384),
                                        (8192, 256, 8, None, -1), (10, 3, 2, 1.0, 6)])
def test_capacity_counting_assignments(T, E, K, cf, C):
    assert O.capacity_assignments(T, E, K, cf) == C


def test_capacity_counting_assignments_balanced_load_never_drops():
    """"Capacity is rarely hit" when the load is even: with the capacity counting
    assignments and capacity_factor 1, an exactly balanced routing drops nothing."""
    T, E, K = 48, 6, 2
    ids = (np.arange(T * K) % E).reshape(T, K).astype(np.int32)  # each expert 16 times
    C = O.capacity_assignments(T, E, K, 1.0)
    plan = O.dispatch_plan(ids, E, C)
    assert C == 16 and plan["R"] == T * K and (plan["slot"] >= 0).all()
    # the capacity as printed (tokens) drops K-1 of every K assignments here
    assert O.dispatch_plan(ids, E, O.capacity(T, E, 1.0))["R"] == E * (T // E)


# ---------------------------------------------------------------- aux-loss backward
def _l_aux_full(L, K, alpha):
    """L_aux recomputed from scratch (routing included) for finite differences."""
    L32 = np.asarray(L, dtype=np.float64)
    z = L32 - L32.max(axis=1, keepdims=True)
    p = np.exp(z) / np.exp(z).sum(axis=1, keepdims=True)
    ids = np.argsort(-L32, axis=1, kind="stable")[:, :K]
    T, E = L32.shape
    f = np.bincount(ids.reshape(-1), minlength=E) / (T * K)
    return alpha * float(np.sum(f * p.mean(axis=0)))


@pytest.mark.parametrize("seed,T,E,K", [(0, 6, 5, 2), (1, 4, 8, 1), (2, 9, 3, 3)])
def test_aux_grad_matches_finite_differences(seed, T, E, K):
    """Central differences of the whole L_aux (top-K counts recomputed) equal the
    analytic gradient: steps far smaller than every logit gap cross no tie."""
    rng = np.random.default_rng(seed)
    L = rng.standard_normal((T, E))
    ids = O.top_k(L.astype(np.float32), K)
    g = O.aux_loss_grad_logits(L, ids, 0.01)
    srt = np.sort(L, axis=1)
    h = 1e-3 * np.min(np.diff(srt, axis=1))
    num = np.zeros_like(L)
    for t in range(T):
        for j in range(E):
            Lp, Lm = L.copy(), L.copy()
            Lp[t, j] += h
            Lm[t, j] -= h
            num[t, j] = (_l_aux_full(Lp, K, 0.01) - _l_aux_full(Lm, K, 0.01)) / (2 * h)
    assert np.allclose(g, num, rtol=1e-5, atol=1e-12)


def test_aux_grad_rows_sum_to_zero_and_balanced_is_zero():
    """Softmax is shift-invariant, so each token's gradient sums to zero; with f uniform
    (balanced routing) the gradient vanishes."""
    rng = np.random.default_rng(4)
    L = rng.standard_normal((12, 6))
    g = O.aux_loss_grad_logits(L, O.top_k(L.astype(np.float32), 2), 0.01)
    assert np.allclose(g.sum(axis=1), 0.0, atol=1e-18)
    ids = (np.arange(24) % 6).reshape(12, 2)
    assert np.allclose(O.aux_loss_grad_logits(L, ids, 0.01), 0.0, atol=1e-18)


# ---------------------------------------------------------------- FP8 (E4M3) quantisation
def _e4m3_table():
    """Every finite E4M3 value, enumerated from the bit fields (bias 7; exponent field 0
    is subnormal; S.1111.111 is NaN and left out)."""
    vals = set()
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
            vals.add(mag)
            vals.add(-mag)
    return np.array(sorted(vals))


def test_e4m3_values_are_the_format():
    t = _e4m3_table()
    assert t.max() == 448.0 and np.min(t[t > 0]) == 2.0 ** -9
    assert np.array_equal(O.round_e4m3(t), t)


def test_e4m3_rounding_nearest_even_and_saturating():
    t = _e4m3_table()
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(-460, 460, 4000), rng.uniform(-0.05, 0.05, 4000),
                        (t[1:] + t[:-1]) / 2])                  # exact midpoints
    q = O.round_e4m3(v)
    for x, y in zip(v, q):
        if abs(x) >= 448:
            assert y == np.sign(x) * 448
            continue
        d = np.abs(t - x)
        best = t[d == d.min()]
        if best.size == 1:
            assert y == best[0]
        else:   # tie: the candidate whose 3-bit mantissa is even
            def even(c):
                a = abs(c)
                if a < 2.0 ** -6:
                    return int(round(a / 2.0 ** -9)) % 2 == 0
                e = np.floor(np.log2(a))
                return int(round(a / 2.0 ** (e - 3))) % 2 == 0
            assert y in best and even(y)


def test_quantize_rows_reconstructs_within_half_step():
    rng = np.random.default_rng(1)
    m = (rng.standard_normal((20, 64)) * rng.uniform(0.01, 50, (20, 1))).astype(np.float32)
    m[3] = 0.0
    codes, scale = O.quantize_rows_e4m3(m)
    assert scale[3] == 0 and (codes[3] == 0).all()
    assert (np.abs(codes).max(axis=1)[np.arange(20) != 3] == 448.0).all()  # amax maps to 448
    rec = codes * scale[:, None]
    # relative spacing of E4M3 normals is 2^-3: rounding error <= 2^-4 of |x| (plus the
    # subnormal spacing 2^-10 * scale for tiny entries)
    assert (np.abs(rec - m) <= 2.0 ** -4 * np.abs(m) + 2.0 ** -10 * scale[:, None] * 1.0001).all()


def test_e4m3_expert_ffn_reduces_to_exact_on_representable_inputs():
    """When every row's entries are E4M3 values times a power of two whose row maximum is
    448 times it, quantisation is exact and the FP8 expert equals the fp64 expert up to
    the fp16 store and quantisation of h (checked by applying both to the exact h)."""
    rng = np.random.default_rng(7)
    t = _e4m3_table()
    def rep(shape):
        m = rng.choice(t[np.abs(t) <= 64], size=shape)
        m[:, 0] = 448.0
        return (m * 2.0 ** -7).astype(np.float32)
    x, w1, w2 = rep((6, 16)), rep((8, 16)), rep((16, 8))
    y8, h8 = O.expert_ffn_e4m3(x, w1, w2)
    h = O.gelu(O.linear(x, w1))
    assert np.allclose(h8, h, rtol=1e-15, atol=0)
    hq, sh = O.quantize_rows_e4m3(h.astype(np.float16).astype(np.float32))
    y = (hq * sh[:, None].astype(np.float64)) @ O.widen(w2).T
    assert np.allclose(y8, y, rtol=1e-12, atol=1e-300)
