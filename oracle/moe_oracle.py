"""Plain, slow, fp64 CPU oracle for the forward pass of one mixture-of-experts FFN layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or run this
module: only the test suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
reference leg of ``bench.py`` use it.  It shares no code with the CUDA library and imports
nothing from it; both sides are fed the same seeded synthetic tensors.

Every step is the plain definition written out in float64 over the *stored* input values
(bf16 or fp32 widened exactly), with numpy's matmul, argsort and bincount and
scipy's erf as library primitives.  Nothing is blocked, fused or reordered beyond the
definition.

Sources (web pages on expert parallelism, cited by title and section):

* [EPM] "Expert Parallelism (MoE)":
    - "MoE Layer Structure"                      -> dense FFN, router, top-K, combine
    - "The All-to-All Communication"             -> the dispatch example (packing)
    - "Load Balancing: The Auxiliary Loss"       -> f_i, P_i, L_aux
    - "Top-K Routing and Capacity Factor"        -> capacity and token dropping
* [EPH] "Expert Parallelism (EP)", "Key math / How it works" and "Load balancing"
        -> the four steps route / dispatch / expert GEMMs / combine; overflow tokens
        skip the expert; DeepSeek-V3's shared expert.

Readings taken where the pages are silent, garbled or inconsistent:

* Logits are computed in fp64 and rounded once to fp32 (``L32``); routing decisions
  (top-K) are taken on ``L32`` so that a GPU kernel fed the same fp32 logits must
  reproduce them bit for bit.
* Softmax over all E experts, then top-K on the logits (softmax is monotone).
* Top-K order: logit descending, exact ties broken by the lower expert id.
* Routing weight = the softmax probability of the chosen expert, no renormalisation
  over the K chosen experts (``renormalize=True`` gives w / sum_k w as a variant).
* Capacity C = floor(T * capacity_factor / E), counting tokens as printed; a negative or
  ``None`` capacity means no dropping.
* An assignment (t, k) is dropped iff it arrives when its expert already holds C
  assignments, in flat token-major order a = t*K + k.  A dropped assignment contributes
  exactly 0; a token with all assignments dropped gets Y = 0 (plus the shared expert).
* Within an expert's packed block, rows are in ascending flat-assignment order.
* GELU is the exact erf form; expert Linears have no bias.
* f_i = fraction of the T*K top-K assignments (before dropping) that chose expert i;
  P_i = mean over tokens of the softmax probability of expert i;
  L_aux = alpha * sum_i f_i * P_i with no extra factor of E.  The loss is reported,
  never added to Y.
* The shared expert (DeepSeek-V3 style) has weight 1 and is added to Y for every token.

Routing variants (readings; the pages name these schemes without fixing them):

* Selection-only expert bias ([EPH] "Load balancing": DeepSeek-V3's auxiliary-loss-free
  bias-adjustment scheme).  A per-expert bias b_i is added to the fp32 logits (one fp32
  addition, round to nearest even) for choosing the top-K experts only; routing weights
  and P_i stay those of the unbiased softmax.  After a step the bias is nudged toward
  balance: b_i <- b_i + gamma * sign(T*K/E - count_i) (raise under-loaded experts, lower
  over-loaded ones; an expert at exactly the mean keeps its bias), one fp32 addition.
* Slot-major drop priority: assignments arrive in the order a' = k*T + t (every token's
  first choice before any second choice), instead of flat token-major order; rows of
  an expert's packed block follow the same arrival order.
* Capacity counted in assignments: C_K = floor((T*K / E) * capacity_factor), the reading
  under which "capacity is rarely hit" when the load is balanced.

Parity is pinned for every function here by the CPU tests (worked dispatch example,
closed forms of the aux loss, the E=1 reduction to the dense FFN, brute-force dense
evaluation, brute-force top-K and capacity, tabulated values of the normal CDF).  The
variants above and ``renormalize=True`` are readings, not fixed by the pages: the tests
pin the oracle to those readings (reductions to the default path, brute force, hand
cases), but parity with the pages is unpinned for them beyond the reading; for the
bias adjustment rule in particular it is "parity unpinned".
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
from scipy.special import erf as _erf


def widen(a) -> np.ndarray:
    """Exact widening of stored values (fp32 / bf16-as-fp32 / int) to float64."""
    return np.asarray(a, dtype=np.float64)


def linear(x, w) -> np.ndarray:
    """A Linear layer without bias in fp64, weights stored [out, in]: x . W^T."""
    return widen(x) @ widen(w).T


# --------------------------------------------------------------------------------------
# Router: [EPM] "MoE Layer Structure" -- Router (Linear d -> N_experts).
# --------------------------------------------------------------------------------------
def router_logits(x, w_r, b_r=None):
    """L = x . W_r^T (+ b_r) in fp64; returns (L64 [T,E] float64, L32 [T,E] float32).

    x: [T, d]; w_r: [E, d] (Linear layout, out x in); b_r: [E] or None.
    """
    L = linear(x, w_r)
    if b_r is not None:
        L = L + widen(b_r)[None, :]
    return L, L.astype(np.float32)


def softmax(L32) -> np.ndarray:
    """Row softmax over all E experts, in fp64, max-subtracted ([EPM] aux-loss section:
    "router probability ... after softmax")."""
    z = widen(L32)
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=1, keepdims=True)


def selection_scores(L32, sel_bias=None) -> np.ndarray:
    """Scores the top-K choice compares: the fp32 logits, or with a selection-only bias
    (DeepSeek-V3's bias-adjustment scheme, [EPH] "Load balancing") the fp32 sum
    L32 + b, rounded once to fp32."""
    L32 = np.asarray(L32, dtype=np.float32)
    if sel_bias is None:
        return L32
    return (L32 + np.asarray(sel_bias, dtype=np.float32)[None, :]).astype(np.float32)


def top_k(L32, K: int, sel_bias=None) -> np.ndarray:
    """Top-K experts per token ([EPM] "MoE Layer Structure": "the top-K experts are
    activated"; [EPH] step 1).  Order: fp32 score descending, ties -> lower expert id;
    the score is the logit, plus the selection-only bias when one is given.

    A stable sort of the negated fp32 values keeps equal values in index order.
    """
    S = selection_scores(L32, sel_bias)
    order = np.argsort(-S, axis=1, kind="stable")
    return order[:, :K].astype(np.int32)


def routing_weights(p, ids, renormalize: bool = False) -> np.ndarray:
    """w[t,k] = p[t, ids[t,k]]; optionally renormalised over the K chosen experts."""
    w = np.take_along_axis(widen(p), np.asarray(ids, dtype=np.int64), axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return w


# --------------------------------------------------------------------------------------
# Capacity and dropping: [EPM] "Top-K Routing and Capacity Factor"; [EPH] "Load balancing".
# --------------------------------------------------------------------------------------
def capacity(T: int, E: int, capacity_factor) -> int:
    """C = floor((T / E) * capacity_factor), exactly (rational arithmetic).

    ``capacity_factor=None`` means no dropping and returns -1.
    """
    if capacity_factor is None:
        return -1
    return math.floor(Fraction(T) / E * Fraction(capacity_factor))


def capacity_assignments(T: int, E: int, K: int, capacity_factor) -> int:
    """C_K = floor((T * K / E) * capacity_factor) exactly: the capacity read as counting
    top-K assignments rather than tokens (variant).  ``None`` -> -1 (no dropping)."""
    if capacity_factor is None:
        return -1
    return math.floor(Fraction(T * K) / E * Fraction(capacity_factor))


def arrival_order(T: int, K: int, order: str = "token") -> np.ndarray:
    """Flat assignment indices a = t*K + k in the order assignments arrive at the
    experts: token-major (t, then k) by default; "slot" is slot-major (k, then t)."""
    a = np.arange(T * K, dtype=np.int64)
    if order == "token":
        return a
    if order == "slot":
        return a.reshape(T, K).T.reshape(-1)
    raise ValueError(order)


def dispatch_plan(ids, E: int, C: int, order: str = "token"):
    """Histogram, capacity, drop mask and the packing permutation.

    Walk the assignments in arrival order (flat order a = t*K + k; ``order="slot"``:
    every token's k-th choice before any (k+1)-th).  An assignment's position in its
    expert is the number of assignments to the same expert that arrived before it; it
    is kept iff that position is below C (C < 0: keep all).  Kept rows of expert e are
    packed contiguously at rows [offsets[e], offsets[e+1]) in arrival order -- on one
    GPU this packing is what the all-to-all dispatch of [EPM] "The All-to-All
    Communication" and [EPH] step 2 amounts to.

    Returns dict with counts [E] (before dropping), kept [E], offsets [E+1], pos [A],
    slot [A] (packed row or -1 if dropped) and src [R] (packed row -> flat assignment).
    """
    ids_arr = np.asarray(ids, dtype=np.int64)
    flat = ids_arr.reshape(-1)
    A = flat.size
    if order == "token":
        arrivals = np.arange(A, dtype=np.int64)
    else:
        if ids_arr.ndim != 2:
            raise ValueError("slot-major arrival needs ids shaped [T, K]")
        arrivals = arrival_order(ids_arr.shape[0], ids_arr.shape[1], order)
    counts = np.zeros(E, dtype=np.int64)
    pos = np.zeros(A, dtype=np.int64)
    for a in arrivals:
        e = flat[a]
        pos[a] = counts[e]
        counts[e] += 1
    if C < 0:
        keep = np.ones(A, dtype=bool)
        kept = counts.copy()
    else:
        keep = pos < C
        kept = np.minimum(counts, C)
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + kept[e]
    R = int(offsets[E])
    slot = np.full(A, -1, dtype=np.int64)
    src = np.zeros(R, dtype=np.int64)
    for a in range(A):
        if keep[a]:
            s = offsets[flat[a]] + pos[a]
            slot[a] = s
            src[s] = a
    return {
        "counts": counts.astype(np.int32),
        "kept": kept.astype(np.int32),
        "offsets": offsets.astype(np.int32),
        "pos": pos.astype(np.int32),
        "keep": keep,
        "slot": slot.astype(np.int32),
        "src": src.astype(np.int32),
        "R": R,
    }


# --------------------------------------------------------------------------------------
# Expert FFN: [EPM] "MoE Layer Structure" -- Linear(d -> 4d) -> GELU -> Linear(4d -> d).
# --------------------------------------------------------------------------------------
def gelu(z) -> np.ndarray:
    """Exact GELU: z * Phi(z) = z * (1 + erf(z / sqrt 2)) / 2, fp64."""
    z = widen(z)
    return z * 0.5 * (1.0 + _erf(z / math.sqrt(2.0)))


def expert_ffn(x_rows, w1, w2):
    """One expert on a block of rows: h = GELU(x . W1^T), y = h . W2^T (no biases).

    x_rows: [n, d]; w1: [F, d]; w2: [d, F] (Linear layouts).  Returns (y [n,d], h [n,F]).
    """
    h = gelu(linear(x_rows, w1))
    y = linear(h, w2)
    return y, h


def dense_ffn(x, w1, w2) -> np.ndarray:
    """The standard transformer FFN of [EPM] "MoE Layer Structure" (the E=1 reduction)."""
    return expert_ffn(x, w1, w2)[0]


# --------------------------------------------------------------------------------------
# Combine: [EPM] "MoE Layer Structure" -- Y = sum over selected experts of
# expert_output[token] * routing_weight[token]; [EPH] step 4.
# --------------------------------------------------------------------------------------
def combine(y_perm, slot, w, T: int, y_shared=None) -> np.ndarray:
    """Y[t] = sum_{k ascending, slot[t,k] >= 0} w[t,k] * y_perm[slot[t,k]] (+ y_shared[t]).

    y_perm: [R, d] packed expert outputs; slot: [T, K]; w: [T, K].  Dropped slots add 0.
    """
    y_perm = widen(y_perm)
    slot = np.asarray(slot, dtype=np.int64).reshape(T, -1)
    w = widen(w).reshape(T, -1)
    d = y_perm.shape[1]
    Y = np.zeros((T, d), dtype=np.float64)
    for k in range(slot.shape[1]):
        m = slot[:, k] >= 0
        Y[m] += w[m, k, None] * y_perm[slot[m, k]]
    if y_shared is not None:
        Y += widen(y_shared)
    return Y


# --------------------------------------------------------------------------------------
# Auxiliary statistics: [EPM] "Load Balancing: The Auxiliary Loss".
# --------------------------------------------------------------------------------------
def aux_stats(ids, p, E: int, alpha: float):
    """f_i = count_i / (T*K) (pre-drop), P_i = mean_t p[t,i], L_aux = alpha * sum f_i P_i.

    With no tokens the fractions and means are empty sums: all statistics are 0."""
    ids = np.asarray(ids, dtype=np.int64)
    if ids.size == 0:
        return np.zeros(E), np.zeros(E), 0.0
    counts = np.bincount(ids.reshape(-1), minlength=E).astype(np.float64)
    f = counts / ids.size
    P = widen(p).mean(axis=0)
    return f, P, float(alpha) * float(np.sum(f * P))


def aux_loss_grad_logits(L32, ids, alpha: float) -> np.ndarray:
    """Gradient of L_aux = alpha * sum_i f_i P_i with respect to the router logits, in fp64
    ([EPM] "Load Balancing": the auxiliary loss "is added to the main task loss and
    backpropagated").

    f_i counts top-K choices, a step function of the logits: its derivative is zero
    wherever no tie is crossed, so only P_i = (1/T) sum_t softmax(L)[t,i] carries
    gradient.  With p = softmax(L[t]) and the softmax Jacobian p_i (delta_ij - p_j):
        dL_aux/dL[t,j] = (alpha / T) * p[t,j] * (f_j - sum_i f_i p[t,i]).
    """
    p = softmax(L32)
    T, E = p.shape
    if T == 0:
        return np.zeros((0, E))
    f, _, _ = aux_stats(ids, p, E, alpha)
    mean_f = p @ f
    return (float(alpha) / T) * p * (f[None, :] - mean_f[:, None])


# --------------------------------------------------------------------------------------
# FP8 expert GEMMs (variant; "Expert Parallelism (EP)", "See also": MoE is the most
# FP8-sensitive architecture).  The pages fix no FP8 recipe; the reading taken here is the
# plainest one: E4M3 values (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
# infinities, largest finite 448, smallest subnormal 2^-9), round to nearest even,
# saturating; one fp32 scale per row of each operand (per token row of the activations,
# per output channel of the weights), amax / 448.
# --------------------------------------------------------------------------------------
E4M3_MAX = 448.0


def round_e4m3(v) -> np.ndarray:
    """Nearest E4M3 value (ties to even), saturating at +-448; returned as float64."""
    v = np.clip(np.asarray(v, dtype=np.float64), -E4M3_MAX, E4M3_MAX)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)                   # below 2^-6 the spacing is that of subnormals
    quantum = np.exp2(e - 3)                # 3 mantissa bits
    q = np.round(v / quantum) * quantum     # np.round rounds halves to even
    return np.clip(q, -E4M3_MAX, E4M3_MAX)


def quantize_rows_e4m3(m):
    """Per-row E4M3 quantisation of an fp32 matrix, in fp32 arithmetic as stated:
    amax = max |row|, inv = 448 / amax, code = e4m3(row * inv), scale = amax / 448
    (a zero row gets inv = scale = 0 and codes 0).  Returns (codes as float64, scale fp32)."""
    m = np.asarray(m, dtype=np.float32)
    amax = np.max(np.abs(m), axis=1) if m.shape[1] else np.zeros(m.shape[0], np.float32)
    nz = amax > 0
    inv = np.zeros_like(amax)
    inv[nz] = (np.float32(E4M3_MAX) / amax[nz]).astype(np.float32)
    scaled = (m * inv[:, None]).astype(np.float32)
    scale = np.zeros_like(amax)
    scale[nz] = (amax[nz] / np.float32(E4M3_MAX)).astype(np.float32)
    return round_e4m3(scaled), scale


def expert_ffn_e4m3(x_rows, w1, w2):
    """One expert on E4M3 operands (variant): x rows and the weight rows quantised per
    row (quantize_rows_e4m3), h = GELU(dequantised product) in fp64 and stored in fp16
    (as the intermediate activation of bf16 layers is), h quantised per row in turn,
    y = dequantised product with W2.  Returns (y [n,d], h [n,F] before the fp16 store)."""
    xq, sx = quantize_rows_e4m3(x_rows)
    w1q, s1 = quantize_rows_e4m3(w1)
    h = gelu((xq @ w1q.T) * widen(sx)[:, None] * widen(s1)[None, :])
    hq, sh = quantize_rows_e4m3(h.astype(np.float16).astype(np.float32))
    w2q, s2 = quantize_rows_e4m3(w2)
    y = (hq @ w2q.T) * widen(sh)[:, None] * widen(s2)[None, :]
    return y, h


# --------------------------------------------------------------------------------------
# Selection-bias adjustment: [EPH] "Load balancing" (DeepSeek-V3's auxiliary-loss-free
# bias-adjustment scheme; the update rule is a reading, see the module docstring).
# --------------------------------------------------------------------------------------
def adjust_selection_bias(sel_bias, counts, T: int, K: int, gamma: float) -> np.ndarray:
    """b_i + gamma * sign(T*K/E - count_i), each sum rounded once to fp32.

    The comparison with the mean load T*K/E is exact (count_i * E against T*K in
    integers): an expert above the mean is lowered by gamma, one below is raised, one at
    the mean keeps its bias."""
    b = np.asarray(sel_bias, dtype=np.float32)
    counts = np.asarray(counts, dtype=np.int64)
    E = b.size
    sign = np.sign(T * K - counts * E).astype(np.float32)
    return (b + np.float32(gamma) * sign).astype(np.float32)


# --------------------------------------------------------------------------------------
# The whole layer.
# --------------------------------------------------------------------------------------
def moe_forward(x, w_r, b_r, w1, w2, K: int, C: int, alpha: float,
                renormalize: bool = False, shared=None, logits32=None, sel_bias=None,
                order: str = "token", experts: str = "exact"):
    """Forward pass of one MoE FFN layer, every intermediate returned.

    x [T,d]; w_r [E,d]; b_r [E] or None; w1 [E,F,d]; w2 [E,d,F];
    shared = (w1s [F,d], w2s [d,F]) or None; logits32 [T,E] float32 replaces the router
    when given (the routing stages are then driven by those exact fp32 values);
    sel_bias [E] fp32: selection-only bias; order: arrival order for dropping;
    experts: "exact" (fp64 on the stored values) or "e4m3" (expert_ffn_e4m3, the FP8
    variant; the router and the combine stay exact).
    """
    ffn = expert_ffn if experts == "exact" else expert_ffn_e4m3
    x = np.asarray(x)
    T = x.shape[0]
    E = w1.shape[0]
    if logits32 is None:
        _, L32 = router_logits(x, w_r, b_r)
    else:
        L32 = np.asarray(logits32, dtype=np.float32)
    p = softmax(L32)
    ids = top_k(L32, K, sel_bias)
    w = routing_weights(p, ids, renormalize)
    plan = dispatch_plan(ids, E, C, order)
    R = plan["R"]
    src = plan["src"].astype(np.int64)
    d = x.shape[1]
    F = w1.shape[1]
    x_perm = widen(x)[src // K] if R else np.zeros((0, d))
    h = np.zeros((R, F))
    y_perm = np.zeros((R, d))
    offs = plan["offsets"]
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            y_perm[lo:hi], h[lo:hi] = ffn(x_perm[lo:hi], w1[e], w2[e])
    y_shared = None
    if shared is not None:
        y_shared = ffn(widen(x), shared[0], shared[1])[0]
    y = combine(y_perm, plan["slot"], w, T, y_shared)
    f, P, l_aux = aux_stats(ids, p, E, alpha)
    out = dict(plan)
    out.update(L32=L32, p=p, ids=ids, w=w, x_perm=x_perm, h=h, y_perm=y_perm,
               y_shared=y_shared, y=y, f=f, P=P, l_aux=l_aux)
    return out
