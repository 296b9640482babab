"""Comparison utilities shared by the GPU parity tests (no method arithmetic: the
expected values always come from the oracle)."""

from __future__ import annotations

import numpy as np
import torch


def to_np(t):
    """Exact host copy of a device tensor (bf16 widened to fp32, which is exact)."""
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def rel_rms_err(got, ref) -> float:
    """max |got - ref| / RMS(ref)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = np.sqrt(np.mean(ref ** 2))
    if rms == 0:
        return float(np.max(np.abs(got - ref)))
    return float(np.max(np.abs(got - ref)) / rms)


def comparable_tokens(L32, ids, K: int, C: int, thr: float = 1e-4) -> np.ndarray:
    """Tokens whose end-to-end output is a fixed function of routing decisions that fp32
    logits from another rounding path cannot flip.

    Excluded: tokens whose K-th and (K+1)-th largest logits differ by less than ``thr``,
    and -- when capacity is finite -- every token with an assignment, later in flat order,
    to an expert that an excluded token picked or could have picked (its arrival position
    may shift, which can change which assignments are dropped)."""
    L32 = np.asarray(L32, dtype=np.float64)
    T, E = L32.shape
    srt = -np.sort(-L32, axis=1)
    if K < E:
        gap = srt[:, K - 1] - srt[:, K]
    else:
        gap = np.full(T, np.inf)
    excl = gap < thr
    keep = ~excl
    if C < 0 or not excl.any():
        return keep
    flat = np.asarray(ids).reshape(-1)
    first = np.full(E, np.iinfo(np.int64).max)
    for t in np.nonzero(excl)[0]:
        cand = np.nonzero(L32[t] >= srt[t, K - 1] - thr)[0]
        first[cand] = np.minimum(first[cand], t * K)
    a = np.arange(flat.size)
    hit = a >= first[flat]
    keep[np.unique(a[hit] // K)] = False
    return keep


def assert_rounded_to(got, ref, dtype: str, acc_rel: float = 1e-4):
    """Elementwise: |got - ref| <= u * |ref| + acc_rel * RMS(ref), with u the unit
    roundoff of the storage type (2^-8 bf16, 2^-11 fp16, 2^-24 fp32): a value stored once in
    that type after an fp32-accumulated computation."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return
    u = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 2.0 ** -24}[dtype]
    rms = np.sqrt(np.mean(ref ** 2))
    bound = u * np.abs(ref) + acc_rel * rms
    excess = np.abs(got - ref) - bound
    i = int(np.argmax(excess))
    assert excess.flat[i] <= 0, (f"element {i}: got {got.flat[i]!r} ref {ref.flat[i]!r} "
                                 f"bound {bound.flat[i]!r}")


def half_ulp(ref, dtype: str):
    """Half a unit in the last place of |ref| in the output type (0 where ref == 0)."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    p = {"bf16": 8, "f16": 11, "f32": 24}[dtype]
    e = np.floor(np.log2(np.where(ref > 0, ref, 1.0)))
    return np.where(ref > 0, 2.0 ** (e - p), 0.0)


def layer_output_error(got, ref, dtype: str):
    """(metric, literal) for a layer output stored in ``dtype``.

    literal = max|got - ref| / RMS(ref).  For bf16 outputs that bound is dominated by the
    output's own rounding (an exactly computed result rounded to bf16 already reaches
    0.02-0.04 on these workloads), so the metric compared with the tolerance is the error
    in excess of half an output ulp: max(|got - ref| - ulp(ref)/2, 0) / RMS(ref).  For
    fp32 outputs metric = literal."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0, 0.0
    rms = np.sqrt(np.mean(ref ** 2))
    rms = rms if rms > 0 else 1.0
    err = np.abs(got - ref)
    literal = float(err.max() / rms)
    if dtype == "f32":
        return literal, literal
    return float(np.maximum(err - half_ulp(ref, dtype), 0).max() / rms), literal
