"""ctypes binding of the C ABI in ``include/moe.h`` -- argument marshalling only.

Every function takes torch tensors (or ``None`` for nullable pointers) and passes their
device addresses, sizes and the current CUDA stream to the library; all work runs in
the library's CUDA kernels.  A non-OK status raises :class:`MoeError`.  The library is
the in-tree ``libmoe.so``; if it is missing, loading raises instead of falling back.
"""

from __future__ import annotations

import ctypes
import math
import os
from fractions import Fraction

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe.so")

MOE_F32, MOE_BF16, MOE_F16 = 0, 1, 2
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_TIMEOUT", 5: "MOE_ERR_DEVICE"}

EXPORTS = ("moe_workspace_size", "moe_rows_capacity", "moe_route", "moe_route_select_bias",
           "moe_route_plan", "moe_dispatch_planned", "moe_adjust_select_bias", "moe_dispatch",
           "moe_dispatch_noalloc", "moe_dispatch_noalloc_status",
           "moe_expert_up", "moe_expert_up_gather", "moe_expert_down", "moe_quantize_e4m3",
           "moe_expert_up_e4m3", "moe_expert_down_e4m3", "moe_grouped_ffn", "moe_combine",
           "moe_aux_stats", "moe_aux_loss_grad", "moe_bf16_to_f16", "moe_sync_status", "moe_status_string", "moe_launch_count",
           "moe_test_arm_scan_timeout", "moe_set_gemm_pairing", "moe_set_gemm_sms")


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("F", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("renormalize", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("drop_order", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_CFG = ctypes.POINTER(MoeConfig)
_SIGS = {
    "moe_workspace_size": (ctypes.c_size_t, [_CFG]),
    "moe_rows_capacity": (ctypes.c_int64, [_CFG]),
    "moe_route": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_route_select_bias": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_route_plan": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_dispatch_planned": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_adjust_select_bias": (ctypes.c_int, [_CFG, _P, _P, ctypes.c_float, _P]),
    "moe_dispatch": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_dispatch_noalloc": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_dispatch_noalloc_status": (ctypes.c_int, [_P]),
    "moe_expert_up": (ctypes.c_int, [_CFG, _P, _P, ctypes.c_int32, ctypes.c_int64, _P, _P, _P, _P]),
    "moe_expert_up_gather": (ctypes.c_int, [_CFG, _P, _P, _P, ctypes.c_int32, ctypes.c_int64, _P, _P,
                                            _P, _P]),
    "moe_expert_down": (ctypes.c_int, [_CFG, _P, _P, ctypes.c_int32, ctypes.c_int64, _P, _P, _P, _P]),
    "moe_quantize_e4m3": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _P, _P, _P,
                                         _P]),
    "moe_expert_up_e4m3": (ctypes.c_int, [_CFG, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_int64, _P, _P,
                                          _P, _P, _P]),
    "moe_expert_down_e4m3": (ctypes.c_int, [_CFG, _P, _P, _P, ctypes.c_int32, ctypes.c_int64, _P, _P,
                                            _P, _P, _P]),
    "moe_grouped_ffn": (ctypes.c_int, [_CFG, _P, _P, ctypes.c_int32, ctypes.c_int64, _P, _P, _P, _P,
                                       _P, _P]),
    "moe_combine": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P]),
    "moe_aux_stats": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P]),
    "moe_aux_loss_grad": (ctypes.c_int, [_CFG, _P, _P, _P, _P]),
    "moe_bf16_to_f16": (ctypes.c_int, [_P, _P, ctypes.c_int64, _P, _P]),
    "moe_sync_status": (ctypes.c_int, [_P, _P]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_launch_count": (ctypes.c_uint64, []),
    "moe_test_arm_scan_timeout": (None, [ctypes.c_int32, ctypes.c_int32]),
    "moe_set_gemm_pairing": (ctypes.c_int, [ctypes.c_int32]),
    "moe_set_gemm_sms": (ctypes.c_int, [ctypes.c_int32]),
}


def lib():
    """Load the in-tree CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library {LIB_PATH} is missing: build it with "
                               "`python -m routing_dispatch_expert_04_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def capacity(T: int, E: int, capacity_factor) -> int:
    """C = floor((T / E) * capacity_factor) exactly; -1 (no dropping) for None."""
    if capacity_factor is None:
        return -1
    return math.floor(Fraction(T) / E * Fraction(capacity_factor))


DROP_TOKEN_MAJOR, DROP_SLOT_MAJOR = 0, 1


def capacity_assignments(T: int, E: int, K: int, capacity_factor) -> int:
    """C_K = floor((T * K / E) * capacity_factor) exactly (capacity counting top-K
    assignments instead of tokens); -1 for None."""
    if capacity_factor is None:
        return -1
    return math.floor(Fraction(T * K) / E * Fraction(capacity_factor))


def make_config(T, d, E, K, F, dtype, capacity=-1, renormalize=False, alpha=0.01,
                drop_order=DROP_TOKEN_MAJOR) -> MoeConfig:
    dt = {"f32": MOE_F32, "bf16": MOE_BF16}[dtype] if isinstance(dtype, str) else int(dtype)
    if isinstance(drop_order, str):
        drop_order = {"token": DROP_TOKEN_MAJOR, "slot": DROP_SLOT_MAJOR}[drop_order]
    return MoeConfig(T, d, E, K, F, dt, capacity, int(bool(renormalize)), alpha, int(drop_order))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(fn: str, st: int):
    if st != 0:
        raise MoeError(fn, st)


def workspace_size(cfg: MoeConfig) -> int:
    return lib().moe_workspace_size(ctypes.byref(cfg))


def rows_capacity(cfg: MoeConfig) -> int:
    return lib().moe_rows_capacity(ctypes.byref(cfg))


def route(cfg, x, w_r, b_r, logits, topk_ids, topk_w, ws, stream=None):
    _check("moe_route", lib().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(b_r), _ptr(logits),
                                         _ptr(topk_ids), _ptr(topk_w), _ptr(ws), _stream(stream)))


def route_select_bias(cfg, x, w_r, b_r, sel_bias, logits, topk_ids, topk_w, ws, stream=None):
    _check("moe_route_select_bias", lib().moe_route_select_bias(
        ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(b_r), _ptr(sel_bias), _ptr(logits),
        _ptr(topk_ids), _ptr(topk_w), _ptr(ws), _stream(stream)))


def route_plan(cfg, x, w_r, b_r, sel_bias, logits, topk_ids, topk_w, counts, offsets, ws,
               stream=None):
    """Routing plus the dispatch plan (counts, offsets, positions in ws) in one kernel."""
    _check("moe_route_plan", lib().moe_route_plan(
        ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(b_r), _ptr(sel_bias), _ptr(logits),
        _ptr(topk_ids), _ptr(topk_w), _ptr(counts), _ptr(offsets), _ptr(ws), _stream(stream)))


def dispatch_planned(cfg, x, topk_ids, offsets, slot, src, x_perm, ws, stream=None):
    """The dispatch permutation (slot, src, row copy) after moe_route_plan on the same ws."""
    _check("moe_dispatch_planned", lib().moe_dispatch_planned(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_ids), _ptr(offsets), _ptr(slot), _ptr(src),
        _ptr(x_perm), _ptr(ws), _stream(stream)))


def adjust_select_bias(cfg, counts, sel_bias, gamma: float, stream=None):
    _check("moe_adjust_select_bias", lib().moe_adjust_select_bias(
        ctypes.byref(cfg), _ptr(counts), _ptr(sel_bias), float(gamma), _stream(stream)))


def dispatch(cfg, x, topk_ids, counts, offsets, slot, src, x_perm, ws, stream=None):
    _check("moe_dispatch", lib().moe_dispatch(ctypes.byref(cfg), _ptr(x), _ptr(topk_ids), _ptr(counts),
                                               _ptr(offsets), _ptr(slot), _ptr(src), _ptr(x_perm),
                                               _ptr(ws), _stream(stream)))


def dispatch_noalloc(cfg, x, topk_ids, counts, offsets, slot, src, x_perm, stream=None):
    """moe_dispatch with its scratch in the library's static device array (no workspace)."""
    _check("moe_dispatch_noalloc", lib().moe_dispatch_noalloc(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_ids), _ptr(counts), _ptr(offsets), _ptr(slot),
        _ptr(src), _ptr(x_perm), _stream(stream)))


def dispatch_noalloc_status(stream=None) -> int:
    """Synchronise and return (then clear) the status code of the moe_dispatch_noalloc
    calls on the current device (0 = OK) without raising."""
    return lib().moe_dispatch_noalloc_status(_stream(stream))


def expert_up(cfg, x_perm, offsets, n_groups, rows_cap, w1, h, ws, stream=None):
    _check("moe_expert_up", lib().moe_expert_up(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), n_groups,
                                                 rows_cap, _ptr(w1), _ptr(h), _ptr(ws), _stream(stream)))


def expert_up_gather(cfg, x, src, offsets, n_groups, rows_cap, w1, h, ws, stream=None):
    """First expert Linear with the dispatch fused in: rows gathered from x by src."""
    _check("moe_expert_up_gather", lib().moe_expert_up_gather(
        ctypes.byref(cfg), _ptr(x), _ptr(src), _ptr(offsets), n_groups, rows_cap, _ptr(w1),
        _ptr(h), _ptr(ws), _stream(stream)))


def quantize_e4m3(src, codes, scales, rows_dev=None, stream=None):
    """Per-row E4M3 codes (uint8 tensor shaped like src) and fp32 scales of a 2-D fp32,
    bf16 or fp16 tensor; ``rows_dev``: optional device int32 bounding the rows done."""
    import torch
    dt = {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16, torch.float16: MOE_F16}[src.dtype]
    rows, cols = src.shape
    _check("moe_quantize_e4m3", lib().moe_quantize_e4m3(_ptr(src), dt, rows, cols, _ptr(rows_dev),
                                                         _ptr(codes), _ptr(scales), _stream(stream)))


def expert_up_e4m3(cfg, xq, x_scale, src, offsets, n_groups, rows_cap, w1q, w1_scale, h, ws,
                   stream=None):
    _check("moe_expert_up_e4m3", lib().moe_expert_up_e4m3(
        ctypes.byref(cfg), _ptr(xq), _ptr(x_scale), _ptr(src), _ptr(offsets), n_groups, rows_cap,
        _ptr(w1q), _ptr(w1_scale), _ptr(h), _ptr(ws), _stream(stream)))


def expert_down_e4m3(cfg, hq, h_scale, offsets, n_groups, rows_cap, w2q, w2_scale, y_perm, ws,
                     stream=None):
    _check("moe_expert_down_e4m3", lib().moe_expert_down_e4m3(
        ctypes.byref(cfg), _ptr(hq), _ptr(h_scale), _ptr(offsets), n_groups, rows_cap, _ptr(w2q),
        _ptr(w2_scale), _ptr(y_perm), _ptr(ws), _stream(stream)))


def expert_down(cfg, h, offsets, n_groups, rows_cap, w2, y_perm, ws, stream=None):
    _check("moe_expert_down", lib().moe_expert_down(ctypes.byref(cfg), _ptr(h), _ptr(offsets), n_groups,
                                                     rows_cap, _ptr(w2), _ptr(y_perm), _ptr(ws),
                                                     _stream(stream)))


def grouped_ffn(cfg, x_perm, offsets, n_groups, rows_cap, w1, w2, h, y_perm, ws, stream=None):
    _check("moe_grouped_ffn", lib().moe_grouped_ffn(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets),
                                                     n_groups, rows_cap, _ptr(w1), _ptr(w2), _ptr(h),
                                                     _ptr(y_perm), _ptr(ws), _stream(stream)))


def combine(cfg, y_perm, slot, topk_w, y_shared, y, stream=None):
    _check("moe_combine", lib().moe_combine(ctypes.byref(cfg), _ptr(y_perm), _ptr(slot), _ptr(topk_w),
                                             _ptr(y_shared), _ptr(y), _stream(stream)))


def aux_stats(cfg, counts, ws, f, P, l_aux, stream=None):
    _check("moe_aux_stats", lib().moe_aux_stats(ctypes.byref(cfg), _ptr(counts), _ptr(ws), _ptr(f),
                                                 _ptr(P), _ptr(l_aux), _stream(stream)))


def aux_loss_grad(cfg, logits, f, grad_logits, stream=None):
    """Gradient of the auxiliary loss with respect to the router logits."""
    _check("moe_aux_loss_grad", lib().moe_aux_loss_grad(ctypes.byref(cfg), _ptr(logits), _ptr(f),
                                                         _ptr(grad_logits), _stream(stream)))


def bf16_to_f16(src, dst, ws, stream=None):
    _check("moe_bf16_to_f16", lib().moe_bf16_to_f16(_ptr(src), _ptr(dst), src.numel(), _ptr(ws),
                                                     _stream(stream)))


def sync_status(ws, stream=None) -> int:
    """Synchronise and return the device status code (0 = OK) without raising."""
    return lib().moe_sync_status(_ptr(ws), _stream(stream))


def launch_count() -> int:
    return lib().moe_launch_count()


GEMM_AUTO, GEMM_SINGLE, GEMM_PAIR, GEMM_SPLIT, GEMM_PAIR_T, GEMM_MIXED = 0, 1, 2, 3, 4, 5


def set_gemm_pairing(mode: int):
    """Kernel choice for the bf16 expert GEMMs: GEMM_AUTO, GEMM_SINGLE, GEMM_PAIR,
    GEMM_SPLIT (pairs for whole 256-row tiles, one CTA for the rest), GEMM_PAIR_T
    (pairs with the tokens on the MMA's N side) or GEMM_MIXED (pairs for whole 256-row
    tiles and transposed pair tiles for the rest, in one launch)."""
    _check("moe_set_gemm_pairing", lib().moe_set_gemm_pairing(mode))


def set_gemm_sms(n: int):
    """SM budget of the expert GEMMs (0: all SMs), read when a GEMM call is made."""
    _check("moe_set_gemm_sms", lib().moe_set_gemm_sms(n))


def num_sms(device=None) -> int:
    import torch
    return torch.cuda.get_device_properties(device if device is not None else
                                            torch.cuda.current_device()).multi_processor_count


def arm_scan_timeout(skip_block: int, spin_limit: int):
    lib().moe_test_arm_scan_timeout(skip_block, spin_limit)
