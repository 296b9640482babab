"""The C-ABI library loads without a GPU and exports exactly what include/moe.h declares;
host-side argument validation rejects bad calls before any CUDA work (CPU only)."""

import ctypes
import os
import re

import pytest

from routing_dispatch_expert_04_b300 import build as B
from routing_dispatch_expert_04_b300 import native as N

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src))


def test_exports_match_header(lib):
    declared = _declared()
    assert declared == set(N.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in N.STATUS.items():
        assert lib.moe_status_string(code).decode() == name


def _cfg(**kw):
    base = dict(T=64, d=128, E=8, K=2, F=256, dtype="bf16", capacity=10)
    base.update(kw)
    return N.make_config(**base)


def test_workspace_and_rows_capacity(lib):
    c = _cfg()
    assert N.rows_capacity(c) == min(64 * 2, 8 * 10)
    assert N.rows_capacity(_cfg(capacity=-1)) == 128
    assert N.workspace_size(c) > 256 and N.workspace_size(c) % 256 == 0
    assert N.workspace_size(_cfg(K=9)) == 0          # K > E is invalid
    assert N.rows_capacity(_cfg(E=300, K=2)) == -1    # E > 256 unsupported


@pytest.mark.parametrize("kw,code", [
    (dict(K=9), 1), (dict(K=0), 1), (dict(T=-1), 1), (dict(dtype=7), 1),
    (dict(E=257, K=2), 2), (dict(K=33, E=64), 2), (dict(d=100), 2), (dict(F=12), 2),
    (dict(dtype="f32", d=6), 2),
])
def test_invalid_configs_rejected_on_host(lib, kw, code):
    c = _cfg(**kw)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    st = lib.moe_route(ctypes.byref(c), fake, fake, None, fake, fake, fake, fake, None)
    assert st == code
    st = lib.moe_combine(ctypes.byref(c), fake, fake, fake, None, fake, None)
    assert st == code


def test_null_and_misaligned_pointers_rejected(lib):
    c = _cfg()
    ok = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p((1 << 20) + 4)
    assert lib.moe_route(ctypes.byref(c), ok, ok, None, None, ok, ok, ok, None) == 1
    assert lib.moe_route(ctypes.byref(c), ok, ok, None, bad, ok, ok, ok, None) == 1
    assert lib.moe_dispatch(ctypes.byref(c), ok, ok, ok, ok, ok, ok, None, ok, None) == 1  # x w/o x_perm
    assert lib.moe_expert_up(ctypes.byref(c), ok, ok, 0, 10, ok, ok, ok, None) == 1      # n_groups 0
    assert lib.moe_expert_down(ctypes.byref(c), ok, ok, 257, 10, ok, ok, ok, None) == 1
    assert lib.moe_aux_stats(ctypes.byref(c), ok, None, ok, ok, ok, None) == 1
    assert lib.moe_sync_status(None, None) == 1


def test_gemm_settings_validated_on_host(lib):
    assert lib.moe_set_gemm_sms(-1) == 1
    assert lib.moe_set_gemm_sms(1) == 1
    assert lib.moe_set_gemm_sms(20) == 0 and lib.moe_set_gemm_sms(0) == 0
    assert lib.moe_set_gemm_pairing(9) == 1
    assert lib.moe_set_gemm_pairing(N.GEMM_AUTO) == 0


def test_capacity_binding_matches_pages_values():
    assert [N.capacity(256, 8, 1.25), N.capacity(4096, 8, 1.25), N.capacity(8192, 256, None),
            N.capacity(16384, 128, 1.5), N.capacity(65536, 8, 1.0)] == [40, 640, -1, 192, 8192]
