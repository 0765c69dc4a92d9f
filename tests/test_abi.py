"""CPU checks of the C ABI: the library builds, loads without a GPU, exports
every entry point that include/*.h declares, and rejects bad arguments on the
host before any CUDA call."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import combine_ep_plan_gb300 as ep
from combine_ep_plan_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ep.load_library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(ep_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["ep_plan", "ep_dispatch", "ep_combine", "ep_dispatch_cached", "ep_dispatch_fresh",
                     "ep_plan_sizes", "ep_handle_destroy", "ep_handle_get", "ep_set_num_sms",
                     "ep_dispatch_async", "ep_combine_async", "ep_pending_wait", "ep_profile_begin",
                     "ep_profile_end"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert lib.ep_abi_version() == 4


def test_status_strings(lib):
    for code in range(7):
        assert lib.ep_status_string(code).startswith(b"EP_")


def test_worst_expanded_rows(lib):
    # T*K + E*(A-1): every real row plus the largest possible padding
    assert ep.worst_expanded_rows(16384, 6, 64, 128) == 16384 * 6 + 64 * 127
    assert ep.worst_expanded_rows(10, 2, 4, 1) == 20
    assert ep.worst_expanded_rows(10, 0, 4, 1) == -1


FAKE = 1 << 20  # never dereferenced: these calls must fail before any CUDA call


@pytest.mark.parametrize("S,P,K,E,A,C", [
    (64, 4, 2, 9, 1, 0),      # E % P != 0
    (64, 4, 2, 8, 0, 0),      # A < 1
    (64, 4, 2, 8, 1, 65),     # C > S
    (64, 4, 17, 32, 1, 0),    # K > EP_MAX_TOPK
    (64, 4, 9, 8, 1, 0),      # K > E
    (64, 0, 2, 8, 1, 0),      # P < 1
    (0, 4, 2, 8, 1, 0),       # S < 1
    (64, 2048, 2, 2048, 1, 0),  # P > EP_MAX_RANKS
    (64, 4, 2, 4096, 1, 0),   # E > EP_MAX_EXPERTS
    (1 << 28, 4, 8, 8, 1, 0),  # worst expanded rows overflow int32
])
def test_plan_rejects_bad_shapes_on_host(lib, S, P, K, E, A, C):
    h = ctypes.c_void_p(123)
    assert lib.ep_plan(FAKE, S, P, K, E, A, C, None, ctypes.byref(h)) == ep.EP_ERR_INVALID
    assert not h.value


def test_plan_rejects_null_and_misaligned(lib):
    h = ctypes.c_void_p()
    assert lib.ep_plan(None, 64, 4, 2, 8, 1, 0, None, ctypes.byref(h)) == ep.EP_ERR_INVALID
    assert lib.ep_plan(FAKE + 4, 64, 4, 2, 8, 1, 0, None, ctypes.byref(h)) == ep.EP_ERR_INVALID
    assert lib.ep_plan(FAKE, 64, 4, 2, 8, 1, 0, None, None) == ep.EP_ERR_INVALID


def test_calls_on_null_handle_are_rejected(lib):
    assert lib.ep_dispatch(None, FAKE, 0, None, 256, 0, 1, FAKE, None, 10, None) == ep.EP_ERR_INVALID
    assert lib.ep_combine(None, FAKE, 10, FAKE, None, 256, FAKE, None) == ep.EP_ERR_INVALID
    assert lib.ep_dispatch_metadata(None, FAKE, FAKE, FAKE, 10, 1, None) == ep.EP_ERR_INVALID
    assert lib.ep_sync_status(None, None) == ep.EP_ERR_INVALID
    assert lib.ep_handle_destroy(None, None) == ep.EP_ERR_INVALID
    assert lib.ep_dispatch_cached(None, 8, 1, 64, FAKE, 0, None, 256, 0, 1, FAKE, None, 10, None) == \
        ep.EP_ERR_INVALID
    h = ctypes.c_void_p()
    # fresh dispatch: bad arguments rejected before planning
    bad = [
        (FAKE, 0, None, 100, 0, 1, FAKE, None),          # H % 8 != 0
        (FAKE, 0, None, 256, 0, 1, FAKE + 8, None),      # misaligned output
        (FAKE, 0, None, 200, 1, 1, FAKE, FAKE),          # fp8 needs H % 128 == 0
        (FAKE, 1, FAKE, 256, 0, 1, FAKE, None),          # fp8 input cannot give bf16 output
        (FAKE, 1, None, 256, 1, 1, FAKE, FAKE),          # fp8 input needs its scales
        (FAKE, 0, FAKE, 256, 1, 1, FAKE, FAKE),          # bf16 input takes no scales
        (FAKE, 0, None, 256, 0, 2, FAKE, None),          # column-major scales need fp8 output
        (FAKE, 0, None, 256, 0, 8, FAKE, None),          # unknown flag
    ]
    for x, xd, xs, H, od, fl, rx, rs in bad:
        assert lib.ep_dispatch_fresh(FAKE, 64, 4, 2, 8, 1, 0, x, xd, xs, H, od, fl, rx, rs, 10, None,
                                     ctypes.byref(h)) == ep.EP_ERR_INVALID
    assert not h.value


def test_async_profile_and_budget_calls_reject_bad_arguments(lib):
    p = ctypes.c_void_p(123)
    assert lib.ep_dispatch_async(None, None, FAKE, 0, None, 256, 0, 1, FAKE, None, 10, None, None, 1,
                                 ctypes.byref(p)) == ep.EP_ERR_INVALID
    assert not p.value
    assert lib.ep_dispatch_async(None, None, FAKE, 0, None, 256, 0, 1, FAKE, None, 10, None, None, 1,
                                 None) == ep.EP_ERR_INVALID
    p = ctypes.c_void_p(123)
    assert lib.ep_combine_async(None, FAKE, 10, FAKE, None, 256, FAKE, None, None, 0,
                                ctypes.byref(p)) == ep.EP_ERR_INVALID
    assert not p.value
    assert lib.ep_pending_wait(None, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_set_num_sms(None, 4) == ep.EP_ERR_INVALID
    assert lib.ep_profile_begin(None, FAKE, 16) == ep.EP_ERR_INVALID
    assert lib.ep_profile_end(None, None, None) == ep.EP_ERR_INVALID
