"""C-ABI library checks that need no GPU: it builds, loads, exports every
entry point include/mhc.h declares, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

from manifold_constrained_hyper_gb300 import build as mbuild
from manifold_constrained_hyper_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return ops.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mhc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mhc_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary_entry_points():
    names = declared_functions()
    for n in ("mhc_prepare_weight", "mhc_pre", "mhc_post", "mhc_boundary_fused"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ops.EXPORTS)


def test_sizes_and_plan(lib):
    assert ops.weight_bytes(7168) == 384 * 7168
    assert ops.weight_bytes(100) == 0                 # unsupported hidden
    assert ops.workspace_bytes(0, 7168) == 0
    for T, H in [(1, 256), (64, 7168), (512, 7168), (8192, 7168), (1024, 4096), (5, 32)]:
        S, w = ops.plan(T, H)
        assert S * w == H and w % 32 == 0
        assert ops.workspace_bytes(T, H) >= S * ((T + 127) // 128) * 28 * 128 * 4
    assert ops.plan(8192, 7168) == (28, 256)
    # every tile's slices fit in one wave of persistent CTAs; item sizes of at
    # most 8 chunks wherever some such size fits
    for H in range(32, 65537, 32):
        for T in (1, 128, 129, 256, 512, 1024, 8192):
            S, w = ops.plan(T, H)
            assert S <= 152 and S * w == H, (T, H, S, w)
            if H <= 152 * 8 * 32 and any((H // 32) % d == 0 and H // 32 // d <= 152
                                         for d in range(1, 9)):
                assert w <= 256, (T, H, S, w)


def test_status_strings(lib):
    for code, name in ops.STATUS_NAMES.items():
        assert ops.mhc_status_string(code).startswith(name)


def _P(v):
    return ctypes.c_void_p(v)


def test_argument_errors_before_any_device_work(lib):
    p = ops.Params().c()
    A = 0x10000                  # an aligned fake address, never dereferenced
    # mhc_post: T == 0 is a no-op; negative T; bad hidden; NULL; misaligned
    assert lib.mhc_post(None, None, None, None, None, 0, 256, None) == 0
    assert lib.mhc_post(_P(A), _P(A), _P(A), _P(A), _P(A), -1, 256, None) == 3
    assert lib.mhc_post(_P(A), _P(A), _P(A), _P(A), _P(A), 4, 100, None) == 4
    assert lib.mhc_post(None, _P(A), _P(A), _P(A), _P(A), 4, 256, None) == 1
    assert lib.mhc_post(_P(A + 8), _P(A), _P(A), _P(A), _P(A), 4, 256, None) == 2
    # partial overlap of output and input
    assert lib.mhc_post(_P(A), _P(A * 16), _P(A * 32), _P(A * 48), _P(A * 16 + 64), 4, 256,
                        None) == 5
    # mhc_pre: iters < 1; workspace too small; NULL outputs
    bad = ops.Params(sinkhorn_iters=0).c()
    args = [_P(A * 1), _P(A * 2), _P(A * 3), _P(A * 4), None, 0]
    outs = [_P(A * 8), _P(A * 9), _P(A * 10), _P(A * 11)]
    assert lib.mhc_pre(*args, ctypes.byref(bad), 4, 256, *outs, _P(A * 12), 1 << 20, None) == 3
    assert lib.mhc_pre(*args, ctypes.byref(p), 4, 256, *outs, _P(A * 12), 16, None) == 8
    assert lib.mhc_pre(*args, ctypes.byref(p), 4, 256, None, *outs[1:], _P(A * 12), 1 << 20,
                       None) == 1
    # fused: shifted needs x/post/comb/residual_out
    assert lib.mhc_boundary_fused(None, _P(A), _P(A * 2), _P(A * 3), _P(A * 4), _P(A * 5),
                                  _P(A * 6), _P(A * 7), None, 0, ctypes.byref(p), 4, 256,
                                  _P(A * 8), _P(A * 9), _P(A * 10), _P(A * 11), _P(A * 12),
                                  _P(A * 13), 1 << 20, None) == 1
    # reciprocal check hook: NULL / misaligned result, range past 2^32
    assert lib.mhc_debug_rcp_check(0, 16, None, None) == 1
    assert lib.mhc_debug_rcp_check(0, 16, _P(A + 4), None) == 2
    assert lib.mhc_debug_rcp_check(0xFFFFFFF0, 17, _P(A), None) == 3
    assert lib.mhc_debug_rcp_check(0, 0, _P(A), None) == 0
    # split-K pre: splits out of range, NULL sums, misaligned mixes, T == 0
    sk = [_P(A), _P(A * 2), _P(A * 3)]
    rest = [_P(A * 4), _P(A * 5), None, 0, ctypes.byref(p), 4, 256, _P(A * 8), _P(A * 9),
            _P(A * 10), _P(A * 11), None]
    assert lib.mhc_pre_split_k(*sk, 0, *rest) == 3
    assert lib.mhc_pre_split_k(*sk, 65, *rest) == 3
    assert lib.mhc_pre_split_k(_P(A), _P(A * 2), None, 4, *rest) == 1
    assert lib.mhc_pre_split_k(_P(A), _P(A * 2 + 4), _P(A * 3), 4, *rest) == 2
    rest0 = list(rest)
    rest0[5] = 0
    assert lib.mhc_pre_split_k(*sk, 4, *rest0) == 0


def test_coef_check_hook_argument_errors():
    """The coefficient-forms hook validates before enqueuing anything (no GPU
    needed): NULL, misaligned, negative count, aliasing outputs, T == 0."""
    lib = ops.load()
    p = ops.Params().c()
    A = 0x100000
    ok = [_P(A), _P(A * 2), _P(A * 3), ctypes.byref(p), 1024]
    assert lib.mhc_debug_coef_check(*ok, 0, _P(A * 4), _P(A * 5), None) == 0
    assert lib.mhc_debug_coef_check(*ok, -1, _P(A * 4), _P(A * 5), None) == 3
    assert lib.mhc_debug_coef_check(None, *ok[1:], 8, _P(A * 4), _P(A * 5), None) == 1
    assert lib.mhc_debug_coef_check(*ok, 8, _P(A * 4 + 8), _P(A * 5), None) == 2
    assert lib.mhc_debug_coef_check(*ok, 8, _P(A * 4), _P(A * 4 + 16), None) == 5
