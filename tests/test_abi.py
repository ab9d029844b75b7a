"""The C-ABI library loads, exports every function include/mita.h declares, and
rejects invalid arguments on the host before touching the GPU (no compute call
runs here: every call below fails validation)."""
import ctypes
import re

import pytest

from sparse_top_landmark_gb300 import build as B
from sparse_top_landmark_gb300 import mita


@pytest.fixture(scope="module")
def lib():
    B.build()
    return mita.load()


def test_every_declared_symbol_is_exported(lib):
    names = mita.declared_functions()
    assert len(names) >= 16
    for required in ["mita_pool", "mita_landmark_topk_shared", "mita_route", "mita_bucket",
                     "mita_expert_attn", "mita_forward"]:
        assert required in names
    for n in names:
        assert hasattr(lib, n), n


def test_no_oracle_in_product_sources():
    import os
    pkg = os.path.dirname(mita.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert not re.search(r"\b(import|from)\s+oracle\b", text), f
                assert "liboracle" not in text, f


def test_status_strings(lib):
    for code in range(6):
        assert len(lib.mita_status_string(code)) > 0


NULL = ctypes.c_void_p(0)
GOOD = ctypes.c_void_p(1 << 20)      # aligned, never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p((1 << 20) + 2)


def _msg(lib):
    return lib.mita_last_error_message().decode()


@pytest.mark.parametrize("args,code", [
    ((0, 1, 64, 16, 1, 64, 4), 1),        # B = 0
    ((1, 1, 64, 48, 1, 64, 4), 2),        # d = 48 unsupported
    ((1, 1, 64, 16, 2, 64, 4), 1),        # grid does not hold N
    ((1, 1, 64, 16, 8, 8, 5), 1),         # 2D needs a square m
    ((1, 1, 64, 16, 1, 64, 65), 1),       # m > N
    ((1, 1, 64, 16, 1, 64, 0), 1),        # m = 0
])
def test_pool_validation(lib, args, code):
    B_, H, N, d, gh, gw, m = args
    rc = lib.mita_pool(GOOD, B_, H, N, d, gh, gw, m, GOOD, NULL)
    assert rc == code, _msg(lib)


def test_pool_rejects_null_and_misaligned(lib):
    assert lib.mita_pool(NULL, 1, 1, 64, 16, 1, 64, 4, GOOD, NULL) == 1
    assert "NULL" in _msg(lib)
    assert lib.mita_pool_f32(MISALIGNED, 1, 1, 64, 16, 1, 64, 4, GOOD, NULL) == 1
    assert "aligned" in _msg(lib)


def test_forward_validation(lib):
    f = lib.mita_forward
    assert f(GOOD, GOOD, GOOD, 1, 1, 64, 16, 1, 64, 4, 0, 1, GOOD, NULL) == 1     # topk 0
    assert f(GOOD, GOOD, GOOD, 1, 1, 64, 16, 1, 64, 4, 65, 1, GOOD, NULL) == 1    # topk > N
    assert f(GOOD, GOOD, GOOD, 1, 1, 8192, 16, 1, 8192, 4, 4097, 1, GOOD, NULL) == 2  # limit
    assert f(GOOD, GOOD, GOOD, 1, 1, 64, 16, 1, 64, 16, 4, 9, GOOD, NULL) == 2    # s > 8
    assert f(GOOD, GOOD, GOOD, 1, 1, 64, 16, 1, 64, 4, 4, 5, GOOD, NULL) == 1     # s > m
    assert f(GOOD, GOOD, NULL, 1, 1, 64, 16, 1, 64, 4, 4, 1, GOOD, NULL) == 1     # v NULL


def test_stage_validation(lib):
    assert lib.mita_route(GOOD, GOOD, NULL, 1, 1, 64, 16, 16, 9, GOOD, NULL, NULL, NULL) == 2
    assert lib.mita_route(GOOD, GOOD, NULL, 1, 1, 64, 16, 4, 5, GOOD, NULL, NULL, NULL) == 1
    assert lib.mita_bucket(GOOD, 1, 1, 64, 16, 9, GOOD, GOOD, NULL) == 2
    assert lib.mita_bucket(NULL, 1, 1, 64, 4, 1, GOOD, GOOD, NULL) == 1
    assert lib.mita_landmark_topk_shared(GOOD, GOOD, GOOD, 1, 1, 64, 16, 4, 0, GOOD, GOOD,
                                         NULL) == 1
    # shared partial must be both-or-neither
    assert lib.mita_expert_attn(GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, NULL,
                                1, 1, 64, 16, 4, 4, 1, GOOD, NULL) == 1


def test_workspace_bytes_query(lib):
    n = lib.mita_forward_workspace_bytes(4, 2, 65536, 64, 128, 128, 1, 0)
    assert n > 4 * 2 * 65536 * 8        # at least the route + bucket arrays
    assert lib.mita_forward_workspace_bytes(1, 1, 64, 48, 4, 4, 1, 0) == 0
    # s = 2: routes and bucket lists twice as long, plus the per-expert partials (fp32 rows)
    n2 = lib.mita_forward_workspace_bytes(4, 2, 65536, 64, 128, 128, 2, 0)
    assert n2 > 4 * 2 * 65536 * (2 * 64 * 4 + 2 * 2 * 4)
    assert lib.mita_forward_workspace_bytes(4, 2, 65536, 64, 128, 128, 9, 0) == 0


def test_launch_counter_is_readable_without_a_gpu(lib):
    lib.mita_kernel_launches.restype = ctypes.c_uint64
    a = lib.mita_kernel_launches()
    assert lib.mita_kernel_launches() == a      # nothing launched in between


def test_forward_ex_and_pool_grid_validation(lib):
    f = lib.mita_forward_ex
    opt = mita.MitaOptions(2, 0, 0, 0)                  # unknown temperature
    assert f(GOOD, GOOD, GOOD, 1, 1, 64, 16, 1, 64, 4, 4, 1, ctypes.byref(opt), GOOD, NULL) == 1
    assert "shared_temperature" in _msg(lib)
    opt = mita.MitaOptions(0, 2, 3, 0)                  # 2 x 3 != m
    assert f(GOOD, GOOD, GOOD, 1, 1, 64, 16, 8, 8, 4, 4, 1, ctypes.byref(opt), GOOD, NULL) == 1
    assert "landmark grid" in _msg(lib)
    opt = mita.MitaOptions(1, 2, 2, 0)                  # 1D sequence onto a 2-row grid
    assert f(GOOD, GOOD, GOOD, 1, 1, 64, 16, 1, 64, 4, 4, 1, ctypes.byref(opt), GOOD, NULL) == 1
    opt = mita.MitaOptions(0, 0, 0, 0)                  # 2D grid, non-square m, no landmark grid
    assert f(GOOD, GOOD, GOOD, 1, 1, 64, 16, 8, 8, 6, 4, 1, ctypes.byref(opt), GOOD, NULL) == 1
    opt = mita.MitaOptions(0, 0, 0, 2)               # unknown branches
    assert f(GOOD, GOOD, GOOD, 1, 1, 64, 16, 1, 64, 4, 4, 1, ctypes.byref(opt), GOOD, NULL) == 1
    assert "branches" in _msg(lib)
    assert lib.mita_dense_attn(GOOD, GOOD, NULL, 1, 1, 64, 16, GOOD, NULL) == 1
    assert lib.mita_dense_attn_f32(GOOD, GOOD, GOOD, 1, 1, 64, 48, GOOD, NULL) == 2
    assert lib.mita_pool_grid(GOOD, 1, 1, 64, 16, 8, 8, 0, 3, GOOD, NULL) == 1
    assert lib.mita_pool_grid_f32(GOOD, 1, 1, 64, 16, 8, 8, 2, 3, NULL, NULL) == 1


def test_backward_validation(lib):
    f = lib.mita_backward
    opt = mita.MitaOptions(0, 0, 0, 0)
    # dq NULL
    assert f(GOOD, GOOD, GOOD, GOOD, 1, 1, 64, 16, 1, 64, 4, 4, 1, ctypes.byref(opt), NULL, GOOD,
             GOOD, NULL) == 1
    assert "dq" in _msg(lib)
    # s above the build's limit, unknown option
    assert f(GOOD, GOOD, GOOD, GOOD, 1, 1, 64, 16, 1, 64, 16, 4, 9, None, GOOD, GOOD, GOOD,
             NULL) == 2
    bad = mita.MitaOptions(0, 0, 0, 5)
    assert f(GOOD, GOOD, GOOD, GOOD, 1, 1, 64, 16, 1, 64, 4, 4, 1, ctypes.byref(bad), GOOD, GOOD,
             GOOD, NULL) == 1
    assert lib.mita_backward_f32(GOOD, GOOD, GOOD, GOOD, 1, 1, 64, 48, 1, 64, 4, 4, 1, None, GOOD,
                                 GOOD, GOOD, NULL) == 2


def test_workspace_limit_setter_returns_the_previous_cap(lib):
    assert mita.workspace_set_limit(1 << 20) == 0
    assert mita.workspace_set_limit(0) == 1 << 20


def test_bounded_wait_probe_rejects_a_null_result(lib):
    assert lib.mita_check_bounded_wait(NULL, NULL) == 1
    assert "gave_up" in _msg(lib)
