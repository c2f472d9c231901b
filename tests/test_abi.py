"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every entry point that include/mita.h declares, and rejects
invalid plans before touching the device."""
import ctypes
import os
import re

import pytest

import mixture_top_attention_mita_b300 as mita
from mixture_top_attention_mita_b300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mita_\w+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mita.load()


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert {"mita_plan", "mita_forward", "mita_destroy"} <= declared
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared <= set(mita.EXPORTS) | declared  # binding lists them


def test_binding_lists_every_declared_symbol():
    assert _declared() == set(mita.EXPORTS)


def test_strerror(lib):
    for code in range(7):
        assert lib.mita_strerror(code)
    assert lib.mita_strerror(999) == b"unknown status"


@pytest.mark.parametrize("args,code", [
    ((1, 1, 196, 64, (14, 14, 5, 5), 25, 197), 1),      # k > N
    ((1, 1, 196, 64, (14, 13, 5, 5), 25, 25), 1),       # gh*gw != N
    ((1, 1, 196, 64, (14, 14, 5, 4), 25, 25), 1),       # ph*pw != m
    ((1, 1, 196, 64, (14, 14, 15, 1), 15, 25), 1),      # ph > gh
    ((0, 1, 196, 64, (14, 14, 5, 5), 25, 25), 1),       # B < 1
    ((1, 1, 196, 64, (14, 14, 5, 5), 25, 0), 1),        # k < 1
    ((1, 1, 196, 96, (14, 14, 5, 5), 25, 25), 2),       # d unsupported
    ((1, 1, 8192, 64, (1, 8192, 1, 2048), 2048, 25), 2),  # m too large
    ((256, 256, 196, 64, (14, 14, 5, 5), 25, 25), 2),   # B*H too large
])
def test_plan_rejects_before_device(lib, args, code):
    B, H, N, d, grid, m, k = args
    h = ctypes.c_void_p(1)
    rc = lib.mita_plan(ctypes.byref(h), B, H, N, d, mita.Grid(*grid), m, k, mita.MITA_BF16)
    assert rc == code
    assert h.value is None


def test_null_handles(lib):
    assert lib.mita_forward(None, None, None, None, None, None, None, None) == 1
    assert lib.mita_set_option(None, 0, 0) == 1
    assert lib.mita_get_status(None) == 1
    lib.mita_destroy(None)


@pytest.mark.parametrize("d", [0, -64])
def test_noalloc_rejects_bad_head_dim_as_invalid(lib, d):
    # the argument checks of mita_plan(): d < 1 is an invalid argument, not
    # an unsupported size; no device is touched
    rc = lib.mita_forward_noalloc(1, 1, 196, d, mita.Grid(14, 14, 5, 5), 25, 25, mita.MITA_BF16,
                                  None, None, None, None, None, None, None)
    assert rc == 1


def test_plan_rejects_bad_head_dim_as_invalid(lib):
    h = ctypes.c_void_p(1)
    assert lib.mita_plan(ctypes.byref(h), 1, 1, 196, 0, mita.Grid(14, 14, 5, 5), 25, 25, mita.MITA_BF16) == 1
    assert h.value is None
