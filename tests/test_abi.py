"""The C-ABI library loads and exports every symbol include/himuon.h declares;
host-only entry points behave as documented. No GPU needed."""

import ctypes
import os
import re

import pytest

import tiled_newton_schulz_03_b300 as hm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "himuon.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(himuon_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from tiled_newton_schulz_03_b300 import build
    build.build()
    return hm.load_library()


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for required in ("himuon_tiled_ns", "himuon_tiled_ns_batched", "himuon_step"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(hm.EXPORTED_SYMBOLS) == declared_functions()


def test_version_and_defaults(lib):
    assert lib.himuon_version() >= 10000
    p = hm.NSParams()
    lib.himuon_default_ns_params(ctypes.byref(p))
    assert (round(p.a, 4), round(p.b, 4), round(p.c, 4)) == (3.4445, -4.775, 2.0315)
    assert p.norm == 0 and abs(p.eps - 1e-7) < 1e-12 and p.path == 0


def test_flop_count(lib):
    assert hm.ns_flops(4096, 4096, 128, 5) == 6 * 4096 * 4096 * 128 * 5
    assert hm.ns_flops(0, 5, 128, 5) == 0.0


def test_tile_schedule(lib):
    s = hm.TSchedule([(0, 64), (1, 128), (2, 256)])
    assert [s(i) for i in range(5)] == [64, 128, 256, 256, 256]
    s = hm.TSchedule([(10, 32), (100, 128)])
    assert s(0) == 32 and s(99) == 32 and s(100) == 128
    with pytest.raises(hm.HimuonError):
        hm.TSchedule([(5, 64), (5, 128)])
    with pytest.raises(hm.HimuonError):
        hm.TSchedule([])


def test_create_without_device_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = ctypes.c_void_p()
    st = lib.himuon_create(ctypes.byref(p))
    assert st == 5 and not p.value
    assert b"device" in lib.himuon_last_error_string().lower() or b"driver" in lib.himuon_last_error_string().lower()


def test_null_handle_is_rejected(lib):
    st = lib.himuon_tiled_ns(None, None, 4, 4, 4, 0, 128, 5, None, None, 4, 0, None)
    assert st == 1
    assert b"handle" in lib.himuon_last_error_string()
