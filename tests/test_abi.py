"""The C-ABI library builds, loads on a machine without a GPU and exports every
function include/halo.h declares; argument checks answer without touching the
GPU.  The library contains none of the oracle's code."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "halo.h")


STENCIL_HEADER = os.path.join(ROOT, "include", "stencil.h")


def declared_functions(header=HEADER, prefix="halo_"):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    pat = r"^[A-Za-z_][\w\s\*]*?\b(%s\w+)\s*\(" % prefix
    return sorted(set(re.findall(pat, text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from domain_decomposition_halo_build_gb300 import _build, halo
    _build.build()
    return halo.load_library()


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("halo_setup", "halo_exchange_x", "halo_exchange_f", "halo_rebuild",
              "halo_query", "halo_status", "halo_destroy", "halo_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header():
    from domain_decomposition_halo_build_gb300 import halo
    assert set(declared_functions()) == set(halo.SIGNATURES)


def test_stencil_header_symbols_exported_and_bound(lib):
    from domain_decomposition_halo_build_gb300 import stencil
    names = declared_functions(STENCIL_HEADER, "stencil_")
    assert {"stencil_setup", "stencil_exchange", "stencil_sweep", "stencil_sweep_fused"} <= set(names)
    assert not [n for n in names if not hasattr(lib, n)]
    assert set(names) == set(stencil.SIGNATURES)


def test_stencil_host_only_checks(lib):
    from domain_decomposition_halo_build_gb300 import halo, stencil
    stencil.load_library()
    h = ctypes.c_void_p()
    assert lib.stencil_setup(2, 2, 6, ctypes.byref(h)) == halo.EINVAL    # n % 4 != 0
    assert lib.stencil_setup(0, 2, 8, ctypes.byref(h)) == halo.EINVAL
    assert lib.stencil_setup(300, 300, 8, ctypes.byref(h)) == halo.EINVAL  # > 65535 tiles
    assert lib.stencil_setup(2, 3, 8, ctypes.byref(h)) == halo.OK
    pitch, rows, col0 = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    tile, total = ctypes.c_int64(), ctypes.c_int64()
    assert lib.stencil_layout(h, ctypes.byref(pitch), ctypes.byref(rows), ctypes.byref(col0),
                              ctypes.byref(tile), ctypes.byref(total)) == halo.OK
    from oracle import stencil as S
    assert (pitch.value, rows.value, col0.value) == (S.pitch(8), 10, S.COL0)
    assert (tile.value, total.value) == (S.tile_floats(8), 6 * S.tile_floats(8))
    # misaligned or aliased fields are refused before any launch
    assert lib.stencil_exchange(h, ctypes.c_void_p(8), None) == halo.EINVAL
    assert lib.stencil_sweep(h, ctypes.c_void_p(16), ctypes.c_void_p(16), None) == halo.EINVAL
    lib.stencil_destroy(h)


def test_host_only_argument_checks(lib):
    from domain_decomposition_halo_build_gb300 import halo
    assert lib.halo_strerror(halo.ETIMEOUT).decode() == "device-side wait timed out"
    assert lib.halo_query(None, None) == halo.EINVAL
    h = ctypes.c_void_p()
    box = (ctypes.c_float * 3)(3, 3, 3)
    grid = (ctypes.c_int32 * 3)(3, 1, 1)
    # null inputs and non-positive sizes are rejected before any CUDA call
    assert lib.halo_setup(box, grid, ctypes.c_float(0.5), None, None, 10, None,
                          ctypes.byref(h)) == halo.EINVAL
    assert lib.halo_setup(box, grid, ctypes.c_float(0.5), ctypes.c_void_p(16),
                          ctypes.c_void_p(16), 0, None, ctypes.byref(h)) == halo.EINVAL
    assert lib.halo_setup(box, grid, ctypes.c_float(2.5), ctypes.c_void_p(16),
                          ctypes.c_void_p(16), 10, None, ctypes.byref(h)) == halo.EPULSES
    bad = (ctypes.c_int32 * 3)(0, 1, 1)
    assert lib.halo_setup(box, bad, ctypes.c_float(0.5), ctypes.c_void_p(16),
                          ctypes.c_void_p(16), 10, None, ctypes.byref(h)) == halo.EINVAL
    assert not h.value


def test_library_has_no_oracle_code(lib):
    from domain_decomposition_halo_build_gb300 import halo
    out = subprocess.run(["nm", "-D", "--defined-only", halo.LIBRARY], capture_output=True,
                         text=True).stdout
    assert "oracle" not in out
    exported = [l.split()[-1] for l in out.splitlines() if " T " in l]
    assert all(not n.startswith("oracle_") for n in exported)
