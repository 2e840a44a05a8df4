"""The C-ABI library builds, loads and exports every symbol include/moe_route.h declares.
Only host-side helpers are called here (no GPU in this environment)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libpath():
    from serving_moe_route_02_gb300 import _build
    return _build.build()


def header_symbols():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:int|const char\s*\*)\s*(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(libpath):
    names = header_symbols()
    assert len(names) >= 10, names
    lib = ctypes.CDLL(libpath)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (moe_\w+)", out))
    assert set(names) <= exported


def test_host_helpers(libpath):
    import serving_moe_route_02_gb300 as mr
    lib = mr.load()
    assert mr.bins(896, 16, 112) == 128
    assert mr.bins(896, 16, 0) == 896
    assert mr.bins(896, 16, 30) == 48
    assert mr.num_experts(896, 16, 336, 112) == 128
    assert mr.num_experts(896, 16, 0, 896) == 896       # not a proper sub-range
    assert mr.num_experts(896, 16, 0, 0) == 896
    assert mr.num_experts(896, 16, 0, 890) == 896       # would not shrink the problem
    assert mr.strerror(0) == "ok" and "invalid" in mr.strerror(-1)
    assert lib.moe_route_set_path(5) == mr.E_INVALID_ARG
    prev = mr.set_path(2)
    assert mr.set_path(prev) == 2
    assert lib.moe_route_set_path(3) >= 0 and mr.set_path(prev) == 3
    # the barrier test hook validates its arguments on the host (and is left disarmed)
    assert lib.moe_route_arm_barrier_timeout(-2, 0) == mr.E_INVALID_ARG
    assert lib.moe_route_arm_barrier_timeout(0, 0) == mr.E_INVALID_ARG
    assert lib.moe_route_arm_barrier_timeout(0, 2000001) == mr.E_INVALID_ARG
    assert lib.moe_route_arm_barrier_timeout(-1, 0) == mr.OK


def test_missing_library_fails_loudly(tmp_path):
    import serving_moe_route_02_gb300 as mr
    with pytest.raises(ImportError):
        mr.load(str(tmp_path / "nope.so"))


def test_route_with_layout_checks_arguments_on_the_host(libpath):
    """moe_route_with_layout rejects a bad tile or a capacity below the bound before it
    touches the device (no GPU here: only the host-side checks run)."""
    import serving_moe_route_02_gb300 as mr
    lib = mr.load()
    T, E, k = 128, 896, 16
    NE = mr.bins(E, k, 0)
    need = mr.padded_capacity(T, k, NE, 128)
    assert need >= T * k
    dummy = ctypes.c_void_p(16)  # never dereferenced: the calls return before any launch

    def call(tile, capacity, rows=True, T=T):
        return lib.moe_route_with_layout(dummy, 1, dummy, T, E, k, 8, 4, 2.5, 0, 0, dummy, dummy, dummy,
                                         dummy, None, None, tile, dummy, dummy if rows else None, None,
                                         capacity, None)

    assert call(0, need) == mr.E_INVALID_ARG
    assert call(128, need - 1) == mr.E_INVALID_ARG
    assert call(-5, need, rows=False) == mr.E_INVALID_ARG
    assert lib.moe_route_with_layout(dummy, 1, dummy, T, E, k, 8, 9, 2.5, 0, 0, dummy, dummy, dummy,
                                     dummy, None, None, 128, dummy, dummy, None, need, None) == mr.E_INVALID_ARG
