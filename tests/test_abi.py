"""The C ABI library loads and exports every entry point include/vr.h declares;
host-side argument checks that need no GPU. (CPU only: no compute calls.)"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vr.h")


def declared_entry_points():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\bVR_API\s+[\w\s\*]*?\b(vr[A-Z]\w*)\s*\(", text)))


@pytest.fixture(scope="module")
def vrlib():
    from ring_allreduce_virtual_gb300 import build
    build.build()
    import ring_allreduce_virtual_gb300 as vr
    return vr


def test_header_declares_the_ring_allreduce_calls():
    names = declared_entry_points()
    for n in ("vrCommCreate", "vrAllReduce", "vrCommDestroy", "vrCommGetAsyncError",
              "vrGetErrorString"):
        assert n in names


def test_library_exports_every_declared_symbol(vrlib):
    lib = ctypes.CDLL(vrlib.LIB_PATH)
    for name in declared_entry_points():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", vrlib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    assert exported == set(declared_entry_points()), exported ^ set(declared_entry_points())


def test_error_strings(vrlib):
    for code in range(6):
        assert vrlib.vrGetErrorString(code)
    assert vrlib.vrGetErrorString(99) == "unknown result code"


@pytest.mark.parametrize("args", [
    (0, 1, "simple", 1024),        # no ranks
    (129, 1, "simple", 1024),      # too many ranks
    (4, 0, "simple", 1024),        # no channels
    (4, 129, "simple", 1024),      # too many channels
    (4, 1, 3, 1024),               # unknown protocol
    (4, 1, "ll", 8),               # chunk below 16 bytes
    (4, 1, "ll128", 1000),         # chunk not a multiple of 16
])
def test_create_rejects_bad_arguments_before_touching_the_device(vrlib, args):
    with pytest.raises(vrlib.VrError) as e:
        vrlib.vrCommCreate(*args)
    assert e.value.code == vrlib.vrInvalidArgument


def test_calls_on_a_handle_that_is_not_a_communicator(vrlib):
    bogus = ctypes.addressof(ctypes.c_uint64(0x7672436f6d6d3031))
    for h in (None, bogus):
        with pytest.raises(vrlib.VrError) as e:
            vrlib.vrAllReduce(h, [1], [1], 1, "float32", "sum")
        assert e.value.code == vrlib.vrInvalidArgument
        with pytest.raises(vrlib.VrError):
            vrlib.vrCommDestroy(h)
        with pytest.raises(vrlib.VrError):
            vrlib.vrCommGetAsyncError(h)
        with pytest.raises(vrlib.VrError):
            vrlib.vrCommSetTimeout(h, 10)
        with pytest.raises(vrlib.VrError):
            vrlib.vrCommGetInfo(h)


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    import ring_allreduce_virtual_gb300 as vr
    monkeypatch.setattr(vr, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(vr, "_lib_handle", None)
    with pytest.raises(ImportError):
        vr.vrCommCreate(2, 1, "simple", 1024)
