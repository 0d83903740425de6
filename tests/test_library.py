"""CPU-side checks of the C ABI library: it builds, loads without a GPU, and
exports every entry point include/mla_decode.h declares. Host-side argument
checks that return before any CUDA call are exercised too."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_decode.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from paged_mla_decode_04_gb300 import _build
    path = _build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["mla_kv_write", "mla_decode_plan", "mla_decode", "mla_decode_workspace_size",
              "mla_uv_project", "mla_get_error", "mla_decode_num_clusters"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_names_match_header():
    import paged_mla_decode_04_gb300 as m
    assert sorted(m.EXPORTED) == declared_functions()


def test_host_argument_checks_need_no_gpu(lib):
    lib.mla_kv_write.restype = ctypes.c_int
    assert lib.mla_kv_write(None, 0, None, None, 1, None, None) == -1
    lib.mla_get_error.restype = ctypes.c_int
    assert lib.mla_get_error(None, None, 0, None) == -1
    lib.mla_uv_project.restype = ctypes.c_int
    assert lib.mla_uv_project(None, None, None, -1, 16, None, None) == -1
    assert lib.mla_uv_project(None, None, None, 4, 16, None, None) == -1
    # a misaligned workspace for the status word is refused before any launch
    buf = ctypes.create_string_buffer(1024)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    assert lib.mla_uv_project(ctypes.c_void_p(base), ctypes.c_void_p(base), ctypes.c_void_p(base), 4, 16,
                              ctypes.c_void_p(base + 8), None) == -3
    # the bounded-wait self-test refuses a null status word and limits outside [1 us, 1 s]
    lib.mla_selftest_bounded_wait.restype = ctypes.c_int
    lib.mla_selftest_bounded_wait.argtypes = [ctypes.c_int, ctypes.c_uint, ctypes.c_void_p, ctypes.c_void_p]
    assert lib.mla_selftest_bounded_wait(0, 1000, None, None) == -1
    assert lib.mla_selftest_bounded_wait(0, 0, ctypes.c_void_p(base), None) == -1
    assert lib.mla_selftest_bounded_wait(0, 1000001, ctypes.c_void_p(base), None) == -1


def test_product_package_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "paged_mla_decode_04_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.lower(), f


def test_tracing_tool_reads_the_event_enum():
    """The trace tool's event ids come from the kernel's header (a rename or
    a new event there cannot leave the tool reading the wrong records)."""
    from paged_mla_decode_04_gb300 import tracing
    ids = tracing.event_ids()
    assert ids["KernelStart"] == 1 and ids["SetupDone"] == 2
    assert sorted(ids.values()) == list(range(1, len(ids) + 1))
    for name in ["SlotAcquired", "TileIssued", "QkTileReady", "QkSFree", "QkIssued", "SmSFull", "SmSent",
                 "SmXFull", "SmComputed", "SmPvDone", "SmOFixed", "PvOFixed", "PvIssued", "GlobalStart",
                 "GlobalEnd"]:
        assert name in ids
    assert tracing.summarize({}, ids) == ""
