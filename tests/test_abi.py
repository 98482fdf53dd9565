"""The C-ABI library builds for sm_103a, loads, and exports every function that
include/qlin.h declares.  Host-only calls; nothing here needs a GPU."""
import ctypes
import os
import re

import pytest

from w4a16_linear_layers_gb300 import build as qbuild
from w4a16_linear_layers_gb300 import qlin

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "qlin.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qlin_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qlin.load()


def test_header_matches_binding():
    assert header_functions() == sorted(qlin.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(qbuild.LIB_PATH)
    for name in header_functions():
        assert hasattr(raw, name), name


def test_status_strings_and_version(lib):
    assert qlin.version() == 103
    codes = [0, -1, -2, -3, -4, -5, -6, -7, -10, -20, -21]
    names = [qlin.status_string(c) for c in codes]
    assert len(set(names)) == len(codes)
    assert qlin.status_string(12345) == "unknown status"


def test_library_does_not_link_torch(lib):
    maps = open(f"/proc/{os.getpid()}/maps").read()
    assert qbuild.LIB_PATH in maps
    needed = os.popen(f"readelf -d {qbuild.LIB_PATH} 2>/dev/null").read()
    assert "torch" not in needed and "c10" not in needed
