"""The C-ABI library builds (nvcc cross-compiles for sm_103a without a GPU),
loads, and exports every function include/*.h declares.  No kernels run."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_125_gb300 as kvp
from paged_kv_cache_125_gb300 import _build

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "kvpaged.h")
SCHED_HEADER = os.path.join(INCLUDE, "kvpaged_sched.h")


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^(?:const\s+)?\w[\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M))


def all_declared():
    return {n for h in sorted(os.listdir(INCLUDE)) if h.endswith(".h")
            for n in declared_functions(os.path.join(INCLUDE, h))}


@pytest.fixture(scope="module")
def lib_path():
    return _build.build()


def test_header_declares_the_three_calls():
    names = declared_functions()
    assert {"kv_store", "attn_prefill_varlen", "attn_decode_paged"} <= names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in all_declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header(lib_path):
    from paged_kv_cache_125_gb300 import scheduler
    assert set(kvp.SIGNATURES) == declared_functions()
    assert set(scheduler.SIGNATURES) == declared_functions(SCHED_HEADER)
    lib = kvp.library()
    assert lib.kvp_version() >= 100
    assert lib.kvp_last_error() == b""
