"""The C ABI without a GPU: the library loads, exports every symbol the public
header declares, and rejects invalid create arguments before touching CUDA."""

import ctypes
import os
import re

import pytest

from tensor_comm_gemm_gb300 import build as tb
from tensor_comm_gemm_gb300 import tpoverlap as t

HEADER = os.path.join(tb.INCLUDE, "tpoverlap.h")


@pytest.fixture(scope="module")
def lib():
    tb.build()
    return t.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tpo_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    assert sorted(t.EXPORTS) == names
    for name in names:
        assert hasattr(lib, name), name


def test_version_names_target(lib):
    assert "sm_103a" in t.tpo_version()


@pytest.mark.parametrize("args,word", [
    ((0, 256, 256, 256, 0), "tp"),
    ((17, 256, 256, 256, 0), "tp"),
    ((2, 256, 256, 256, 7), "dtype"),
    ((2, 0, 256, 256, 0), "sizes"),
    ((3, 256, 256, 256, 0), "n="),        # unequal row chunks (n % tp)
    ((2, 256, 256, 100, 0), "m="),        # bf16 output rows not a multiple of 16 bytes
    ((2, 256, 100, 256, 0), "k="),        # bf16 rows of 200 bytes
    ((2, 256, 200, 256, 1), "k="),        # e4m3 rows of 200 bytes
])
def test_create_rejects_bad_arguments(lib, args, word):
    assert not lib.tpo_ctx_create(*args)
    assert word in t.tpo_last_error()


def test_null_handles_are_safe(lib):
    assert lib.tpo_ctx_destroy(None) == 0
    assert lib.tpo_sync_status(None) == 1
    assert lib.tpo_set_opt(None, b"mode", 0) == 1
    assert lib.tpo_staging_ptr(None) is None
    arr = (ctypes.c_void_p * 2)()
    assert lib.tpo_ag_gemm(None, arr, None, None, None, None, None) == 1
