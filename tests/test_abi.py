"""The C ABI: libsbt.so builds for sm_103a, loads without a GPU and exports every
symbol include/sbt.h declares (no compute call is made here)."""
import ctypes
import os
import re
import subprocess

import pytest

import scatter_boundary_tile_gb300 as sbt
from scatter_boundary_tile_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "sbt.h")).read()
    return sorted(set(re.findall(r"^SBT_API\s+[\w\s\*]+?\b(sbt_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sbt.load_library()


def test_header_and_binding_agree():
    assert header_functions() == sorted(sbt.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(sbt_\w+)", out))
    assert exported == set(header_functions())


def test_no_driver_dependency_at_load_time():
    out = subprocess.run(["ldd", _build.LIB], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart.so" not in out


def test_built_for_sm_103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)


def test_null_context_is_rejected_before_cuda(lib):
    st = lib.sbt_gather_rows(None, 0, None, 0, 0, 0, None, 0, 0, 0, 1, None, 0, None, 1, None, None)
    assert st == sbt.SBT_ERR_INVALID_ARG
    assert b"ctx" in lib.sbt_last_error_message()


def test_create_without_a_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = lib.sbt_create(0, ctypes.byref(h))
    assert st in (sbt.SBT_ERR_CUDA, sbt.SBT_ERR_INVALID_ARG) and not h.value
    assert lib.sbt_last_error_message()


def test_noalloc_scratch_size_matches_header():
    """The binding's size check and the library's fixed GEMM scratch are the same number."""
    text = open(os.path.join(ROOT, "include", "sbt.h")).read()
    m = re.search(r"#define\s+SBT_GEMM_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "SBT_GEMM_NOALLOC_SCRATCH_BYTES not found in include/sbt.h"
    assert int(m.group(1)) << int(m.group(2)) == sbt.GEMM_NOALLOC_SCRATCH_BYTES
