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


# --------------------------------------------------------------------------- pointer alignment
# Every call refuses an array pointer that is not a multiple of its element size before it
# touches the device.  The calls are made with a zero-filled host buffer standing in for the
# context (the calls test it only for NULL before validating) and addresses that are never
# dereferenced; with a GPU present the test does not run, so a stand-in context never
# reaches a device.
F32, BF16 = 0, 1
E4M3, E8M0 = 0, 2
X = 1 << 20  # an address on a 1 MiB boundary; every pointer below is X + a multiple of 4096


def _alignment_cases():
    p = lambda k: X + 4096 * k
    return {  # call: (positional arguments after ctx, {argument index: required alignment})
        "sbt_tile_load_padded": ([F32, p(0), 4, 4, 4, 1, 0, 0, 4, 4, 1, 1, 4, 4, p(1), None, None], {1: 4, 14: 4}),
        "sbt_tile_store_clipped": ([F32, p(0), 1, 1, 4, 4, p(1), 4, 4, 4, 1, 0, 0, 4, 4, None], {1: 4, 6: 4}),
        "sbt_gather_rows": ([F32, p(0), 4, 4, 4, p(1), 2, 0, 0, 4, None, 0, p(2), 4, None, None],
                            {1: 4, 5: 4, 12: 4}),
        "sbt_scatter_rows_masked": ([F32, p(0), 4, 4, 4, p(1), 2, 0, 0, p(2), 4, 4, None, 0, None],
                                    {1: 4, 5: 4, 9: 4}),
        "sbt_gather_cols": ([F32, p(0), 4, 4, 4, p(1), 2, 0, 0, 4, p(2), 2, None, None], {1: 4, 5: 4, 10: 4}),
        "sbt_scatter_add_rows": ([BF16, p(0), 4, 4, 4, p(1), 2, 0, 0, p(2), 4, 4, None], {1: 2, 5: 4, 9: 2}),
        "sbt_ragged_tile_load": ([BF16, p(0), 8, 2, 4, 8, 4, p(1), 2, 4, p(2), None], {1: 2, 7: 4, 10: 2}),
        "sbt_ragged_tile_store": ([BF16, p(0), 2, 2, 4, 4, p(1), p(2), 8, 8, 4, None], {1: 2, 6: 4, 7: 2}),
        "sbt_gemm_bounded": ([p(0), 8, p(1), 8, p(2), 8, F32, 4, 4, 4, p(16), 1 << 30, None], {0: 2, 2: 2, 4: 4}),
        "sbt_gemm_block_scaled": ([E4M3, p(0), 32, E4M3, p(1), 4, E8M0, p(2), 1, p(3), 4, 1, p(4), 4, p(5), 4,
                                   4, 4, 32, p(16), 1 << 30, None], {12: 4, 14: 4}),
    }


@pytest.mark.parametrize("name", sorted(_alignment_cases()))
def test_misaligned_pointers_are_refused_before_the_device(lib, name):
    import torch
    if torch.cuda.is_available():
        pytest.skip("CPU-only check: a stand-in context must never reach a device")
    ctx = ctypes.create_string_buffer(4096)
    args, align = _alignment_cases()[name]
    fn = getattr(lib, name)
    for i, a in align.items():
        for off in range(1, a):
            bad = list(args)
            bad[i] = args[i] + off
            assert fn(ctx, *bad) == sbt.SBT_ERR_ALIGNMENT, (i, off)
            assert b"aligned" in lib.sbt_last_error_message()
    # aligned pointers pass validation and stop only at device selection (no GPU here)
    assert fn(ctx, *args) == sbt.SBT_ERR_CUDA, lib.sbt_last_error_message()
