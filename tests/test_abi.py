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


# --------------------------------------------------------------------------- argument validation
# Each case changes one argument of a valid call (the alignment cases above) and expects the
# status the host returns before touching the device: SBT_OK for an empty call (nothing is
# launched), an error code otherwise.  Same stand-in context, same CPU-only guard.
F16 = 2
E5M2, E2M1 = 1, 3


def _validation_cases():
    base = {name: args for name, (args, _) in _alignment_cases().items()}
    ok, bad, uns, aln = sbt.SBT_OK, sbt.SBT_ERR_INVALID_ARG, sbt.SBT_ERR_UNSUPPORTED, sbt.SBT_ERR_ALIGNMENT
    return [  # (call, {argument index: value}, expected status, what)
        ("sbt_tile_load_padded", {0: 7}, uns, "dtype"),
        ("sbt_tile_load_padded", {2: -1}, bad, "negative rows"),
        ("sbt_tile_load_padded", {12: 0}, bad, "tile_r 0"),
        ("sbt_tile_load_padded", {13: 257}, bad, "tile_c 257"),
        ("sbt_tile_load_padded", {5: 0}, bad, "stride_c 0"),
        ("sbt_tile_load_padded", {14: None}, bad, "dst_tiles NULL"),
        ("sbt_tile_load_padded", {1: None}, bad, "src NULL"),
        ("sbt_tile_load_padded", {10: 0}, ok, "empty grid"),
        ("sbt_tile_store_clipped", {2: -1}, bad, "negative grid"),
        ("sbt_tile_store_clipped", {4: 0}, bad, "tile_r 0"),
        ("sbt_tile_store_clipped", {10: 0}, bad, "stride_r 0"),
        ("sbt_tile_store_clipped", {6: None}, bad, "dst NULL"),
        ("sbt_tile_store_clipped", {7: 0}, ok, "empty array"),
        ("sbt_gather_rows", {4: 2}, bad, "ld_src < cols"),
        ("sbt_gather_rows", {13: 2}, bad, "ld_out < tile_c"),
        ("sbt_gather_rows", {5: None}, bad, "idx NULL"),
        ("sbt_gather_rows", {9: 0}, bad, "tile_c 0"),
        ("sbt_gather_rows", {10: X + 4096 * 9, 11: 2}, bad, "ld_mask < tile_c"),
        ("sbt_gather_rows", {6: 0}, ok, "no indices"),
        ("sbt_gather_cols", {11: 1}, bad, "ld_out < n_idx"),
        ("sbt_gather_cols", {9: 0}, bad, "tile_r 0"),
        ("sbt_gather_cols", {6: -1}, bad, "negative n_idx"),
        ("sbt_gather_cols", {6: 0}, ok, "no indices"),
        ("sbt_scatter_rows_masked", {4: 2}, bad, "ld_dst < cols"),
        ("sbt_scatter_rows_masked", {10: 2}, bad, "ld_src < tile_c"),
        ("sbt_scatter_rows_masked", {1: None}, bad, "dst NULL"),
        ("sbt_scatter_rows_masked", {6: 0}, ok, "no indices"),
        ("sbt_scatter_add_rows", {0: 7}, uns, "dtype"),
        ("sbt_scatter_add_rows", {4: 2}, bad, "ld_dst < cols"),
        ("sbt_scatter_add_rows", {11: 0}, bad, "tile_c 0"),
        ("sbt_scatter_add_rows", {2: 0}, ok, "empty destination"),
        ("sbt_ragged_tile_load", {3: -1}, bad, "negative heads"),
        ("sbt_ragged_tile_load", {5: 0}, bad, "ld_row 0"),
        ("sbt_ragged_tile_load", {7: None}, bad, "cu_seqlens NULL"),
        ("sbt_ragged_tile_load", {8: 0}, ok, "no sequences"),
        ("sbt_ragged_tile_store", {9: 0}, bad, "ld_row 0"),
        ("sbt_ragged_tile_store", {7: None}, bad, "x NULL"),
        ("sbt_ragged_tile_store", {8: 0}, ok, "empty packed array"),
        ("sbt_gemm_bounded", {1: 2}, bad, "lda < K"),
        ("sbt_gemm_bounded", {5: 2}, bad, "ldc < N"),
        ("sbt_gemm_bounded", {6: F16}, uns, "c_dtype"),
        ("sbt_gemm_bounded", {7: -1}, bad, "negative M"),
        ("sbt_gemm_bounded", {4: None}, bad, "C NULL"),
        ("sbt_gemm_bounded", {11: 16}, aln, "workspace too small"),
        ("sbt_gemm_bounded", {10: X + 4096 * 16 + 16}, aln, "workspace not 256-byte aligned"),
        ("sbt_gemm_bounded", {7: 0}, ok, "empty C"),
        ("sbt_gemm_block_scaled", {0: E8M0}, uns, "operand format E8M0"),
        ("sbt_gemm_block_scaled", {6: E5M2}, uns, "scale format E5M2"),
        ("sbt_gemm_block_scaled", {11: 3}, bad, "K_s does not divide K"),
        ("sbt_gemm_block_scaled", {0: E2M1, 2: 33}, bad, "E2M1 A with an odd lda"),
        ("sbt_gemm_block_scaled", {8: 0}, bad, "ld_sa < K_s"),
        ("sbt_gemm_block_scaled", {12: X + 4096 * 5, 13: 5, 15: 4}, bad, "acc aliasing D with another ld"),
        ("sbt_gemm_block_scaled", {20: 16}, aln, "workspace too small"),
        ("sbt_gemm_block_scaled", {16: 0}, ok, "empty D"),
    ], base


@pytest.mark.parametrize("i", range(len(_validation_cases()[0])))
def test_argument_validation_before_the_device(lib, i):
    import torch
    if torch.cuda.is_available():
        pytest.skip("CPU-only check: a stand-in context must never reach a device")
    cases, base = _validation_cases()
    name, change, want, what = cases[i]
    args = list(base[name])
    for k, v in change.items():
        args[k] = v
    ctx = ctypes.create_string_buffer(4096)
    assert getattr(lib, name)(ctx, *args) == want, (what, lib.sbt_last_error_message())


def test_workspace_queries_validate_on_the_host(lib):
    ctx = ctypes.create_string_buffer(4096)
    n = ctypes.c_size_t(0)
    assert lib.sbt_gemm_bounded_workspace_size(ctx, 8, 8, 8, 8, 8, ctypes.byref(n)) == sbt.SBT_OK
    assert lib.sbt_gemm_bounded_workspace_size(ctx, 8, 8, 8, 4, 8, ctypes.byref(n)) == sbt.SBT_ERR_INVALID_ARG
    assert lib.sbt_gemm_bounded_workspace_size(ctx, -1, 8, 8, 8, 8, ctypes.byref(n)) == sbt.SBT_ERR_INVALID_ARG
    assert lib.sbt_gemm_bounded_workspace_size(None, 8, 8, 8, 8, 8, ctypes.byref(n)) == sbt.SBT_ERR_INVALID_ARG
    assert lib.sbt_gemm_block_scaled_workspace_size(ctx, 8, 8, -8, ctypes.byref(n)) == sbt.SBT_ERR_INVALID_ARG
    assert lib.sbt_gemm_block_scaled_workspace_size(ctx, 8, 8, 64, ctypes.byref(n)) == sbt.SBT_OK


def test_noalloc_refuses_a_shape_beyond_its_scratch_on_the_host(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("CPU-only check: a stand-in context must never reach a device")
    ctx = ctypes.create_string_buffer(4096)
    p = lambda k: X + 4096 * k
    # odd leading dimensions at 4096^3 need staging far beyond the fixed 16 MiB array
    st = lib.sbt_gemm_bounded_noalloc(ctx, p(0), 4097, p(1), 4097, p(2), 4097, BF16, 4096, 4096, 4096, None)
    assert st == sbt.SBT_ERR_INVALID_ARG and b"fixed" in lib.sbt_last_error_message()
    assert lib.sbt_gemm_bounded_noalloc(None, p(0), 8, p(1), 8, p(2), 8, BF16, 4, 4, 4, None) == sbt.SBT_ERR_INVALID_ARG
