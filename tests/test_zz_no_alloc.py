"""sbt_gemm_bounded_noalloc: the bounded GEMM for callers that cannot allocate.

Some callers cannot call cudaMalloc when they multiply -- code running while a
stream is captured into a CUDA graph, plugins confined to another framework's
memory pool, latency-critical paths that cannot take cudaMalloc's implicit
synchronisation.  For them the library keeps the GEMM's staging scratch in a
fixed device array of its own.  These tests call that entry point through the
C ABI and compare it with the workspace entry point, twice in a row (the
second call finds the first call's data left in the shared array), and check
that a shape too large for the fixed array is refused before any launch.

This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import scatter_boundary_tile_gb300 as sbt
import synth
import synth.workloads as wl
from gpu_helpers import sync

pytestmark = pytest.mark.gpu
TOL = 1e-3  # relative Frobenius, as in the other GEMM tests


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8).copy()).to("cuda")


def compare_with_workspace_entry(ctx, M, N, K, c_dtype, tag):
    g = wl.gemm_bf16(M=M, N=N, K=K, tag=tag)
    lda, ldb, ldc = g["lda"], g["ldb"], g["ldc"]
    es = 2 if c_dtype == "bf16" else 4
    A, B = to_dev(g["A"]), to_dev(g["B"])
    ws_n = sbt.gemm_bounded_workspace_size(ctx, M, N, K, lda, ldb)
    assert 0 < ws_n <= sbt.GEMM_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    c_ref = torch.full((M * ldc * es,), 0x5A, dtype=torch.uint8, device="cuda")
    c_new = torch.full((M * ldc * es,), 0x5A, dtype=torch.uint8, device="cuda")
    sbt.gemm_bounded(ctx, A, lda, B, ldb, c_ref, ldc, M, N, K, ws, ws_n, c_dtype=c_dtype)
    sbt.gemm_bounded_noalloc(ctx, A, lda, B, ldb, c_new, ldc, M, N, K, c_dtype=c_dtype)
    sync()
    ctx.check_status()
    dt = np.uint16 if es == 2 else np.float32
    ref = c_ref.cpu().numpy().view(dt).reshape(M, ldc)
    new = c_new.cpu().numpy().view(dt).reshape(M, ldc)
    if es == 2:
        r = synth.bf16_bits_to_f32(ref[:, :N]).astype(np.float64)
        n = synth.bf16_bits_to_f32(new[:, :N]).astype(np.float64)
    else:
        r, n = ref[:, :N].astype(np.float64), new[:, :N].astype(np.float64)
    err = np.linalg.norm(n - r) / np.linalg.norm(r)
    assert err <= TOL, err
    # elements past N in each row of C are never written
    assert np.all(new[:, N:].view(np.uint8) == 0x5A)


def test_two_calls_in_a_row_match_workspace_entry_point(ctx):
    compare_with_workspace_entry(ctx, 1000, 1000, 1000, "bf16", tag=11)
    compare_with_workspace_entry(ctx, 65, 97, 73, "bf16", tag=12)


def test_fp32_output_two_calls(ctx):
    compare_with_workspace_entry(ctx, 300, 257, 129, "f32", tag=13)
    compare_with_workspace_entry(ctx, 129, 600, 64, "f32", tag=14)


def test_shape_beyond_fixed_scratch_is_refused(ctx):
    M, N, K = 8191, 8193, 4097
    need = sbt.gemm_bounded_workspace_size(ctx, M, N, K, K + 1, N)
    assert need > sbt.GEMM_NOALLOC_SCRATCH_BYTES
    A = torch.empty(16, dtype=torch.uint8, device="cuda")
    before = ctx.launch_count
    with pytest.raises(sbt.SbtError) as e:
        sbt.gemm_bounded_noalloc(ctx, A, K + 1, A, N, A, N, M, N, K)
    assert e.value.status == sbt.SBT_ERR_INVALID_ARG
    assert "scratch" in str(e.value)
    assert ctx.launch_count == before
