"""sbt_gemm_bounded_noalloc: the bounded GEMM for callers that cannot allocate.

Some callers cannot call cudaMalloc when they multiply -- plugins confined to
another framework's memory pool, code under a device-memory budget committed
up front, latency-critical paths that cannot take cudaMalloc's implicit
synchronisation.  For them the library keeps the GEMM's staging scratch in a
fixed device array of its own.  These tests call that entry point through the
C ABI and check:

* its C equals, bit for bit, what the workspace entry point writes on the same
  inputs (both run the same kernels), on two calls in a row -- the second call
  finds the first call's data left in the shared array;
* one case against the oracle (fp64 reference, the GEMM gate of the other GEMM
  tests);
* the largest shape whose staging still fits the fixed array, and the refusal,
  before any launch, of the next larger one;
* that a call allocates nothing: free device memory is unchanged around it and
  it launches exactly the kernels the workspace entry point launches.

This file is collected last on purpose.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import scatter_boundary_tile_gb300 as sbt
import synth
import synth.workloads as wl
from gpu_helpers import sync

pytestmark = pytest.mark.gpu
GATE = 1e-3  # relative Frobenius error against the bf16-rounded fp64 reference, as in the other GEMM tests


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8).copy()).to("cuda")


def run_both(ctx, M, N, K, c_dtype, tag):
    """C from the workspace entry point and from the no-alloc one (same inputs), as host arrays."""
    g = wl.gemm_bf16(M=M, N=N, K=K, tag=tag)
    lda, ldb, ldc = g["lda"], g["ldb"], g["ldc"]
    es = 2 if c_dtype == "bf16" else 4
    A, B = to_dev(g["A"]), to_dev(g["B"])
    ws_n = sbt.gemm_bounded_workspace_size(ctx, M, N, K, lda, ldb)
    assert ws_n <= sbt.GEMM_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda")
    c_ref = torch.full((M * ldc * es,), 0x5A, dtype=torch.uint8, device="cuda")
    c_new = torch.full((M * ldc * es,), 0x5A, dtype=torch.uint8, device="cuda")
    sbt.gemm_bounded(ctx, A, lda, B, ldb, c_ref, ldc, M, N, K, ws, ws_n, c_dtype=c_dtype)
    sbt.gemm_bounded_noalloc(ctx, A, lda, B, ldb, c_new, ldc, M, N, K, c_dtype=c_dtype)
    sync()
    ctx.check_status()
    dt = np.uint16 if es == 2 else np.uint32
    ref = c_ref.cpu().numpy().view(dt).reshape(M, ldc)
    new = c_new.cpu().numpy().view(dt).reshape(M, ldc)
    # elements past N in each row of C are never written
    assert np.all(new[:, N:].view(np.uint8) == 0x5A)
    return g, ref[:, :N], new[:, :N]


def test_two_calls_in_a_row_equal_workspace_entry_point(ctx):
    for (M, N, K, tag) in [(1000, 1000, 1000, 11), (65, 97, 73, 12)]:
        _, ref, new = run_both(ctx, M, N, K, "bf16", tag)
        assert np.array_equal(ref, new), (M, N, K)


def test_fp32_output_two_calls(ctx):
    for (M, N, K, tag) in [(300, 257, 129, 13), (129, 600, 64, 14)]:
        _, ref, new = run_both(ctx, M, N, K, "f32", tag)
        assert np.array_equal(ref, new), (M, N, K)


def test_against_the_oracle(ctx):
    M, N, K = 333, 517, 291
    g, _, new = run_both(ctx, M, N, K, "bf16", 15)
    ref = oracle.gemm_f64(g["A"], g["lda"], g["B"], g["ldb"], M, N, K)
    ref_b = synth.bf16_bits_to_f32(oracle.round_bf16(ref)).astype(np.float64)
    got = synth.bf16_bits_to_f32(new).astype(np.float64)
    err = np.linalg.norm(got - ref_b) / np.linalg.norm(ref)
    assert err <= GATE, err


def largest_k_that_fits(ctx, M, N):
    """Largest K (up to 2^16) whose staging fits the fixed scratch, for odd leading dimensions."""
    lo, hi = 1, 1 << 16
    fits = lambda k: sbt.gemm_bounded_workspace_size(ctx, M, N, k, k | 1, N | 1) <= sbt.GEMM_NOALLOC_SCRATCH_BYTES
    assert fits(lo)
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if fits(mid):
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_largest_shape_that_fits(ctx):
    M, N = 1531, 1533
    K = largest_k_that_fits(ctx, M, N)
    assert K > 1000
    _, ref, new = run_both(ctx, M, N, K, "bf16", 16)
    assert np.array_equal(ref, new)
    # one more K step no longer fits: refused before any launch
    A = torch.empty(16, dtype=torch.uint8, device="cuda")
    before = ctx.launch_count
    with pytest.raises(sbt.SbtError) as e:
        sbt.gemm_bounded_noalloc(ctx, A, (K + 1) | 1, A, N | 1, A, N | 1, M, N, K + 64)
    assert e.value.status == sbt.SBT_ERR_INVALID_ARG
    assert ctx.launch_count == before


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


def test_call_allocates_nothing(ctx):
    M, N, K = 1000, 1000, 1000
    g = wl.gemm_bf16(M=M, N=N, K=K, tag=17)
    A, B = to_dev(g["A"]), to_dev(g["B"])
    ws_n = sbt.gemm_bounded_workspace_size(ctx, M, N, K, g["lda"], g["ldb"])
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    C = torch.empty(M * g["ldc"] * 2, dtype=torch.uint8, device="cuda")
    sbt.gemm_bounded_noalloc(ctx, A, g["lda"], B, g["ldb"], C, g["ldc"], M, N, K)  # warm-up: set-up done
    sync()
    n0 = ctx.launch_count
    sbt.gemm_bounded(ctx, A, g["lda"], B, g["ldb"], C, g["ldc"], M, N, K, ws, ws_n)
    sync()
    per_call = ctx.launch_count - n0
    # tensors of earlier tests freed by the garbage collector inside the window would move the
    # counters: collect first and keep the collector off while measuring
    gc.collect()
    sync()
    gc.disable()
    try:
        free0, _ = torch.cuda.mem_get_info()
        alloc0 = torch.cuda.memory_allocated()
        n0 = ctx.launch_count
        for _ in range(3):
            sbt.gemm_bounded_noalloc(ctx, A, g["lda"], B, g["ldb"], C, g["ldc"], M, N, K)
        sync()
        ctx.check_status()
        free1, _ = torch.cuda.mem_get_info()
        alloc1 = torch.cuda.memory_allocated()
    finally:
        gc.enable()
    assert ctx.launch_count - n0 == 3 * per_call
    assert free1 == free0
    assert alloc1 == alloc0
