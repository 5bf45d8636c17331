"""Bounded device waits: a withheld copy makes a consumer's wait run out.

The test hook makes the GEMM's TMA producer (or the bulk row kernels'
producer warp) skip its first copy, so the barrier that copy would complete is
never armed.  Nothing faults and nothing hangs: the waiting warp gives up
after the context's wait limit, the kernel sets the device status flag, drains
its copies in flight (bounded), frees its TMEM and returns.  The host reads
SBT_ERR_DEVICE_TIMEOUT from sbt_check_status, and the same context then runs
the same call correctly.
"""
import numpy as np
import pytest
import torch

import oracle
import scatter_boundary_tile_gb300 as sbt
import synth
import synth.workloads as wl
from gpu_helpers import dev, host, sync

pytestmark = pytest.mark.gpu
LIMIT_NS = 20_000_000  # 20 ms


def expect_timeout(ctx, launch):
    ctx.set_wait_limit_ns(LIMIT_NS)
    ctx.set_test_hook(True)
    try:
        launch()
        with pytest.raises(sbt.SbtError) as e:
            ctx.check_status()
        assert e.value.status == sbt.SBT_ERR_DEVICE_TIMEOUT
    finally:
        ctx.set_test_hook(False)
        ctx.set_wait_limit_ns(2_000_000_000)
    ctx.check_status()  # the flag was cleared by the read above


@pytest.mark.parametrize("mnk", [(1000, 1000, 1000), (2048, 2560, 256), (4096, 2560, 256)],
                         ids=["single_cta", "cta_pair", "cta_pair_512_rows"])
def test_gemm_wait_runs_out_then_recovers(ctx, mnk):
    M, N, K = mnk
    g = wl.gemm_bf16(M=M, N=N, K=K, tag=21)
    A, B = dev(g["A"]), dev(g["B"])
    C = torch.empty(M * g["ldc"] * 2, dtype=torch.uint8, device="cuda")
    ws_n = sbt.gemm_bounded_workspace_size(ctx, M, N, K, g["lda"], g["ldb"])
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    run = lambda: sbt.gemm_bounded(ctx, A, g["lda"], B, g["ldb"], C, g["ldc"], M, N, K, ws, ws_n)
    expect_timeout(ctx, run)
    run()
    sync()
    ctx.check_status()
    got = synth.bf16_bits_to_f32(host(C, np.uint16, (M, g["ldc"]))[:, :N]).astype(np.float64)
    ref = oracle.gemm_f64(g["A"], g["lda"], g["B"], g["ldb"], M, N, K)
    ref_b = synth.bf16_bits_to_f32(oracle.round_bf16(ref)).astype(np.float64)
    assert np.linalg.norm(got - ref_b) / np.linalg.norm(ref) <= 1e-3


@pytest.mark.parametrize("mnk,fmts", [((600, 700, 256), ("e4m3", "e8m0", 32)), ((600, 8320, 128), ("e4m3", "e8m0", 32)),
                                      ((600, 8320, 512), ("e2m1", "e8m0", 32)), ((600, 700, 512), ("e2m1", "e4m3", 16))],
                         ids=["few_tiles", "many_tiles", "mxf4_many_tiles", "mxf4nvf4_few_tiles"])
def test_block_scaled_mma_wait_runs_out_then_recovers(ctx, mnk, fmts):
    # the tcgen05 block-scaled CTA-pair kernel in its three forms (E4M3 with E8M0 scales per 32;
    # packed E2M1 with E8M0 per 32 or E4M3 per 16), with fewer tiles than CTA pairs and with
    # several tiles per pair
    M, N, K = mnk
    fmt, sfmt, block = fmts
    g = wl.gemm_block_scaled(M=M, N=N, K=K, block=block, afmt=fmt, bfmt=fmt, sfmt=sfmt, tag=22)
    A, B, SA, SB = (dev(g[k]) for k in ("A", "B", "SA", "SB"))
    D = torch.empty(M * g["ldd"] * 4, dtype=torch.uint8, device="cuda")
    ws_n = sbt.gemm_block_scaled_workspace_size(ctx, M, N, K)
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    run = lambda: sbt.gemm_block_scaled(ctx, A, g["lda"], B, g["ldb"], SA, g["ld_sa"], SB, g["ld_sb"], g["Ks"], D,
                                        g["ldd"], M, N, K, workspace=ws, workspace_bytes=ws_n, a_fmt=fmt, b_fmt=fmt,
                                        s_fmt=sfmt)
    expect_timeout(ctx, run)
    run()
    sync()
    ctx.check_status()
    got = host(D, np.float32, (M, g["ldd"]))[:, :N].astype(np.float64)
    ref = oracle.gemm_block_scaled_f64(g["A"], g["lda"], g["SA"], g["ld_sa"], g["B"], g["ldb"], g["SB"], g["ld_sb"],
                                       M, N, K, block, afmt=fmt, bfmt=fmt, sfmt=sfmt)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 1e-5


def test_bulk_scatter_wait_runs_out_then_recovers(ctx):
    d = wl.scatter_rows_f32(dst_rows=20000, n_idx=5000, cols=256)
    rows, n = d["dst_rows"], d["idx"].size
    dst = torch.zeros(rows * 256 * 4, dtype=torch.uint8, device="cuda")
    s_, i, m = dev(d["src"]), dev(d["idx"]), dev(d["mask"])
    ctx.set_path("tma")
    run = lambda: sbt.scatter_rows_masked(ctx, dst, rows, 256, 256, i, n, s_, 256, 256, mask=m, ld_mask=256,
                                          dtype="f32")
    expect_timeout(ctx, run)
    dst.zero_()
    run()
    sync()
    ctx.check_status()
    want = oracle.scatter_rows_masked(np.zeros((rows, 256), np.float32), rows, 256, 256, d["idx"], d["src"], 256, 256,
                                      mask=d["mask"])
    assert np.array_equal(host(dst, np.uint32, (rows, 256)), want.view(np.uint32))


def test_bulk_gather_wait_runs_out_then_recovers(ctx):
    d = wl.gather_rows_bf16(n_rows=5000, n_idx=3000, cols=512)
    t, idx = dev(d["table"]), dev(d["idx"])
    out = torch.empty(3000 * 512 * 2, dtype=torch.uint8, device="cuda")
    ctx.set_path("tma")
    run = lambda: sbt.gather_rows(ctx, t, 5000, 512, 512, idx, 3000, out, 512, 512, dtype="bf16")
    expect_timeout(ctx, run)
    run()
    sync()
    ctx.check_status()
    want = oracle.gather_rows(d["table"], 5000, 512, 512, d["idx"], 512)
    assert np.array_equal(host(out, np.uint16, (3000, 512)), want)
