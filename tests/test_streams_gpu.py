"""Calls are asynchronous on the caller's stream.

Every call enqueues its kernels on the stream it is given (the binding passes
torch's current stream) and returns.  These tests run chains of dependent
calls on side streams with no synchronisation between the calls, while the
default stream is kept busy, and check the final results bit for bit against
the oracle; they also run two independent chains on two streams at once.
"""
import numpy as np
import pytest
import torch

import oracle
import scatter_boundary_tile_gb300 as sbt
import synth
import synth.workloads as wl
from gpu_helpers import dev, host

pytestmark = pytest.mark.gpu


def busy_default_stream():
    """Queue a few milliseconds of unrelated work on the default stream."""
    a = torch.randn(4096, 4096, device="cuda")
    for _ in range(4):
        a = a @ a
        a = a / a.norm()
    return a


def gather_scatter_buffers(d):
    """Device buffers of one gather -> scatter chain, made (and synchronised) up front."""
    rows, cols, n = d["n_rows"], d["cols"], d["idx"].size
    bufs = (dev(d["table"]), dev(d["idx"]), torch.empty(n * cols * 2, dtype=torch.uint8, device="cuda"),
            torch.zeros(rows * cols * 2, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    return bufs


def gather_then_scatter(ctx, d, bufs, stream):
    """gather rows of a table, then scatter them into a fresh array: with unique
    valid indices the destination rows equal the gathered rows."""
    rows, cols, n = d["n_rows"], d["cols"], d["idx"].size
    table, idx, out, back = bufs
    with torch.cuda.stream(stream):
        sbt.gather_rows(ctx, table, rows, cols, cols, idx, n, out, cols, cols, dtype="bf16")
        sbt.scatter_rows_masked(ctx, back, rows, cols, cols, idx, n, out, cols, cols, dtype="bf16")
    return out, back


def unique_gather(seed, rows=20000, n=6000, cols=512):
    d = wl.gather_rows_bf16(n_rows=rows, n_idx=1, cols=cols)
    d["idx"] = synth.permutation_prefix(seed, rows, n).astype(np.int32)
    return d


def check_gather_scatter(d, out, back):
    rows, cols, n = d["n_rows"], d["cols"], d["idx"].size
    want = oracle.gather_rows(d["table"], rows, cols, cols, d["idx"], cols)
    assert np.array_equal(host(out, np.uint16, (n, cols)), want)
    got_back = host(back, np.uint16, (rows, cols))
    assert np.array_equal(got_back[d["idx"]], want)
    others = np.ones(rows, bool)
    others[d["idx"]] = False
    assert not got_back[others].any()


def test_dependent_calls_on_a_side_stream(ctx):
    d = unique_gather(701)
    bufs = gather_scatter_buffers(d)
    s = torch.cuda.Stream()
    busy = busy_default_stream()
    out, back = gather_then_scatter(ctx, d, bufs, s)
    ctx.check_status(s)  # synchronises s only
    check_gather_scatter(d, out, back)
    torch.cuda.synchronize()
    del busy


def test_two_streams_at_once(ctx):
    d1, d2 = unique_gather(702), unique_gather(703)
    bufs1, bufs2 = gather_scatter_buffers(d1), gather_scatter_buffers(d2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    o1, b1 = gather_then_scatter(ctx, d1, bufs1, s1)
    o2, b2 = gather_then_scatter(ctx, d2, bufs2, s2)
    s1.synchronize()
    s2.synchronize()
    ctx.check_status()
    check_gather_scatter(d1, o1, b1)
    check_gather_scatter(d2, o2, b2)


def test_tile_load_store_and_gemm_chain_on_a_side_stream(ctx):
    # padded load -> clipped store round trip, then a GEMM reading the stored array,
    # all queued on one side stream without synchronising in between
    M, N, K = 200, 300, 160
    g = wl.gemm_bf16(M=M, N=N, K=K, tag=11)
    A_src = dev(g["A"])
    gr, gc = -(-M // 64), -(-g["lda"] // 32)
    tiles = torch.empty(gr * gc * 64 * 32 * 2, dtype=torch.uint8, device="cuda")
    A_copy = torch.zeros(M * g["lda"] * 2, dtype=torch.uint8, device="cuda")
    B = dev(g["B"])
    C = torch.empty(M * g["ldc"] * 2, dtype=torch.uint8, device="cuda")
    ws_n = sbt.gemm_bounded_workspace_size(ctx, M, N, K, g["lda"], g["ldb"])
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()  # inputs in place before the side stream starts
    s = torch.cuda.Stream()
    busy = busy_default_stream()
    with torch.cuda.stream(s):
        sbt.tile_load_padded(ctx, A_src, M, g["lda"], g["lda"], 1, 0, 0, 64, 32, gr, gc, 64, 32, tiles, dtype="bf16")
        sbt.tile_store_clipped(ctx, tiles, gr, gc, 64, 32, A_copy, M, g["lda"], g["lda"], 1, 0, 0, 64, 32,
                               dtype="bf16")
        sbt.gemm_bounded(ctx, A_copy, g["lda"], B, g["ldb"], C, g["ldc"], M, N, K, ws, ws_n)
    s.synchronize()
    ctx.check_status()
    assert np.array_equal(host(A_copy, np.uint16, (M, g["lda"])), g["A"])
    got = synth.bf16_bits_to_f32(host(C, np.uint16, (M, g["ldc"]))[:, :N]).astype(np.float64)
    ref = oracle.gemm_f64(g["A"], g["lda"], g["B"], g["ldb"], M, N, K)
    ref_b = synth.bf16_bits_to_f32(oracle.round_bf16(ref)).astype(np.float64)
    assert np.linalg.norm(got - ref_b) / np.linalg.norm(ref) <= 1e-3
    torch.cuda.synchronize()
    del busy
