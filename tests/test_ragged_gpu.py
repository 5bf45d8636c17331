"""GPU parity of sbt_ragged_tile_load against the CPU oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
import scatter_boundary_tile_gb300 as sbt
import synth
import synth.workloads as wl
from gpu_helpers import Canvas, dev, host, sync

pytestmark = pytest.mark.gpu


def gpu_ragged(ctx, x, total_rows, heads, depth, ld_row, ld_head, cu, t_pad, dtype, path="auto"):
    batch = cu.size - 1
    es = x.dtype.itemsize
    canvas = Canvas(batch * heads * t_pad * depth * es)
    xd, cd = dev(x), dev(cu.astype(np.int32))
    ctx.set_path(path)
    sbt.ragged_tile_load(ctx, xd, total_rows, heads, depth, ld_row, ld_head, cd, batch, t_pad, canvas.ptr,
                         dtype=dtype)
    sync()
    assert canvas.guards_intact()
    return canvas.inner(x.dtype, (batch, heads, t_pad, depth))


@pytest.mark.parametrize("t_pad", [300, 256, 100, 129])
@pytest.mark.parametrize("depth", [128, 24, 20])
def test_small_batches(ctx, t_pad, depth):
    d = wl.ragged_bf16(batch=5, max_len=300, heads=3, depth=depth)
    x, cu = d["x"], d["cu_seqlens"]
    want = oracle.ragged_tile_load(x, d["total_rows"], 3, depth, 3 * depth, depth, cu, t_pad)
    for path in ("auto", "scalar"):
        got = gpu_ragged(ctx, x, d["total_rows"], 3, depth, 3 * depth, depth, cu, t_pad, "bf16", path=path)
        assert np.array_equal(got, want), path


def test_fp32_strided_heads(ctx):
    # heads interleaved with padding: ld_head 40 > depth 32, ld_row 4*40 + 8
    total, H, D, ldh, ldr = 90, 4, 32, 40, 168
    x = synth.uniform_f32(401, (total, ldr))
    cu = np.array([0, 10, 10, 70, 90], np.int32)
    want = oracle.ragged_tile_load(x, total, H, D, ldr, ldh, cu, 64)
    got = gpu_ragged(ctx, x, total, H, D, ldr, ldh, cu, 64, "f32")
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_inconsistent_metadata_reads_zero(ctx):
    x = synth.normal_bf16(402, (10, 2, 8))
    cu = np.array([0, 0, 8, 14, 3, -5, 4], np.int32)  # empty, past total_rows, negative length, negative start
    want = oracle.ragged_tile_load(x, 10, 2, 8, 16, 8, cu, 6)
    got = gpu_ragged(ctx, x, 10, 2, 8, 16, 8, cu, 6, "bf16")
    assert np.array_equal(got, want)


def test_equal_lengths_is_transpose(ctx):
    B, T, H, D = 4, 256, 8, 128
    x = synth.normal_bf16(403, (B * T, H, D))
    cu = np.arange(B + 1, dtype=np.int32) * T
    got = gpu_ragged(ctx, x, B * T, H, D, H * D, D, cu, T, "bf16")
    assert np.array_equal(got, x.reshape(B, T, H, D).transpose(0, 2, 1, 3))


def test_full_size_workload_bit_exact(ctx):
    """batch 64, lengths uniform in [1, 4096], 8 heads, depth 128, bf16 -> [64][8][4096][128]:
    the launch the benchmark times; the whole output is compared."""
    d = wl.ragged_bf16()
    x, cu = d["x"], d["cu_seqlens"]
    out = torch.empty(64 * 8 * 4096 * 128 * 2, dtype=torch.uint8, device="cuda")
    xd, cd = dev(x), dev(cu)
    sbt.ragged_tile_load(ctx, xd, d["total_rows"], 8, 128, 8 * 128, 128, cd, 64, 4096, out, dtype="bf16")
    got = host(out, np.uint16, (64, 8, 4096, 128))
    want = oracle.ragged_tile_load(x, d["total_rows"], 8, 128, 1024, 128, cu, 4096)
    assert np.array_equal(got, want)


# ----------------------------------------------------------------------------- ragged store (the inverse)

def gpu_ragged_store(ctx, tiles, x_init, total_rows, ld_row, ld_head, cu, dtype, path="auto"):
    batch, heads, t_pad, depth = tiles.shape
    canvas = Canvas(x_init.nbytes, fill=x_init)
    td, cd = dev(tiles), dev(cu.astype(np.int32))
    ctx.set_path(path)
    sbt.ragged_tile_store(ctx, td, batch, heads, depth, t_pad, cd, canvas.ptr, total_rows, ld_row, ld_head,
                          dtype=dtype)
    sync()
    assert canvas.guards_intact()
    return canvas.inner(x_init.dtype, x_init.shape)


@pytest.mark.parametrize("t_pad", [300, 256, 100, 129])
@pytest.mark.parametrize("depth", [128, 24, 20])
def test_store_small_batches(ctx, t_pad, depth):
    d = wl.ragged_bf16(batch=5, max_len=300, heads=3, depth=depth)
    cu, total = d["cu_seqlens"], d["total_rows"]
    tiles = synth.normal_bf16(404, (5, 3, t_pad, depth))
    x0 = np.full((total, 3, depth), 0xDEAD, np.uint16)
    want = oracle.ragged_tile_store(tiles, x0.copy(), total, 3 * depth, depth, cu)
    for path in ("auto", "scalar"):
        got = gpu_ragged_store(ctx, tiles, x0, total, 3 * depth, depth, cu, "bf16", path=path)
        assert np.array_equal(got, want), path


def test_store_fp32_strided_heads_and_bad_metadata(ctx):
    total, H, D, ldh, ldr = 90, 4, 32, 40, 168
    # negative start (rows -3..4), an empty sequence, one running past total_rows; none overlap
    cu = np.array([-3, 5, 10, 10, 70, 90, 95], np.int32)
    tiles = synth.uniform_f32(405, (6, H, 64, D), 1.0, 2.0)
    x0 = np.full((total, ldr), wl.F32_CANARY_BITS, np.uint32).view(np.float32)
    want = oracle.ragged_tile_store(tiles, x0.copy(), total, ldr, ldh, cu)
    got = gpu_ragged_store(ctx, tiles, x0, total, ldr, ldh, cu, "f32")
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_store_leaves_spare_rows_after_the_last_sequence(ctx):
    # every tile row (also those past a length) holds data; the packed buffer has 6 spare rows
    cu = np.array([0, 3, 3, 40, 45], np.int32)  # lengths 3, 0, 37, 5, all below t_pad = 48
    total, H, D = 51, 2, 16
    tiles = synth.normal_bf16(407, (4, H, 48, D))
    x0 = np.full((total, H, D), 0xDEAD, np.uint16)
    want = oracle.ragged_tile_store(tiles, x0.copy(), total, H * D, D, cu)
    assert np.all(want[45:] == 0xDEAD)
    for path in ("auto", "scalar"):
        got = gpu_ragged_store(ctx, tiles, x0, total, H * D, D, cu, "bf16", path=path)
        assert np.array_equal(got, want), path


def test_store_round_trip(ctx):
    d = wl.ragged_bf16(batch=9, max_len=700, heads=8, depth=128)
    x, cu, total = d["x"], d["cu_seqlens"], d["total_rows"]
    tiles = gpu_ragged(ctx, x, total, 8, 128, 1024, 128, cu, 700, "bf16")
    back = gpu_ragged_store(ctx, tiles, np.zeros_like(x), total, 1024, 128, cu, "bf16")
    assert np.array_equal(back, x)


def test_store_full_size_workload_bit_exact(ctx):
    """batch 64, lengths uniform in [1, 4096], 8 heads, depth 128: [64][8][4096][128] bf16 tiles
    stored back into the packed array; the whole packed array is compared."""
    d = wl.ragged_bf16()
    cu, total = d["cu_seqlens"], d["total_rows"]
    tiles = synth.normal_bf16(406, (64, 8, 4096, 128))
    xd = torch.zeros(total * 1024 * 2, dtype=torch.uint8, device="cuda")
    sbt.ragged_tile_store(ctx, dev(tiles), 64, 8, 128, 4096, dev(cu), xd, total, 1024, 128, dtype="bf16")
    got = host(xd, np.uint16, (total, 8, 128))
    want = oracle.ragged_tile_store(tiles, np.zeros((total, 8, 128), np.uint16), total, 1024, 128, cu)
    assert np.array_equal(got, want)


def test_grouped_ragged_tiles(ctx):
    """group > 1: packed [rows][middle=8][group=4][depth=32] read as tiles of (position, group member)
    rows, i.e. the ragged load with depth' = group * depth."""
    d = wl.ragged_bf16(batch=6, max_len=500, heads=8, depth=128)  # 128 = group 4 x depth 32
    x, cu = d["x"], d["cu_seqlens"]
    got = gpu_ragged(ctx, x, d["total_rows"], 8, 128, 1024, 128, cu, 512, "bf16")
    want = oracle.ragged_tile_load(x, d["total_rows"], 8, 128, 1024, 128, cu, 512)
    assert np.array_equal(got, want)
    g = got.reshape(6, 8, 512, 4, 32)
    xg = x.reshape(-1, 8, 4, 32)
    b, m, s, gi = 2, 5, 3, 1
    if s < d["lens"][b]:
        np.testing.assert_array_equal(g[b, m, s, gi], xg[cu[b] + s, m, gi])
