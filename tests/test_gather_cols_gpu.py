"""GPU parity of sbt_gather_cols (the gather along axis 1) against the CPU oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
import scatter_boundary_tile_gb300 as sbt
import synth
from gpu_helpers import Canvas, dev, host, sync

pytestmark = pytest.mark.gpu
I32_MIN, I32_MAX = np.iinfo(np.int32).min, np.iinfo(np.int32).max


def gpu_gather_cols(ctx, a, rows, cols, ld, idx, tile_r, dtype, row_offset=0, col_offset=0, pad=None, ld_out=None):
    n = idx.size
    ld_out = n if ld_out is None else ld_out
    canvas = Canvas(tile_r * ld_out * a.dtype.itemsize)
    sbt.gather_cols(ctx, dev(a), rows, cols, ld, dev(idx.astype(np.int32)), n, canvas.ptr, ld_out, tile_r,
                    row_offset=row_offset, col_offset=col_offset, pad=pad, dtype=dtype)
    sync()
    assert canvas.guards_intact()
    return canvas.inner(a.dtype, (tile_r, ld_out)), canvas.original(a.dtype, (tile_r, ld_out))


@pytest.mark.parametrize("row_offset,col_offset", [(0, 0), (-3, 2), (10, -5), (2**32, 0)])
def test_fp32_sentinels_and_offsets(ctx, row_offset, col_offset):
    a = synth.uniform_f32(701, (40, 70), -1.0, 1.0)
    idx = np.array([-1, 0, 63, 64, 65, I32_MIN, I32_MAX, 5, 5, 30, 2, 61, 62, 17], np.int32)
    got, _ = gpu_gather_cols(ctx, a, 40, 64, 70, idx, 37, "f32", row_offset, col_offset, pad=-1.0)
    want = oracle.gather_cols(a, 40, 64, 70, idx, 37, row_offset=row_offset, col_offset=col_offset,
                              pad=np.float32(-1.0))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("n_idx,tile_r", [(1, 1), (255, 33), (256, 32), (257, 70), (3000, 9)])
def test_bf16_shapes_and_untouched_columns(ctx, n_idx, tile_r):
    a = synth.normal_bf16(702, (100, 1031))
    idx = synth.int_below(703, n_idx, 1040, lo=-4).astype(np.int32)
    got, orig = gpu_gather_cols(ctx, a, 100, 1031, 1031, idx, tile_r, "bf16", row_offset=5, ld_out=n_idx + 3)
    want = oracle.gather_cols(a, 100, 1031, 1031, idx, tile_r, row_offset=5, ld_out=n_idx + 3)
    assert np.array_equal(got[:, :n_idx], want[:, :n_idx])
    assert np.array_equal(got[:, n_idx:], orig[:, n_idx:])


def test_empty_and_invalid(ctx):
    before = ctx.launch_count
    b = dev(np.zeros(64, np.float32))
    sbt.gather_cols(ctx, b, 4, 8, 8, b, 0, b, 8, 2, dtype="f32")
    with pytest.raises(sbt.SbtError):
        sbt.gather_cols(ctx, b, 4, 8, 8, b, 9, b, 8, 2, dtype="f32")  # ld_out < n_idx
    with pytest.raises(sbt.SbtError):
        sbt.gather_cols(ctx, b, 4, 8, 4, b, 2, b, 8, 2, dtype="f32")  # ld_src < cols
    assert ctx.launch_count == before


def test_large_column_gather(ctx):
    """4,096 random columns (1% -1) of every row of a 2,048 x 100,003 bf16 matrix."""
    rows, cols = 2048, 100_003
    a = synth.normal_bf16(704, (rows, cols))
    idx = synth.int_below(705, 4096, cols).astype(np.int32)
    idx[::100] = -1
    out = torch.empty(rows * 4096 * 2, dtype=torch.uint8, device="cuda")
    sbt.gather_cols(ctx, dev(a), rows, cols, cols, dev(idx), 4096, out, 4096, rows, dtype="bf16")
    assert np.array_equal(host(out, np.uint16, (rows, 4096)), oracle.gather_cols(a, rows, cols, cols, idx, rows))
