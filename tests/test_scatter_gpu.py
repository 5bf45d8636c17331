"""GPU parity of sbt_scatter_rows_masked against the CPU oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
import scatter_boundary_tile_gb300 as sbt
import synth
import synth.workloads as wl
from gpu_helpers import Canvas, dev, host, sync

pytestmark = pytest.mark.gpu


def gpu_scatter(ctx, dst_init, rows, cols, ld_dst, idx, src, ld_src, tile_c, dtype, row_offset=0, col_offset=0,
                mask=None, ld_mask=0, path="auto"):
    canvas = Canvas(dst_init.nbytes, fill=dst_init)
    s, i = dev(src), dev(idx.astype(np.int32))
    m = dev(mask) if mask is not None else None
    ctx.set_path(path)
    sbt.scatter_rows_masked(ctx, canvas.ptr, rows, cols, ld_dst, i, idx.size, s, ld_src, tile_c,
                            row_offset=row_offset, col_offset=col_offset, mask=m, ld_mask=ld_mask, dtype=dtype)
    sync()
    assert canvas.guards_intact()
    return canvas.inner(dst_init.dtype, dst_init.shape)


@pytest.mark.parametrize("n_idx", [1, 33, 1000])
def test_unique_rows_fp32(ctx, n_idx):
    d = wl.scatter_rows_f32(dst_rows=5000, n_idx=n_idx, cols=256)
    dst = np.zeros((5000, 256), np.float32)
    want = oracle.scatter_rows_masked(dst.copy(), 5000, 256, 256, d["idx"], d["src"], 256, 256, mask=d["mask"])
    for path in ("auto", "tma", "vector", "scalar"):
        got = gpu_scatter(ctx, dst, 5000, 256, 256, d["idx"], d["src"], 256, 256, "f32", mask=d["mask"],
                          ld_mask=256, path=path)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), path


@pytest.mark.parametrize("tile_c,dtype", [(4096, "f32"), (3000, "f32"), (8192, "bf16")])
def test_wide_rows_one_row_per_chunk(ctx, tile_c, dtype):
    # Rows of up to 16 KiB plus a 4 KiB mask: the bulk ring holds one row per stage.
    rows, n = 70, 23
    idx = synth.permutation_prefix(311, rows, n).astype(np.int32)
    if dtype == "f32":
        src = synth.uniform_f32(312, (n, tile_c), -1.0, 1.0)
        dst = np.full((rows, tile_c), wl.F32_CANARY_BITS, np.uint32).view(np.float32)
    else:
        src = synth.normal_bf16(312, (n, tile_c))
        dst = np.full((rows, tile_c), 0xDEAD, np.uint16)
    mask = synth.bernoulli_u8(313, (n, tile_c), 0.9)
    want = oracle.scatter_rows_masked(dst.copy(), rows, tile_c, tile_c, idx, src, tile_c, tile_c, mask=mask,
                                      ld_mask=tile_c)
    for path in ("auto", "tma", "vector"):
        got = gpu_scatter(ctx, dst, rows, tile_c, tile_c, idx, src, tile_c, tile_c, dtype, mask=mask, ld_mask=tile_c,
                          path=path)
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), path


CASES = [
    # rows, cols, ld_dst, tile_c, ld_src, col_offset, row_offset, ld_mask (0 = no mask)
    (300, 64, 64, 64, 64, 0, 0, 64),
    (300, 64, 72, 64, 64, 8, 0, 67),      # unaligned mask rows
    (300, 64, 64, 64, 64, -8, 3, 64),     # columns clipped on the left
    (300, 61, 64, 64, 64, 0, -2, 0),      # partial last vector, no mask
    (300, 50, 53, 37, 41, 5, 0, 37),      # unaligned everything
    # masked rows through the bulk ring: destination units not 4-byte aligned (bf16), odd clips
    (300, 64, 72, 64, 64, 3, 0, 64),      # odd column offset, right clip
    (300, 64, 65, 64, 64, 0, 0, 64),      # odd destination stride
    (300, 61, 64, 64, 64, -2, 0, 64),     # left clip by a whole unit, right clip inside one
    (300, 60, 64, 64, 64, -3, 5, 64),     # odd left clip
    (300, 16, 16, 16, 16, 0, 0, 16),      # narrow rows: a block step spans many rows
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_edge_cases(ctx, case, dtype):
    rows, cols, ld_dst, tile_c, ld_src, col_offset, row_offset, ld_mask = case
    n = 97
    idx = synth.permutation_prefix(301, rows + 40, n).astype(np.int64) - 20  # some out of range on both sides
    idx = idx.astype(np.int32)
    if dtype == "f32":
        src = synth.uniform_f32(302, (n, ld_src), 1.0, 2.0)
        dst = np.full((rows, ld_dst), wl.F32_CANARY_BITS, np.uint32).view(np.float32)
    else:
        src = synth.normal_bf16(302, (n, ld_src))
        dst = np.full((rows, ld_dst), 0xDEAD, np.uint16)
    mask = synth.bernoulli_u8(303, (n, ld_mask), 0.85) if ld_mask else None
    want = oracle.scatter_rows_masked(dst.copy(), rows, cols, ld_dst, idx, src, ld_src, tile_c,
                                      row_offset=row_offset, col_offset=col_offset, mask=mask, ld_mask=ld_mask or None)
    for path in ("auto", "tma", "vector", "scalar"):
        got = gpu_scatter(ctx, dst, rows, cols, ld_dst, idx, src, ld_src, tile_c, dtype, row_offset=row_offset,
                          col_offset=col_offset, mask=mask, ld_mask=ld_mask, path=path)
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), path


def test_duplicate_indices_land_one_candidate(ctx):
    rows, cols, n = 16, 64, 200
    idx = synth.int_below(304, n, 4).astype(np.int32)  # heavy duplication into rows 0..3
    src = synth.uniform_f32(305, (n, cols), 1.0, 2.0)
    mask = synth.bernoulli_u8(306, (n, cols), 0.5)
    dst = np.full((rows, cols), -1.0, np.float32)
    got = gpu_scatter(ctx, dst, rows, cols, cols, idx, src, cols, cols, "f32", mask=mask, ld_mask=cols)
    for r in range(rows):
        for j in range(cols):
            cands = {-1.0} | {float(src[k, j]) for k in np.nonzero(idx == r)[0] if mask[k, j]}
            assert float(got[r, j]) in cands
    assert np.all(got[4:] == -1.0)


def test_empty_and_invalid(ctx):
    before = ctx.launch_count
    sbt.scatter_rows_masked(ctx, None, 0, 0, 0, None, 0, None, 8, 8, dtype="f32")
    b = dev(np.zeros(64, np.float32))
    with pytest.raises(sbt.SbtError):
        sbt.scatter_rows_masked(ctx, b, 4, 8, 4, b, 2, b, 8, 8, dtype="f32")  # ld_dst < cols
    with pytest.raises(sbt.SbtError):
        sbt.scatter_rows_masked(ctx, b, 4, 8, 8, b, 2, b, 4, 8, dtype="f32")  # ld_src < tile_c
    assert ctx.launch_count == before


@pytest.mark.parametrize("path", ["auto", "tma", "vector"])
def test_full_size_workload_bit_exact(ctx, path):
    """4,194,304 x 256 fp32 destination (zero), 1,048,576 unique rows, Bernoulli(0.9) mask:
    the launch the benchmark times; the whole 4 GiB destination is compared."""
    d = wl.scatter_rows_f32()
    rows, cols = d["dst_rows"], d["cols"]
    dst_dev = torch.zeros(rows * cols * 4, dtype=torch.uint8, device="cuda")
    s, i, m = dev(d["src"]), dev(d["idx"]), dev(d["mask"])
    ctx.set_path(path)
    sbt.scatter_rows_masked(ctx, dst_dev, rows, cols, cols, i, d["idx"].size, s, cols, cols, mask=m, ld_mask=cols,
                            dtype="f32")
    got = host(dst_dev, np.uint32, (rows, cols))
    del dst_dev, s, m
    want = np.zeros((rows, cols), np.float32)
    oracle.scatter_rows_masked(want, rows, cols, cols, d["idx"], d["src"], cols, cols, mask=d["mask"])
    assert np.array_equal(got, want.view(np.uint32))
