"""GPU parity of sbt_scatter_add_rows (the gather's backward) against the CPU oracle.

Every destination element that receives one addition must match bit for bit
(the addition is one rounding to nearest even in the element type on both
sides).  With repeated indices the order of additions is unspecified, so
those cases use integer-valued data (every partial sum exact, hence
order-independent and bit-exact), or random data within a rounding bound.
"""
import numpy as np
import pytest
import torch

import oracle
import scatter_boundary_tile_gb300 as sbt
import synth
import synth.workloads as wl
from gpu_helpers import Canvas, dev, host, sync

pytestmark = pytest.mark.gpu
TDT = {"bf16": torch.bfloat16, "f16": torch.float16}


def bits_of(vals, kind):
    if kind == "f32":
        return np.asarray(vals, np.float32)
    return torch.from_numpy(np.asarray(vals, np.float32)).to(TDT[kind]).view(torch.int16).numpy().view(np.uint16)


def gpu_scatter_add(ctx, dst_init, rows, cols, ld_dst, idx, src, ld_src, tile_c, kind, row_offset=0, col_offset=0,
                    path="auto"):
    canvas = Canvas(dst_init.nbytes, fill=dst_init)
    ctx.set_path(path)
    sbt.scatter_add_rows(ctx, canvas.ptr, rows, cols, ld_dst, dev(idx.astype(np.int32)), idx.size, dev(src), ld_src,
                         tile_c, row_offset=row_offset, col_offset=col_offset, dtype=kind)
    sync()
    assert canvas.guards_intact()
    return canvas.inner(dst_init.dtype, dst_init.shape)


@pytest.mark.parametrize("kind", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("case", [(400, 64, 64, 64, 0), (400, 61, 70, 48, 5), (400, 64, 64, 64, -8)])
def test_unique_targets_bit_exact(ctx, kind, case):
    rows, cols, ld, tile_c, col_offset = case
    n = 150
    idx = synth.permutation_prefix(601, rows + 20, n).astype(np.int32) - 10  # some rows out of range
    dst = bits_of(synth.normal_f32(602, (rows, ld)), kind)
    src = bits_of(synth.normal_f32(603, (n, tile_c)) * np.float32(2.0), kind)
    want = oracle.scatter_add_rows(dst.copy(), rows, cols, ld, idx, src, tile_c, tile_c, col_offset=col_offset,
                                   kind=kind)
    for path in ("auto", "scalar"):
        got = gpu_scatter_add(ctx, dst, rows, cols, ld, idx, src, tile_c, tile_c, kind, col_offset=col_offset,
                              path=path)
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), path


@pytest.mark.parametrize("kind", ["f32", "bf16", "f16"])
def test_repeated_indices_integer_values_bit_exact(ctx, kind):
    rows, cols, n = 37, 128, 3000
    idx = synth.int_below(604, n, rows + 4, lo=-2).astype(np.int32)
    dst = bits_of(synth.int_below(605, rows * cols, 9, lo=-4).reshape(rows, cols), kind)
    src = bits_of(synth.int_below(606, n * cols, 3, lo=-1).reshape(n, cols), kind)
    want = oracle.scatter_add_rows(dst.copy(), rows, cols, cols, idx, src, cols, cols, kind=kind)
    for path in ("auto", "scalar"):
        got = gpu_scatter_add(ctx, dst, rows, cols, cols, idx, src, cols, cols, kind, path=path)
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), path


def test_repeated_indices_random_fp32_within_rounding(ctx):
    rows, cols, n = 50, 256, 4000
    idx = synth.int_below(607, n, rows).astype(np.int32)
    src = synth.normal_f32(608, (n, cols))
    dst = np.zeros((rows, cols), np.float32)
    got = gpu_scatter_add(ctx, dst, rows, cols, cols, idx, src, cols, cols, "f32")
    exact = np.zeros((rows, cols), np.float64)
    np.add.at(exact, idx, src.astype(np.float64))
    count = np.bincount(idx, minlength=rows)[:, None]
    # each of `count` fp32 additions rounds once: |error| <= count * 2^-24 * max partial sum
    bound = count * 2.0**-24 * (np.abs(exact) + 4.0 * np.sqrt(count)) + 1e-30
    assert np.all(np.abs(got - exact) <= bound)


def test_invalid_arguments(ctx):
    b = dev(np.zeros(64, np.float32))
    before = ctx.launch_count
    with pytest.raises(sbt.SbtError) as e:
        sbt.scatter_add_rows(ctx, b, 4, 8, 4, b, 2, b, 8, 8, dtype="f32")
    assert e.value.status == sbt.SBT_ERR_INVALID_ARG
    with pytest.raises(sbt.SbtError) as e:
        sbt.scatter_add_rows(ctx, b, 4, 8, 8, b, 2, b, 8, 8, dtype=sbt.SBT_F32 + 7)
    assert e.value.status == sbt.SBT_ERR_UNSUPPORTED
    sbt.scatter_add_rows(ctx, b, 4, 8, 8, b, 0, b, 8, 8, dtype="f32")  # nothing to add
    assert ctx.launch_count == before


def test_full_size_gather_backward_bit_exact(ctx):
    """The backward of the 1,000,000 x 512 bf16 row gather: 1,048,576 gradient rows added into
    a zero gradient table through the same indices (many rows repeat).  Integer-valued
    gradients keep every partial sum exact, so the whole table is compared bit for bit."""
    d = wl.gather_rows_bf16()
    idx, n = d["idx"], d["idx"].size
    grad = bits_of(synth.int_below(609, n * 512, 5, lo=-2).reshape(n, 512), "bf16")
    table = torch.zeros(1_000_000 * 512 * 2, dtype=torch.uint8, device="cuda")
    sbt.scatter_add_rows(ctx, table, 1_000_000, 512, 512, dev(idx), n, dev(grad), 512, 512, dtype="bf16")
    got = host(table, np.uint16, (1_000_000, 512))
    want = oracle.scatter_add_rows(np.zeros((1_000_000, 512), np.uint16), 1_000_000, 512, 512, idx, grad, 512, 512)
    assert np.array_equal(got, want)
