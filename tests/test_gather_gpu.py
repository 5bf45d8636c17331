"""GPU parity of sbt_gather_rows against the CPU oracle (bit-exact)."""
import os

import numpy as np
import pytest

import oracle
import scatter_boundary_tile_gb300 as sbt
import synth
import synth.workloads as wl
from gpu_helpers import Canvas, dev, host, sync

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
I32_MIN, I32_MAX = np.iinfo(np.int32).min, np.iinfo(np.int32).max
GATHER_LAST_CANVAS = []


def run_gather(ctx, table, rows, cols, ld, idx, tile_c, dtype, row_offset=0, col_offset=0, mask=None, ld_mask=0,
               pad=None, ld_out=None, path="auto", table_byte_offset=0):
    ld_out = tile_c if ld_out is None else ld_out
    es = table.dtype.itemsize
    n = idx.size
    t_dev = dev(table)
    i_dev = dev(idx.astype(np.int32))
    m_dev = dev(mask) if mask is not None else None
    canvas = Canvas(n * ld_out * es)
    GATHER_LAST_CANVAS[:] = [canvas]
    ctx.set_path(path)
    sbt.gather_rows(ctx, t_dev.data_ptr() + table_byte_offset, rows, cols, ld, i_dev, n, canvas.ptr, ld_out, tile_c,
                    row_offset=row_offset, col_offset=col_offset, mask=m_dev, ld_mask=ld_mask, pad=pad, dtype=dtype)
    sync()
    assert canvas.guards_intact()
    return canvas.inner(table.dtype, (n, ld_out))


def oracle_gather(table, rows, cols, ld, idx, tile_c, row_offset=0, col_offset=0, mask=None, ld_mask=None, pad=0,
                  ld_out=None):
    return oracle.gather_rows(table, rows, cols, ld, idx, tile_c, row_offset=row_offset, col_offset=col_offset,
                              mask=mask, ld_mask=ld_mask, pad=pad, ld_out=ld_out)


def test_warp_worked_example(ctx):
    vals = {}
    for line in open(os.path.join(GOLDEN, "warp_gather_even_rows.txt")):
        if "=" in line and not line.startswith("#"):
            k, v = line.split("=")
            vals[k.strip()] = [int(t) for t in v.split()]
    x = np.array(vals["x"], np.float32).reshape(4, 4)
    out = run_gather(ctx, x, 4, 4, 4, np.array(vals["indices"], np.int32), 4, "f32")
    np.testing.assert_array_equal(out, np.array(vals["expected"], np.float32).reshape(2, 4))


@pytest.mark.parametrize("path", ["auto", "scalar"])
def test_small_fp32_table_pad_minus_one(ctx, path):
    d = wl.gather_small()
    a, idx = d["table"], d["idx"]
    got = run_gather(ctx, a, 65, 73, 73, idx, 73, "f32", pad=-1.0, path=path)
    want = oracle_gather(a, 65, 73, 73, idx, 73, pad=np.float32(-1.0))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("row_offset", [0, 5, -3, 2**32 + 1])
def test_sentinels_and_offsets(ctx, row_offset):
    a = synth.uniform_f32(101, (40, 64), -1.0, 1.0)
    idx = np.array([-1, 0, 39, 40, 41, I32_MIN, I32_MAX, -2, 3, -5, 7, 35, 36, 37, 1, 2, 11], np.int32)
    for path in ("auto", "tma", "vector", "scalar"):
        got = run_gather(ctx, a, 40, 64, 64, idx, 64, "f32", row_offset=row_offset, pad=-1.0, path=path)
        want = oracle_gather(a, 40, 64, 64, idx, 64, row_offset=row_offset, pad=np.float32(-1.0))
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), path


@pytest.mark.parametrize("n_idx", [1, 31, 32, 33, 3001])
@pytest.mark.parametrize("col_offset,tile_c", [(0, 512), (8, 496), (-16, 512), (24, 512), (3, 509), (-5, 40)])
def test_bf16_rows_vector_and_edges(ctx, n_idx, col_offset, tile_c):
    d = wl.gather_rows_bf16(n_rows=5000, n_idx=n_idx, cols=512)
    t, idx = d["table"], d["idx"]
    for path in ("auto", "tma", "vector", "scalar"):
        got = run_gather(ctx, t, 5000, 512, 512, idx, tile_c, "bf16", col_offset=col_offset, path=path)
        want = oracle_gather(t, 5000, 512, 512, idx, tile_c, col_offset=col_offset, pad=0)
        assert np.array_equal(got, want), path


@pytest.mark.parametrize("ld_mask_extra", [0, 3])
def test_bf16_mask_and_wide_output(ctx, ld_mask_extra):
    d = wl.gather_rows_bf16(n_rows=700, n_idx=257, cols=128)
    t, idx = d["table"], d["idx"]
    ld_mask = 128 + ld_mask_extra
    mask = synth.bernoulli_u8(102, (257, ld_mask), 0.8)
    ld_out = 136  # columns >= tile_c of the output must stay untouched
    for path in ("auto", "tma", "vector", "scalar"):
        got = run_gather(ctx, t, 700, 128, 128, idx, 128, "bf16", mask=mask, ld_mask=ld_mask, pad=0xBF80,
                         ld_out=ld_out, path=path)
        want = oracle_gather(t, 700, 128, 128, idx, 128, mask=mask, ld_mask=ld_mask, pad=0xBF80, ld_out=ld_out)
        assert np.array_equal(got[:, :128], want[:, :128]), path
        assert np.array_equal(got[:, 128:], GATHER_LAST_CANVAS[0].original(np.uint16, (257, ld_out))[:, 128:]), path


def test_raw_bits_preserved(ctx):
    special = np.array([0x7FC1, 0xFFFF, 0x8000, 0x0001, 0x7F80, 0xFF80, 0x3F80, 0x0000], np.uint16)
    t = np.tile(special, (16, 4))  # 16 x 32
    idx = np.arange(16, dtype=np.int32)[::-1].copy()
    got = run_gather(ctx, t, 16, 32, 32, idx, 32, "bf16")
    assert np.array_equal(got, t[::-1])


def test_unaligned_table_pointer_takes_element_path(ctx):
    # A table starting 2 bytes into its buffer: no 16-byte vector is aligned.
    base = synth.normal_bf16(103, (1 + 300 * 64,))
    t = base[1:].reshape(300, 64)
    idx = synth.int_below(104, 100, 320, lo=-10).astype(np.int32)
    t_dev = dev(base)
    i_dev = dev(idx)
    canvas = Canvas(100 * 64 * 2)
    sbt.gather_rows(ctx, t_dev.data_ptr() + 2, 300, 64, 64, i_dev, 100, canvas.ptr, 64, 64, dtype="bf16")
    sync()
    assert canvas.guards_intact()
    assert np.array_equal(canvas.inner(np.uint16, (100, 64)), oracle_gather(np.ascontiguousarray(t), 300, 64, 64, idx, 64))


def test_empty_inputs(ctx):
    before = ctx.launch_count
    sbt.gather_rows(ctx, None, 0, 0, 0, None, 0, None, 8, 8, dtype="f32")
    assert ctx.launch_count == before
    # an empty table: every index is out of range -> all pad
    idx = np.array([0, 1, -1], np.int32)
    canvas = Canvas(3 * 8 * 4)
    sbt.gather_rows(ctx, None, 0, 8, 8, dev(idx), 3, canvas.ptr, 8, 8, pad=2.5, dtype="f32")
    sync()
    assert np.all(canvas.inner(np.float32, (3, 8)) == 2.5)


def test_invalid_arguments_launch_nothing(ctx):
    before = ctx.launch_count
    buf = dev(np.zeros(64, np.float32))
    with pytest.raises(sbt.SbtError) as e:
        sbt.gather_rows(ctx, buf, 4, 8, 4, buf, 2, buf, 8, 8, dtype="f32")  # ld_src < cols
    assert e.value.status == sbt.SBT_ERR_INVALID_ARG
    with pytest.raises(sbt.SbtError):
        sbt.gather_rows(ctx, buf, 4, 8, 8, buf, 2, buf, 4, 8, dtype="f32")  # ld_out < tile_c
    with pytest.raises(sbt.SbtError):
        sbt.gather_rows(ctx, buf, 4, 8, 8, None, 2, buf, 8, 8, dtype="f32")  # idx NULL
    with pytest.raises(sbt.SbtError):
        sbt.gather_rows(ctx, buf, -4, 8, 8, buf, 2, buf, 8, 8, dtype="f32")
    with pytest.raises(sbt.SbtError):
        sbt.gather_rows(ctx, buf, 4, 8, 8, buf, 2, buf, 8, 0, dtype="f32")  # tile_c 0
    assert ctx.launch_count == before


@pytest.mark.parametrize("path", ["auto", "tma", "vector"])
def test_full_size_workload_bit_exact(ctx, path):
    """1,000,000 x 512 bf16 table, 1,048,576 indices (1 % -1, 0.5 % past the end), the
    launch the benchmark times; the whole 1 GiB output is compared with the oracle."""
    d = wl.gather_rows_bf16()
    t, idx = d["table"], d["idx"]
    n = idx.size
    t_dev, i_dev = dev(t), dev(idx)
    import torch
    out = torch.empty(n * 512 * 2, dtype=torch.uint8, device="cuda")
    ctx.set_path(path)
    sbt.gather_rows(ctx, t_dev, 1_000_000, 512, 512, i_dev, n, out, 512, 512, dtype="bf16")
    got = host(out, np.uint16, (n, 512))
    del t_dev, out
    want = oracle_gather(t, 1_000_000, 512, 512, idx, 512)
    assert np.array_equal(got, want)
    assert (idx == -1).sum() > 0 and (idx >= 1_000_000).sum() > 0
