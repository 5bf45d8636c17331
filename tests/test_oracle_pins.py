"""Pins of the CPU oracle to facts fixed outside it (CPU only).

Each test checks the oracle against something it does not itself compute:
values printed on the pages (tests/golden/), numpy library routines on the
special cases they cover, closed forms and invariants.  A plausible mistake
in the oracle (dropped padding, swapped row/column, an offset applied after
instead of before the bounds check, a transposed GEMM operand, a wrong
rounding rule) fails at least one of them.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = [int(t) for t in v.split()]
    return out


def padded_reference(a, pad, margin):
    """numpy's np.pad: the array surrounded by `margin` pad elements on every side."""
    return np.pad(a, margin, mode="constant", constant_values=pad)


# ----------------------------------------------------------------------------- generator

def test_splitmix64_published_vector():
    # SplitMix64 seeded with 0: the first three outputs of the reference generator
    # (Steele, Lea & Flood 2014; the sequence used to seed xoshiro).
    assert [synth.h(0, i) for i in range(3)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_generator_distributions():
    u = synth.uniform_f32(7, 100000, -1.0, 1.0)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 0.01
    z = synth.bf16_bits_to_f32(synth.normal_bf16(8, 200000)).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    k = synth.int_below(9, 100000, 82, lo=-1)
    assert k.min() == -1 and k.max() == 80
    p = synth.permutation_prefix(10, 1000, 1000)
    assert sorted(p.tolist()) == list(range(1000))


# ----------------------------------------------------------------------------- gather

def test_gather_warp_example():
    g = read_golden("warp_gather_even_rows.txt")
    x = np.array(g["x"], np.float32).reshape(g["x_rows"][0], g["x_cols"][0])
    idx = np.array(g["indices"], np.int32)
    rows, cols = x.shape
    out = oracle.gather_rows(x, rows, cols, cols, idx, tile_c=g["tile_shape"][1])
    np.testing.assert_array_equal(out, np.array(g["expected"], np.float32).reshape(g["tile_shape"]))


@pytest.mark.parametrize("bad", [-1, -2, np.iinfo(np.int32).min, 65, 66, np.iinfo(np.int32).max])
def test_gather_sentinel_reads_pad(bad):
    # warp.tile_load_indexed: a negative or past-the-end source index reads the padding value.
    a = synth.uniform_f32(11, (65, 73), -1.0, 1.0)
    idx = np.array([3, bad, 64], np.int32)
    out = oracle.gather_rows(a, 65, 73, 73, idx, tile_c=73, pad=-1.0)
    np.testing.assert_array_equal(out[0], a[3])
    np.testing.assert_array_equal(out[1], np.full(73, -1.0, np.float32))
    np.testing.assert_array_equal(out[2], a[64])


def test_gather_offset_added_before_check_in_64bit():
    a = synth.uniform_f32(12, (10, 8), -1.0, 1.0)
    idx = np.array([np.iinfo(np.int32).max, -5, 2], np.int32)
    out = oracle.gather_rows(a, 10, 8, 8, idx, tile_c=8, row_offset=5, pad=7.0)
    # INT32_MAX + 5 overflows int32 but not int64: past the end -> pad.  -5 + 5 = row 0.
    np.testing.assert_array_equal(out[0], np.full(8, 7.0, np.float32))
    np.testing.assert_array_equal(out[1], a[0])
    np.testing.assert_array_equal(out[2], a[7])
    # An offset that needs more than 32 bits: truncating it would land on row 5.
    out = oracle.gather_rows(a, 10, 8, 8, np.array([2], np.int32), tile_c=8, row_offset=2**32 + 3, pad=7.0)
    np.testing.assert_array_equal(out[0], np.full(8, 7.0, np.float32))


def test_gather_all_valid_equals_numpy_fancy_indexing():
    a = synth.uniform_f32(13, (300, 50), -1.0, 1.0)
    idx = synth.int_below(14, 97, 300).astype(np.int32)
    out = oracle.gather_rows(a, 300, 50, 50, idx, tile_c=40, col_offset=6)
    np.testing.assert_array_equal(out, a[idx][:, 6:46])


def test_gather_general_equals_numpy_pad_and_clip():
    # Out-of-range rows and columns, negative column offset, strided source, mask.
    rows, cols, ld = 40, 30, 37
    buf = synth.uniform_f32(15, (rows, ld), -1.0, 1.0)
    idx = synth.int_below(16, 200, 60, lo=-10).astype(np.int32)
    mask = synth.bernoulli_u8(17, (200, 45), 0.7)
    pad = np.float32(-3.5)
    for col_offset in (-7, 0, 5):
        out = oracle.gather_rows(buf, rows, cols, ld, idx, tile_c=45, col_offset=col_offset, mask=mask,
                                 pad=pad)
        logical = buf[:, :cols]
        big = padded_reference(logical, pad, 1)  # one pad row/column on each side
        r = np.clip(idx.astype(np.int64), -1, rows) + 1
        c = np.clip(np.arange(45) + col_offset, -1, cols) + 1
        want = big[r][:, c]
        want = np.where(mask != 0, want, pad)
        np.testing.assert_array_equal(out, want)


def test_gather_with_its_own_output_and_mask_leading_dimensions():
    # warp.tile_load_indexed with a per-element mask (cuTile.jl "Memory"): out[k*ld_out + j] and
    # mask[k*ld_mask + j] for j < tile_c, every leading dimension wider than the tile; the mask's extra
    # columns are all ones, so reading them for the real ones would show.
    rows, cols, ld, n, tile_c, ld_out, ld_mask = 30, 24, 29, 50, 20, 27, 23
    a = synth.uniform_f32(18, (rows, ld), -1.0, 1.0)
    idx = synth.int_below(19, n, rows + 6, lo=-3).astype(np.int32)
    mask = np.ones((n, ld_mask), np.uint8)
    mask[:, :tile_c] = synth.bernoulli_u8(20, (n, tile_c), 0.5)
    pad = np.float32(9.0)
    out = oracle.gather_rows(a, rows, cols, ld, idx, tile_c=tile_c, col_offset=2, mask=mask, ld_mask=ld_mask,
                             pad=pad, ld_out=ld_out)
    big = padded_reference(a[:, :cols], pad, 1)
    r = np.clip(idx.astype(np.int64), -1, rows) + 1
    c = np.clip(np.arange(tile_c) + 2, -1, cols) + 1
    want = np.where(mask[:, :tile_c] != 0, big[r][:, c], pad)
    np.testing.assert_array_equal(out[:, :tile_c], want)
    assert not out[:, tile_c:].any()  # columns past the tile are never written


def test_gather_cols_equals_numpy_fancy_indexing_and_pad_clip():
    rows, cols, ld = 30, 50, 53
    a = synth.uniform_f32(71, (rows, ld), -1.0, 1.0)
    logical = a[:, :cols]
    idx = synth.int_below(72, 40, 50).astype(np.int32)
    out = oracle.gather_cols(a, rows, cols, ld, idx, tile_r=25, row_offset=3)
    np.testing.assert_array_equal(out, logical[3:28][:, idx])  # numpy: all coordinates valid
    # out-of-range rows and columns (both sides), via np.pad with one pad row/column around the array
    idx = np.array([-1, 0, 49, 50, np.iinfo(np.int32).min, 7, 52], np.int32)
    pad = np.float32(-2.0)
    out = oracle.gather_cols(a, rows, cols, ld, idx, tile_r=34, row_offset=-2, col_offset=1, pad=pad)
    big = padded_reference(logical, pad, 1)
    r = np.clip(np.arange(34) - 2, -1, rows) + 1
    c = np.clip(idx.astype(np.int64) + 1, -1, cols) + 1
    np.testing.assert_array_equal(out, big[r][:, c])


def test_gather_cols_with_its_own_output_leading_dimension():
    rows, cols, n, tile_r, ld_out = 14, 20, 9, 12, 13
    a = synth.uniform_f32(74, (rows, cols), -1.0, 1.0)
    idx = synth.int_below(75, n, cols + 4, lo=-2).astype(np.int32)
    out = oracle.gather_cols(a, rows, cols, cols, idx, tile_r=tile_r, row_offset=1, pad=4.0, ld_out=ld_out)
    big = padded_reference(a, np.float32(4.0), 1)
    r = np.clip(np.arange(tile_r) + 1, -1, rows) + 1
    c = np.clip(idx.astype(np.int64), -1, cols) + 1
    np.testing.assert_array_equal(out[:, :n], big[r][:, c])
    assert not out[:, n:].any()


def test_gather_cols_is_row_gather_of_the_transpose():
    a = synth.uniform_f32(73, (12, 9), -1.0, 1.0)
    idx = np.array([8, -1, 3, 3, 9, 0], np.int32)
    by_cols = oracle.gather_cols(a, 12, 9, 9, idx, tile_r=12, pad=5.0)
    at = np.ascontiguousarray(a.T)
    by_rows = oracle.gather_rows(at, 9, 12, 12, idx, tile_c=12, pad=np.float32(5.0))
    np.testing.assert_array_equal(by_cols, by_rows.T)


def test_gather_bf16_raw_bits_nan_negzero():
    a = np.array([[0x7FC1, 0x8000, 0x3F80, 0xFF81]], np.uint16)  # NaN payload, -0.0, 1.0, -NaN
    out = oracle.gather_rows(a, 1, 4, 4, np.array([0, -1], np.int32), tile_c=4, pad=0xBF80)
    np.testing.assert_array_equal(out[0], a[0])
    np.testing.assert_array_equal(out[1], np.full(4, 0xBF80, np.uint16))


# ----------------------------------------------------------------------------- tile load / store

def test_tile_load_tylo_concrete_edge():
    g = read_golden("tylo_concrete_edge.txt")
    M, K = g["a_shape"]
    tr, tc = g["tile_shape"]
    r0, c0 = g["origin"]
    # bf16 values that are never zero, so "valid" == "nonzero"
    a = (np.arange(M * K, dtype=np.uint32) % 0x3F00 + 0x0100).astype(np.uint16).reshape(M, K)
    t = oracle.tile_load_padded(a, M, K, K, 1, r0, c0, 0, 0, 1, 1, tr, tc, pad=0)[0, 0]
    nz_rows = np.nonzero(t.any(axis=1))[0]
    nz_cols = np.nonzero(t.any(axis=0))[0]
    assert nz_rows.size == g["valid_rows"][0] and nz_cols.size == g["valid_cols"][0]
    assert np.count_nonzero(t) == g["valid_rows"][0] * g["valid_cols"][0]
    np.testing.assert_array_equal(t[0, :9], a[64, 64:73])
    v = g["vector_elems"][0]
    # one full 16-byte vector of valid K values, then a vector with one valid element
    assert np.count_nonzero(t[0, :v]) == v * g["full_vectors_in_valid_row"][0]
    assert np.count_nonzero(t[0, v:2 * v]) == g["partial_vector_valid_elems"][0]
    # the same tile as tile (1, 2) of the ceil-div grid of (64, 32) tiles over (65, 73)
    gr, gc = -(-M // tr), -(-K // tc)
    assert (gr, gc) == (2, 3)
    grid = oracle.tile_load_padded(a, M, K, K, 1, 0, 0, tr, tc, gr, gc, tr, tc, pad=0)
    np.testing.assert_array_equal(grid[1, 2], t)


@pytest.mark.parametrize("origin", [(0, 0), (-5, -3), (3, 7), (-70, 2), (60, -40)])
@pytest.mark.parametrize("stride_c", [1, 2])
def test_tile_load_equals_numpy_pad_slice(origin, stride_c):
    rows, cols = 65, 73
    buf = synth.uniform_f32(21, (rows, cols * stride_c + 3), -1.0, 1.0)
    ld = buf.shape[1]
    logical = buf[:, : cols * stride_c : stride_c]
    pad = np.float32(9.25)
    tr, tc, sr, sc, gr, gc = 16, 8, 20, 12, 5, 8
    tiles = oracle.tile_load_padded(buf, rows, cols, ld, stride_c, origin[0], origin[1], sr, sc, gr, gc, tr, tc,
                                    pad=pad)
    m = 200
    big = padded_reference(logical, pad, m)
    for ti in range(gr):
        for tj in range(gc):
            r, c = origin[0] + ti * sr + m, origin[1] + tj * sc + m
            np.testing.assert_array_equal(tiles[ti, tj], big[r:r + tr, c:c + tc])


def test_tile_load_valid_count_closed_form():
    rows, cols = 37, 51
    a = synth.uniform_f32(22, (rows, cols), 1.0, 2.0)  # no zero in the data
    tr, tc = 16, 16
    for r0, c0 in [(-9, -9), (30, 40), (0, 0), (-16, 10)]:
        t = oracle.tile_load_padded(a, rows, cols, cols, 1, r0, c0, 0, 0, 1, 1, tr, tc, pad=0)[0, 0]
        vr = max(0, min(r0 + tr, rows) - max(r0, 0))
        vc = max(0, min(c0 + tc, cols) - max(c0, 0))
        assert np.count_nonzero(t) == vr * vc


def test_tile_grid_covers_array_once():
    rows, cols = 65, 73
    a = np.arange(rows * cols, dtype=np.int32).reshape(rows, cols)
    gr, gc = -(-rows // 64), -(-cols // 32)
    t = oracle.tile_load_padded(a, rows, cols, cols, 1, 0, 0, 64, 32, gr, gc, 64, 32, pad=-1)
    vals = t[t >= 0]
    assert vals.size == rows * cols and np.array_equal(np.sort(vals), np.arange(rows * cols))


def test_tile_store_round_trip_and_clipping():
    rows, cols = 65, 73
    a = synth.uniform_f32(23, (rows, cols), -1.0, 1.0)
    tr, tc = 64, 32
    gr, gc = 2, 3
    tiles = oracle.tile_load_padded(a, rows, cols, cols, 1, 0, 0, tr, tc, gr, gc, tr, tc, pad=5.0)
    canary = np.array([synth.workloads.F32_CANARY_BITS], np.uint32).view(np.float32)[0]
    canvas = np.full((70, 81), canary, np.float32)
    view_off = 2 * 81 + 3
    flat = canvas.reshape(-1)
    sub = flat[view_off:]
    oracle.tile_store_clipped(tiles, sub, rows, cols, 81, 1, 0, 0, tr, tc)
    got = canvas[2:2 + rows, 3:3 + cols]
    np.testing.assert_array_equal(got, a)
    mask = np.ones(canvas.shape, bool)
    mask[2:2 + rows, 3:3 + cols] = False
    assert np.all(canvas.view(np.uint32)[mask] == synth.workloads.F32_CANARY_BITS)


def test_tile_store_numpy_slice_assignment_with_negative_origin():
    rows, cols = 30, 20
    dst = np.zeros((rows, cols), np.float32)
    tiles = synth.uniform_f32(24, (2, 2, 8, 8), 1.0, 2.0)
    oracle.tile_store_clipped(tiles, dst, rows, cols, cols, 1, -4, 15, 26, 8)
    want = np.zeros((rows + 100, cols + 100), np.float32)
    m = 50
    for ti in range(2):
        for tj in range(2):
            r, c = -4 + ti * 26 + m, 15 + tj * 8 + m
            want[r:r + 8, c:c + 8] = tiles[ti, tj]
    np.testing.assert_array_equal(dst, want[m:m + rows, m:m + cols])


# ----------------------------------------------------------------------------- scatter

def test_scatter_unique_equals_numpy_where():
    rows, cols, n = 500, 40, 120
    dst = synth.uniform_f32(31, (rows, cols), -1.0, 1.0)
    before = dst.copy()
    idx = synth.permutation_prefix(32, rows, n)
    src = synth.uniform_f32(33, (n, cols), 5.0, 6.0)
    mask = synth.bernoulli_u8(34, (n, cols), 0.9)
    oracle.scatter_rows_masked(dst, rows, cols, cols, idx, src, cols, cols, mask=mask)
    want = before.copy()
    want[idx] = np.where(mask != 0, src, before[idx])
    np.testing.assert_array_equal(dst, want)


def test_scatter_out_of_bounds_rows_and_columns_clipped():
    rows, cols = 10, 6
    dst = np.zeros((rows, cols), np.float32)
    idx = np.array([-1, 10, np.iinfo(np.int32).min, 4], np.int32)
    src = np.arange(4 * 8, dtype=np.float32).reshape(4, 8) + 1
    oracle.scatter_rows_masked(dst, rows, cols, cols, idx, src, 8, 8, col_offset=-1)
    want = np.zeros((rows, cols), np.float32)
    want[4, 0:6] = src[3, 1:7]
    np.testing.assert_array_equal(dst, want)


def test_scatter_rows_past_the_end_leave_the_memory_after_the_array():
    # cuTile.jl "Memory": a bounds-checked store never writes outside the array.  The array is the first
    # 10 rows of a 12-row buffer; indices 10 and 11 name the two rows after it, which must stay zero.
    buf = np.zeros((12, 6), np.float32)
    idx = np.array([10, 11, 3], np.int32)
    src = np.arange(3 * 6, dtype=np.float32).reshape(3, 6) + 1
    oracle.scatter_rows_masked(buf[:10], 10, 6, 6, idx, src, 6, 6)
    want = np.zeros((12, 6), np.float32)
    want[3] = src[2]
    np.testing.assert_array_equal(buf, want)


def test_scatter_duplicates_take_a_candidate():
    rows, cols = 8, 4
    dst = np.full((rows, cols), -1.0, np.float32)
    idx = np.array([2, 2, 5, 2], np.int32)
    src = synth.uniform_f32(35, (4, cols), 1.0, 2.0)
    mask = synth.bernoulli_u8(36, (4, cols), 0.5)
    oracle.scatter_rows_masked(dst, rows, cols, cols, idx, src, cols, cols, mask=mask)
    for j in range(cols):
        cands = {-1.0} | {float(src[k, j]) for k in (0, 1, 3) if mask[k, j]}
        assert float(dst[2, j]) in cands


# ----------------------------------------------------------------------------- scatter-add (gather backward)

def test_scatter_with_row_and_column_offsets_equals_numpy():
    # cuTile.jl "Memory", "Sparse views": source element (k, j) goes to row row_offset + idx[k],
    # column col_offset + j, clipped to the array.  Written out with numpy fancy indexing on the
    # valid (row, column) pairs; the leading dimension is wider than the array.
    rows, cols, ld, n, tile_c, row_offset, col_offset = 60, 30, 33, 40, 31, -5, 2
    idx = (synth.permutation_prefix(37, rows, n) + 5).astype(np.int32)  # rows idx - 5: a permutation prefix
    idx[0], idx[1] = 2, rows + 5                                         # rows -3 and `rows`: clipped
    dst = synth.uniform_f32(38, (rows, ld), -1.0, 1.0)
    before = dst.copy()
    src = synth.uniform_f32(39, (n, tile_c), 5.0, 6.0)
    mask = synth.bernoulli_u8(40, (n, tile_c), 0.8)
    oracle.scatter_rows_masked(dst, rows, cols, ld, idx, src, tile_c, tile_c, row_offset=row_offset,
                               col_offset=col_offset, mask=mask)
    want = before.copy()
    r = idx.astype(np.int64) + row_offset
    c = col_offset + np.arange(tile_c)
    keep_r, keep_c = (r >= 0) & (r < rows), (c >= 0) & (c < cols)
    rr, cc = r[keep_r][:, None], c[keep_c][None, :]
    m = mask[keep_r][:, keep_c] != 0
    want[rr, cc] = np.where(m, src[keep_r][:, keep_c], before[rr, cc])
    np.testing.assert_array_equal(dst, want)


def test_scatter_with_its_own_source_and_mask_leading_dimensions():
    # src[k*ld_src + j] and mask[k*ld_mask + j] for j < tile_c, both wider than the tile; their extra
    # columns hold values (and all-one mask bytes) that a wrong leading dimension would pick up.
    rows, cols, n, tile_c, ld_src, ld_mask = 80, 16, 30, 16, 21, 19
    dst = synth.uniform_f32(41, (rows, cols), -1.0, 1.0)
    before = dst.copy()
    idx = synth.permutation_prefix(42, rows, n)
    src = np.full((n, ld_src), 100.0, np.float32)
    src[:, :tile_c] = synth.uniform_f32(43, (n, tile_c), 5.0, 6.0)
    mask = np.ones((n, ld_mask), np.uint8)
    mask[:, :tile_c] = synth.bernoulli_u8(44, (n, tile_c), 0.5)
    oracle.scatter_rows_masked(dst, rows, cols, cols, idx, src, ld_src, tile_c, mask=mask, ld_mask=ld_mask)
    want = before.copy()
    want[idx] = np.where(mask[:, :tile_c] != 0, src[:, :tile_c], before[idx])
    np.testing.assert_array_equal(dst, want)


def test_scatter_add_with_its_own_source_leading_dimension():
    rows, cols, n, tile_c, ld_src = 20, 8, 60, 8, 11
    dst = synth.int_below(74, rows * cols, 9, lo=-4).astype(np.float32).reshape(rows, cols)
    idx = synth.int_below(75, n, rows).astype(np.int32)
    src = np.full((n, ld_src), 1000.0, np.float32)
    src[:, :tile_c] = synth.int_below(76, n * tile_c, 7, lo=-3).astype(np.float32).reshape(n, tile_c)
    want = dst.astype(np.int64)
    np.add.at(want, idx, src[:, :tile_c].astype(np.int64))
    oracle.scatter_add_rows(dst, rows, cols, cols, idx, src, ld_src, tile_c)
    np.testing.assert_array_equal(dst, want.astype(np.float32))


def test_scatter_add_unique_fp32_equals_numpy_rounding():
    rows, cols, n = 300, 40, 120
    dst = synth.uniform_f32(61, (rows, cols), -1.0, 1.0)
    before = dst.copy()
    idx = synth.permutation_prefix(62, rows, n)
    src = synth.uniform_f32(63, (n, cols), -1.0, 1.0)
    oracle.scatter_add_rows(dst, rows, cols, cols, idx, src, cols, cols)
    want = before.copy()
    want[idx] = (before[idx].astype(np.float64) + src.astype(np.float64)).astype(np.float32)
    np.testing.assert_array_equal(dst, want)


def test_scatter_add_duplicates_integer_values_equal_numpy_add_at():
    rows, cols, n = 10, 16, 500
    dst = synth.int_below(64, rows * cols, 9, lo=-4).astype(np.float32).reshape(rows, cols)
    idx = synth.int_below(65, n, 14, lo=-2).astype(np.int32)   # duplicates and out-of-range rows
    src = synth.int_below(66, n * cols, 7, lo=-3).astype(np.float32).reshape(n, cols)
    want = dst.astype(np.int64)
    ok = (idx >= 0) & (idx < rows)
    np.add.at(want, idx[ok], src[ok].astype(np.int64))
    oracle.scatter_add_rows(dst, rows, cols, cols, idx, src, cols, cols)
    np.testing.assert_array_equal(dst, want.astype(np.float32))


@pytest.mark.parametrize("kind,tdt", [("bf16", torch.bfloat16), ("f16", torch.float16)])
def test_scatter_add_half_types_equal_torch(kind, tdt):
    rows, cols, n = 200, 24, 90
    base = torch.from_numpy(synth.normal_f32(67, (rows, cols))).to(tdt)
    add = torch.from_numpy(synth.normal_f32(68, (n, cols)) * np.float32(3.0)).to(tdt)
    idx = synth.permutation_prefix(69, rows, n)
    dst = base.view(torch.int16).numpy().view(np.uint16).copy()
    src = add.view(torch.int16).numpy().view(np.uint16).copy()
    oracle.scatter_add_rows(dst, rows, cols, cols, idx, src, cols, cols, kind=kind)
    want = base.clone()
    want[torch.from_numpy(idx.astype(np.int64))] = (base[torch.from_numpy(idx.astype(np.int64))].float()
                                                   + add.float()).to(tdt)
    np.testing.assert_array_equal(dst, want.view(torch.int16).numpy().view(np.uint16))


def test_scatter_add_fp16_subnormals_equal_torch():
    # binary16 subnormals (exponent field 0: m * 2^-24) on both sides of the addition, and sums that
    # cross into and out of the subnormal range; torch adds in fp32 and rounds once to fp16, which is
    # exact rounding for two fp16 operands
    a_bits = np.array([0x0001, 0x03FF, 0x8200, 0x0400, 0x8001, 0x0155, 0x3C00, 0x83FF], np.uint16)
    b_bits = np.array([0x0001, 0x0001, 0x0300, 0x8001, 0x8001, 0x02AB, 0x0001, 0x0400], np.uint16)
    dst = a_bits.reshape(1, 8).copy()
    oracle.scatter_add_rows(dst, 1, 8, 8, np.array([0], np.int32), b_bits.reshape(1, 8), 8, 8, kind="f16")
    ta = torch.from_numpy(a_bits.view(np.int16)).view(torch.float16)
    tb = torch.from_numpy(b_bits.view(np.int16)).view(torch.float16)
    want = (ta.float() + tb.float()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(dst.reshape(8), want)


def test_scatter_add_fp16_overflow_threshold_equals_torch():
    # binary16 sums next to the overflow threshold 65520 (the largest finite 65504 plus half an ulp):
    # below it they round to 65504, at and above it to infinity; torch adds in fp32 and rounds once
    a_bits = np.array([0x7BFF, 0x7BFF, 0x7BFF, 0x7BFF, 0xFBFF, 0xFBFF, 0x7BFE, 0x7BFF], np.uint16)
    b_bits = np.array([0x4800, 0x4B80, 0x4C00, 0x4C80, 0xC800, 0xCC00, 0x4C00, 0x0000], np.uint16)
    dst = a_bits.reshape(1, 8).copy()
    oracle.scatter_add_rows(dst, 1, 8, 8, np.array([0], np.int32), b_bits.reshape(1, 8), 8, 8, kind="f16")
    ta = torch.from_numpy(a_bits.view(np.int16)).view(torch.float16)
    tb = torch.from_numpy(b_bits.view(np.int16)).view(torch.float16)
    want = (ta.float() + tb.float()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert (want == 0x7C00).any() and (want == 0x7BFF).any()  # both sides of the threshold occur
    np.testing.assert_array_equal(dst.reshape(8), want)


def test_scatter_add_with_row_and_column_offsets_equals_numpy_add_at():
    # The gather's backward with both offsets: source element (k, j) adds into row row_offset + idx[k],
    # column col_offset + j when that is inside the array.  Integer values keep every sum exact.
    rows, cols, ld, n, tile_c, row_offset, col_offset = 12, 10, 13, 300, 9, -2, 3
    dst = synth.int_below(70, rows * ld, 9, lo=-4).astype(np.float32).reshape(rows, ld)
    idx = synth.int_below(71, n, rows + 4, lo=0).astype(np.int32)  # rows -2 .. rows + 1: some clipped
    src = synth.int_below(72, n * tile_c, 7, lo=-3).astype(np.float32).reshape(n, tile_c)
    want = dst.astype(np.int64)
    r = idx.astype(np.int64) + row_offset
    c = col_offset + np.arange(tile_c)
    keep_r, keep_c = (r >= 0) & (r < rows), (c >= 0) & (c < cols)
    np.add.at(want, (r[keep_r][:, None], c[keep_c][None, :]), src[keep_r][:, keep_c].astype(np.int64))
    oracle.scatter_add_rows(dst, rows, cols, ld, idx, src, tile_c, tile_c, row_offset=row_offset,
                            col_offset=col_offset)
    np.testing.assert_array_equal(dst, want.astype(np.float32))


def test_scatter_add_clips_rows_and_columns():
    dst = np.zeros((6, 5), np.float32)
    idx = np.array([-1, 6, 2, np.iinfo(np.int32).max], np.int32)
    src = np.ones((4, 7), np.float32)
    oracle.scatter_add_rows(dst, 6, 5, 5, idx, src, 7, 7, col_offset=-1)
    want = np.zeros((6, 5), np.float32)
    want[2, :] = 1.0   # window columns -1..5 -> 0..4 inside
    np.testing.assert_array_equal(dst, want)


# ----------------------------------------------------------------------------- ragged

def test_ragged_equal_lengths_is_a_transpose():
    B, T, H, D = 3, 20, 4, 16
    x = synth.normal_bf16(41, (B * T, H, D))
    cu = np.arange(B + 1, dtype=np.int32) * T
    out = oracle.ragged_tile_load(x, B * T, H, D, H * D, D, cu, T)
    np.testing.assert_array_equal(out, x.reshape(B, T, H, D).transpose(0, 2, 1, 3))


def test_ragged_prefix_and_zero_rows():
    d = synth.workloads.ragged_bf16(batch=6, max_len=50, heads=3, depth=8)
    x, cu, lens = d["x"], d["cu_seqlens"], d["lens"]
    t_pad = 40  # shorter than some sequences: rows >= t_pad are dropped
    out = oracle.ragged_tile_load(x, d["total_rows"], 3, 8, 24, 8, cu, t_pad)
    for b in range(6):
        L = min(int(lens[b]), t_pad)
        np.testing.assert_array_equal(out[b, :, :L], x[cu[b]:cu[b] + L].transpose(1, 0, 2))
        assert not out[b, :, L:].any()


def test_grouped_ragged_is_the_ragged_load_with_merged_depth():
    # Mojo "RaggedTMA3DTile", group > 1: the packed array is [rows][middle][group][depth] and a
    # tile holds (sequence position, group member) rows.  The grouped tile, written out directly
    # with numpy, equals the ragged load with depth' = group * depth.
    B, M, G, D, t_pad = 4, 3, 2, 8, 12
    lens = np.array([5, 12, 0, 9])
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    x = synth.normal_bf16(45, (int(cu[-1]), M, G, D))
    want = np.zeros((B, M, t_pad, G, D), np.uint16)
    for b in range(B):
        L = min(int(lens[b]), t_pad)
        want[b, :, :L] = x[cu[b]:cu[b] + L].transpose(1, 0, 2, 3)
    got = oracle.ragged_tile_load(x, int(cu[-1]), M, G * D, M * G * D, G * D, cu, t_pad)
    np.testing.assert_array_equal(got.reshape(B, M, t_pad, G, D), want)


def test_ragged_empty_and_out_of_range_metadata():
    x = synth.normal_bf16(42, (10, 2, 4))
    cu = np.array([0, 0, 8, 14], np.int32)  # empty sequence; the last one runs past total_rows=10
    out = oracle.ragged_tile_load(x, 10, 2, 4, 8, 4, cu, 6)
    assert not out[0].any()
    np.testing.assert_array_equal(out[1], x[0:6].transpose(1, 0, 2))
    np.testing.assert_array_equal(out[2, :, :2], x[8:10].transpose(1, 0, 2))
    assert not out[2, :, 2:].any()


def test_ragged_store_inverts_the_load_and_writes_nothing_else():
    d = synth.workloads.ragged_bf16(batch=7, max_len=60, heads=3, depth=8)
    x, cu, lens, total = d["x"], d["cu_seqlens"], d["lens"], d["total_rows"]
    t_pad = 64
    tiles = synth.normal_bf16(43, (7, 3, t_pad, 8))
    canvas = np.full((total, 3, 8), 0xDEAD, np.uint16)
    oracle.ragged_tile_store(tiles, canvas, total, 24, 8, cu)
    for b in range(7):
        L = int(lens[b])
        # numpy slicing: packed rows of sequence b are the first L rows of its tiles
        np.testing.assert_array_equal(canvas[cu[b]:cu[b] + L], tiles[b, :, :L].transpose(1, 0, 2))
    # every packed row belongs to one sequence, so nothing keeps the canary
    assert not np.any(canvas == 0xDEAD)
    # load then store reproduces the packed array exactly
    back = np.zeros_like(x)
    oracle.ragged_tile_store(oracle.ragged_tile_load(x, total, 3, 8, 24, 8, cu, t_pad), back, total, 24, 8, cu)
    np.testing.assert_array_equal(back, x)


def test_ragged_store_clips_long_sequences_and_bad_metadata():
    tiles = synth.normal_bf16(44, (3, 2, 4, 4))
    x = np.full((12, 2, 4), 0x1234, np.uint16)
    cu = np.array([0, 6, 6, 14], np.int32)  # len 6 > t_pad 4; an empty sequence; len 8 > t_pad
    oracle.ragged_tile_store(tiles, x, 12, 8, 4, cu)
    np.testing.assert_array_equal(x[0:4], tiles[0].transpose(1, 0, 2))
    assert np.all(x[4:6] == 0x1234)          # rows past t_pad of sequence 0: not written
    np.testing.assert_array_equal(x[6:10], tiles[2].transpose(1, 0, 2))
    assert np.all(x[10:12] == 0x1234)        # sequence 2's rows 4.. are past t_pad


def test_ragged_store_leaves_rows_outside_every_sequence():
    # Mojo "RaggedTMA3DTile", async_copy_from_col: only the first dynamic_dim rows of a tile are written.
    # The packed buffer has 4 spare rows after the last sequence, and every tile row (also those past a
    # sequence's length) holds data: only rows [cu[b], cu[b] + len_b) may change.
    cu = np.array([0, 3, 3, 8], np.int32)  # lengths 3, 0, 5, all below t_pad = 6
    tiles = synth.normal_bf16(45, (3, 2, 6, 4))
    x = np.full((12, 2, 4), 0x1234, np.uint16)
    oracle.ragged_tile_store(tiles, x, 12, 8, 4, cu)
    np.testing.assert_array_equal(x[0:3], tiles[0, :, :3].transpose(1, 0, 2))
    np.testing.assert_array_equal(x[3:8], tiles[2, :, :5].transpose(1, 0, 2))
    assert np.all(x[8:12] == 0x1234)


def test_ragged_load_and_store_with_padded_packed_rows():
    # Mojo "RaggedTMA3DTile": the packed array is addressed through its own strides: element (row, h, d)
    # at row*ld_row + h*ld_head + d.  Here heads are 3 apart beyond their depth and rows 5 beyond their
    # heads, so a stride read as the dense one lands elsewhere; expected positions come from numpy index
    # arithmetic on the flat buffer.
    heads, depth, ld_head = 3, 4, 7
    ld_row = heads * ld_head + 5
    cu = np.array([0, 5, 5, 11], np.int32)
    total, t_pad, batch = 11, 8, 3
    flat = synth.normal_bf16(47, total * ld_row)
    out = oracle.ragged_tile_load(flat, total, heads, depth, ld_row, ld_head, cu, t_pad)
    lens = np.diff(cu)
    b, h, r, d = np.meshgrid(np.arange(batch), np.arange(heads), np.arange(t_pad), np.arange(depth), indexing="ij")
    valid = r < lens[b]
    pos = (cu[b] + r) * ld_row + h * ld_head + d
    want = np.where(valid, flat[np.where(valid, pos, 0)], 0).astype(np.uint16)
    np.testing.assert_array_equal(out, want)
    # the store writes exactly those positions back, from other tiles, and nothing else of the buffer
    tiles = synth.normal_bf16(48, (batch, heads, t_pad, depth))
    canvas = np.full(total * ld_row, 0xBEEF, np.uint16)
    oracle.ragged_tile_store(tiles, canvas, total, ld_row, ld_head, cu)
    want_c = np.full(total * ld_row, 0xBEEF, np.uint16)
    want_c[pos[valid]] = tiles[valid]
    np.testing.assert_array_equal(canvas, want_c)


def test_ragged_store_stops_at_the_packed_array_end():
    # A sequence whose rows run past total_rows: the packed array is the first 10 rows of a 14-row
    # buffer, and the rows after it must keep their bits (a store never writes outside the array).
    cu = np.array([0, 6, 13], np.int32)  # sequence 1 claims packed rows 6..12
    tiles = synth.normal_bf16(46, (2, 2, 8, 4))
    buf = np.full((14, 2, 4), 0x1234, np.uint16)
    oracle.ragged_tile_store(tiles, buf[:10], 10, 8, 4, cu)
    np.testing.assert_array_equal(buf[0:6], tiles[0, :, :6].transpose(1, 0, 2))
    np.testing.assert_array_equal(buf[6:10], tiles[1, :, :4].transpose(1, 0, 2))
    assert np.all(buf[10:] == 0x1234)


# ----------------------------------------------------------------------------- GEMM and bf16 rounding

def _bits_of(vals):
    return (np.asarray(vals, np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("mnk", [(1, 1, 1), (3, 5, 7), (17, 13, 11), (16, 16, 64)])
def test_gemm_integer_inputs_exact_vs_numpy_int_matmul(mnk):
    M, N, K = mnk
    a_int = synth.int_below(51, M * K, 5, lo=-2).reshape(M, K)
    b_int = synth.int_below(52, K * N, 5, lo=-2).reshape(K, N)
    lda, ldb = K + 1, N + 2
    A = np.zeros((M, lda), np.uint16)
    B = np.zeros((K, ldb), np.uint16)
    A[:, :K] = _bits_of(a_int)
    B[:, :N] = _bits_of(b_int)
    C = oracle.gemm_f64(A, lda, B, ldb, M, N, K)
    np.testing.assert_array_equal(C, (a_int @ b_int).astype(np.float64))


def test_gemm_identity_and_random_vs_numpy():
    M, N, K = 9, 14, 9
    B = synth.normal_bf16(53, (K, N))
    eye = np.zeros((M, K), np.uint16)
    eye[np.arange(M), np.arange(M)] = 0x3F80
    C = oracle.gemm_f64(eye, K, B, N, M, N, K)
    np.testing.assert_array_equal(C, synth.bf16_bits_to_f32(B).astype(np.float64))
    A = synth.normal_bf16(54, (21, 33))
    B = synth.normal_bf16(55, (33, 12))
    C = oracle.gemm_f64(A, 33, B, 12, 21, 12, 33)
    want = synth.bf16_bits_to_f32(A).astype(np.float64) @ synth.bf16_bits_to_f32(B).astype(np.float64)
    np.testing.assert_allclose(C, want, rtol=1e-12, atol=1e-12)
    ms = np.array([0, 20, 7]); ns = np.array([11, 0, 5])
    np.testing.assert_array_equal(oracle.gemm_f64_at(A, 33, B, 12, 33, ms, ns), C[ms, ns])


@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80), (1.0 + 2**-8, 0x3F80), (1.0 + 3 * 2**-8, 0x3F82), (1.0 + 2**-8 + 2**-30, 0x3F81),
    (-2.5, 0xC020), (0.0, 0x0000), (-0.0, 0x8000), (float("inf"), 0x7F80), (float("-inf"), 0xFF80),
    (2**127 * (2 - 2**-7), 0x7F7F), (2**127 * (2 - 2**-8), 0x7F80), (2**127 * (2 - 2**-8) * (1 - 2**-40), 0x7F7F),
    (2**-133, 0x0001), (2**-134, 0x0000), (1.5 * 2**-134, 0x0001), (3 * 2**-134, 0x0002), (2**-126, 0x0080),
])
def test_bf16_rne_pins(x, bits):
    assert oracle.bf16_rne(x) == bits


def test_bf16_rne_nan():
    assert oracle.bf16_rne(float("nan")) & 0x7FC0 == 0x7FC0


def test_bf16_rne_matches_torch_on_binary32_values():
    # Values exactly representable in binary32 round identically through torch's
    # float32 -> bfloat16 conversion (round to nearest even).
    f = synth.normal_f32(56, 200000) * np.float32(1000.0)
    f[:5] = [1.0 + 2**-8, 1.0 + 3 * 2**-8, -1.0 - 2**-8, 3.0e38, 1e-40]
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(f.astype(np.float64))
    np.testing.assert_array_equal(got, want)


# ----------------------------------------------------------------------------- block-scaled GEMM
# Formats: OCP 8-bit floating point / microscaling formats; the GEMM is
# cuTile.jl "Operations", muladd_scaled.

E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # the format's whole positive value set


@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2),
                                     ("e8m0", torch.float8_e8m0fnu)])
def test_fp8_decode_all_codes_equal_torch(fmt, tdt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(tdt).to(torch.float64).numpy()
    got = np.array([oracle.fp8_decode(fmt, c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])
    np.testing.assert_array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def test_e2m1_decode_is_the_format_table():
    got = [oracle.fp8_decode("e2m1", c) for c in range(16)]
    assert got[:8] == E2M1_VALUES
    assert got[8:] == [-v for v in E2M1_VALUES]
    assert np.signbit(got[8])  # code 0b1000 is -0


def _fp8_codes(seed, shape):
    """Uniform E4M3 codes with the two NaN codes replaced by 1.0 (0x38)."""
    c = synth.int_below(seed, int(np.prod(shape)), 256).astype(np.uint8).reshape(shape)
    c[(c & 0x7F) == 0x7F] = 0x38
    return c


def _e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_block_scaled_unit_scales_equal_numpy_matmul():
    M, N, K, bs = 7, 9, 64, 32
    A, B = _fp8_codes(81, (M, K)), _fp8_codes(82, (K, N))
    SA = np.full((M, K // bs), 127, np.uint8)
    SB = np.full((K // bs, N), 127, np.uint8)
    C = oracle.gemm_block_scaled_f64(A, K, SA, K // bs, B, N, SB, N, M, N, K, bs)
    np.testing.assert_allclose(C, _e4m3(A) @ _e4m3(B), rtol=1e-12, atol=1e-9)


def test_block_scaled_e4m3_scales_equal_broadcast_matmul():
    # Scales E4M3 over blocks of 16 along K, odd leading dimensions everywhere:
    # (A * repeat(SA, 16, axis=1)) @ (B * repeat(SB, 16, axis=0)) in numpy.
    M, N, K, bs = 11, 13, 80, 16
    Ks = K // bs
    lda, ldb, ldsa, ldsb = K + 3, N + 5, Ks + 1, N + 2
    A, B = _fp8_codes(83, (M, lda)), _fp8_codes(84, (K, ldb))
    SA = (0x30 + synth.int_below(85, M * ldsa, 16)).astype(np.uint8).reshape(M, ldsa)  # scales in [0.5, 1.875]
    SB = (0x30 + synth.int_below(86, Ks * ldsb, 16)).astype(np.uint8).reshape(Ks, ldsb)
    C = oracle.gemm_block_scaled_f64(A, lda, SA, ldsa, B, ldb, SB, ldsb, M, N, K, bs, sfmt="e4m3")
    a = _e4m3(A[:, :K]) * np.repeat(_e4m3(SA[:, :Ks]), bs, axis=1)
    b = _e4m3(B[:, :N]) * np.repeat(_e4m3(SB[:, :N]), bs, axis=0)
    np.testing.assert_allclose(C, a @ b, rtol=1e-12, atol=1e-9)


def test_block_scaled_e2m1_with_signed_e4m3_scales_equal_broadcast_matmul():
    # The NVFP4 combination: packed E2M1 operands, E4M3 scales per 16, the scale codes drawn
    # over the whole format (negative, +0 and -0, subnormal, up to 448; NaN excluded), and
    # a different leading dimension for every array. The expected value is the definition
    # in numpy: operand values from the E2M1 table, scale values from torch's E4M3 decode,
    # the scales repeated over their blocks of 16, then one matmul.
    M, N, K, bs = 9, 14, 96, 16
    Ks = K // bs
    lda, ldb, ldsa, ldsb = K + 10, N + 4, Ks + 3, N + 1
    ca = synth.int_below(89, M * lda, 16).astype(np.uint8).reshape(M, lda)
    cb = synth.int_below(90, K * ldb, 16).astype(np.uint8).reshape(K, ldb)
    pack = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    SA, SB = _fp8_codes(91, (M, ldsa)), _fp8_codes(92, (Ks, ldsb))
    SA[0, :3] = [0x00, 0x80, 0x01]   # +0, -0, the smallest subnormal
    SB[1, :3] = [0xFE, 0x7E, 0x81]   # -448, 448, the smallest negative subnormal
    table = np.array(E2M1_VALUES + [-v for v in E2M1_VALUES])
    C = oracle.gemm_block_scaled_f64(pack(ca), lda, SA, ldsa, pack(cb), ldb, SB, ldsb, M, N, K, bs,
                                     afmt="e2m1", bfmt="e2m1", sfmt="e4m3")
    a = table[ca[:, :K]] * np.repeat(_e4m3(SA[:, :Ks]), bs, axis=1)
    b = table[cb[:, :N]] * np.repeat(_e4m3(SB[:, :N]), bs, axis=0)
    assert (a < 0).any() and (_e4m3(SA[:, :Ks]) < 0).any() and (_e4m3(SB[:, :N]) < 0).any()
    # every product is exact in double; the two sums differ only in their order of addition
    np.testing.assert_array_less(np.abs(C - a @ b), 1e-13 * (np.abs(a) @ np.abs(b)) + 1e-300)


def test_block_scaled_e2m1_packed_equal_table_matmul():
    # E2M1 operands, two per byte along each row, even element in the low nibble.
    M, N, K, bs = 6, 10, 64, 32
    ca = synth.int_below(87, M * K, 16).astype(np.uint8).reshape(M, K)
    cb = synth.int_below(88, K * N, 16).astype(np.uint8).reshape(K, N)
    pack = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    table = np.array(E2M1_VALUES + [-v for v in E2M1_VALUES])
    SA = np.full((M, K // bs), 128, np.uint8)   # 2.0
    SB = np.full((K // bs, N), 126, np.uint8)   # 0.5
    C = oracle.gemm_block_scaled_f64(pack(ca), K, SA, K // bs, pack(cb), N, SB, N, M, N, K, bs,
                                     afmt="e2m1", bfmt="e2m1")
    np.testing.assert_array_equal(C, table[ca] @ table[cb])


def test_block_scaled_closed_form_with_acc():
    # ones times ones with scale_a[m][j] = 2^(m % 3) and scale_b[j][n] = 2^(j % 2), plus acc:
    # D[m][n] = bs * 2^(m % 3) * (1 + 2 + 1) + acc[m][n]
    M, N, K, bs = 5, 4, 96, 32   # 3 blocks: j = 0, 1, 2
    A = np.full((M, K), 0x38, np.uint8)
    B = np.full((K, N), 0x38, np.uint8)
    SA = np.array([[127 + (m % 3)] * 3 for m in range(M)], np.uint8)
    SB = np.array([[127 + (j % 2)] * N for j in range(3)], np.uint8)
    acc = np.arange(M * N, dtype=np.float32).reshape(M, N) - 7.5
    C = oracle.gemm_block_scaled_f64(A, K, SA, 3, B, N, SB, N, M, N, K, bs, acc=acc, ld_acc=N)
    want = np.array([[bs * 2.0 ** (m % 3) * 4 for n in range(N)] for m in range(M)]) + acc
    np.testing.assert_array_equal(C, want)


def test_block_scaled_acc_with_its_own_leading_dimension():
    # acc is an (M, N) view with its own leading dimension: D = closed form + acc[:, :N]
    M, N, K, bs, ld_acc = 5, 4, 64, 32, 7
    A = np.full((M, K), 0x38, np.uint8)
    B = np.full((K, N), 0x38, np.uint8)
    SA = np.full((M, 2), 127, np.uint8)
    SB = np.full((2, N), 128, np.uint8)   # 2.0
    acc = synth.uniform_f32(73, (M, ld_acc), -4.0, 4.0)
    C = oracle.gemm_block_scaled_f64(A, K, SA, 2, B, N, SB, N, M, N, K, bs, acc=acc, ld_acc=ld_acc)
    np.testing.assert_array_equal(C, 2.0 * K + acc[:, :N].astype(np.float64))


def test_block_scaled_nan_stays_in_its_row_and_column():
    M, N, K, bs = 4, 5, 32, 32
    A = np.full((M, K), 0x38, np.uint8)
    B = np.full((K, N), 0x38, np.uint8)
    A[2, 7] = 0x7F            # E4M3 NaN
    SA = np.full((M, 1), 127, np.uint8)
    SB = np.full((1, N), 127, np.uint8)
    SB[0, 3] = 0xFF           # E8M0 NaN
    C = oracle.gemm_block_scaled_f64(A, K, SA, 1, B, N, SB, N, M, N, K, bs)
    nan = np.zeros((M, N), bool)
    nan[2, :] = True
    nan[:, 3] = True
    np.testing.assert_array_equal(np.isnan(C), nan)
    np.testing.assert_array_equal(C[~nan], 32.0)
