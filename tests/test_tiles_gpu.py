"""GPU parity of sbt_tile_load_padded / sbt_tile_store_clipped against the CPU oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
import scatter_boundary_tile_gb300 as sbt
import synth
import synth.workloads as wl
from gpu_helpers import Canvas, dev, host, sync

pytestmark = pytest.mark.gpu


def gpu_load(ctx, buf, rows, cols, sr, sc, r0, c0, str_, stc, gr, gc, tr, tc, dtype, pad=None, path="auto",
             byte_offset=0):
    es = buf.dtype.itemsize
    b = dev(buf)
    canvas = Canvas(gr * gc * tr * tc * es)
    ctx.set_path(path)
    sbt.tile_load_padded(ctx, b.data_ptr() + byte_offset, rows, cols, sr, sc, r0, c0, str_, stc, gr, gc, tr, tc,
                         canvas.ptr, pad=pad, dtype=dtype)
    sync()
    assert canvas.guards_intact()
    return canvas.inner(buf.dtype, (gr, gc, tr, tc))


def gpu_store(ctx, tiles, dst_init, rows, cols, sr, sc, r0, c0, str_, stc, dtype, path="auto", byte_offset=0):
    gr, gc, tr, tc = tiles.shape
    t = dev(tiles)
    canvas = Canvas(dst_init.nbytes, fill=dst_init)
    ctx.set_path(path)
    sbt.tile_store_clipped(ctx, t, gr, gc, tr, tc, canvas.ptr + byte_offset, rows, cols, sr, sc, r0, c0, str_, stc,
                           dtype=dtype)
    sync()
    assert canvas.guards_intact()
    return canvas.inner(dst_init.dtype, dst_init.shape)


def same_bits(a, b):
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


@pytest.mark.parametrize("path", ["auto", "tma", "vector", "scalar"])
def test_small_fp32_grid_load_and_store(ctx, path):
    a = wl.tiles_small()["a"]
    got = gpu_load(ctx, a, 65, 73, 73, 1, 0, 0, 64, 32, 2, 3, 64, 32, "f32", pad=0.0, path=path)
    want = oracle.tile_load_padded(a, 65, 73, 73, 1, 0, 0, 64, 32, 2, 3, 64, 32, pad=np.float32(0))
    assert same_bits(got, want)
    # store into a 65x73 view at (2, 3) of a 70x81 canvas pre-filled with a canary
    canvas = np.full((70, 81), wl.F32_CANARY_BITS, np.uint32).view(np.float32)
    off = (2 * 81 + 3) * 4
    got_c = gpu_store(ctx, got, canvas, 65, 73, 81, 1, 0, 0, 64, 32, "f32", path=path, byte_offset=off)
    want_c = canvas.copy()
    oracle.tile_store_clipped(want, want_c.reshape(-1)[2 * 81 + 3:], 65, 73, 81, 1, 0, 0, 64, 32)
    assert same_bits(got_c, want_c)
    np.testing.assert_array_equal(got_c[2:67, 3:76], a)
    # the bare ld-73 case
    bare = np.zeros((65, 73), np.float32)
    got_b = gpu_store(ctx, got, bare, 65, 73, 73, 1, 0, 0, 64, 32, "f32", path=path)
    np.testing.assert_array_equal(got_b, a)


@pytest.mark.parametrize("aligned", [True, False])
def test_tylo_concrete_edge_bf16(ctx, aligned):
    # A (65, 73) bf16; tile (64, 32) at (64, 64): 1 valid row, 9 valid K values.
    ld = 80 if aligned else 73
    A = synth.normal_bf16(201, (65, ld))
    got = gpu_load(ctx, A, 65, 73, ld, 1, 64, 64, 0, 0, 1, 1, 64, 32, "bf16", pad=0)
    want = oracle.tile_load_padded(A, 65, 73, ld, 1, 64, 64, 0, 0, 1, 1, 64, 32, pad=0)
    assert same_bits(got, want)
    t = got[0, 0]
    assert np.count_nonzero(t) == np.count_nonzero(A[64, 64:73])
    assert not t[1:].any() and not t[0, 9:].any()


CASES = [
    # rows, cols, ld, stride_c, origin, step, grid, tile
    (65, 73, 80, 1, (0, 0), (64, 32), (2, 3), (64, 32)),        # vector path, edge tiles
    (65, 73, 80, 1, (-5, -8), (20, 24), (5, 4), (16, 16)),      # negative origins, gaps
    (65, 73, 80, 1, (-64, -32), (10, 8), (9, 12), (64, 32)),    # tiles wholly outside, overlap (load only)
    (65, 73, 73, 1, (3, 7), (13, 11), (6, 8), (13, 11)),        # unaligned everything
    (40, 37, 90, 2, (-3, 5), (8, 8), (6, 5), (8, 8)),           # column stride 2
    (30, 20, 20, 1, (0, 0), (0, 0), (1, 1), (256, 256)),        # tile larger than the array
    (1, 1, 1, 1, (0, 0), (1, 1), (3, 3), (1, 1)),               # 1x1
    (70, 72, 80, 1, (0, 0), (64, 32), (2, 3), (64, 32)),        # 16-byte row width: TMA tiles, edge tiles
    (70, 72, 80, 1, (-6, -8), (30, 24), (4, 4), (32, 16)),      # TMA with negative origins and gaps
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_load_edge_cases(ctx, case, dtype):
    rows, cols, ld, sc, (r0, c0), (str_, stc), (gr, gc), (tr, tc) = case
    npdt = np.float32 if dtype == "f32" else np.uint16
    buf = (synth.uniform_f32(202, (rows, ld)) if dtype == "f32" else synth.normal_bf16(202, (rows, ld))).astype(npdt)
    pad = 7.5 if dtype == "f32" else 0x40F0
    pad_np = np.float32(7.5) if dtype == "f32" else 0x40F0
    want = oracle.tile_load_padded(buf, rows, cols, ld, sc, r0, c0, str_, stc, gr, gc, tr, tc, pad=pad_np)
    for path in ("auto", "tma", "scalar"):
        got = gpu_load(ctx, buf, rows, cols, ld, sc, r0, c0, str_, stc, gr, gc, tr, tc, dtype, pad=pad, path=path)
        assert same_bits(got, want), path


STORE_CASES = [
    (65, 73, 80, 1, (0, 0), (64, 32), (2, 3), (64, 32)),
    (65, 73, 80, 1, (-5, -8), (20, 24), (5, 4), (16, 16)),
    (65, 73, 73, 1, (3, 7), (13, 11), (6, 8), (13, 11)),
    (40, 37, 90, 2, (-3, 5), (8, 8), (6, 5), (8, 8)),
    (30, 20, 24, 1, (-100, -100), (64, 64), (2, 2), (8, 8)),  # wholly outside: writes nothing
    (70, 72, 80, 1, (0, 0), (64, 32), (2, 3), (64, 32)),        # TMA store, partial edge tiles
    (70, 72, 80, 1, (3, 40), (34, 24), (3, 2), (32, 16)),       # TMA store, gaps, rows and columns past the end
    # unaligned destination rows (every row offset mod 16), tile rows of 1 to 32 vectors
    (65, 73, 73, 1, (0, 0), (64, 32), (2, 3), (64, 32)),        # every row offset mod 16, partial edge tiles
    (50, 70, 71, 1, (-3, -5), (16, 16), (4, 5), (16, 16)),      # negative origin, odd column steps
    (40, 300, 301, 1, (1, 3), (8, 128), (5, 3), (8, 128)),      # 32 (fp32) / 16 (bf16) vectors per tile row
    (33, 37, 37, 1, (0, 1), (3, 8), (11, 5), (3, 8)),           # 2 (fp32) / 1 (bf16) vectors per tile row
    (40, 100, 101, 1, (0, 0), (8, 48), (5, 3), (8, 48)),        # 12 / 6 vectors per row: element rows
    (5, 8200, 8201, 1, (-1, -9), (2, 256), (3, 33), (2, 256)),  # runs of 2,112 (fp32) / 1,056 vectors: chunks
    (3, 5000, 5003, 1, (0, 0), (1, 256), (3, 20), (1, 256)),    # 1,280 / 640 vectors per run
]


@pytest.mark.parametrize("case", STORE_CASES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_store_edge_cases(ctx, case, dtype):
    rows, cols, ld, sc, (r0, c0), (str_, stc), (gr, gc), (tr, tc) = case
    if dtype == "f32":
        tiles = synth.uniform_f32(203, (gr, gc, tr, tc), 1.0, 2.0)
        dst = np.full((rows, ld), wl.F32_CANARY_BITS, np.uint32).view(np.float32)
    else:
        tiles = synth.normal_bf16(203, (gr, gc, tr, tc))
        dst = np.full((rows, ld), 0xDEAD, np.uint16)
    want = dst.copy()
    oracle.tile_store_clipped(tiles, want, rows, cols, ld, sc, r0, c0, str_, stc)
    for path in ("auto", "tma", "vector", "scalar"):  # unaligned rows: bulk copies, lane-shifted runs, elements
        got = gpu_store(ctx, tiles, dst, rows, cols, ld, sc, r0, c0, str_, stc, dtype, path=path)
        assert same_bits(got, want), path


def test_round_trip_identity_bf16(ctx):
    a = synth.normal_bf16(204, (300, 264))
    tiles = gpu_load(ctx, a, 300, 260, 264, 1, 0, 0, 64, 64, 5, 5, 64, 64, "bf16")
    back = gpu_store(ctx, tiles, np.zeros((300, 264), np.uint16), 300, 260, 264, 1, 0, 0, 64, 64, "bf16")
    np.testing.assert_array_equal(back[:, :260], a[:, :260])
    assert not back[:, 260:].any()


def test_validation(ctx):
    before = ctx.launch_count
    b = dev(np.zeros(16, np.float32))
    for bad in [dict(tile_r=0), dict(tile_c=257), dict(stride_c=0), dict(rows=-1)]:
        kw = dict(rows=4, cols=4, stride_r=4, stride_c=1, tile_r=4, tile_c=4)
        kw.update(bad)
        with pytest.raises(sbt.SbtError) as e:
            sbt.tile_load_padded(ctx, b, kw["rows"], kw["cols"], kw["stride_r"], kw["stride_c"], 0, 0, 4, 4, 1, 1,
                                 kw["tile_r"], kw["tile_c"], b, dtype="f32")
        assert e.value.status == sbt.SBT_ERR_INVALID_ARG
    sbt.tile_load_padded(ctx, b, 4, 4, 4, 1, 0, 0, 4, 4, 0, 5, 4, 4, b, dtype="f32")  # empty grid: no launch
    assert ctx.launch_count == before


@pytest.mark.parametrize("shape,path", [((16381, 16411, 16411), "auto"), ((16381, 16411, 16411), "vector"),
                                        ((16384, 16416, 16416), "auto"),
                                        ((16384, 16416, 16416), "tma"), ((16384, 16416, 16416), "vector"),
                                        ((16381, 16411, 16416), "auto")])
def test_large_fp32_grid(ctx, shape, path):
    """fp32 arrays over a ceil-div grid of 64 x 32 tiles: 16,381 x 16,411 with ld 16,411
    (unaligned rows: realigned loads, stores along whole destination rows), 16,384 x 16,416 with ld 16,416 (16-byte
    rows: vector or TMA tiles), and 16,381 x 16,411 with ld 16,416 (aligned rows, ragged edge)."""
    rows, cols, ld = shape
    a = synth.uniform_f32(205, (rows, ld), -1.0, 1.0)
    gr, gc = -(-rows // 64), -(-cols // 32)
    a_dev = dev(a)
    tiles = torch.empty(gr * gc * 64 * 32 * 4, dtype=torch.uint8, device="cuda")
    ctx.set_path(path)
    sbt.tile_load_padded(ctx, a_dev, rows, cols, ld, 1, 0, 0, 64, 32, gr, gc, 64, 32, tiles, dtype="f32")
    want = oracle.tile_load_padded(a, rows, cols, ld, 1, 0, 0, 64, 32, gr, gc, 64, 32, pad=np.float32(0))
    assert same_bits(host(tiles, np.float32, want.shape), want)
    del want
    a_dev.zero_()
    sbt.tile_store_clipped(ctx, tiles, gr, gc, 64, 32, a_dev, rows, cols, ld, 1, 0, 0, 64, 32, dtype="f32")
    back = host(a_dev, np.float32, (rows, ld))
    assert same_bits(back[:, :cols], a[:, :cols])
    assert not back[:, cols:].any()
