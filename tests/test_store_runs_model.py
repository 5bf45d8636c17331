"""CPU model of the lane logic of the row-run tile store (k_tiles_runs.cu).

The clipped store into unaligned destination rows numbers tile vectors along
whole destination rows; each lane takes its left neighbour's vector and writes
the aligned 16-byte chunk that starts inside it, and the ends of a warp's run
go out element by element.  This model replays that logic lane by lane (32
lanes per warp, the kernel's grid-stride loop) over a byte image of the
destination and checks, for several shapes, origins and pointer offsets, that
every byte written belongs to an element inside the array, that every 16-byte
store is 16-byte aligned, and that the result equals plain element stores.  It
checks the algorithm, not the CUDA code; the GPU tests check the kernel
against the oracle.
"""
import numpy as np
import pytest


def model_store(tiles, rows, cols, ld, r0, c0, step_r, es, base_off, blocks=3, threads=64):
    gr, gc, tr, tc = tiles.shape
    V = 16 // es
    per_row = tc // V
    width = gc * per_row
    ntasks = gr * tr * width
    tile_bytes = tiles.view(np.uint8).reshape(gr, gc, tr, tc * es)
    mem = np.zeros(base_off + rows * ld * es + 64, np.uint8)

    def store(addr, data):
        n = len(data)
        if n == 16:
            assert addr % 16 == 0, "unaligned 16-byte store"
        for b in range(n):
            off = addr + b - base_off
            assert 0 <= off < rows * ld * es, "byte outside the array"
            rr, cc = divmod(off // es, ld)
            assert rr < rows and cc < cols, "byte outside the rows x cols window"
        mem[addr:addr + n] = data

    stride = blocks * threads
    for blk in range(blocks):
        for warp in range(threads // 32):
            wbase = blk * threads + warp * 32
            while wbase < ntasks:
                lanes = []
                for lane in range(32):
                    t = wbase + lane
                    d = {"live": t < ntasks, "run": -1, "inside": False, "v": None, "r": -1, "c": 0}
                    if d["live"]:
                        run, vc = divmod(t, width)
                        ti, i = divmod(run, tr)
                        tj, j = divmod(vc, per_row)
                        d.update(run=run, v=tile_bytes[ti, tj, i, 16 * j:16 * j + 16].copy(),
                                 r=r0 + ti * step_r + i, c=c0 + vc * V)
                        d["inside"] = 0 <= d["r"] < rows and d["c"] >= 0 and d["c"] + V <= cols
                    lanes.append(d)
                for lane, d in enumerate(lanes):
                    if not d["live"] or not 0 <= d["r"] < rows:
                        continue
                    if not d["inside"]:
                        for e in range(V):
                            ce = d["c"] + e
                            if 0 <= ce < cols:
                                store(base_off + (d["r"] * ld + ce) * es, d["v"][e * es:(e + 1) * es])
                        continue
                    a = base_off + (d["r"] * ld + d["c"]) * es
                    sh = a % 16
                    if sh == 0:
                        store(a, d["v"])
                        continue
                    prev = lanes[lane - 1] if lane > 0 else None
                    nxt = lanes[lane + 1] if lane < 31 else None
                    prev_ok = prev is not None and prev["run"] == d["run"] and prev["inside"]
                    next_ok = nxt is not None and nxt["run"] == d["run"] and nxt["inside"]
                    if prev_ok:
                        store(a - sh, np.concatenate([prev["v"], d["v"]])[16 - sh:32 - sh])
                    head = (16 - sh) // es
                    for e in range(V):
                        if (not prev_ok) if e < head else (not next_ok):
                            store(a + e * es, d["v"][e * es:(e + 1) * es])
                wbase += stride
    return mem[base_off:base_off + rows * ld * es]


SHAPES = [  # rows, cols, ld, r0, c0, tile_r, tile_c, grid_r, grid_c
    (65, 73, 73, 0, 0, 64, 32, 2, 3),
    (50, 70, 71, -3, -5, 16, 16, 4, 5),
    (40, 300, 301, 1, 3, 8, 128, 5, 3),
    (33, 37, 37, 0, 1, 3, 8, 11, 5),
    (20, 50, 53, 2, -7, 5, 24, 5, 4),
    (9, 17, 19, -2, 2, 4, 8, 4, 4),
]


@pytest.mark.parametrize("es", [4, 2])
@pytest.mark.parametrize("shape", SHAPES)
def test_row_run_store_model_equals_element_stores(es, shape):
    rows, cols, ld, r0, c0, tr, tc, gr, gc = shape
    V = 16 // es
    if tc % V:
        pytest.skip("tile rows are not whole 16-byte vectors: the element kernel takes these")
    dtype = np.uint32 if es == 4 else np.uint16
    rng = np.random.default_rng(rows * 1000 + cols)
    tiles = rng.integers(1, 2 ** (8 * es) - 1, size=(gr, gc, tr, tc), dtype=np.uint64).astype(dtype)
    want = np.zeros((rows, ld), dtype)
    for ti in range(gr):
        for tj in range(gc):
            for i in range(tr):
                for j in range(tc):
                    r, c = r0 + ti * tr + i, c0 + tj * tc + j
                    if 0 <= r < rows and 0 <= c < cols:
                        want[r, c] = tiles[ti, tj, i, j]
    for base_off in (0, es, 2 * es, 16 - es):  # destination pointer offset within 16 bytes
        got = model_store(tiles, rows, cols, ld, r0, c0, tr, es, base_off)
        assert np.array_equal(got.view(dtype).reshape(rows, ld), want), base_off


# ----------------------------------------------------------------------------- bulk-copy variant
# The default kernel cuts each run into chunks of at most 1,024 vectors (equal sizes rounded
# up to whole warps) and writes the chunk's aligned destination words whose bytes are all in
# bounds with one bulk copy; the other words, and the bytes of the run's last vector past its
# last word, go out element by element.  This model follows its index arithmetic and lane
# logic (256 threads, four vectors each, the previous vector from the next lane down, from the
# edge slots across warps and from one extra load before the chunk) and checks every bulk copy
# for 16-byte alignment at both ends, and every byte written for being in bounds and written
# once.
BULK_THREADS, BULK_PER = 256, 4


def model_store_bulk(tiles, rows, cols, ld, r0, c0, step_r, es, base_off):
    gr, gc, tr, tc = tiles.shape
    V = 16 // es
    per_row = tc // V
    width = gc * per_row
    tile_bytes = tiles.view(np.uint8).reshape(gr, gc, tr, tc * es)
    size = rows * ld * es
    mem = np.zeros(base_off + size + 64, np.uint8)
    count = np.zeros_like(mem, dtype=np.int32)
    bulk_vec = BULK_THREADS * BULK_PER
    n = -(-width // bulk_vec)
    chunk = min(bulk_vec, (-(-width // n) + 31) // 32 * 32)
    n_chunks = -(-width // chunk)
    lo = max(0, -c0) * es
    hi = max(min(width * V, cols - c0), 0) * es

    def write(addr, data):
        for b in range(len(data)):
            off = addr + b - base_off
            assert 0 <= off < size, "byte outside the array"
            rr, cc = divmod(off // es, ld)
            assert rr < rows and cc < cols, "byte outside the rows x cols window"
        mem[addr:addr + len(data)] = data
        count[addr:addr + len(data)] += 1

    def vec(ti, i, q):
        tj, j = divmod(q, per_row)
        return tile_bytes[ti, tj, i, 16 * j:16 * j + 16].copy()

    for item in range(gr * tr * n_chunks):
        run, k = divmod(item, n_chunks)
        ti, i = divmod(run, tr)
        r = r0 + ti * step_r + i
        if not 0 <= r < rows:
            continue
        v0 = k * chunk
        nv = min(chunk, width - v0)
        row = base_off + (r * ld + c0) * es
        sh = row % 16
        bo = 16 * v0 - sh
        dlo, dhi = lo - bo, hi - bo
        j_lo = min(0 if dlo <= 0 else (dlo + 15) // 16, nv)
        j_hi = max(min(0 if dhi < 16 else dhi // 16, nv), j_lo)
        v = {}
        for t in range(BULK_THREADS):
            for u in range(BULK_PER):
                j = t + BULK_THREADS * u
                v[t, u] = vec(ti, i, v0 + j) if j < nv else np.zeros(16, np.uint8)
        before = vec(ti, i, v0 - 1) if sh and v0 > 0 else np.zeros(16, np.uint8)
        words = np.zeros((nv, 16), np.uint8)
        for t in range(BULK_THREADS):
            lane, warp = t % 32, t // 32
            for u in range(BULK_PER):
                j = t + BULK_THREADS * u
                if lane > 0:
                    prev = v[t - 1, u]
                elif warp > 0:
                    prev = v[t - 1, u]                    # lane 31 of the warp below, same u
                else:
                    prev = v[BULK_THREADS - 1, u - 1] if u > 0 else before
                if j >= nv:
                    continue
                w = v[t, u] if sh == 0 else np.concatenate([prev, v[t, u]])[16 - sh:32 - sh]
                if j_lo <= j < j_hi:
                    words[j] = w
                else:
                    wo = bo + 16 * j
                    for e in range(V):
                        o = wo + e * es
                        if lo <= o < hi:
                            write(row + o, w[e * es:(e + 1) * es])
                if sh and v0 + j == width - 1:
                    vo = 16 * (v0 + j)
                    for e in range(V):
                        o = vo + e * es
                        if e * es >= 16 - sh and lo <= o < hi:
                            write(row + o, v[t, u][e * es:(e + 1) * es])
        if j_hi > j_lo:
            dst = row + bo + 16 * j_lo
            assert dst % 16 == 0 and (16 * (j_hi - j_lo)) % 16 == 0, "unaligned bulk copy"
            write(dst, words[j_lo:j_hi].reshape(-1))
    assert count.max() <= 1, "a byte written twice"
    return mem[base_off:base_off + size]


BULK_SHAPES = SHAPES + [  # runs of several chunks: 1,280 and 2,056 vectors (fp32) per run
    (3, 5000, 5003, 0, 0, 1, 256, 3, 20),
    (5, 8200, 8201, -1, -9, 2, 256, 3, 33),
]


@pytest.mark.parametrize("es", [4, 2])
@pytest.mark.parametrize("shape", BULK_SHAPES)
def test_bulk_row_run_store_model_equals_element_stores(es, shape):
    rows, cols, ld, r0, c0, tr, tc, gr, gc = shape
    V = 16 // es
    if tc % V:
        pytest.skip("tile rows are not whole 16-byte vectors: the element kernel takes these")
    dtype = np.uint32 if es == 4 else np.uint16
    rng = np.random.default_rng(rows * 1000 + cols + es)
    tiles = rng.integers(1, 2 ** (8 * es) - 1, size=(gr, gc, tr, tc), dtype=np.uint64).astype(dtype)
    want = np.zeros((rows, ld), dtype)
    for ti in range(gr):
        for tj in range(gc):
            for i in range(tr):
                r = r0 + ti * tr + i
                if not 0 <= r < rows:
                    continue
                c = c0 + tj * tc + np.arange(tc)
                ok = (c >= 0) & (c < cols)
                want[r, c[ok]] = tiles[ti, tj, i, ok]
    for base_off in (0, es, 2 * es, 16 - es):  # destination pointer offset within 16 bytes
        got = model_store_bulk(tiles, rows, cols, ld, r0, c0, tr, es, base_off)
        assert np.array_equal(got.view(dtype).reshape(rows, ld), want), base_off


def test_bulk_model_constants_match_the_kernel():
    import os
    import re
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "scatter_boundary_tile_gb300",
                            "csrc", "k_tiles_runs.cu")).read()
    threads = int(re.search(r"constexpr int kBulkThreads = (\d+);", src).group(1))
    per = int(re.search(r"constexpr int kBulkPer = (\d+);", src).group(1))
    assert (threads, per) == (BULK_THREADS, BULK_PER)
