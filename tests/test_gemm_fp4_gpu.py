"""GPU parity of the packed 4-bit block-scaled forms against the fp64 CPU oracle.

cuTile.jl "Operations", muladd_scaled with f4e2m1fn operands: E2M1 x E2M1 with
E8M0 scales over blocks of 32 runs on tcgen05.mma kind::mxf4 (two scales per
K = 64 instruction), and with E4M3 scales over blocks of 16 on
kind::mxf4nvf4 (four per instruction).  The tensor cores read the latter
scales unsigned, so staging moves a negative scale's sign onto its 16 codes
and the epilogue writes NaN where a scale was NaN; these tests give the
kernel signed, zero, subnormal and NaN scales.

Bounds as in the 8-bit tests: every scaled operand and every product is exact
in fp32, so each element must lie within (K + 2) * 2^-23 * (|A'| |B'|)[m][n]
of the oracle's exact result, |A'| |B'| being the oracle run on the codes and
scales with their sign bits cleared; the relative Frobenius error must stay
under 1e-3; integer-valued inputs must match bit for bit.
"""
import numpy as np
import pytest

import oracle
import synth
import synth.workloads as wl
from test_gemm_block_scaled_gpu import run, sampled_check

pytestmark = pytest.mark.gpu
TOL = 1e-3

FORMS = [("e8m0", 32), ("e4m3", 16)]
FORM_IDS = ["mxf4_e8m0_per32", "mxf4nvf4_e4m3_per16"]


def packed(M, N, K, form, tag):
    sfmt, block = form
    return wl.gemm_block_scaled(M=M, N=N, K=K, block=block, afmt="e2m1", bfmt="e2m1", sfmt=sfmt, tag=tag)


def abs_scales(codes, sfmt):
    """Scale codes with the sign cleared (E4M3); NaN codes stay NaN."""
    return codes & 0x7F if sfmt == "e4m3" else codes


def oracle_pair(g, acc=None):
    """The exact result and the bound |A'| |B'| (codes and scales without signs)."""
    ld_acc = g["N"] if acc is not None else 0
    args = dict(afmt="e2m1", bfmt="e2m1", sfmt=g["sfmt"])
    ref = oracle.gemm_block_scaled_f64(g["A"], g["lda"], g["SA"], g["ld_sa"], g["B"], g["ldb"], g["SB"], g["ld_sb"],
                                       g["M"], g["N"], g["K"], g["block"], acc=acc, ld_acc=ld_acc, **args)
    bound = oracle.gemm_block_scaled_f64(g["A"] & 0x77, g["lda"], abs_scales(g["SA"], g["sfmt"]), g["ld_sa"],
                                         g["B"] & 0x77, g["ldb"], abs_scales(g["SB"], g["sfmt"]), g["ld_sb"],
                                         g["M"], g["N"], g["K"], g["block"], **args)
    return ref, bound


def check(got, g, acc=None):
    ref, bound = oracle_pair(g, acc)
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), ~fin), "NaN pattern differs from the oracle's"
    slack = (g["K"] + 2) * 2.0 ** -23 * bound + (np.abs(acc) * 2.0 ** -23 if acc is not None else 0) + 1e-30
    bad = fin & ~(np.abs(got - ref) <= slack)
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref[bad][:5])
    if fin.any():
        err = float(np.linalg.norm((got - ref)[fin]) / max(np.linalg.norm(ref[fin]), 1e-300))
        assert err <= TOL, err


# K blocks of the packed forms are 256 deep (four instructions of 64): these cut M, N and K
# at every kind of edge (one scale block; a K tail of 32 or 16 in the last instruction; several
# 256 x 208 tiles with one-row or one-column tails).
SHAPES = [(1, 1, 32), (7, 9, 64), (65, 97, 96), (256, 208, 256), (257, 209, 288), (300, 420, 544),
          (513, 417, 1056)]


@pytest.mark.parametrize("path", ["auto", "scalar"], ids=["block_scale_mma", "bf16_staging"])
@pytest.mark.parametrize("form", FORMS, ids=FORM_IDS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_packed_forms_both_paths_vs_oracle(ctx, path, form, shape):
    M, N, K = shape
    ctx.set_path(path)
    g = packed(M, N, K, form, tag=30)
    check(run(ctx, g), g)


@pytest.mark.parametrize("K", [16, 48, 80, 272])
def test_nvf4_k_tails(ctx, K):
    # blocks of 16: a last instruction holding one, three or five scale blocks of real data
    g = packed(130, 220, K, ("e4m3", 16), tag=31)
    check(run(ctx, g), g)


@pytest.mark.parametrize("form", FORMS, ids=FORM_IDS)
def test_integer_values_exact(ctx, form):
    # every E2M1 code (multiples of 0.5 up to 6), scales 1 and 2: each product is a multiple of
    # 0.25 and every partial sum stays below 2^18, so fp32 sums are exact in any order
    M, N, K = 150, 230, 512
    g = packed(M, N, K, form, tag=32)
    sfmt = form[0]
    one, two = (127, 128) if sfmt == "e8m0" else (0x38, 0x40)
    Ks = g["Ks"]
    g["SA"][:, :Ks] = np.where(synth.int_below(631, M * Ks, 2) == 0, one, two).reshape(M, Ks)
    g["SB"][:, :N] = np.where(synth.int_below(632, Ks * N, 2) == 0, one, two).reshape(Ks, N)
    got = run(ctx, g)
    ref, _ = oracle_pair(g)
    assert np.array_equal(got, ref)


def test_nvf4_signed_zero_and_subnormal_scales(ctx):
    # E4M3 scales drawn over every code but NaN: negative scales (their sign moves onto the
    # operand codes), +-0, subnormals and the largest magnitude 448
    M, N, K = 300, 430, 320
    g = packed(M, N, K, ("e4m3", 16), tag=33)
    Ks = g["Ks"]

    def codes(seed, n):
        c = synth.int_below(seed, n, 256).astype(np.uint8)
        c[(c & 0x7F) == 0x7F] = 0x80  # NaN -> -0
        return c

    g["SA"][:, :Ks] = codes(641, M * Ks).reshape(M, Ks)
    g["SB"][:, :N] = codes(642, Ks * N).reshape(Ks, N)
    g["SA"][3, :Ks] = np.arange(Ks, dtype=np.uint8) % 8  # +0 and the positive subnormals
    g["SB"][:, 7] = 0x80 | (np.arange(Ks, dtype=np.uint8) % 8)  # -0 and the negative subnormals
    check(run(ctx, g), g)


@pytest.mark.parametrize("form", FORMS, ids=FORM_IDS)
def test_nan_scales_propagate_to_their_row_and_column(ctx, form):
    M, N, K = 300, 430, 128
    g = packed(M, N, K, form, tag=34)
    nan = 0xFF if form[0] == "e8m0" else 0x7F
    g["SA"][5, 1] = nan                      # first row tile
    g["SA"][270, 0] = 0xFF                   # second row tile (E4M3: negative NaN)
    g["SB"][1, 33] = nan                     # first column tile
    g["SB"][0, 415] = 0xFF                   # second column tile
    got = run(ctx, g)
    want = np.zeros((M, N), bool)
    want[[5, 270], :] = True
    want[:, [33, 415]] = True
    np.testing.assert_array_equal(np.isnan(got), want)
    check(got, g)


@pytest.mark.parametrize("form", FORMS, ids=FORM_IDS)
@pytest.mark.parametrize("case", ["tail_rows", "acc_in_place"])
def test_many_tiles_sampled(ctx, form, case):
    """CTA-pair kernel over many tiles and K blocks, on sampled rows and columns: (600, 8320)
    has a last row tile of 88 rows, one of its CTAs wholly past M; acc is added in place."""
    M, N, K = (600, 8320, 768) if case == "tail_rows" else (1100, 8400, 1312)
    g = packed(M, N, K, form, tag=35)
    acc = None
    if case == "acc_in_place":
        acc = synth.uniform_f32(synth.stream_seed(wl.SEED_GEMM_SCALED, 93), (M, g["ldd"]), -10.0, 10.0)
    got = run(ctx, g, acc=acc, in_place=acc is not None)
    rows = np.concatenate([[0, 1, 127, 128, 255, 256, 511, 512, 513, M - 2, M - 1], synth.int_below(652, 30, M)])
    cols = np.concatenate([[0, 1, 207, 208, 415, 416, N - 2, N - 1], synth.int_below(653, 24, N)])
    sampled_check(got, g, rows, cols, acc=None if acc is None else acc[:, :N])


@pytest.mark.parametrize("form", FORMS, ids=FORM_IDS)
def test_full_size_sampled_rows_and_columns(ctx, form):
    # 8191 x 8193 x 4096: the launch configuration the benchmark times, on 48 rows x 40 columns
    M, N, K = 8191, 8193, 4096
    g = packed(M, N, K, form, tag=0)
    got = run(ctx, g)
    rows = np.concatenate([[0, 1, 127, 128, 255, 256, M - 2, M - 1], synth.int_below(660, 40, M)])
    cols = np.concatenate([[0, 1, 207, 208, 415, 416, N - 2, N - 1], synth.int_below(661, 32, N)])
    sampled_check(got, g, rows, cols)


@pytest.mark.parametrize("lda_extra,offset,launches", [(0, 0, 3), (0, 16, 3), (2, 0, 4), (0, 2, 4)],
                         ids=["aligned_rows_in_place", "offset_16_in_place", "row_stride_staged",
                              "offset_2_staged"])
def test_mxf4_a_read_in_place_or_staged(ctx, lda_extra, offset, launches):
    # kind::mxf4 reads packed A where it lies when its rows start on 16-byte boundaries (lda a
    # multiple of 32 codes, base 16-byte aligned): three launches (B, scales, tensor kernel);
    # otherwise A is staged first (four).  M, N and K cut tiles, K blocks and the 128-byte box.
    import torch
    import scatter_boundary_tile_gb300 as sbt
    from gpu_helpers import Canvas, dev, sync
    M, N, K = 300, 230, 544
    g = packed(M, N, K, ("e8m0", 32), tag=36)
    lda = K + lda_extra
    codes = np.stack([g["A"] & 15, g["A"] >> 4], axis=-1).reshape(M, -1)[:, :K]
    A = np.zeros((M, lda // 2), np.uint8)
    A[:, :K // 2] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    if lda_extra:
        A[:, K // 2:] = 0x77  # padding codes 6.0: a read past K would show
    g["A"], g["lda"] = A, lda
    buf = torch.zeros(A.size + 64, dtype=torch.uint8, device="cuda")
    buf[offset:offset + A.size] = dev(A.reshape(-1))
    canvas = Canvas(M * g["ldd"] * 4)
    ws_n = sbt.gemm_block_scaled_workspace_size(ctx, M, N, K)
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    before = ctx.launch_count
    sbt.gemm_block_scaled(ctx, buf[offset:], lda, dev(g["B"]), g["ldb"], dev(g["SA"]), g["ld_sa"], dev(g["SB"]),
                          g["ld_sb"], g["Ks"], canvas.ptr, g["ldd"], M, N, K, workspace=ws, workspace_bytes=ws_n,
                          a_fmt="e2m1", b_fmt="e2m1", s_fmt="e8m0")
    sync()
    ctx.check_status()
    assert ctx.launch_count - before == launches
    assert canvas.guards_intact()
    got = canvas.inner(np.float32, (M, g["ldd"]))[:, :N].astype(np.float64)
    check(got, g)


@pytest.mark.parametrize("fmts", [("e4m3", "e8m0", 32), ("e2m1", "e8m0", 32), ("e2m1", "e4m3", 16)],
                         ids=["mxf8f6f4", "mxf4", "mxf4nvf4"])
def test_repeated_calls_bit_identical(ctx, fmts):
    # each tile's K order is fixed by the kernel, so the same inputs give the same bits on every call
    fmt, sfmt, block = fmts
    g = wl.gemm_block_scaled(M=700, N=650, K=1024, block=block, afmt=fmt, bfmt=fmt, sfmt=sfmt, tag=37)
    first = run(ctx, g)
    again = run(ctx, g)
    assert np.array_equal(first.view(np.uint64), again.view(np.uint64))
