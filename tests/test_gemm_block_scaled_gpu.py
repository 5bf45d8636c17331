"""GPU parity of sbt_gemm_block_scaled against the fp64 CPU oracle.

cuTile.jl "Operations", muladd_scaled: D = (A .* a_scale)(B .* b_scale) + acc
with fp32 accumulation.  Every scaled operand and every product is exact in
fp32 for these inputs, so the only error is fp32 summation: each element must
lie within (K + 2) * 2^-23 * (|A'| |B'|)[m][n] of the exact result, |A'| |B'|
being the oracle run on the codes with their sign bits cleared.  The
relative Frobenius error must also stay under 1e-3, the GEMM gate.
Integer-valued inputs must match bit for bit.  Leading-dimension padding of
operands and scales holds NaN codes, so a read past K, K_s or N would show.
"""
import numpy as np
import pytest
import torch

import oracle
import scatter_boundary_tile_gb300 as sbt
import synth
import synth.workloads as wl
from gpu_helpers import Canvas, dev, sync

pytestmark = pytest.mark.gpu
TOL = 1e-3


def abs_codes(codes, fmt):
    return codes & (0x77 if fmt == "e2m1" else 0x7F)


def oracle_of(g, acc=None, ld_acc=0, absolute=False):
    A, B = g["A"], g["B"]
    if absolute:
        A, B = abs_codes(A, g["afmt"]), abs_codes(B, g["bfmt"])
    return oracle.gemm_block_scaled_f64(A, g["lda"], g["SA"], g["ld_sa"], B, g["ldb"], g["SB"], g["ld_sb"], g["M"],
                                        g["N"], g["K"], g["block"], afmt=g["afmt"], bfmt=g["bfmt"], sfmt=g["sfmt"],
                                        acc=acc, ld_acc=ld_acc)


def run(ctx, g, acc=None, in_place=False, ws_pad=0):
    M, N, K, ldd = g["M"], g["N"], g["K"], g["ldd"]
    canvas = Canvas(M * ldd * 4, fill=acc if in_place else None)
    acc_t = dev(acc) if (acc is not None and not in_place) else None
    ws_n = sbt.gemm_block_scaled_workspace_size(ctx, M, N, K)
    ws = torch.empty(max(ws_n + ws_pad, 256), dtype=torch.uint8, device="cuda")
    acc_ptr = canvas.ptr if in_place else acc_t
    sbt.gemm_block_scaled(ctx, dev(g["A"]), g["lda"], dev(g["B"]), g["ldb"], dev(g["SA"]), g["ld_sa"], dev(g["SB"]),
                          g["ld_sb"], g["Ks"], canvas.ptr, ldd, M, N, K,
                          acc=acc_ptr if acc is not None else None, ld_acc=ldd if acc is not None else 0,
                          workspace=ws, workspace_bytes=ws_n, a_fmt=g["afmt"], b_fmt=g["bfmt"], s_fmt=g["sfmt"])
    sync()
    ctx.check_status()
    assert canvas.guards_intact()
    full = canvas.inner(np.float32, (M, ldd))
    orig = canvas.original(np.float32, (M, ldd))
    assert np.array_equal(full[:, N:].view(np.uint32), orig[:, N:].view(np.uint32)), "padding columns of D written"
    return full[:, :N].astype(np.float64)


def check(got, g, acc=None):
    ref = oracle_of(g, acc=acc, ld_acc=g["N"] if acc is not None else 0)
    bound = oracle_of(g, absolute=True)
    slack = (g["K"] + 2) * 2.0 ** -23 * bound + (np.abs(acc) * 2.0 ** -23 if acc is not None else 0) + 1e-30
    bad = np.abs(got - ref) > slack
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref[bad][:5])
    err = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    assert err <= TOL, err


FORMATS = [("e4m3", "e4m3", "e8m0"), ("e5m2", "e5m2", "e8m0"), ("e4m3", "e5m2", "e4m3"), ("e2m1", "e2m1", "e8m0"),
           ("e2m1", "e4m3", "e4m3"), ("e2m1", "e2m1", "e4m3")]
SHAPES = [(1, 1, 32, 32), (3, 5, 64, 32), (65, 97, 96, 32), (128, 256, 64, 16), (129, 257, 160, 32),
          (300, 17, 48, 1), (17, 300, 200, 200)]


@pytest.mark.parametrize("fmts", FORMATS, ids=lambda f: "x".join(f))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_shapes_and_formats_vs_oracle(ctx, fmts, shape):
    M, N, K, block = shape
    g = wl.gemm_block_scaled(M=M, N=N, K=K, block=block, afmt=fmts[0], bfmt=fmts[1], sfmt=fmts[2], tag=3)
    check(run(ctx, g), g)


MX_FORMATS = [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3"), ("e2m1", "e2m1"),
              ("e2m1", "e4m3"), ("e5m2", "e2m1")]
MX_SHAPES = [(1, 1, 32), (7, 9, 96), (65, 97, 160), (256, 224, 128), (257, 225, 256), (300, 449, 544),
             (513, 448, 32)]


@pytest.mark.parametrize("path", ["auto", "scalar"], ids=["block_scale_mma", "bf16_staging"])
@pytest.mark.parametrize("fmts", MX_FORMATS, ids=lambda f: "x".join(f))
@pytest.mark.parametrize("shape", MX_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_e8m0_block32_both_paths_vs_oracle(ctx, path, fmts, shape):
    # E4M3/E5M2/E2M1 with E8M0 scales per 32 along K: "auto" takes the
    # tcgen05 block-scaled kernel (kind::mxf8f6f4 with 128-deep K blocks, or
    # kind::mxf4 with 256-deep ones for E2M1 x E2M1; 256 x 208 tiles, so these
    # shapes cut tiles and K blocks at every kind of edge), "scalar" forces the
    # bf16 staging path; both must meet the same bounds.
    M, N, K = shape
    ctx.set_path(path)
    g = wl.gemm_block_scaled(M=M, N=N, K=K, block=32, afmt=fmts[0], bfmt=fmts[1], sfmt="e8m0", tag=8)
    check(run(ctx, g), g)


def test_several_tiles_ragged_tail(ctx):
    # 3 x 3 tiles of 128 x 256 (or 2 x 3 CTA-pair tiles) with one-row / one-column tails, 32 K blocks
    g = wl.gemm_block_scaled(M=257, N=513, K=1024, block=32, tag=4)
    check(run(ctx, g), g)


@pytest.mark.parametrize("in_place", [False, True])
def test_acc_added(ctx, in_place):
    g = wl.gemm_block_scaled(M=70, N=90, K=128, block=32, tag=5)
    acc = synth.uniform_f32(synth.stream_seed(wl.SEED_GEMM_SCALED, 90), (g["M"], g["ldd"]), -100.0, 100.0)
    got = run(ctx, g, acc=acc, in_place=in_place)
    check(got, g, acc=np.ascontiguousarray(acc[:, :g["N"]]))


def test_k_zero_gives_acc_or_zero(ctx):
    M, N, ldd = 33, 45, 47
    acc = synth.uniform_f32(synth.stream_seed(wl.SEED_GEMM_SCALED, 91), (M, ldd), -1.0, 1.0)
    for use_acc in (False, True):
        canvas = Canvas(M * ldd * 4)
        acc_t = dev(acc)
        sbt.gemm_block_scaled(ctx, None, 0, None, N, None, 0, None, N, 0, canvas.ptr, ldd, M, N, 0,
                              acc=acc_t if use_acc else None, ld_acc=ldd if use_acc else 0)
        sync()
        d = canvas.inner(np.float32, (M, ldd))
        want = acc[:, :N] if use_acc else np.zeros((M, N), np.float32)
        assert np.array_equal(d[:, :N], want)
        assert np.array_equal(d[:, N:].view(np.uint32), canvas.original(np.float32, (M, ldd))[:, N:].view(np.uint32))
        assert canvas.guards_intact()


def test_integer_values_exact(ctx):
    # E4M3 integers -4..4 (codes 0x00, 0x38, 0x40, 0x44, 0x48 and negatives), scales 2^0 / 2^1:
    # every product and partial sum is an integer below 2^24.
    M, N, K, block = 96, 80, 256, 32
    g = wl.gemm_block_scaled(M=M, N=N, K=K, block=block, tag=6)
    ints = np.array([0x00, 0x38, 0x40, 0x44, 0x48], np.uint8)
    pick = lambda seed, n: ints[synth.int_below(seed, n, 5)] | (synth.int_below(seed + 1, n, 2) << 7).astype(np.uint8)
    g["A"][:, :K] = pick(611, M * K).reshape(M, K)
    g["B"][:, :N] = pick(613, K * N).reshape(K, N)
    g["SA"][:, :g["Ks"]] = 127 + synth.int_below(615, M * g["Ks"], 2).reshape(M, g["Ks"])
    g["SB"][:, :N] = 127 + synth.int_below(616, g["Ks"] * N, 2).reshape(g["Ks"], N)
    got = run(ctx, g)
    ref = oracle_of(g)
    assert np.array_equal(got, ref)


def test_nan_codes_propagate_to_their_row_and_column(ctx):
    g = wl.gemm_block_scaled(M=40, N=50, K=64, block=32, tag=7)
    g["A"][5, 9] = 0x7F       # E4M3 NaN in row 5 of A
    g["SB"][1, 33] = 0xFF     # E8M0 NaN scale of column 33, block 1
    got = run(ctx, g)
    nan = np.zeros((40, 50), bool)
    nan[5, :] = True
    nan[:, 33] = True
    np.testing.assert_array_equal(np.isnan(got), nan)


def sampled_check(got, g, rows, cols, acc=None):
    """The oracle on the sampled rows and columns only, held to the same bound as check()."""
    K, block = g["K"], g["block"]
    Ar, SAr = np.ascontiguousarray(g["A"][rows]), np.ascontiguousarray(g["SA"][rows])
    Bc = np.ascontiguousarray(g["B"][:, cols]) if g["bfmt"] != "e2m1" else None
    if Bc is None:  # packed E2M1 columns cannot be sliced bytewise: unpack, slice, repack
        codes = np.stack([g["B"] & 15, g["B"] >> 4], axis=-1).reshape(g["B"].shape[0], -1)[:, cols]
        codes = np.pad(codes, ((0, 0), (0, len(cols) % 2)))
        Bc = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    SBc = np.ascontiguousarray(g["SB"][:, cols])
    R, C = len(rows), len(cols)
    ldb = C + (C % 2 if g["bfmt"] == "e2m1" else 0)
    accs = None if acc is None else np.ascontiguousarray(acc[np.ix_(rows, cols)])
    ref = oracle.gemm_block_scaled_f64(Ar, g["lda"], SAr, g["ld_sa"], Bc, ldb, SBc, C, R, C, K, block,
                                       afmt=g["afmt"], bfmt=g["bfmt"], sfmt=g["sfmt"], acc=accs, ld_acc=C)
    bound = oracle.gemm_block_scaled_f64(abs_codes(Ar, g["afmt"]), g["lda"], SAr, g["ld_sa"],
                                         abs_codes(Bc, g["bfmt"]), ldb, SBc, C, R, C, K, block,
                                         afmt=g["afmt"], bfmt=g["bfmt"], sfmt=g["sfmt"])
    d = got[np.ix_(rows, cols)]
    slack = (K + 2) * 2.0 ** -23 * bound + (np.abs(accs) * 2.0 ** -23 if accs is not None else 0) + 1e-30
    assert np.all(np.abs(d - ref) <= slack)


@pytest.mark.parametrize("case", ["e4m3_tail_rows", "e2m1_acc_in_place", "e5m2_acc"])
def test_many_tiles_sampled(ctx, case):
    """CTA-pair kernel over many tiles, checked on sampled rows and columns: (600, 8320) has a
    last row tile of 88 rows, one of its CTAs wholly past M; acc is added (also in place,
    D = acc); E2M1 and E5M2 operands."""
    M, N, K = {"e4m3_tail_rows": (600, 8320, 256), "e2m1_acc_in_place": (600, 8320, 256),
               "e5m2_acc": (1100, 8400, 384)}[case]
    fmt = {"e4m3_tail_rows": "e4m3", "e2m1_acc_in_place": "e2m1", "e5m2_acc": "e5m2"}[case]
    g = wl.gemm_block_scaled(M=M, N=N, K=K, block=32, afmt=fmt, bfmt=fmt, tag=8)
    acc = None
    if case != "e4m3_tail_rows":
        acc = synth.uniform_f32(synth.stream_seed(wl.SEED_GEMM_SCALED, 92), (M, g["ldd"]), -10.0, 10.0)
    got = run(ctx, g, acc=acc, in_place=case == "e2m1_acc_in_place")
    rows = np.concatenate([[0, 1, 127, 128, 255, 256, 511, 512, 513, M - 2, M - 1], synth.int_below(622, 30, M)])
    cols = np.concatenate([[0, 1, 207, 208, 415, 416, N - 2, N - 1], synth.int_below(623, 24, N)])
    sampled_check(got, g, rows, cols, acc=None if acc is None else acc[:, :N])


def test_full_size_sampled_rows_and_columns(ctx):
    # 8191 x 8193 x 4096, E4M3 operands, E8M0 scales over blocks of 32: the
    # launch configuration the benchmark times (CTA pairs), checked on 48 rows
    # x 40 columns computed by the oracle one by one.
    M, N, K, block = 8191, 8193, 4096, 32
    g = wl.gemm_block_scaled(M=M, N=N, K=K, block=block, tag=0)
    got = run(ctx, g)
    rows = np.concatenate([[0, 1, 127, 128, 255, 256, M - 2, M - 1], synth.int_below(620, 40, M)])
    cols = np.concatenate([[0, 1, 255, 256, 511, 512, N - 2, N - 1], synth.int_below(621, 32, N)])
    Ar, SAr = g["A"][rows], np.ascontiguousarray(g["SA"][rows])
    Bc, SBc = np.ascontiguousarray(g["B"][:, cols]), np.ascontiguousarray(g["SB"][:, cols])
    R, C = len(rows), len(cols)
    ref = oracle.gemm_block_scaled_f64(Ar, g["lda"], SAr, g["ld_sa"], Bc, C, SBc, C, R, C, K, block)
    bound = oracle.gemm_block_scaled_f64(abs_codes(Ar, "e4m3"), g["lda"], SAr, g["ld_sa"], abs_codes(Bc, "e4m3"), C,
                                         SBc, C, R, C, K, block)
    d = got[np.ix_(rows, cols)]
    assert np.all(np.abs(d - ref) <= (K + 2) * 2.0 ** -23 * bound + 1e-30)


@pytest.mark.parametrize("case,status", [
    ("ks_not_dividing", sbt.SBT_ERR_INVALID_ARG), ("odd_ld_e2m1", sbt.SBT_ERR_INVALID_ARG),
    ("scale_e5m2", sbt.SBT_ERR_UNSUPPORTED), ("operand_e8m0", sbt.SBT_ERR_UNSUPPORTED),
    ("small_workspace", sbt.SBT_ERR_ALIGNMENT), ("acc_alias_other_ld", sbt.SBT_ERR_INVALID_ARG)])
def test_rejected_before_launch(ctx, case, status):
    M, N, K = 16, 16, 64
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    D = torch.zeros(M * 40, dtype=torch.float32, device="cuda")
    ws_n = sbt.gemm_block_scaled_workspace_size(ctx, M, N, K)
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    kw = dict(a_fmt="e4m3", b_fmt="e4m3", s_fmt="e8m0", workspace=ws, workspace_bytes=ws_n)
    Ks, lda, ldd, acc, ld_acc = 2, K, N, None, 0
    if case == "ks_not_dividing":
        Ks = 3
    elif case == "odd_ld_e2m1":
        kw["a_fmt"], lda = "e2m1", K + 1
    elif case == "scale_e5m2":
        kw["s_fmt"] = "e5m2"
    elif case == "operand_e8m0":
        kw["b_fmt"] = "e8m0"
    elif case == "small_workspace":
        kw["workspace_bytes"] = ws_n - 1
    elif case == "acc_alias_other_ld":
        acc, ld_acc, ldd = D, N + 1, N
    before = ctx.launch_count
    with pytest.raises(sbt.SbtError) as e:
        sbt.gemm_block_scaled(ctx, buf, lda, buf, N, buf, Ks, buf, N, Ks, D, ldd, M, N, K, acc=acc, ld_acc=ld_acc,
                              **kw)
    assert e.value.status == status
    assert ctx.launch_count == before
