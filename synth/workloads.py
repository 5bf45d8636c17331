"""Input recipes of the benchmark workloads (seeded, synthetic).

Each function returns plain numpy buffers (bf16 as uint16 bits) plus the
scalar parameters of the call.  Sizes default to the full workloads; tests
pass smaller sizes with the same value distributions and structure.

Seeds: workload *i* (1..5, in the order tiles, gather, scatter, ragged, GEMM)
uses ``0x5B7000 + i``; every buffer draws from its own sub-stream.
"""
from __future__ import annotations

import numpy as np

from . import bernoulli_u8, int_below, normal_bf16, permutation_prefix, stream_seed, uniform_f32, uniform_f64

SEED_TILES = 0x5B7001
SEED_GATHER = 0x5B7002
SEED_SCATTER = 0x5B7003
SEED_RAGGED = 0x5B7004
SEED_GEMM = 0x5B7005

BF16_NAN_BITS = 0x7FC1  # fill of leading-dimension padding: any read of it poisons a GEMM result
F32_CANARY_BITS = 0x7FC0DEAD


def smallest_odd_at_least(n: int) -> int:
    return n if n % 2 == 1 else n + 1


def tiles_small(seed: int = SEED_TILES, rows: int = 65, cols: int = 73):
    """fp32 ``rows x cols`` matrix, row-major with ld = cols, uniform [-1, 1)."""
    a = uniform_f32(stream_seed(seed, 1), (rows, cols), -1.0, 1.0)
    return {"a": a, "rows": rows, "cols": cols, "ld": cols}


def gather_small(seed: int = SEED_TILES, rows: int = 65, cols: int = 73, n_idx: int = 16):
    """16 int32 indices uniform in [-1, 80] into the 65x73 fp32 table; pad -1.0."""
    t = tiles_small(seed, rows, cols)
    idx = (int_below(stream_seed(seed, 2), n_idx, 82, lo=-1)).astype(np.int32)
    return {"table": t["a"], "idx": idx, "pad": np.float32(-1.0)}


def gather_rows_bf16(seed: int = SEED_GATHER, n_rows: int = 1_000_000, n_idx: int = 1_048_576, cols: int = 512):
    """bf16 table N(0,1); indices: 1 % are -1, 0.5 % are >= n_rows, the rest uniform in [0, n_rows)."""
    table = normal_bf16(stream_seed(seed, 1), (n_rows, cols))
    u = uniform_f64(stream_seed(seed, 2), n_idx)
    valid = int_below(stream_seed(seed, 3), n_idx, n_rows)
    past = int_below(stream_seed(seed, 4), n_idx, (2**31 - 1) - n_rows, lo=n_rows)
    idx = np.where(u < 0.01, -1, np.where(u < 0.015, past, valid)).astype(np.int32)
    return {"table": table, "idx": idx, "n_rows": n_rows, "cols": cols}


def scatter_rows_f32(seed: int = SEED_SCATTER, dst_rows: int = 4_194_304, n_idx: int = 1_048_576,
                     cols: int = 256, p: float = 0.9):
    """Unique destination rows (prefix of a seeded permutation), uniform [-1,1) source,
    Bernoulli(p) per-element uint8 mask.  The destination starts at zero (the caller's fill)."""
    idx = permutation_prefix(stream_seed(seed, 1), dst_rows, n_idx)
    src = uniform_f32(stream_seed(seed, 2), (n_idx, cols), -1.0, 1.0)
    mask = bernoulli_u8(stream_seed(seed, 3), (n_idx, cols), p)
    return {"idx": idx, "src": src, "mask": mask, "dst_rows": dst_rows, "cols": cols}


def ragged_bf16(seed: int = SEED_RAGGED, batch: int = 64, max_len: int = 4096, heads: int = 8, depth: int = 128):
    """Packed sequences [sum(len)][heads][depth] bf16 N(0,1), lengths uniform in [1, max_len]."""
    lens = 1 + int_below(stream_seed(seed, 1), batch, max_len)
    cu = np.zeros(batch + 1, np.int64)
    cu[1:] = np.cumsum(lens)
    total = int(cu[-1])
    x = normal_bf16(stream_seed(seed, 2), (total, heads, depth))
    return {"x": x, "cu_seqlens": cu.astype(np.int32), "lens": lens, "t_pad": max_len,
            "heads": heads, "depth": depth, "total_rows": total}


def gemm_bf16(seed: int = SEED_GEMM, M: int = 65, N: int = 97, K: int = 73, tag: int = 0):
    """A (M,K) and B (K,N) bf16 N(0,1) stored row-major with odd leading dimensions
    lda = smallest odd >= K, ldb = ldc = smallest odd >= N.  Leading-dimension padding
    holds a bf16 NaN so that any read past the logical extent shows in the result."""
    lda, ldb, ldc = smallest_odd_at_least(K), smallest_odd_at_least(N), smallest_odd_at_least(N)
    A = np.full((M, lda), BF16_NAN_BITS, np.uint16)
    B = np.full((K, ldb), BF16_NAN_BITS, np.uint16)
    A[:, :K] = normal_bf16(stream_seed(seed, 2 * tag + 1), (M, K))
    B[:, :N] = normal_bf16(stream_seed(seed, 2 * tag + 2), (K, N))
    return {"A": A, "B": B, "M": M, "N": N, "K": K, "lda": lda, "ldb": ldb, "ldc": ldc}


GEMM_SHAPES = [(65, 97, 73), (1000, 1000, 1000), (8191, 8193, 4097)]

SEED_GEMM_SCALED = 0x5B7006


def lowp_codes(seed: int, shape, fmt: str) -> np.ndarray:
    """Uniformly drawn codes of a low-precision format with NaN/infinity codes
    replaced by the code of 1.0, so that magnitudes are log-uniform over the
    format's whole range (zeros and subnormals included).  E2M1 returns one
    nibble per uint8 (unpacked)."""
    n = int(np.prod(shape))
    if fmt == "e2m1":
        return int_below(seed, n, 16).astype(np.uint8).reshape(shape)
    c = int_below(seed, n, 256).astype(np.uint8).reshape(shape)
    if fmt == "e4m3":
        c[(c & 0x7F) == 0x7F] = 0x38
    elif fmt == "e5m2":
        c[(c & 0x7C) == 0x7C] = 0x3C
    else:
        raise ValueError(fmt)
    return c


def pack_e2m1(nibbles: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte along each row (even column in the low nibble); columns must be even."""
    assert nibbles.shape[-1] % 2 == 0
    return (nibbles[..., 0::2] | (nibbles[..., 1::2] << 4)).astype(np.uint8)


def scale_codes(seed: int, shape, fmt: str) -> np.ndarray:
    """E8M0 scales 2^-4 .. 2^4 (codes 123..131), or positive normal E4M3 scales 0.125 .. 7.5 (codes 0x20..0x4F)."""
    n = int(np.prod(shape))
    if fmt == "e8m0":
        return (123 + int_below(seed, n, 9)).astype(np.uint8).reshape(shape)
    if fmt == "e4m3":
        return (0x20 + int_below(seed, n, 0x30)).astype(np.uint8).reshape(shape)
    raise ValueError(fmt)


def gemm_block_scaled(seed: int = SEED_GEMM_SCALED, M: int = 65, N: int = 97, K: int = 96, block: int = 32,
                      afmt: str = "e4m3", bfmt: str = "e4m3", sfmt: str = "e8m0", tag: int = 0):
    """A (M,K) and B (K,N) codes (see lowp_codes), a_scale (M,K/block), b_scale (K/block,N).
    Leading dimensions: the smallest odd >= the extent for byte formats and the
    smallest even for E2M1 (packed, ld in elements); ld_sa = smallest odd >= K_s,
    ld_sb = smallest odd >= N, ldd = smallest odd >= N.  Padding codes are NaN
    (0x7F) for byte formats and 0xFF (NaN in E8M0 and E4M3) for scales, so that
    any read past K, K_s or N shows."""
    Ks = K // block
    even = lambda n: n + (n % 2)
    lda = even(K) if afmt == "e2m1" else smallest_odd_at_least(K)
    ldb = even(N) if bfmt == "e2m1" else smallest_odd_at_least(N)
    ld_sa, ld_sb = smallest_odd_at_least(Ks), smallest_odd_at_least(N)
    a = lowp_codes(stream_seed(seed, 4 * tag + 1), (M, K), afmt)
    b = lowp_codes(stream_seed(seed, 4 * tag + 2), (K, N), bfmt)
    if afmt == "e2m1":
        A = pack_e2m1(np.pad(a, ((0, 0), (0, lda - K))))
    else:
        A = np.full((M, lda), 0x7F, np.uint8)
        A[:, :K] = a
    if bfmt == "e2m1":
        B = pack_e2m1(np.pad(b, ((0, 0), (0, ldb - N))))
    else:
        B = np.full((K, ldb), 0x7F, np.uint8)
        B[:, :N] = b
    SA = np.full((M, ld_sa), 0xFF, np.uint8)
    SB = np.full((Ks, ld_sb), 0xFF, np.uint8)
    SA[:, :Ks] = scale_codes(stream_seed(seed, 4 * tag + 3), (M, Ks), sfmt)
    SB[:, :N] = scale_codes(stream_seed(seed, 4 * tag + 4), (Ks, N), sfmt)
    return {"A": A, "B": B, "SA": SA, "SB": SB, "M": M, "N": N, "K": K, "Ks": Ks, "block": block,
            "lda": lda, "ldb": ldb, "ld_sa": ld_sa, "ld_sb": ld_sb, "ldd": smallest_odd_at_least(N),
            "afmt": afmt, "bfmt": bfmt, "sfmt": sfmt}
