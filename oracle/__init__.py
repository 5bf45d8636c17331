"""CPU oracle (test infrastructure only).

Plain single-threaded C (``sbt_oracle.c``) behind ctypes, taking numpy
arrays.  Only the tests, the smoke check and the benchmark's CPU-baseline
leg import this package; the product library never does, and the two share
no code.  bf16 data is carried as numpy uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sbt_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no OpenMP, no vector intrinsics)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, i32, p, ci = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int
            lib.oracle_tile_load_padded.argtypes = [ci, p, i64, i64, i64, i64, i64, i64, i64, i64,
                                                    i32, i32, i32, i32, p, p]
            lib.oracle_tile_store_clipped.argtypes = [ci, p, i32, i32, i32, i32, p, i64, i64, i64, i64,
                                                      i64, i64, i64, i64]
            lib.oracle_gather_rows.argtypes = [ci, p, i64, i64, i64, p, i64, i64, i64, i32, p, i64, p, i64, p]
            lib.oracle_gather_cols.argtypes = [ci, p, i64, i64, i64, p, i64, i64, i64, i32, p, i64, p]
            lib.oracle_gather_cols.restype = None
            lib.oracle_scatter_rows_masked.argtypes = [ci, p, i64, i64, i64, p, i64, i64, i64, p, i64, i32,
                                                       p, i64]
            lib.oracle_ragged_tile_load.argtypes = [ci, p, i64, i32, i32, i64, i64, p, i32, i32, p]
            lib.oracle_scatter_add_rows.argtypes = [ci, p, i64, i64, i64, p, i64, i64, i64, p, i64, i32]
            lib.oracle_scatter_add_rows.restype = None
            lib.oracle_ragged_tile_store.argtypes = [ci, p, i32, i32, i32, i32, p, p, i64, i64, i64]
            lib.oracle_gemm_f64.argtypes = [p, i64, p, i64, i64, i64, i64, p, i64]
            lib.oracle_gemm_f64_at.argtypes = [p, i64, p, i64, i64, p, p, i64, p]
            lib.oracle_fp8_decode.argtypes = [ci, ctypes.c_uint8]
            lib.oracle_fp8_decode.restype = ctypes.c_double
            lib.oracle_gemm_block_scaled_f64.argtypes = [ci, ci, ci, p, i64, p, i64, p, i64, p, i64, p, i64, i64,
                                                         i64, i64, i64, p, i64]
            lib.oracle_gemm_block_scaled_f64.restype = None
            lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
            lib.oracle_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_round_bf16.argtypes = [p, i64, p]
            for f in (lib.oracle_tile_load_padded, lib.oracle_tile_store_clipped, lib.oracle_gather_rows,
                      lib.oracle_scatter_rows_masked, lib.oracle_ragged_tile_load, lib.oracle_ragged_tile_store, lib.oracle_gemm_f64,
                      lib.oracle_gemm_f64_at, lib.oracle_round_bf16):
                f.restype = None
            _lib = lib
    return _lib


def _es(a: np.ndarray) -> int:
    if a.dtype.itemsize not in (2, 4):
        raise TypeError("movement ops take 2- or 4-byte elements")
    return a.dtype.itemsize


def _p(a):
    return None if a is None else a.ctypes.data


def _pad_bits(pad, dtype) -> np.ndarray:
    return np.array([pad], dtype=dtype).reshape(1)


def _flat_buffer(a: np.ndarray) -> np.ndarray:
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle buffers must be C-contiguous (strides are passed explicitly)")
    return a


def tile_load_padded(src, rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c,
                     grid_r, grid_c, tile_r, tile_c, pad=0):
    """Padded loads of a grid of tiles; returns [grid_r][grid_c][tile_r][tile_c]."""
    src = _flat_buffer(src)
    out = np.empty((grid_r, grid_c, tile_r, tile_c), src.dtype)
    padb = _pad_bits(pad, src.dtype)
    _load().oracle_tile_load_padded(_es(src), _p(src), rows, cols, stride_r, stride_c, origin_r, origin_c,
                                    step_r, step_c, grid_r, grid_c, tile_r, tile_c, _p(out), _p(padb))
    return out


def tile_store_clipped(tiles, dst, rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c):
    """Clipped stores of a [grid_r][grid_c][tile_r][tile_c] tile grid into ``dst`` (in place)."""
    tiles, dst = _flat_buffer(tiles), _flat_buffer(dst)
    assert tiles.dtype == dst.dtype and tiles.ndim == 4
    gr, gc, tr, tc = tiles.shape
    _load().oracle_tile_store_clipped(_es(dst), _p(tiles), gr, gc, tr, tc, _p(dst), rows, cols, stride_r,
                                      stride_c, origin_r, origin_c, step_r, step_c)
    return dst


def gather_rows(src, rows, cols, ld_src, idx, tile_c, row_offset=0, col_offset=0, mask=None, ld_mask=None,
                pad=0, ld_out=None):
    """Row gather; returns out[n_idx][ld_out] (columns >= tile_c left as zero)."""
    src = _flat_buffer(src)
    idx = np.ascontiguousarray(idx, np.int32)
    n = idx.size
    ld_out = tile_c if ld_out is None else ld_out
    out = np.zeros((n, ld_out), src.dtype)
    if mask is not None:
        mask = _flat_buffer(np.asarray(mask, np.uint8))
        ld_mask = tile_c if ld_mask is None else ld_mask
    padb = _pad_bits(pad, src.dtype)
    _load().oracle_gather_rows(_es(src), _p(src), rows, cols, ld_src, _p(idx), n, row_offset, col_offset,
                               tile_c, _p(mask), ld_mask or 0, _p(out), ld_out, _p(padb))
    return out


def gather_cols(src, rows, cols, ld_src, idx, tile_r, row_offset=0, col_offset=0, pad=0, ld_out=None):
    """Column gather; returns out[tile_r][ld_out] (columns >= n_idx left as zero)."""
    src = _flat_buffer(src)
    idx = np.ascontiguousarray(idx, np.int32)
    n = idx.size
    ld_out = n if ld_out is None else ld_out
    out = np.zeros((tile_r, ld_out), src.dtype)
    padb = _pad_bits(pad, src.dtype)
    _load().oracle_gather_cols(_es(src), _p(src), rows, cols, ld_src, _p(idx), n, row_offset, col_offset, tile_r,
                               _p(out), ld_out, _p(padb))
    return out


def scatter_rows_masked(dst, rows, cols, ld_dst, idx, src, ld_src, tile_c, row_offset=0, col_offset=0,
                        mask=None, ld_mask=None):
    """Masked row scatter into ``dst`` (in place)."""
    dst, src = _flat_buffer(dst), _flat_buffer(src)
    assert dst.dtype == src.dtype
    idx = np.ascontiguousarray(idx, np.int32)
    if mask is not None:
        mask = _flat_buffer(np.asarray(mask, np.uint8))
        ld_mask = tile_c if ld_mask is None else ld_mask
    _load().oracle_scatter_rows_masked(_es(dst), _p(dst), rows, cols, ld_dst, _p(idx), idx.size, row_offset,
                                       col_offset, _p(src), ld_src, tile_c, _p(mask), ld_mask or 0)
    return dst


def ragged_tile_load(x, total_rows, heads, depth, ld_row, ld_head, cu_seqlens, t_pad):
    """Ragged 3D load; returns dense [batch][heads][t_pad][depth]."""
    x = _flat_buffer(x)
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    batch = cu.size - 1
    out = np.empty((batch, heads, t_pad, depth), x.dtype)
    _load().oracle_ragged_tile_load(_es(x), _p(x), total_rows, heads, depth, ld_row, ld_head, _p(cu), batch,
                                    t_pad, _p(out))
    return out


def scatter_add_rows(dst, rows, cols, ld_dst, idx, src, ld_src, tile_c, row_offset=0, col_offset=0, kind=None):
    """Row scatter-add into ``dst`` (in place).  kind: 'f32', 'bf16' or 'f16' (2-byte arrays
    default to bf16)."""
    dst, src = _flat_buffer(dst), _flat_buffer(src)
    assert dst.dtype == src.dtype
    if kind is None:
        kind = "f32" if dst.dtype.itemsize == 4 else "bf16"
    code = {"f32": 4, "bf16": 2, "f16": 3}[kind]
    idx = np.ascontiguousarray(idx, np.int32)
    _load().oracle_scatter_add_rows(code, _p(dst), rows, cols, ld_dst, _p(idx), idx.size, row_offset, col_offset,
                                    _p(src), ld_src, tile_c)
    return dst


def ragged_tile_store(tiles, x, total_rows, ld_row, ld_head, cu_seqlens):
    """Ragged 3D store of dense tiles [batch][heads][t_pad][depth] into packed ``x`` (in place)."""
    tiles, x = _flat_buffer(tiles), _flat_buffer(x)
    assert tiles.dtype == x.dtype and tiles.ndim == 4
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    batch, heads, t_pad, depth = tiles.shape
    assert batch == cu.size - 1
    _load().oracle_ragged_tile_store(_es(x), _p(tiles), batch, heads, depth, t_pad, _p(cu), _p(x), total_rows,
                                     ld_row, ld_head)
    return x


def gemm_f64(A, lda, B, ldb, M, N, K):
    """C = A.B in double from bf16 bit arrays; returns (M, N) float64."""
    A = _flat_buffer(np.ascontiguousarray(A, np.uint16))
    B = _flat_buffer(np.ascontiguousarray(B, np.uint16))
    C = np.empty((M, N), np.float64)
    _load().oracle_gemm_f64(_p(A), lda, _p(B), ldb, M, N, K, _p(C), N)
    return C


def gemm_f64_at(A, lda, B, ldb, K, ms, ns):
    """C[m, n] in double at the listed positions."""
    A = _flat_buffer(np.ascontiguousarray(A, np.uint16))
    B = _flat_buffer(np.ascontiguousarray(B, np.uint16))
    ms = np.ascontiguousarray(ms, np.int64)
    ns = np.ascontiguousarray(ns, np.int64)
    out = np.empty(ms.size, np.float64)
    _load().oracle_gemm_f64_at(_p(A), lda, _p(B), ldb, K, _p(ms), _p(ns), ms.size, _p(out))
    return out


LOWP_FORMATS = {"e4m3": 0, "e5m2": 1, "e8m0": 2, "e2m1": 3}


def fp8_decode(fmt: str, code: int) -> float:
    """Value of one code of a low-precision format (E2M1: the low 4 bits)."""
    return float(_load().oracle_fp8_decode(LOWP_FORMATS[fmt], code))


def gemm_block_scaled_f64(A, lda, SA, ldsa, B, ldb, SB, ldsb, M, N, K, block, afmt="e4m3", bfmt="e4m3",
                          sfmt="e8m0", acc=None, ld_acc=0):
    """(A .* scale_a)(B .* scale_b) + acc in double from raw codes; returns (M, N) float64.

    A, B: uint8 buffers of codes (E2M1: two per byte, even element in the low
    nibble, element index row * ld + col).  acc: optional float32 buffer."""
    arrs = [_flat_buffer(np.ascontiguousarray(x, np.uint8)) for x in (A, SA, B, SB)]
    accp = None
    if acc is not None:
        acc = _flat_buffer(np.ascontiguousarray(acc, np.float32))
        accp = _p(acc)
    C = np.empty((M, N), np.float64)
    _load().oracle_gemm_block_scaled_f64(LOWP_FORMATS[afmt], LOWP_FORMATS[bfmt], LOWP_FORMATS[sfmt], _p(arrs[0]),
                                         lda, _p(arrs[1]), ldsa, _p(arrs[2]), ldb, _p(arrs[3]), ldsb, accp, ld_acc,
                                         M, N, K, block, _p(C), N)
    return C


def bf16_rne(x: float) -> int:
    return int(_load().oracle_bf16_rne(float(x)))


def round_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_round_bf16(_p(x), x.size, _p(out))
    return out
