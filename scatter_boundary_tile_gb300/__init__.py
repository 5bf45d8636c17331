"""Python binding of libsbt.so (bounds-checked tile movement and the boundary-tile GEMM).

Argument marshalling only: every op runs in the library's CUDA kernels on the
caller's current torch stream.  torch supplies device memory and streams.
There is no fallback: if ``libsbt.so`` is missing or fails to load, importing
an op raises.

Op names match the C ABI in ``include/sbt.h`` without the ``sbt_`` prefix:
``tile_load_padded``, ``tile_store_clipped``, ``gather_rows``, ``gather_cols``,
``scatter_rows_masked``, ``scatter_add_rows``, ``ragged_tile_load``, ``ragged_tile_store``, ``gemm_bounded`` (plus
``gemm_bounded_workspace_size``), ``gemm_bounded_noalloc``, ``gemm_block_scaled`` (plus
``gemm_block_scaled_workspace_size``).  Arrays are torch tensors on the device
(only their data pointer is used; shapes and strides are the explicit
arguments, in elements).
"""
from __future__ import annotations

import ctypes
import os
import struct
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsbt.so")

SBT_OK, SBT_ERR_INVALID_ARG, SBT_ERR_UNSUPPORTED, SBT_ERR_ALIGNMENT = 0, 1, 2, 3
SBT_ERR_TENSOR_MAP, SBT_ERR_CUDA, SBT_ERR_DEVICE_TIMEOUT = 4, 5, 6
STATUS_NAMES = {0: "SBT_OK", 1: "SBT_ERR_INVALID_ARG", 2: "SBT_ERR_UNSUPPORTED", 3: "SBT_ERR_ALIGNMENT",
                4: "SBT_ERR_TENSOR_MAP", 5: "SBT_ERR_CUDA", 6: "SBT_ERR_DEVICE_TIMEOUT"}
SBT_F32, SBT_BF16, SBT_F16 = 0, 1, 2
PATHS = {"auto": 0, "scalar": 1, "vector": 2, "tma": 3}

# Every symbol include/sbt.h declares.
EXPORTS = ("sbt_create", "sbt_destroy", "sbt_set_path", "sbt_set_wait_limit_ns", "sbt_set_test_hook", "sbt_launch_count",
           "sbt_check_status", "sbt_last_error_message", "sbt_tile_load_padded", "sbt_tile_store_clipped",
           "sbt_gather_rows", "sbt_gather_cols", "sbt_scatter_rows_masked", "sbt_scatter_add_rows", "sbt_ragged_tile_load", "sbt_ragged_tile_store", "sbt_gemm_bounded_workspace_size",
           "sbt_gemm_bounded", "sbt_gemm_block_scaled_workspace_size", "sbt_gemm_block_scaled",
           "sbt_gemm_bounded_noalloc")
LOWP_FORMATS = {"e4m3": 0, "e5m2": 1, "e8m0": 2, "e2m1": 3}  # sbt_lowp_format
GEMM_NOALLOC_SCRATCH_BYTES = 16 << 20  # SBT_GEMM_NOALLOC_SCRATCH_BYTES in include/sbt.h


class SbtError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH):
    """Load libsbt.so and declare its signatures (no CUDA call is made)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libsbt.so not built ({path}); run `python -m scatter_boundary_tile_gb300._build`")
        lib = ctypes.CDLL(path)
        p, i64, i32, u64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_int
        sig = {
            "sbt_create": [ci, ctypes.POINTER(p)],
            "sbt_destroy": [p],
            "sbt_set_path": [p, ci],
            "sbt_set_wait_limit_ns": [p, u64],
            "sbt_set_test_hook": [p, ci],
            "sbt_check_status": [p, p],
            "sbt_tile_load_padded": [p, ci, p, i64, i64, i64, i64, i64, i64, i64, i64, i32, i32, i32, i32, p, p, p],
            "sbt_tile_store_clipped": [p, ci, p, i32, i32, i32, i32, p, i64, i64, i64, i64, i64, i64, i64, i64, p],
            "sbt_gather_rows": [p, ci, p, i64, i64, i64, p, i64, i64, i64, i32, p, i64, p, i64, p, p],
            "sbt_scatter_rows_masked": [p, ci, p, i64, i64, i64, p, i64, i64, i64, p, i64, i32, p, i64, p],
            "sbt_gather_cols": [p, ci, p, i64, i64, i64, p, i64, i64, i64, i32, p, i64, p, p],
            "sbt_scatter_add_rows": [p, ci, p, i64, i64, i64, p, i64, i64, i64, p, i64, i32, p],
            "sbt_ragged_tile_load": [p, ci, p, i64, i32, i32, i64, i64, p, i32, i32, p, p],
            "sbt_ragged_tile_store": [p, ci, p, i32, i32, i32, i32, p, p, i64, i64, i64, p],
            "sbt_gemm_bounded_workspace_size": [p, i64, i64, i64, i64, i64, ctypes.POINTER(ctypes.c_size_t)],
            "sbt_gemm_bounded": [p, p, i64, p, i64, p, i64, ci, i64, i64, i64, p, ctypes.c_size_t, p],
            "sbt_gemm_bounded_noalloc": [p, p, i64, p, i64, p, i64, ci, i64, i64, i64, p],
            "sbt_gemm_block_scaled_workspace_size": [p, i64, i64, i64, ctypes.POINTER(ctypes.c_size_t)],
            "sbt_gemm_block_scaled": [p, ci, p, i64, ci, p, i64, ci, p, i64, p, i64, i64, p, i64, p, i64, i64, i64,
                                      i64, p, ctypes.c_size_t, p],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ci
        lib.sbt_launch_count.argtypes = [p]
        lib.sbt_launch_count.restype = u64
        lib.sbt_last_error_message.argtypes = []
        lib.sbt_last_error_message.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int):
    if status != SBT_OK:
        msg = load_library().sbt_last_error_message().decode(errors="replace")
        raise SbtError(status, msg)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t, dtype):
    if dtype is not None:
        return {"f32": SBT_F32, "bf16": SBT_BF16, "f16": SBT_F16}[dtype] if isinstance(dtype, str) else int(dtype)
    import torch
    if t.dtype == torch.float16:
        return SBT_F16
    return {4: SBT_F32, 2: SBT_BF16}[t.element_size()]


def _pad_bytes(pad, code):
    """One element's bits: an int is taken as raw bits, a float is converted to the dtype."""
    if pad is None:
        return None
    if isinstance(pad, (bytes, bytearray)):
        return ctypes.create_string_buffer(bytes(pad), len(pad))
    if code == SBT_F32:
        raw = struct.pack("<I", pad & 0xFFFFFFFF) if isinstance(pad, int) else struct.pack("<f", pad)
    else:
        if isinstance(pad, int):
            raw = struct.pack("<H", pad & 0xFFFF)
        else:
            import torch
            tdt = torch.bfloat16 if code == SBT_BF16 else torch.float16
            bits = torch.tensor([float(pad)], dtype=torch.float32).to(tdt).view(torch.int16).item()
            raw = struct.pack("<H", bits & 0xFFFF)
    return ctypes.create_string_buffer(raw, len(raw))


class Context:
    """An ``sbt_context`` bound to one CUDA device."""

    def __init__(self, device: int = 0):
        lib = load_library()
        h = ctypes.c_void_p()
        _check(lib.sbt_create(device, ctypes.byref(h)))
        self._h = h
        self.device = device

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            load_library().sbt_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_path(self, path: str):
        _check(load_library().sbt_set_path(self._h, PATHS[path]))

    def set_wait_limit_ns(self, ns: int):
        _check(load_library().sbt_set_wait_limit_ns(self._h, ns))

    def set_test_hook(self, withhold_load: bool):
        """Test only: make the next GEMM / bulk row launches withhold their first copy."""
        _check(load_library().sbt_set_test_hook(self._h, 1 if withhold_load else 0))

    @property
    def launch_count(self) -> int:
        return int(load_library().sbt_launch_count(self._h))

    def check_status(self, stream=None):
        _check(load_library().sbt_check_status(self._h, _stream(stream)))


def tile_load_padded(ctx, src, rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c, grid_r, grid_c,
                     tile_r, tile_c, dst_tiles, pad=None, dtype=None, stream=None):
    code = _dtype_code(dst_tiles, dtype)
    _check(load_library().sbt_tile_load_padded(ctx.handle, code, _ptr(src), rows, cols, stride_r, stride_c, origin_r,
                                               origin_c, step_r, step_c, grid_r, grid_c, tile_r, tile_c,
                                               _ptr(dst_tiles), _pad_bytes(pad, code), _stream(stream)))


def tile_store_clipped(ctx, src_tiles, grid_r, grid_c, tile_r, tile_c, dst, rows, cols, stride_r, stride_c, origin_r,
                       origin_c, step_r, step_c, dtype=None, stream=None):
    code = _dtype_code(src_tiles, dtype)
    _check(load_library().sbt_tile_store_clipped(ctx.handle, code, _ptr(src_tiles), grid_r, grid_c, tile_r, tile_c,
                                                 _ptr(dst), rows, cols, stride_r, stride_c, origin_r, origin_c,
                                                 step_r, step_c, _stream(stream)))


def gather_rows(ctx, src, rows, cols, ld_src, idx, n_idx, out, ld_out, tile_c, row_offset=0, col_offset=0,
                mask=None, ld_mask=0, pad=None, dtype=None, stream=None):
    code = _dtype_code(out, dtype)
    _check(load_library().sbt_gather_rows(ctx.handle, code, _ptr(src), rows, cols, ld_src, _ptr(idx), n_idx,
                                          row_offset, col_offset, tile_c, _ptr(mask), ld_mask, _ptr(out), ld_out,
                                          _pad_bytes(pad, code), _stream(stream)))


def gather_cols(ctx, src, rows, cols, ld_src, idx, n_idx, out, ld_out, tile_r, row_offset=0, col_offset=0, pad=None,
                dtype=None, stream=None):
    code = _dtype_code(out, dtype)
    _check(load_library().sbt_gather_cols(ctx.handle, code, _ptr(src), rows, cols, ld_src, _ptr(idx), n_idx, row_offset,
                                          col_offset, tile_r, _ptr(out), ld_out, _pad_bytes(pad, code),
                                          _stream(stream)))


def scatter_rows_masked(ctx, dst, rows, cols, ld_dst, idx, n_idx, src, ld_src, tile_c, row_offset=0, col_offset=0,
                        mask=None, ld_mask=0, dtype=None, stream=None):
    code = _dtype_code(dst, dtype)
    _check(load_library().sbt_scatter_rows_masked(ctx.handle, code, _ptr(dst), rows, cols, ld_dst, _ptr(idx), n_idx,
                                                  row_offset, col_offset, _ptr(src), ld_src, tile_c, _ptr(mask),
                                                  ld_mask, _stream(stream)))


def scatter_add_rows(ctx, dst, rows, cols, ld_dst, idx, n_idx, src, ld_src, tile_c, row_offset=0, col_offset=0,
                     dtype=None, stream=None):
    code = _dtype_code(dst, dtype)
    _check(load_library().sbt_scatter_add_rows(ctx.handle, code, _ptr(dst), rows, cols, ld_dst, _ptr(idx), n_idx,
                                               row_offset, col_offset, _ptr(src), ld_src, tile_c, _stream(stream)))


def ragged_tile_load(ctx, x, total_rows, heads, depth, ld_row, ld_head, cu_seqlens, batch, t_pad, out, dtype=None,
                     stream=None):
    code = _dtype_code(out, dtype)
    _check(load_library().sbt_ragged_tile_load(ctx.handle, code, _ptr(x), total_rows, heads, depth, ld_row, ld_head,
                                               _ptr(cu_seqlens), batch, t_pad, _ptr(out), _stream(stream)))


def ragged_tile_store(ctx, tiles, batch, heads, depth, t_pad, cu_seqlens, x, total_rows, ld_row, ld_head, dtype=None,
                      stream=None):
    code = _dtype_code(tiles, dtype)
    _check(load_library().sbt_ragged_tile_store(ctx.handle, code, _ptr(tiles), batch, heads, depth, t_pad,
                                                _ptr(cu_seqlens), _ptr(x), total_rows, ld_row, ld_head,
                                                _stream(stream)))


def gemm_bounded_workspace_size(ctx, M, N, K, lda, ldb) -> int:
    n = ctypes.c_size_t()
    _check(load_library().sbt_gemm_bounded_workspace_size(ctx.handle, M, N, K, lda, ldb, ctypes.byref(n)))
    return int(n.value)


def gemm_bounded(ctx, A, lda, B, ldb, C, ldc, M, N, K, workspace=None, workspace_bytes=0, c_dtype="bf16",
                 stream=None):
    code = {"bf16": SBT_BF16, "f32": SBT_F32}[c_dtype] if isinstance(c_dtype, str) else int(c_dtype)
    _check(load_library().sbt_gemm_bounded(ctx.handle, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, code, M, N, K,
                                           _ptr(workspace), workspace_bytes, _stream(stream)))


def gemm_block_scaled_workspace_size(ctx, M, N, K) -> int:
    n = ctypes.c_size_t()
    _check(load_library().sbt_gemm_block_scaled_workspace_size(ctx.handle, M, N, K, ctypes.byref(n)))
    return int(n.value)


def gemm_block_scaled(ctx, A, lda, B, ldb, a_scale, ld_sa, b_scale, ld_sb, K_s, D, ldd, M, N, K, acc=None, ld_acc=0,
                      workspace=None, workspace_bytes=0, a_fmt="e4m3", b_fmt="e4m3", s_fmt="e8m0", stream=None):
    """sbt_gemm_block_scaled: D = (A .* a_scale)(B .* b_scale) + acc; formats by name (see LOWP_FORMATS)."""
    fmt = lambda f: LOWP_FORMATS[f] if isinstance(f, str) else int(f)
    _check(load_library().sbt_gemm_block_scaled(ctx.handle, fmt(a_fmt), _ptr(A), lda, fmt(b_fmt), _ptr(B), ldb,
                                                fmt(s_fmt), _ptr(a_scale), ld_sa, _ptr(b_scale), ld_sb, K_s,
                                                _ptr(acc), ld_acc, _ptr(D), ldd, M, N, K, _ptr(workspace),
                                                workspace_bytes, _stream(stream)))


def gemm_bounded_noalloc(ctx, A, lda, B, ldb, C, ldc, M, N, K, c_dtype="bf16", stream=None):
    """sbt_gemm_bounded_noalloc: the bounded GEMM with the library's fixed staging scratch.

    For callers that cannot allocate device memory at the call: plugins
    confined to another framework's memory pool, code under a device-memory
    budget committed up front, or paths that cannot take cudaMalloc's implicit
    synchronisation.  Shapes needing more than GEMM_NOALLOC_SCRATCH_BYTES of
    staging are rejected; calls that may overlap on the GPU race on the shared
    scratch.
    """
    code = {"bf16": SBT_BF16, "f32": SBT_F32}[c_dtype] if isinstance(c_dtype, str) else int(c_dtype)
    _check(load_library().sbt_gemm_bounded_noalloc(ctx.handle, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, code, M, N,
                                                   K, _stream(stream)))
