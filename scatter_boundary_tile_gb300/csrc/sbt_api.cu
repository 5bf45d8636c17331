// C ABI of libsbt.so: context, argument validation and dispatch.
// Every check here runs before any launch; a failing call launches nothing.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <string>

#include <algorithm>

#include "sbt_internal.cuh"

// Per-device status flag set by kernels whose bounded waits ran out.
__device__ unsigned int g_sbt_status_flag;

static thread_local std::string t_last_error;

sbt_status sbt_fail(sbt_status st, const std::string& msg) {
    t_last_error = msg;
    return st;
}

sbt_status sbt_ok() { return SBT_OK; }

sbt_status sbt_cuda_check(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return SBT_OK;
    return sbt_fail(SBT_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

sbt_status sbt_use_device(sbt_context* ctx) { return sbt_cuda_check(cudaSetDevice(ctx->device), "cudaSetDevice"); }

uint32_t sbt_pad_word(const void* pad, int es) {
    if (!pad) return 0u;
    if (es == 4) {
        uint32_t w;
        memcpy(&w, pad, 4);
        return w;
    }
    uint16_t h;
    memcpy(&h, pad, 2);
    return (uint32_t)h | ((uint32_t)h << 16);
}

int sbt_persistent_grid(const sbt_context* ctx, const void* kernel, int threads, size_t smem, int64_t work_units) {
    int per_sm = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    int64_t g = (int64_t)ctx->sm_count * per_sm;
    if (work_units < g) g = work_units;
    return (int)(g < 1 ? 1 : g);
}

sbt_status sbt_after_launch(sbt_context* ctx, const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return sbt_fail(SBT_ERR_CUDA, std::string(what) + " launch: " + cudaGetErrorString(e));
    ctx->launches++;
    return SBT_OK;
}

#define SBT_REQUIRE(cond, msg)                                          \
    do {                                                                \
        if (!(cond)) return sbt_fail(SBT_ERR_INVALID_ARG, (msg));       \
    } while (0)

// Every array starts on a multiple of its element size (int32 indices and
// cu_seqlens on 4 bytes): the kernels' element accesses are naturally aligned,
// so a pointer that is not is refused here, before anything touches the device.
#define SBT_REQUIRE_ALIGNED(ptr, bytes, msg)                                                    \
    do {                                                                                        \
        if ((reinterpret_cast<uintptr_t>(ptr) % (uintptr_t)(bytes)) != 0)                       \
            return sbt_fail(SBT_ERR_ALIGNMENT, (msg));                                          \
    } while (0)

extern "C" {

const char* sbt_last_error_message(void) { return t_last_error.c_str(); }

sbt_status sbt_create(int device, sbt_context** out) {
    if (!out) return sbt_fail(SBT_ERR_INVALID_ARG, "sbt_create: out is NULL");
    *out = nullptr;
    int n = 0;
    sbt_status st = sbt_cuda_check(cudaGetDeviceCount(&n), "cudaGetDeviceCount");
    if (st) return st;
    if (device < 0 || device >= n) return sbt_fail(SBT_ERR_INVALID_ARG, "sbt_create: no such device");
    if ((st = sbt_cuda_check(cudaSetDevice(device), "cudaSetDevice"))) return st;
    sbt_context* c = new sbt_context();
    c->device = device;
    cudaDeviceProp prop;
    if ((st = sbt_cuda_check(cudaGetDeviceProperties(&prop, device), "cudaGetDeviceProperties"))) {
        delete c;
        return st;
    }
    c->sm_count = prop.multiProcessorCount;
    c->cc_major = prop.major;
    c->cc_minor = prop.minor;
    c->smem_optin = prop.sharedMemPerBlockOptin;
    if (!(prop.major == 10 && prop.minor == 3)) {
        delete c;
        return sbt_fail(SBT_ERR_UNSUPPORTED, "sbt_create: libsbt is built for sm_103a (compute capability 10.3)");
    }
    void* flag = nullptr;
    if ((st = sbt_cuda_check(cudaGetSymbolAddress(&flag, g_sbt_status_flag), "cudaGetSymbolAddress(status)"))) {
        delete c;
        return st;
    }
    c->status = (unsigned int*)flag;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if ((st = sbt_cuda_check(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                              cudaEnableDefault, &q),
                             "cudaGetDriverEntryPointByVersion")) ||
        q != cudaDriverEntryPointSuccess || !fn) {
        delete c;
        return st ? st : sbt_fail(SBT_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
    }
    c->encode_tiled = (sbt_encode_tiled_fn)fn;
    *out = c;
    return SBT_OK;
}

sbt_status sbt_destroy(sbt_context* ctx) {
    delete ctx;
    return SBT_OK;
}

sbt_status sbt_set_path(sbt_context* ctx, sbt_path path) {
    if (!ctx) return sbt_fail(SBT_ERR_INVALID_ARG, "ctx is NULL");
    if (path < SBT_PATH_AUTO || path > SBT_PATH_TMA) return sbt_fail(SBT_ERR_INVALID_ARG, "unknown path");
    ctx->path = path;
    return SBT_OK;
}

sbt_status sbt_set_wait_limit_ns(sbt_context* ctx, uint64_t ns) {
    if (!ctx) return sbt_fail(SBT_ERR_INVALID_ARG, "ctx is NULL");
    if (ns == 0) return sbt_fail(SBT_ERR_INVALID_ARG, "wait limit must be positive");
    ctx->wait_limit_ns = ns;
    return SBT_OK;
}

sbt_status sbt_set_test_hook(sbt_context* ctx, sbt_test_hook hook) {
    if (!ctx) return sbt_fail(SBT_ERR_INVALID_ARG, "ctx is NULL");
    if (hook != SBT_TEST_NONE && hook != SBT_TEST_WITHHOLD_LOAD) return sbt_fail(SBT_ERR_INVALID_ARG, "unknown test hook");
    ctx->test_hook = hook;
    return SBT_OK;
}

uint64_t sbt_launch_count(const sbt_context* ctx) { return ctx ? ctx->launches : 0; }

sbt_status sbt_check_status(sbt_context* ctx, void* stream) {
    if (!ctx) return sbt_fail(SBT_ERR_INVALID_ARG, "ctx is NULL");
    sbt_status st = sbt_use_device(ctx);
    if (st) return st;
    if ((st = sbt_cuda_check(cudaStreamSynchronize((cudaStream_t)stream), "cudaStreamSynchronize"))) return st;
    unsigned int flag = 0, zero = 0;
    if ((st = sbt_cuda_check(cudaMemcpy(&flag, ctx->status, 4, cudaMemcpyDeviceToHost), "read status"))) return st;
    if (flag) {
        if ((st = sbt_cuda_check(cudaMemcpy(ctx->status, &zero, 4, cudaMemcpyHostToDevice), "clear status")))
            return st;
        return sbt_fail(SBT_ERR_DEVICE_TIMEOUT, "a bounded device-side wait ran out (code " + std::to_string(flag) + ")");
    }
    return SBT_OK;
}

static sbt_status check_dtype_move(sbt_dtype dtype, int* es) {
    *es = sbt_dtype_size(dtype);
    if (*es != 2 && *es != 4) return sbt_fail(SBT_ERR_UNSUPPORTED, "unsupported dtype");
    return SBT_OK;
}

sbt_status sbt_tile_load_padded(sbt_context* ctx, sbt_dtype dtype, const void* src, int64_t rows, int64_t cols,
                                int64_t stride_r, int64_t stride_c, int64_t origin_r, int64_t origin_c,
                                int64_t step_r, int64_t step_c, int32_t grid_r, int32_t grid_c, int32_t tile_r,
                                int32_t tile_c, void* dst_tiles, const void* pad_value, void* stream) {
    SBT_REQUIRE(ctx, "ctx is NULL");
    int es;
    sbt_status st = check_dtype_move(dtype, &es);
    if (st) return st;
    SBT_REQUIRE(rows >= 0 && cols >= 0, "tile_load_padded: negative extent");
    SBT_REQUIRE(grid_r >= 0 && grid_c >= 0, "tile_load_padded: negative grid");
    SBT_REQUIRE(tile_r >= 1 && tile_r <= 256 && tile_c >= 1 && tile_c <= 256, "tile_load_padded: tile dims must be in [1, 256]");
    if ((int64_t)grid_r * grid_c == 0) return SBT_OK;
    SBT_REQUIRE(dst_tiles, "tile_load_padded: dst_tiles is NULL");
    SBT_REQUIRE(stride_r != 0 && stride_c != 0, "tile_load_padded: strides must be nonzero");
    SBT_REQUIRE(rows * cols == 0 || src, "tile_load_padded: src is NULL");
    SBT_REQUIRE_ALIGNED(src, es, "tile_load_padded: src is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(dst_tiles, es, "tile_load_padded: dst_tiles is not aligned to its element size");
    if ((st = sbt_use_device(ctx))) return st;
    return sbt_launch_tile_load(ctx, es, src, rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c,
                                grid_r, grid_c, tile_r, tile_c, dst_tiles, sbt_pad_word(pad_value, es),
                                (cudaStream_t)stream);
}

sbt_status sbt_tile_store_clipped(sbt_context* ctx, sbt_dtype dtype, const void* src_tiles, int32_t grid_r,
                                  int32_t grid_c, int32_t tile_r, int32_t tile_c, void* dst, int64_t rows,
                                  int64_t cols, int64_t stride_r, int64_t stride_c, int64_t origin_r,
                                  int64_t origin_c, int64_t step_r, int64_t step_c, void* stream) {
    SBT_REQUIRE(ctx, "ctx is NULL");
    int es;
    sbt_status st = check_dtype_move(dtype, &es);
    if (st) return st;
    SBT_REQUIRE(rows >= 0 && cols >= 0, "tile_store_clipped: negative extent");
    SBT_REQUIRE(grid_r >= 0 && grid_c >= 0, "tile_store_clipped: negative grid");
    SBT_REQUIRE(tile_r >= 1 && tile_r <= 256 && tile_c >= 1 && tile_c <= 256, "tile_store_clipped: tile dims must be in [1, 256]");
    if ((int64_t)grid_r * grid_c == 0 || rows * cols == 0) return SBT_OK;
    SBT_REQUIRE(src_tiles && dst, "tile_store_clipped: NULL pointer");
    SBT_REQUIRE(stride_r != 0 && stride_c != 0, "tile_store_clipped: strides must be nonzero");
    SBT_REQUIRE_ALIGNED(src_tiles, es, "tile_store_clipped: src_tiles is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(dst, es, "tile_store_clipped: dst is not aligned to its element size");
    if ((st = sbt_use_device(ctx))) return st;
    if (sbt_tile_store_runs_ok(ctx, es, src_tiles, grid_r, grid_c, tile_r, tile_c, dst, stride_r, stride_c, origin_c,
                               step_c))
        return sbt_launch_tile_store_runs(ctx, es, src_tiles, grid_r, grid_c, tile_r, tile_c, dst, rows, cols,
                                          stride_r, origin_r, origin_c, step_r, (cudaStream_t)stream);
    return sbt_launch_tile_store(ctx, es, src_tiles, grid_r, grid_c, tile_r, tile_c, dst, rows, cols, stride_r,
                                 stride_c, origin_r, origin_c, step_r, step_c, (cudaStream_t)stream);
}

sbt_status sbt_gather_rows(sbt_context* ctx, sbt_dtype dtype, const void* src, int64_t rows, int64_t cols,
                           int64_t ld_src, const int32_t* idx, int64_t n_idx, int64_t row_offset,
                           int64_t col_offset, int32_t tile_c, const uint8_t* mask, int64_t ld_mask, void* out,
                           int64_t ld_out, const void* pad_value, void* stream) {
    SBT_REQUIRE(ctx, "ctx is NULL");
    int es;
    sbt_status st = check_dtype_move(dtype, &es);
    if (st) return st;
    SBT_REQUIRE(rows >= 0 && cols >= 0 && n_idx >= 0, "gather_rows: negative extent");
    SBT_REQUIRE(tile_c >= 1 && tile_c <= 65536, "gather_rows: tile_c must be in [1, 65536]");
    SBT_REQUIRE(ld_out >= tile_c, "gather_rows: ld_out < tile_c");
    if (n_idx == 0) return SBT_OK;
    SBT_REQUIRE(idx && out, "gather_rows: NULL idx or out");
    SBT_REQUIRE(rows * cols == 0 || src, "gather_rows: src is NULL");
    SBT_REQUIRE(rows * cols == 0 || ld_src >= cols, "gather_rows: ld_src < cols");
    SBT_REQUIRE(!mask || ld_mask >= tile_c, "gather_rows: ld_mask < tile_c");
    SBT_REQUIRE_ALIGNED(src, es, "gather_rows: src is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(out, es, "gather_rows: out is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(idx, 4, "gather_rows: idx is not 4-byte aligned");
    if ((st = sbt_use_device(ctx))) return st;
    return sbt_launch_gather(ctx, es, src, rows, cols, ld_src, idx, n_idx, row_offset, col_offset, tile_c, mask,
                             ld_mask, out, ld_out, sbt_pad_word(pad_value, es), (cudaStream_t)stream);
}

sbt_status sbt_gather_cols(sbt_context* ctx, sbt_dtype dtype, const void* src, int64_t rows, int64_t cols,
                           int64_t ld_src, const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                           int32_t tile_r, void* out, int64_t ld_out, const void* pad_value, void* stream) {
    SBT_REQUIRE(ctx, "ctx is NULL");
    int es;
    sbt_status st = check_dtype_move(dtype, &es);
    if (st) return st;
    SBT_REQUIRE(rows >= 0 && cols >= 0 && n_idx >= 0, "gather_cols: negative extent");
    SBT_REQUIRE(tile_r >= 1 && tile_r <= 65536, "gather_cols: tile_r must be in [1, 65536]");
    SBT_REQUIRE(ld_out >= n_idx, "gather_cols: ld_out < n_idx");
    if (n_idx == 0) return SBT_OK;
    SBT_REQUIRE(idx && out, "gather_cols: NULL idx or out");
    SBT_REQUIRE(rows * cols == 0 || src, "gather_cols: src is NULL");
    SBT_REQUIRE(rows * cols == 0 || ld_src >= cols, "gather_cols: ld_src < cols");
    SBT_REQUIRE_ALIGNED(src, es, "gather_cols: src is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(out, es, "gather_cols: out is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(idx, 4, "gather_cols: idx is not 4-byte aligned");
    if ((st = sbt_use_device(ctx))) return st;
    return sbt_launch_gather_cols(ctx, es, src, rows, cols, ld_src, idx, n_idx, row_offset, col_offset, tile_r, out,
                                  ld_out, sbt_pad_word(pad_value, es), (cudaStream_t)stream);
}

sbt_status sbt_scatter_rows_masked(sbt_context* ctx, sbt_dtype dtype, void* dst, int64_t rows, int64_t cols,
                                   int64_t ld_dst, const int32_t* idx, int64_t n_idx, int64_t row_offset,
                                   int64_t col_offset, const void* src, int64_t ld_src, int32_t tile_c,
                                   const uint8_t* mask, int64_t ld_mask, void* stream) {
    SBT_REQUIRE(ctx, "ctx is NULL");
    int es;
    sbt_status st = check_dtype_move(dtype, &es);
    if (st) return st;
    SBT_REQUIRE(rows >= 0 && cols >= 0 && n_idx >= 0, "scatter_rows_masked: negative extent");
    SBT_REQUIRE(tile_c >= 1 && tile_c <= 65536, "scatter_rows_masked: tile_c must be in [1, 65536]");
    if (n_idx == 0 || rows * cols == 0) return SBT_OK;
    SBT_REQUIRE(dst && idx && src, "scatter_rows_masked: NULL pointer");
    SBT_REQUIRE(ld_dst >= cols, "scatter_rows_masked: ld_dst < cols");
    SBT_REQUIRE(ld_src >= tile_c, "scatter_rows_masked: ld_src < tile_c");
    SBT_REQUIRE(!mask || ld_mask >= tile_c, "scatter_rows_masked: ld_mask < tile_c");
    SBT_REQUIRE_ALIGNED(dst, es, "scatter_rows_masked: dst is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(src, es, "scatter_rows_masked: src is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(idx, 4, "scatter_rows_masked: idx is not 4-byte aligned");
    if ((st = sbt_use_device(ctx))) return st;
    return sbt_launch_scatter(ctx, es, dst, rows, cols, ld_dst, idx, n_idx, row_offset, col_offset, src, ld_src,
                              tile_c, mask, ld_mask, (cudaStream_t)stream);
}

sbt_status sbt_ragged_tile_load(sbt_context* ctx, sbt_dtype dtype, const void* x, int64_t total_rows, int32_t heads,
                                int32_t depth, int64_t ld_row, int64_t ld_head, const int32_t* cu_seqlens,
                                int32_t batch, int32_t t_pad, void* out, void* stream) {
    SBT_REQUIRE(ctx, "ctx is NULL");
    int es;
    sbt_status st = check_dtype_move(dtype, &es);
    if (st) return st;
    SBT_REQUIRE(total_rows >= 0 && heads >= 0 && depth >= 0 && batch >= 0 && t_pad >= 0,
                "ragged_tile_load: negative extent");
    if ((int64_t)batch * heads * t_pad * depth == 0) return SBT_OK;
    SBT_REQUIRE(out && cu_seqlens, "ragged_tile_load: NULL out or cu_seqlens");
    SBT_REQUIRE(total_rows == 0 || x, "ragged_tile_load: x is NULL");
    SBT_REQUIRE(ld_row > 0 && ld_head > 0, "ragged_tile_load: strides must be positive");
    SBT_REQUIRE_ALIGNED(x, es, "ragged_tile_load: x is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(out, es, "ragged_tile_load: out is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(cu_seqlens, 4, "ragged_tile_load: cu_seqlens is not 4-byte aligned");
    if ((st = sbt_use_device(ctx))) return st;
    return sbt_launch_ragged(ctx, es, x, total_rows, heads, depth, ld_row, ld_head, cu_seqlens, batch, t_pad, out,
                             (cudaStream_t)stream);
}

sbt_status sbt_scatter_add_rows(sbt_context* ctx, sbt_dtype dtype, void* dst, int64_t rows, int64_t cols,
                                int64_t ld_dst, const int32_t* idx, int64_t n_idx, int64_t row_offset,
                                int64_t col_offset, const void* src, int64_t ld_src, int32_t tile_c, void* stream) {
    SBT_REQUIRE(ctx, "ctx is NULL");
    const int kind = dtype == SBT_F32 ? 4 : dtype == SBT_BF16 ? 2 : dtype == SBT_F16 ? 3 : 0;
    if (!kind) return sbt_fail(SBT_ERR_UNSUPPORTED, "scatter_add_rows: dtype must be SBT_F32, SBT_BF16 or SBT_F16");
    SBT_REQUIRE(rows >= 0 && cols >= 0 && n_idx >= 0, "scatter_add_rows: negative extent");
    SBT_REQUIRE(tile_c >= 1 && tile_c <= 65536, "scatter_add_rows: tile_c must be in [1, 65536]");
    if (n_idx == 0 || rows * cols == 0) return SBT_OK;
    SBT_REQUIRE(dst && idx && src, "scatter_add_rows: NULL pointer");
    SBT_REQUIRE(ld_dst >= cols, "scatter_add_rows: ld_dst < cols");
    SBT_REQUIRE(ld_src >= tile_c, "scatter_add_rows: ld_src < tile_c");
    const int es = kind == 4 ? 4 : 2;
    SBT_REQUIRE_ALIGNED(dst, es, "scatter_add_rows: dst is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(src, es, "scatter_add_rows: src is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(idx, 4, "scatter_add_rows: idx is not 4-byte aligned");
    sbt_status st = sbt_use_device(ctx);
    if (st) return st;
    return sbt_launch_scatter_add(ctx, kind, dst, rows, cols, ld_dst, idx, n_idx, row_offset, col_offset, src, ld_src,
                                  tile_c, (cudaStream_t)stream);
}

sbt_status sbt_ragged_tile_store(sbt_context* ctx, sbt_dtype dtype, const void* tiles, int32_t batch, int32_t heads,
                                 int32_t depth, int32_t t_pad, const int32_t* cu_seqlens, void* x, int64_t total_rows,
                                 int64_t ld_row, int64_t ld_head, void* stream) {
    SBT_REQUIRE(ctx, "ctx is NULL");
    int es;
    sbt_status st = check_dtype_move(dtype, &es);
    if (st) return st;
    SBT_REQUIRE(total_rows >= 0 && heads >= 0 && depth >= 0 && batch >= 0 && t_pad >= 0,
                "ragged_tile_store: negative extent");
    if ((int64_t)batch * heads * t_pad * depth == 0 || total_rows == 0) return SBT_OK;
    SBT_REQUIRE(tiles && cu_seqlens && x, "ragged_tile_store: NULL pointer");
    SBT_REQUIRE(ld_row > 0 && ld_head > 0, "ragged_tile_store: strides must be positive");
    SBT_REQUIRE_ALIGNED(tiles, es, "ragged_tile_store: tiles is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(x, es, "ragged_tile_store: x is not aligned to its element size");
    SBT_REQUIRE_ALIGNED(cu_seqlens, 4, "ragged_tile_store: cu_seqlens is not 4-byte aligned");
    if ((st = sbt_use_device(ctx))) return st;
    return sbt_launch_ragged_store(ctx, es, tiles, batch, heads, depth, t_pad, cu_seqlens, x, total_rows, ld_row,
                                   ld_head, (cudaStream_t)stream);
}

sbt_status sbt_gemm_bounded_workspace_size(sbt_context* ctx, int64_t M, int64_t N, int64_t K, int64_t lda,
                                           int64_t ldb, size_t* bytes) {
    SBT_REQUIRE(ctx && bytes, "NULL argument");
    SBT_REQUIRE(M >= 0 && N >= 0 && K >= 0, "gemm_bounded: negative extent");
    SBT_REQUIRE(lda >= K && ldb >= N, "gemm_bounded: leading dimension smaller than the extent");
    *bytes = sbt_gemm_workspace_bytes(M, N, K);
    return SBT_OK;
}

sbt_status sbt_gemm_bounded(sbt_context* ctx, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                            int64_t ldc, sbt_dtype c_dtype, int64_t M, int64_t N, int64_t K, void* workspace,
                            size_t workspace_bytes, void* stream) {
    SBT_REQUIRE(ctx, "ctx is NULL");
    SBT_REQUIRE(M >= 0 && N >= 0 && K >= 0, "gemm_bounded: negative extent");
    if (c_dtype != SBT_BF16 && c_dtype != SBT_F32)
        return sbt_fail(SBT_ERR_UNSUPPORTED, "gemm_bounded: c_dtype must be SBT_BF16 or SBT_F32");
    SBT_REQUIRE(lda >= K && ldb >= N && ldc >= N, "gemm_bounded: leading dimension smaller than the extent");
    if (M == 0 || N == 0) return SBT_OK;
    SBT_REQUIRE(C, "gemm_bounded: C is NULL");
    SBT_REQUIRE(K == 0 || (A && B), "gemm_bounded: NULL A or B");
    SBT_REQUIRE_ALIGNED(A, 2, "gemm_bounded: A is not 2-byte aligned");
    SBT_REQUIRE_ALIGNED(B, 2, "gemm_bounded: B is not 2-byte aligned");
    SBT_REQUIRE_ALIGNED(C, c_dtype == SBT_F32 ? 4 : 2, "gemm_bounded: C is not aligned to its element size");
    size_t need = sbt_gemm_workspace_bytes(M, N, K);
    if (need > 0) {
        if (!workspace || workspace_bytes < need)
            return sbt_fail(SBT_ERR_ALIGNMENT, "gemm_bounded: workspace smaller than sbt_gemm_bounded_workspace_size()");
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return sbt_fail(SBT_ERR_ALIGNMENT, "gemm_bounded: workspace must be 256-byte aligned");
    }
    sbt_status st = sbt_use_device(ctx);
    if (st) return st;
    return sbt_launch_gemm(ctx, A, lda, B, ldb, C, ldc, c_dtype, M, N, K, workspace, workspace_bytes,
                           (cudaStream_t)stream);
}

static bool is_operand_format(sbt_lowp_format f) {
    return f == SBT_FMT_E4M3 || f == SBT_FMT_E5M2 || f == SBT_FMT_E2M1;
}

sbt_status sbt_gemm_block_scaled_workspace_size(sbt_context* ctx, int64_t M, int64_t N, int64_t K, size_t* bytes) {
    SBT_REQUIRE(ctx && bytes, "NULL argument");
    SBT_REQUIRE(M >= 0 && N >= 0 && K >= 0, "gemm_block_scaled: negative extent");
    *bytes = std::max(sbt_gemm_workspace_bytes(M, N, K), sbt_gemm_mx_workspace_bytes(M, N, K));
    return SBT_OK;
}

sbt_status sbt_gemm_block_scaled(sbt_context* ctx, sbt_lowp_format a_fmt, const void* A, int64_t lda,
                                 sbt_lowp_format b_fmt, const void* B, int64_t ldb, sbt_lowp_format s_fmt,
                                 const void* a_scale, int64_t ld_sa, const void* b_scale, int64_t ld_sb, int64_t K_s,
                                 const float* acc, int64_t ld_acc, float* D, int64_t ldd, int64_t M, int64_t N,
                                 int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
    SBT_REQUIRE(ctx, "ctx is NULL");
    SBT_REQUIRE(M >= 0 && N >= 0 && K >= 0, "gemm_block_scaled: negative extent");
    if (!is_operand_format(a_fmt) || !is_operand_format(b_fmt))
        return sbt_fail(SBT_ERR_UNSUPPORTED, "gemm_block_scaled: operands must be E4M3, E5M2 or E2M1");
    if (s_fmt != SBT_FMT_E8M0 && s_fmt != SBT_FMT_E4M3)
        return sbt_fail(SBT_ERR_UNSUPPORTED, "gemm_block_scaled: scales must be E8M0 or E4M3");
    SBT_REQUIRE(K == 0 || (K_s >= 1 && K % K_s == 0), "gemm_block_scaled: K_s must divide K");
    SBT_REQUIRE(lda >= K && ldb >= N && ldd >= N, "gemm_block_scaled: leading dimension smaller than the extent");
    SBT_REQUIRE(K == 0 || (ld_sa >= K_s && ld_sb >= N), "gemm_block_scaled: scale leading dimension too small");
    SBT_REQUIRE(!acc || ld_acc >= N, "gemm_block_scaled: ld_acc smaller than N");
    SBT_REQUIRE(a_fmt != SBT_FMT_E2M1 || lda % 2 == 0, "gemm_block_scaled: E2M1 A needs an even lda");
    SBT_REQUIRE(b_fmt != SBT_FMT_E2M1 || ldb % 2 == 0, "gemm_block_scaled: E2M1 B needs an even ldb");
    SBT_REQUIRE(!acc || (const void*)acc != (const void*)D || ld_acc == ldd,
                "gemm_block_scaled: acc aliasing D needs ld_acc == ldd");
    if (M == 0 || N == 0) return SBT_OK;
    SBT_REQUIRE(D, "gemm_block_scaled: D is NULL");
    SBT_REQUIRE(K == 0 || (A && B && a_scale && b_scale), "gemm_block_scaled: NULL operand or scale");
    SBT_REQUIRE_ALIGNED(acc, 4, "gemm_block_scaled: acc is not 4-byte aligned");
    SBT_REQUIRE_ALIGNED(D, 4, "gemm_block_scaled: D is not 4-byte aligned");
    const size_t need = std::max(sbt_gemm_workspace_bytes(M, N, K), sbt_gemm_mx_workspace_bytes(M, N, K));
    if (need > 0) {
        if (!workspace || workspace_bytes < need)
            return sbt_fail(SBT_ERR_ALIGNMENT,
                            "gemm_block_scaled: workspace smaller than sbt_gemm_block_scaled_workspace_size()");
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return sbt_fail(SBT_ERR_ALIGNMENT, "gemm_block_scaled: workspace must be 256-byte aligned");
    }
    sbt_status st = sbt_use_device(ctx);
    if (st) return st;
    return sbt_launch_gemm_block_scaled(ctx, (int)a_fmt, A, lda, (int)b_fmt, B, ldb, (int)s_fmt, a_scale, ld_sa,
                                        b_scale, ld_sb, K_s, acc, ld_acc, D, ldd, M, N, K, workspace,
                                        (cudaStream_t)stream);
}

}  // extern "C"
