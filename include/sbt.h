/*
 * sbt.h -- bounds-checked tile movement and a boundary-tile bf16 GEMM on one
 * NVIDIA GB300 (sm_103a).  C ABI of libsbt.so.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Coordinates are zero-based and signed 64-bit; negative origins are legal
 *    (Tylo.jl "Boundary tiles": the origin and all coordinates are zero-based,
 *    negative crop origins are supported).
 *  - Arrays are row-major with explicit strides counted in ELEMENTS.  A
 *    column-major array is the same call with the strides swapped.
 *  - Movement calls copy raw element bits (dtype only fixes the element size);
 *    NaN payloads and -0.0 are preserved bit for bit.
 *  - All array pointers are DEVICE pointers (cudaMalloc'd or otherwise
 *    device-addressable).  `pad_value` is a HOST pointer to one element's bits.
 *    The caller owns every buffer; the library allocates no device memory.
 *  - Every array pointer is a multiple of its element size (int32 indices and
 *    cu_seqlens: 4 bytes; 8-bit codes, scales and masks: any address); a call
 *    given one that is not returns SBT_ERR_ALIGNMENT before any launch.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and returns after enqueueing.  Arguments are validated on
 *    the host before anything is launched; on error nothing is launched and
 *    sbt_last_error_message() says why.  A call whose output is empty returns
 *    SBT_OK without launching.
 *  - Metadata that lives on the device (indices, cu_seqlens) cannot be checked
 *    on the host: out-of-range values are handled by the semantics (pad on
 *    load, clip on store), never by faulting.
 *  - Kernels that wait on hardware barriers bound every wait; a wait that runs
 *    out sets a per-device status flag, the kernel returns early and
 *    sbt_check_status() reports SBT_ERR_DEVICE_TIMEOUT.
 */
#ifndef SBT_H_
#define SBT_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SBT_API __attribute__((visibility("default")))
#else
#define SBT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SBT_OK = 0,
    SBT_ERR_INVALID_ARG = 1,    /* null pointer, negative extent, bad stride, tile too large, ... */
    SBT_ERR_UNSUPPORTED = 2,    /* dtype or combination this op does not take */
    SBT_ERR_ALIGNMENT = 3,      /* array pointer not on a multiple of its element size; workspace not
                                   256-byte aligned or too small */
    SBT_ERR_TENSOR_MAP = 4,     /* the driver refused a TMA descriptor (Mojo "RaggedTMA3DTile": create raises) */
    SBT_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed */
    SBT_ERR_DEVICE_TIMEOUT = 6  /* a bounded device-side wait ran out (see sbt_check_status) */
} sbt_status;

typedef enum { SBT_F32 = 0, SBT_BF16 = 1, SBT_F16 = 2 } sbt_dtype;

/* Which copy path the host may pick.  AUTO chooses per call from alignment:
 * TMA for aligned interior tiles, 16-byte vectors where the addresses allow,
 * scalar bounds-checked elements otherwise.  The others force one path where
 * the call allows it (tests and measurements); results are identical.  The
 * clipped store into rows that are not 16-byte aligned (tiles side by side
 * along the row) writes realigned row chunks with TMA bulk copies under AUTO
 * and TMA, and lane-shifted 16-byte stores under VECTOR. */
typedef enum { SBT_PATH_AUTO = 0, SBT_PATH_SCALAR = 1, SBT_PATH_VECTOR = 2, SBT_PATH_TMA = 3 } sbt_path;

typedef struct sbt_context sbt_context;

/* Create a context bound to CUDA device `device` (made current by every call
 * that takes the context).  Host memory only.  Returns SBT_ERR_CUDA if the
 * device cannot be queried, SBT_ERR_UNSUPPORTED if it is not compute 10.3. */
SBT_API sbt_status sbt_create(int device, sbt_context** out);
SBT_API sbt_status sbt_destroy(sbt_context* ctx);

/* Path policy for later calls on this context (default SBT_PATH_AUTO). */
SBT_API sbt_status sbt_set_path(sbt_context* ctx, sbt_path path);
/* Limit of every bounded device-side wait, in nanoseconds (default 2e9). */
SBT_API sbt_status sbt_set_wait_limit_ns(sbt_context* ctx, uint64_t ns);
/* Test hook for the bounded device waits.  SBT_TEST_WITHHOLD_LOAD makes the
 * next GEMM (bf16 or block-scaled tensor path) and bulk row launches on this
 * context skip their first copy, so
 * a consumer's bounded wait runs out (no fault, no hang): the kernel sets the
 * status flag, drains and returns, and sbt_check_status() reports
 * SBT_ERR_DEVICE_TIMEOUT.  Stays set until reset with SBT_TEST_NONE. */
typedef enum { SBT_TEST_NONE = 0, SBT_TEST_WITHHOLD_LOAD = 1 } sbt_test_hook;
SBT_API sbt_status sbt_set_test_hook(sbt_context* ctx, sbt_test_hook hook);
/* Number of kernels this context has launched so far. */
SBT_API uint64_t sbt_launch_count(const sbt_context* ctx);
/* Synchronise `stream`, then read and clear the device status flag of the
 * context's device: SBT_ERR_DEVICE_TIMEOUT if a bounded wait ran out since
 * the last check, SBT_ERR_CUDA if the stream reports an error, else SBT_OK. */
SBT_API sbt_status sbt_check_status(sbt_context* ctx, void* stream);
/* Message of the last failing call on this thread ("" if none). */
SBT_API const char* sbt_last_error_message(void);

/*
 * Padded tile load over a grid of tiles.
 * cuTile.jl "Memory", section "Bounds checking" (loads are padded where the
 * tile extends past the array) and section "Tile windows" (tile origins move
 * by a per-dimension step; the host counts tiles with ceiling division).
 *
 *   tile (ti, tj), ti < grid_r, tj < grid_c, starts at
 *     (origin_r + ti*step_r, origin_c + tj*step_c);
 *   dst_tiles[((ti*grid_c + tj)*tile_r + i)*tile_c + j] =
 *     src[r*stride_r + c*stride_c]  if 0 <= r < rows and 0 <= c < cols
 *     *pad_value                    otherwise,
 *   with r = tile origin row + i, c = tile origin column + j.
 *
 * src: device, logical rows x cols with element strides (stride_r, stride_c),
 * both nonzero (negative allowed).  dst_tiles: device, contiguous
 * [grid_r][grid_c][tile_r][tile_c].  1 <= tile_r, tile_c <= 256.
 * pad_value: host pointer to one element of `dtype` (NULL means all-zero bits).
 */
SBT_API sbt_status sbt_tile_load_padded(sbt_context* ctx, sbt_dtype dtype, const void* src, int64_t rows, int64_t cols,
                                int64_t stride_r, int64_t stride_c, int64_t origin_r, int64_t origin_c,
                                int64_t step_r, int64_t step_c, int32_t grid_r, int32_t grid_c, int32_t tile_r,
                                int32_t tile_c, void* dst_tiles, const void* pad_value, void* stream);

/*
 * Clipped tile store: the inverse of sbt_tile_load_padded.
 * cuTile.jl "Memory", section "Bounds checking" (stores are clipped) and
 * Tylo.jl "Boundary tiles", section "Accumulator stores and GEMM" (invalid
 * coordinates are suppressed; memory outside the array is left unchanged).
 * Element (i, j) of tile (ti, tj) is written to dst only when its (r, c) is
 * inside rows x cols; nothing else of dst is touched.  Where windows overlap
 * (step < tile) which write lands is undefined.
 */
SBT_API sbt_status sbt_tile_store_clipped(sbt_context* ctx, sbt_dtype dtype, const void* src_tiles, int32_t grid_r,
                                  int32_t grid_c, int32_t tile_r, int32_t tile_c, void* dst, int64_t rows,
                                  int64_t cols, int64_t stride_r, int64_t stride_c, int64_t origin_r,
                                  int64_t origin_c, int64_t step_r, int64_t step_c, void* stream);

/*
 * Row gather through an int32 index tile.
 * warp.tile_load_indexed, description and "Parameters": element (k, j) reads
 * row row_offset + idx[k] (the offset is added before the check, in 64-bit)
 * and column col_offset + j; every coordinate is checked against both bounds
 * and an element outside reads the padding value, so -1 is a sentinel.
 * cuTile.jl "Memory": an optional per-element mask; masked-out elements read
 * the padding value.
 *
 *   out[k*ld_out + j] = src[(row_offset+idx[k])*ld_src + col_offset + j]
 *                         if mask[k][j] (or no mask) and the coordinate is in
 *                         rows x cols;   *pad_value otherwise,
 *   for k < n_idx, j < tile_c.
 *
 * src: device rows x cols, row stride ld_src >= cols.  idx: device int32[n_idx].
 * mask: device uint8 [n_idx][ld_mask] (nonzero = true) or NULL.  out: device
 * [n_idx][ld_out], ld_out >= tile_c; columns >= tile_c are not written.
 * 1 <= tile_c <= 65536.
 */
SBT_API sbt_status sbt_gather_rows(sbt_context* ctx, sbt_dtype dtype, const void* src, int64_t rows, int64_t cols,
                           int64_t ld_src, const int32_t* idx, int64_t n_idx, int64_t row_offset,
                           int64_t col_offset, int32_t tile_c, const uint8_t* mask, int64_t ld_mask, void* out,
                           int64_t ld_out, const void* pad_value, void* stream);

/*
 * Column gather: the gather along axis 1.
 * warp.tile_load_indexed, description and "Parameters" with axis = 1: element
 * (i, k) reads row row_offset + i and column col_offset + idx[k] (the offset
 * added before the check, in 64-bit); every coordinate is checked against both
 * bounds and an element outside reads the padding value.
 *
 *   out[i*ld_out + k] = src[(row_offset+i)*ld_src + col_offset + idx[k]] or *pad_value,
 *   for i < tile_r, k < n_idx.
 *
 * src: device rows x cols, row stride ld_src >= cols.  idx: device int32[n_idx].
 * out: device [tile_r][ld_out], ld_out >= n_idx.  1 <= tile_r <= 65536.
 */
SBT_API sbt_status sbt_gather_cols(sbt_context* ctx, sbt_dtype dtype, const void* src, int64_t rows, int64_t cols,
                                   int64_t ld_src, const int32_t* idx, int64_t n_idx, int64_t row_offset,
                                   int64_t col_offset, int32_t tile_r, void* out, int64_t ld_out,
                                   const void* pad_value, void* stream);

/*
 * Masked row scatter.
 * cuTile.jl "Memory": scatter writes only where the mask is true and is
 * bounds-checked like every tile memory operation (out-of-range elements are
 * clipped); section "Sparse views": conflicting stores to a repeated index
 * are undefined -- here exactly one of the candidate values lands.
 *
 *   for k < n_idx, j < tile_c: if (mask == NULL or mask[k*ld_mask + j] != 0)
 *   and r = row_offset + idx[k] in [0, rows) and c = col_offset + j in
 *   [0, cols):  dst[r*ld_dst + c] = src[k*ld_src + j].
 *
 * Every other element of dst keeps its bits.
 */
SBT_API sbt_status sbt_scatter_rows_masked(sbt_context* ctx, sbt_dtype dtype, void* dst, int64_t rows, int64_t cols,
                                   int64_t ld_dst, const int32_t* idx, int64_t n_idx, int64_t row_offset,
                                   int64_t col_offset, const void* src, int64_t ld_src, int32_t tile_c,
                                   const uint8_t* mask, int64_t ld_mask, void* stream);

/*
 * Row scatter-add: the adjoint (backward) of sbt_gather_rows.
 * warp.tile_load_indexed, description: in a backward pass the adjoint of the
 * gathered tile is accumulated atomically into the array's gradient at the
 * gathered locations.
 *
 *   for k < n_idx, j < tile_c: if r = row_offset + idx[k] in [0, rows) and
 *   c = col_offset + j in [0, cols):  dst[r*ld_dst + c] += src[k*ld_src + j]
 *
 * Each addition is done in the element type (SBT_F32, SBT_BF16 or SBT_F16)
 * with one rounding to nearest even, by the memory system's atomic add, so
 * repeated indices accumulate; their order is unspecified (results with
 * repeats may differ in the last bits from run to run).  Elements that read
 * padding in the forward pass contribute nothing.  Subnormal fp32 results
 * are outside the contract (the GPU's fp32 atomic add may flush them).
 */
SBT_API sbt_status sbt_scatter_add_rows(sbt_context* ctx, sbt_dtype dtype, void* dst, int64_t rows, int64_t cols,
                                        int64_t ld_dst, const int32_t* idx, int64_t n_idx, int64_t row_offset,
                                        int64_t col_offset, const void* src, int64_t ld_src, int32_t tile_c,
                                        void* stream);

/*
 * Ragged 3D tile load.
 * Mojo "RaggedTMA3DTile", struct description: a packed array
 * [total_rows][heads][depth] whose leading dimension concatenates sequences,
 * read as 2D tiles per head with only the first `dynamic_dim` rows of a tile
 * valid.  Sequence b owns packed rows [cu_seqlens[b], cu_seqlens[b+1]).
 *
 *   out[((b*heads + h)*t_pad + r)*depth + d] =
 *     x[(cu[b]+r)*ld_row + h*ld_head + d]  if r < cu[b+1]-cu[b] and
 *                                            0 <= cu[b]+r < total_rows,
 *     0 (all-zero bits)                    otherwise,
 *   for b < batch, h < heads, r < t_pad, d < depth.
 *
 * x: device; cu_seqlens: device int32[batch+1]; out: device, dense
 * [batch][heads][t_pad][depth].  Sequences longer than t_pad are clipped.
 */
SBT_API sbt_status sbt_ragged_tile_load(sbt_context* ctx, sbt_dtype dtype, const void* x, int64_t total_rows, int32_t heads,
                                int32_t depth, int64_t ld_row, int64_t ld_head, const int32_t* cu_seqlens,
                                int32_t batch, int32_t t_pad, void* out, void* stream);

/*
 * Ragged 3D tile store: the inverse of sbt_ragged_tile_load.
 * Mojo "RaggedTMA3DTile", async_copy_from_col / async_copy_batched: tiles go
 * back to the packed ragged array, only the first `dynamic_dim` rows of a tile
 * (valid sequence positions) are written, and what overhangs is masked off.
 *
 *   x[(cu[b]+r)*ld_row + h*ld_head + d] = tiles[((b*heads + h)*t_pad + r)*depth + d]
 *     for r < min(cu[b+1]-cu[b], t_pad) with 0 <= cu[b]+r < total_rows;
 *   every other element of x keeps its bits.
 *
 * tiles: device, dense [batch][heads][t_pad][depth]; cu_seqlens: device
 * int32[batch+1]; x: device packed [total_rows] rows with strides (ld_row,
 * ld_head), both positive.  Sequences whose packed rows overlap get one of the
 * candidate values (undefined which).
 */
SBT_API sbt_status sbt_ragged_tile_store(sbt_context* ctx, sbt_dtype dtype, const void* tiles, int32_t batch,
                                         int32_t heads, int32_t depth, int32_t t_pad, const int32_t* cu_seqlens,
                                         void* x, int64_t total_rows, int64_t ld_row, int64_t ld_head, void* stream);

/*
 * Boundary-tile GEMM  C = A * B.
 * cuTile.jl "Operations", muladd: (M,K) x (K,N) -> (M,N) with bf16 inputs
 * accumulating in fp32.  Tylo.jl "Boundary tiles", section "Accumulator
 * stores and GEMM": ceiling-division K loop and output grid, boundary tiles
 * zero-filled, the fp32 accumulator converted to the output type at the store
 * (round to nearest even) and stores outside M x N suppressed.
 *
 * A: device bf16, M x K, row stride lda >= K.  B: device bf16, K x N, row
 * stride ldb >= N.  C: device, M x N, row stride ldc >= N, c_dtype SBT_BF16
 * or SBT_F32.  Any leading dimension is accepted (odd ones included); C
 * elements outside M x N (padding columns) are never written.
 * workspace: device scratch of at least sbt_gemm_bounded_workspace_size()
 * bytes, 256-byte aligned, owned by the caller; it holds re-laid-out copies of
 * A and B and may be reused once the call has completed on `stream`.
 */
SBT_API sbt_status sbt_gemm_bounded_workspace_size(sbt_context* ctx, int64_t M, int64_t N, int64_t K, int64_t lda,
                                           int64_t ldb, size_t* bytes);
SBT_API sbt_status sbt_gemm_bounded(sbt_context* ctx, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                            int64_t ldc, sbt_dtype c_dtype, int64_t M, int64_t N, int64_t K, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * Block-scaled GEMM  D = (A .* a_scale) * (B .* b_scale) + acc.
 * cuTile.jl "Operations", muladd_scaled: A (M x K) and B (K x N) in a
 * low-precision float format, a_scale (M x K_s) and b_scale (K_s x N) in
 * E8M0 or E4M3; scale element j of a row of a_scale (of a column of b_scale)
 * multiplies the contiguous block of K / K_s elements k = j*K/K_s ..
 * (j+1)*K/K_s - 1 of that row of A (column of B).  fp32 accumulator, fp32
 * acc and D.
 *
 * Formats (OCP 8-bit floating point and microscaling formats):
 *   SBT_FMT_E4M3  1-4-3, bias 7, no infinities, S.1111.111 is NaN
 *   SBT_FMT_E5M2  1-5-2, bias 15, IEEE infinities and NaNs
 *   SBT_FMT_E8M0  unsigned power of two 2^(e-127), 0xFF is NaN (scales only)
 *   SBT_FMT_E2M1  4-bit 1-2-1, bias 1, values 0, 0.5, 1, 1.5, 2, 3, 4, 6
 *                 (operands only); two per byte, element i of a row-major
 *                 array (i = row * ld + col) in byte i / 2, the even element
 *                 in the low nibble; ld must be even.
 *
 * a_fmt, b_fmt: E4M3, E5M2 or E2M1 (they may differ).  s_fmt: E8M0 or E4M3,
 * both scale arrays.  A: device, row stride lda >= K (elements).  B: device,
 * row stride ldb >= N.  a_scale: device bytes, row stride ld_sa >= K_s.
 * b_scale: device bytes, row stride ld_sb >= N.  K_s >= 1 must divide K
 * (K_s is ignored when K = 0).  acc: device fp32, row stride ld_acc >= N, or
 * NULL for zero; it may be D itself (then ld_acc == ldd) but may not
 * otherwise overlap D.  D: device fp32, row stride ldd >= N; elements outside
 * M x N are never written.
 *
 * Accuracy: each scaled operand value (code value times its scale) is formed
 * exactly and the products are summed in fp32, provided every scaled operand
 * lies in the normal range of bf16/fp32 (E8M0 scale exponents from 2^-124 to
 * 2^119 with E4M3 operands; any E4M3 scale).  NaN codes propagate to the row
 * (A, a_scale) or column (B, b_scale) of D they feed.
 *
 * Paths: under SBT_PATH_AUTO or SBT_PATH_TMA the call runs on the tensor
 * cores' block scaling when the formats allow it: E2M1 x E2M1 with E8M0 scales
 * and K / K_s = 32 on tcgen05.mma kind::mxf4 (packed 4-bit operands), E2M1 x
 * E2M1 with E4M3 scales and K / K_s = 16 on kind::mxf4nvf4 (the scales' signs
 * are moved onto the operand codes first), and any other mix of E4M3 / E5M2 /
 * E2M1 with E8M0 scales and K / K_s = 32 on kind::mxf8f6f4 (8-bit staging).
 * Every other combination, and any combination under SBT_PATH_SCALAR or
 * SBT_PATH_VECTOR, stages the scaled operands as bf16 for the bf16
 * tensor-core kernel.  The paths meet the same accuracy statement; they may
 * differ in the order of the fp32 sums.
 *
 * workspace: device scratch of at least sbt_gemm_block_scaled_workspace_size()
 * bytes (enough for either path), 256-byte aligned, owned by the caller
 * (re-laid-out copies of the operands and scales).
 */
typedef enum { SBT_FMT_E4M3 = 0, SBT_FMT_E5M2 = 1, SBT_FMT_E8M0 = 2, SBT_FMT_E2M1 = 3 } sbt_lowp_format;
SBT_API sbt_status sbt_gemm_block_scaled_workspace_size(sbt_context* ctx, int64_t M, int64_t N, int64_t K,
                                                        size_t* bytes);
SBT_API sbt_status sbt_gemm_block_scaled(sbt_context* ctx, sbt_lowp_format a_fmt, const void* A, int64_t lda,
                                         sbt_lowp_format b_fmt, const void* B, int64_t ldb, sbt_lowp_format s_fmt,
                                         const void* a_scale, int64_t ld_sa, const void* b_scale, int64_t ld_sb,
                                         int64_t K_s, const float* acc, int64_t ld_acc, float* D, int64_t ldd,
                                         int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                                         void* stream);

/*
 * Boundary-tile GEMM without any device allocation.
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory when they multiply: plugins confined to
 * another framework's memory pool (they may not call the CUDA allocator
 * themselves), code running under a device-memory budget committed up front,
 * and latency-critical paths that cannot take the implicit device
 * synchronisation of cudaMalloc and cudaFree.
 *
 * Same arguments and result as sbt_gemm_bounded, minus the workspace: the
 * operand-staging scratch is a fixed array of SBT_GEMM_NOALLOC_SCRATCH_BYTES
 * inside the library (one per device, held from module load until process
 * exit).  Shapes whose sbt_gemm_bounded_workspace_size() exceeds that size
 * are rejected with SBT_ERR_INVALID_ARG before anything is launched.  The
 * call itself allocates nothing (no cudaMalloc, no cudaFree, no allocating
 * library routine).
 *
 * Set-up: the first call on a device (whatever its shape) looks up the
 * array's device address with cudaGetSymbolAddress, with that device current,
 * and caches it; make that first call before any stream capture.  Like every
 * call of this library it leaves ctx's device current on the calling thread.
 * All calls share the one array and it keeps the previous call's contents
 * (the call rewrites every byte it reads, so nothing needs clearing); calls
 * that can overlap on the GPU -- different streams, or unsynchronised host
 * threads -- race on it.
 */
#define SBT_GEMM_NOALLOC_SCRATCH_BYTES (16u << 20)
SBT_API sbt_status sbt_gemm_bounded_noalloc(sbt_context* ctx, const void* A, int64_t lda, const void* B, int64_t ldb,
                                            void* C, int64_t ldc, sbt_dtype c_dtype, int64_t M, int64_t N, int64_t K,
                                            void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SBT_H_ */
