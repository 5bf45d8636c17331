// Internal declarations shared by the translation units of libsbt.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/sbt.h"

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------

typedef CUresult (*sbt_encode_tiled_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                        const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                        CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct sbt_context {
    int device = 0;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    size_t smem_optin = 0;
    sbt_path path = SBT_PATH_AUTO;
    uint64_t wait_limit_ns = 2000000000ull;
    unsigned int* status = nullptr;  // device address of this device's status flag
    sbt_encode_tiled_fn encode_tiled = nullptr;
    uint64_t launches = 0;
    int test_hook = 0;  // sbt_test_hook
};

// Thread-local error message; returns `st` so call sites can `return sbt_fail(...)`.
sbt_status sbt_fail(sbt_status st, const std::string& msg);
sbt_status sbt_ok();
sbt_status sbt_cuda_check(cudaError_t e, const char* what);
// Makes ctx->device current.
sbt_status sbt_use_device(sbt_context* ctx);

inline int sbt_dtype_size(sbt_dtype t) {
    switch (t) {
        case SBT_F32: return 4;
        case SBT_BF16: return 2;
        case SBT_F16: return 2;
    }
    return 0;
}

inline bool sbt_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool sbt_mul16(int64_t elems, int es) { return ((elems * es) % 16) == 0; }
inline int64_t sbt_cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Replicates one element's bits into a 32-bit word (es = 2 or 4).
uint32_t sbt_pad_word(const void* pad, int es);

// Grid size for a persistent kernel: SMs x resident blocks, capped by the work.
int sbt_persistent_grid(const sbt_context* ctx, const void* kernel, int threads, size_t smem, int64_t work_units);

// Launchers of the movement kernels (one translation unit each).
sbt_status sbt_launch_tile_load(sbt_context* ctx, int es, const void* src, int64_t rows, int64_t cols,
                                int64_t stride_r, int64_t stride_c, int64_t origin_r, int64_t origin_c,
                                int64_t step_r, int64_t step_c, int32_t grid_r, int32_t grid_c, int32_t tile_r,
                                int32_t tile_c, void* dst, uint32_t pad_word, cudaStream_t stream);
sbt_status sbt_launch_tile_store(sbt_context* ctx, int es, const void* src_tiles, int32_t grid_r, int32_t grid_c,
                                 int32_t tile_r, int32_t tile_c, void* dst, int64_t rows, int64_t cols,
                                 int64_t stride_r, int64_t stride_c, int64_t origin_r, int64_t origin_c,
                                 int64_t step_r, int64_t step_c, cudaStream_t stream);
// Clipped store along whole destination runs when the destination rows are not
// 16-byte aligned and the tiles sit side by side along the row (k_tiles_runs.cu).
bool sbt_tile_store_runs_ok(sbt_context* ctx, int es, const void* src_tiles, int32_t grid_r, int32_t grid_c,
                            int32_t tile_r, int32_t tile_c, const void* dst, int64_t stride_r, int64_t stride_c,
                            int64_t origin_c, int64_t step_c);
sbt_status sbt_launch_tile_store_runs(sbt_context* ctx, int es, const void* src_tiles, int32_t grid_r,
                                      int32_t grid_c, int32_t tile_r, int32_t tile_c, void* dst, int64_t rows,
                                      int64_t cols, int64_t stride_r, int64_t origin_r, int64_t origin_c,
                                      int64_t step_r, cudaStream_t stream);
sbt_status sbt_launch_gather(sbt_context* ctx, int es, const void* src, int64_t rows, int64_t cols, int64_t ld_src,
                             const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                             int32_t tile_c, const uint8_t* mask, int64_t ld_mask, void* out, int64_t ld_out,
                             uint32_t pad_word, cudaStream_t stream);
sbt_status sbt_launch_scatter(sbt_context* ctx, int es, void* dst, int64_t rows, int64_t cols, int64_t ld_dst,
                              const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                              const void* src, int64_t ld_src, int32_t tile_c, const uint8_t* mask, int64_t ld_mask,
                              cudaStream_t stream);
sbt_status sbt_launch_ragged(sbt_context* ctx, int es, const void* x, int64_t total_rows, int32_t heads,
                             int32_t depth, int64_t ld_row, int64_t ld_head, const int32_t* cu_seqlens,
                             int32_t batch, int32_t t_pad, void* out, cudaStream_t stream);
sbt_status sbt_launch_gather_cols(sbt_context* ctx, int es, const void* src, int64_t rows, int64_t cols, int64_t ld_src,
                                  const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                                  int32_t tile_r, void* out, int64_t ld_out, uint32_t pad_word, cudaStream_t stream);
// kind: 4 = fp32, 2 = bf16, 3 = fp16
sbt_status sbt_launch_scatter_add(sbt_context* ctx, int kind, void* dst, int64_t rows, int64_t cols, int64_t ld_dst,
                                  const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                                  const void* src, int64_t ld_src, int32_t tile_c, cudaStream_t stream);
sbt_status sbt_launch_ragged_store(sbt_context* ctx, int es, const void* tiles, int32_t batch, int32_t heads,
                                   int32_t depth, int32_t t_pad, const int32_t* cu_seqlens, void* x,
                                   int64_t total_rows, int64_t ld_row, int64_t ld_head, cudaStream_t stream);
sbt_status sbt_launch_gemm(sbt_context* ctx, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                           int64_t ldc, sbt_dtype c_dtype, int64_t M, int64_t N, int64_t K, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);
// K-major padded operand copies of the tensor-core GEMM: A' [Mp][Kp] and
// B'^T [Np][Kp] bf16, zero past M, N, K; B' starts a_bytes into the workspace.
struct sbt_gemm_layout {
    int64_t Mp, Np, Kp;
    size_t a_bytes, b_bytes;
};
sbt_gemm_layout sbt_gemm_layout_of(int64_t M, int64_t N, int64_t K);
// The tensor-core kernel over already staged operands; C (fp32 or bf16) gets
// A'B'^T (+ acc, fp32 C only) for m < M, n < N.
sbt_status sbt_launch_gemm_main(sbt_context* ctx, const uint16_t* Ap, const uint16_t* Bp, const sbt_gemm_layout& d,
                                void* C, int64_t ldc, bool c_f32, const float* acc, int64_t ld_acc, int64_t M,
                                int64_t N, int64_t K, cudaStream_t stream);
// C = acc (or 0): the K = 0 result.
sbt_status sbt_launch_gemm_zero_k(sbt_context* ctx, void* C, int64_t ldc, bool c_f32, const float* acc,
                                  int64_t ld_acc, int64_t M, int64_t N, cudaStream_t stream);
// Block-scaled GEMM on tcgen05's own block scaling: E4M3 / E5M2 / E2M1
// operands with E8M0 scales per 32 along K (kind::mxf8f6f4, or kind::mxf4
// when both are E2M1), and E2M1 x E2M1 with E4M3 scales per 16
// (kind::mxf4nvf4); the caller checks that the call is one of these.
size_t sbt_gemm_mx_workspace_bytes(int64_t M, int64_t N, int64_t K);
sbt_status sbt_launch_gemm_mx(sbt_context* ctx, int a_fmt, const void* A, int64_t lda, int b_fmt, const void* B,
                              int64_t ldb, int s_fmt, const void* SA, int64_t ld_sa, const void* SB, int64_t ld_sb,
                              const float* acc, int64_t ld_acc, float* D, int64_t ldd, int64_t M, int64_t N,
                              int64_t K, void* workspace, cudaStream_t stream);
// Block-scaled GEMM (formats as sbt_lowp_format): the block-scaled tensor-core
// kernel where it applies (AUTO / TMA path), else bf16 staging of the scaled operands.
sbt_status sbt_launch_gemm_block_scaled(sbt_context* ctx, int a_fmt, const void* A, int64_t lda, int b_fmt,
                                        const void* B, int64_t ldb, int s_fmt, const void* SA, int64_t ld_sa,
                                        const void* SB, int64_t ld_sb, int64_t Ks, const float* acc, int64_t ld_acc,
                                        float* D, int64_t ldd, int64_t M, int64_t N, int64_t K, void* workspace,
                                        cudaStream_t stream);
size_t sbt_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
// TMA tensor-copy variants of the tile load / store (k_tiles_tma.cu) and their preconditions.
bool sbt_tile_tma_ok(int es, const void* arr, int64_t rows, int64_t cols, int64_t stride_r, int64_t stride_c,
                     int64_t origin_r, int64_t origin_c, int64_t step_r, int64_t step_c, int32_t grid_r,
                     int32_t grid_c, int32_t tile_r, int32_t tile_c, const void* tiles, bool store);
sbt_status sbt_launch_tile_load_tma(sbt_context* ctx, int es, const void* src, int64_t rows, int64_t cols,
                                    int64_t stride_r, int64_t origin_r, int64_t origin_c, int64_t step_r,
                                    int64_t step_c, int32_t grid_r, int32_t grid_c, int32_t tile_r, int32_t tile_c,
                                    void* dst, uint32_t pad_word, cudaStream_t stream);
sbt_status sbt_launch_tile_store_tma(sbt_context* ctx, int es, const void* src_tiles, int32_t grid_r, int32_t grid_c,
                                     int32_t tile_r, int32_t tile_c, void* dst, int64_t rows, int64_t cols,
                                     int64_t stride_r, int64_t origin_r, int64_t origin_c, int64_t step_r,
                                     int64_t step_c, cudaStream_t stream);
// TMA bulk-copy variants of the row gather / scatter (k_bulk.cu) and their preconditions.
bool sbt_gather_bulk_ok(int es, const void* src, int64_t cols, int64_t ld_src, int64_t col_offset, int32_t tile_c,
                        const uint8_t* mask, const void* out, int64_t ld_out);
bool sbt_scatter_bulk_ok(int es, const void* src, int64_t ld_src, int32_t tile_c, const uint8_t* mask,
                         int64_t ld_mask);
sbt_status sbt_launch_gather_bulk(sbt_context* ctx, int es, const void* src, int64_t rows, int64_t ld_src,
                                  const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                                  int32_t tile_c, void* out, int64_t ld_out, uint32_t pad_word, cudaStream_t stream);
sbt_status sbt_launch_scatter_bulk(sbt_context* ctx, int es, void* dst, int64_t rows, int64_t cols, int64_t ld_dst,
                                   const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                                   const void* src, int64_t ld_src, int32_t tile_c, const uint8_t* mask,
                                   int64_t ld_mask, cudaStream_t stream);

// Checks the launch that was just enqueued and counts it.
sbt_status sbt_after_launch(sbt_context* ctx, const char* what);

// Enqueues `kern` as a programmatic dependent of the kernel ahead of it in the
// stream: its blocks may start (and run their set-up) while that kernel drains;
// the kernel itself must call griddep_wait() before it touches memory the
// earlier kernel writes.  Cluster shapes come from the kernel's __cluster_dims__.
template <typename... KArgs, typename... Args>
cudaError_t sbt_launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// ----------------------------------------------------------------------------
// Device side: raw element types and 16-byte vector accesses
// ----------------------------------------------------------------------------

template <int ES> struct sbt_elem;
template <> struct sbt_elem<2> { typedef uint16_t T; };
template <> struct sbt_elem<4> { typedef uint32_t T; };

// Read-only 16-byte load that does not allocate in L1 (streamed data).
__device__ __forceinline__ uint4 sbt_ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Read-only 16-byte load that may allocate in L1 (neighbouring tasks reuse it).
__device__ __forceinline__ uint4 sbt_ld_nc_v4_l1(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Eight bytes p..p+7, all inside the caller's array, through aligned 8-byte
// loads: the word holding p and, when p is unaligned, the one holding p+7 each
// contain a byte of the array, so neither reaches past its pages.
__device__ __forceinline__ uint64_t sbt_load8_any(const void* ptr) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
    const int sh = (int)(a & 7u) * 8;
    const uint64_t* w = reinterpret_cast<const uint64_t*>(a & ~(uintptr_t)7);
    const uint64_t lo = __ldg(w);
    if (sh == 0) return lo;
    return (lo >> sh) | (__ldg(w + 1) << (64 - sh));
}

// Streaming (evict-first) 16-byte store, for outputs this kernel never reads back.
__device__ __forceinline__ void sbt_st_v4_cs(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void sbt_st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// n / d for 0 <= n < 2^31 by one 64-bit multiply and a shift (division by an
// invariant integer, Granlund & Montgomery 1994): with s = ceil(log2 d) and
// m = ceil(2^(32+s) / d), floor(n * m / 2^(32+s)) = floor(n / d) because the
// rounding error of m contributes less than 2^-(1+s) <= 1/(2d).
struct sbt_fastdiv {
    uint32_t d;
    uint32_t shift;
    uint64_t mul;
};

inline sbt_fastdiv sbt_make_fastdiv(uint32_t d) {
    sbt_fastdiv f;
    uint32_t s = 0;
    while ((1ull << s) < d) ++s;
    f.d = d;
    f.shift = 32 + s;
    f.mul = ((1ull << f.shift) + d - 1) / d;
    return f;
}

__device__ __forceinline__ uint32_t sbt_div(const sbt_fastdiv& f, uint32_t n) {
    return (uint32_t)(((uint64_t)n * f.mul) >> f.shift);
}

// Element e (0..16/ES-1) of a 16-byte vector.
template <int ES>
__device__ __forceinline__ typename sbt_elem<ES>::T sbt_vec_get(const uint4& v, int e) {
    uint32_t w = e * ES / 4 == 0 ? v.x : e * ES / 4 == 1 ? v.y : e * ES / 4 == 2 ? v.z : v.w;
    if (ES == 4) return (typename sbt_elem<ES>::T)w;
    return (typename sbt_elem<ES>::T)((e & 1) ? (w >> 16) : (w & 0xFFFFu));
}

template <int ES>
__device__ __forceinline__ void sbt_vec_set(uint4& v, int e, typename sbt_elem<ES>::T x) {
    uint32_t* w = e * ES / 4 == 0 ? &v.x : e * ES / 4 == 1 ? &v.y : e * ES / 4 == 2 ? &v.z : &v.w;
    if (ES == 4) {
        *w = (uint32_t)x;
    } else if (e & 1) {
        *w = (*w & 0x0000FFFFu) | ((uint32_t)x << 16);
    } else {
        *w = (*w & 0xFFFF0000u) | (uint32_t)x;
    }
}
