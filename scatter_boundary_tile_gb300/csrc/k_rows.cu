// Row gather through an int32 index tile, and masked row scatter.
//
// Both kernels are persistent: the grid is (SMs x resident blocks), and each
// block walks chunks of kChunkRows indices.  A chunk's indices are staged in
// shared memory (double-buffered) by one warp, which also checks every row
// against the array bounds (64-bit, offset added first --
// warp.tile_load_indexed, description) and builds the chunk's row-valid mask
// with a warp ballot.  The block then
// moves the chunk's rows with 16-byte vectors (when the host has checked that
// every vector address is 16-byte aligned) or element by element.
//
// Per 16-byte vector the bounds decision follows the vector/scalar split of
// Tylo.jl "Boundary tiles" (a vector wholly inside the array takes one
// vector access; a partial vector goes element by element, and no pointer is
// formed for an element outside the array).
#include "sbt_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kChunkRows = 32;
constexpr int kUnroll = 8;
// Vector gather: one 16-byte vector per thread and trip.  Measured on the 1 KiB
// bf16 rows of the headline gather: 0.322 ms at 1, 0.341 at 2, 0.333 at 8.
constexpr int kGatherVecUnroll = 1;

enum MaskMode { kNoMask = 0, kMaskVec = 1, kMaskBytes = 2 };

struct RowParams {
    const char* src;   // gather: table;  scatter: source rows
    char* dst;         // gather: output; scatter: destination array
    const int32_t* idx;
    const uint8_t* mask;
    int64_t rows, cols;        // bounds of the indexed array (table / destination)
    int64_t ld_arr;            // row stride of the indexed array
    int64_t ld_dense;          // row stride of the dense side (gather out / scatter src)
    int64_t ld_mask;
    int64_t n_idx, row_offset, col_offset;
    int32_t tile_c;
    int32_t nvec;              // tile_c / (16 / ES) on the vector path
    uint32_t pad_word;
};

// Index staging, double-buffered across chunks.  Warp 0 issues the loads of
// the next chunk's indices before the block moves the current chunk, and
// finishes staging them (row = row_offset + idx in 64-bit, bounds check,
// ballot of the rows inside [0, rows)) afterwards, so their latency hides
// behind the data movement.
__device__ __forceinline__ int32_t issue_index_load(const RowParams& p, int64_t chunk, int64_t nchunks) {
    const int lane = threadIdx.x & 31;
    const int64_t k = chunk * kChunkRows + lane;
    return (chunk < nchunks && k < p.n_idx) ? __ldg(p.idx + k) : 0;
}

__device__ __forceinline__ void finish_index_stage(const RowParams& p, int64_t chunk, int64_t nchunks, int32_t raw,
                                                   int64_t* s_row, uint32_t* s_valid) {
    const int lane = threadIdx.x & 31;
    const int64_t k = chunk * kChunkRows + lane;
    const bool present = chunk < nchunks && k < p.n_idx;
    const int64_t r = present ? (int64_t)raw + p.row_offset : -1;
    const bool v = present && r >= 0 && r < p.rows;
    const uint32_t ballot = __ballot_sync(0xffffffffu, v);
    s_row[lane] = r;
    if (lane == 0) *s_valid = ballot;
}

// Bit e set <=> mask element e of the vector starting at column j0 of row k is true.
template <int ES, int MM>
__device__ __forceinline__ uint32_t mask_bits(const RowParams& p, int64_t k, int64_t j0) {
    constexpr int V = 16 / ES;
    constexpr uint32_t kAll = (1u << V) - 1u;
    if (MM == kNoMask) return kAll;
    const uint8_t* m = p.mask + k * p.ld_mask + j0;
    uint32_t bits = 0;
    if (MM == kMaskVec) {
        if (V == 8) {
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(m));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                bits |= ((w.x >> (8 * e)) & 0xFFu) ? (1u << e) : 0u;
                bits |= ((w.y >> (8 * e)) & 0xFFu) ? (1u << (e + 4)) : 0u;
            }
        } else {
            const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(m));
#pragma unroll
            for (int e = 0; e < V; ++e) bits |= ((w >> (8 * e)) & 0xFFu) ? (1u << e) : 0u;
        }
    } else {
#pragma unroll
        for (int e = 0; e < V; ++e) bits |= __ldg(m + e) ? (1u << e) : 0u;
    }
    return bits;
}

template <int ES>
__device__ __forceinline__ typename sbt_elem<ES>::T ld_elem(const char* base, int64_t off) {
    return __ldg(reinterpret_cast<const typename sbt_elem<ES>::T*>(base) + off);
}

template <int ES>
__device__ __forceinline__ void st_elem(char* base, int64_t off, typename sbt_elem<ES>::T v) {
    reinterpret_cast<typename sbt_elem<ES>::T*>(base)[off] = v;
}

// ---------------------------------------------------------------------------- gather

template <int ES, int MM>
__device__ __forceinline__ uint4 gather_vector(const RowParams& p, int64_t k, int64_t r, bool row_ok, int vc) {
    constexpr int V = 16 / ES;
    constexpr uint32_t kAll = (1u << V) - 1u;
    const uint4 padv = make_uint4(p.pad_word, p.pad_word, p.pad_word, p.pad_word);
    if (!row_ok) return padv;
    const int64_t j0 = (int64_t)vc * V;
    const uint32_t mb = mask_bits<ES, MM>(p, k, j0);
    if (mb == 0) return padv;
    const int64_t c0 = p.col_offset + j0;
    if (c0 >= 0 && c0 + V <= p.cols) {
        uint4 v = sbt_ld_nc_v4(p.src + (r * p.ld_arr + c0) * ES);
        if (mb != kAll) {
#pragma unroll
            for (int e = 0; e < V; ++e)
                if (!((mb >> e) & 1u)) sbt_vec_set<ES>(v, e, (typename sbt_elem<ES>::T)p.pad_word);
        }
        return v;
    }
    if (c0 + V <= 0 || c0 >= p.cols) return padv;
    uint4 v = padv;
#pragma unroll
    for (int e = 0; e < V; ++e) {
        const int64_t c = c0 + e;
        if (c >= 0 && c < p.cols && ((mb >> e) & 1u)) sbt_vec_set<ES>(v, e, ld_elem<ES>(p.src, r * p.ld_arr + c));
    }
    return v;
}

template <int ES, bool VEC, int MM>
__global__ void __launch_bounds__(kThreads) k_gather_rows(const RowParams p) {
    __shared__ int64_t s_row[2][kChunkRows];
    __shared__ uint32_t s_valid[2];
    constexpr int V = 16 / ES;
    typedef typename sbt_elem<ES>::T T;
    const int64_t nchunks = (p.n_idx + kChunkRows - 1) / kChunkRows;
    const bool stager = threadIdx.x < 32;
    if (stager) finish_index_stage(p, blockIdx.x, nchunks, issue_index_load(p, blockIdx.x, nchunks), s_row[0], &s_valid[0]);
    __syncthreads();
    int buf = 0;
    for (int64_t chunk = blockIdx.x; chunk < nchunks; chunk += gridDim.x, buf ^= 1) {
        const int64_t next = chunk + gridDim.x;
        const int32_t next_raw = stager ? issue_index_load(p, next, nchunks) : 0;
        const int64_t k0 = chunk * kChunkRows;
        const int nrows = (int)(p.n_idx - k0 < kChunkRows ? p.n_idx - k0 : kChunkRows);
        const uint32_t valid = s_valid[buf];
        const int64_t* rows_of = s_row[buf];
        if (VEC) {
            const int nvec = p.nvec;
            const int ntask = nrows * nvec;
            for (int base = threadIdx.x; base < ntask; base += kThreads * kGatherVecUnroll) {
                uint4 val[kGatherVecUnroll];
#pragma unroll
                for (int u = 0; u < kGatherVecUnroll; ++u) {
                    const int t = base + u * kThreads;
                    if (t < ntask) {
                        const int row = t / nvec;
                        const int vc = t - row * nvec;
                        val[u] = gather_vector<ES, MM>(p, k0 + row, rows_of[row], (valid >> row) & 1u, vc);
                    }
                }
#pragma unroll
                for (int u = 0; u < kGatherVecUnroll; ++u) {
                    const int t = base + u * kThreads;
                    if (t < ntask) {
                        const int row = t / nvec;
                        const int vc = t - row * nvec;
                        // streaming store: the output is not read again here (2.5% faster than a plain store)
                        sbt_st_v4_cs(p.dst + ((k0 + row) * p.ld_dense + (int64_t)vc * V) * ES, val[u]);
                    }
                }
            }
        } else {
            const int tc = p.tile_c;
            const int ntask = nrows * tc;
            for (int base = threadIdx.x; base < ntask; base += kThreads * kUnroll) {
                T val[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int t = base + u * kThreads;
                    val[u] = (T)p.pad_word;
                    if (t < ntask) {
                        const int row = t / tc;
                        const int j = t - row * tc;
                        const int64_t c = p.col_offset + j;
                        const bool m = MM == kNoMask ? true : __ldg(p.mask + (k0 + row) * p.ld_mask + j) != 0;
                        if (((valid >> row) & 1u) && m && c >= 0 && c < p.cols)
                            val[u] = ld_elem<ES>(p.src, rows_of[row] * p.ld_arr + c);
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int t = base + u * kThreads;
                    if (t < ntask) {
                        const int row = t / tc;
                        const int j = t - row * tc;
                        st_elem<ES>(p.dst, (k0 + row) * p.ld_dense + j, val[u]);
                    }
                }
            }
        }
        if (stager) finish_index_stage(p, next, nchunks, next_raw, s_row[buf ^ 1], &s_valid[buf ^ 1]);
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------- scatter

template <int ES, bool VEC, int MM>
__global__ void __launch_bounds__(kThreads) k_scatter_rows(const RowParams p) {
    __shared__ int64_t s_row[2][kChunkRows];
    __shared__ uint32_t s_valid[2];
    constexpr int V = 16 / ES;
    constexpr uint32_t kAll = (1u << V) - 1u;
    typedef typename sbt_elem<ES>::T T;
    const int64_t nchunks = (p.n_idx + kChunkRows - 1) / kChunkRows;
    const bool stager = threadIdx.x < 32;
    if (stager) finish_index_stage(p, blockIdx.x, nchunks, issue_index_load(p, blockIdx.x, nchunks), s_row[0], &s_valid[0]);
    __syncthreads();
    int buf = 0;
    for (int64_t chunk = blockIdx.x; chunk < nchunks; chunk += gridDim.x, buf ^= 1) {
        const int64_t next = chunk + gridDim.x;
        const int32_t next_raw = stager ? issue_index_load(p, next, nchunks) : 0;
        const int64_t k0 = chunk * kChunkRows;
        const int nrows = (int)(p.n_idx - k0 < kChunkRows ? p.n_idx - k0 : kChunkRows);
        const uint32_t valid = s_valid[buf];
        const int64_t* rows_of = s_row[buf];
        if (VEC) {
            const int nvec = p.nvec;
            const int ntask = nrows * nvec;
            for (int base = threadIdx.x; base < ntask; base += kThreads * kUnroll) {
                uint4 val[kUnroll];
                uint32_t mb[kUnroll];
                // Source vector and mask bits are loaded side by side (no dependence
                // between them); a vector whose row or columns lie outside is skipped.
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int t = base + u * kThreads;
                    mb[u] = 0;
                    if (t < ntask) {
                        const int row = t / nvec;
                        const int vc = t - row * nvec;
                        const int64_t j0 = (int64_t)vc * V;
                        const int64_t c0 = p.col_offset + j0;
                        if (((valid >> row) & 1u) && c0 + V > 0 && c0 < p.cols) {
                            val[u] = sbt_ld_nc_v4(p.src + ((k0 + row) * p.ld_dense + j0) * ES);
                            mb[u] = mask_bits<ES, MM>(p, k0 + row, j0);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    if (!mb[u]) continue;
                    const int t = base + u * kThreads;
                    const int row = t / nvec;
                    const int vc = t - row * nvec;
                    const int64_t c0 = p.col_offset + (int64_t)vc * V;
                    char* drow = p.dst + rows_of[row] * p.ld_arr * ES;
                    if (mb[u] == kAll && c0 >= 0 && c0 + V <= p.cols) {
                        sbt_st_v4(drow + c0 * ES, val[u]);
                    } else {
#pragma unroll
                        for (int e = 0; e < V; ++e) {
                            const int64_t c = c0 + e;
                            if (((mb[u] >> e) & 1u) && c >= 0 && c < p.cols)
                                st_elem<ES>(drow, c, sbt_vec_get<ES>(val[u], e));
                        }
                    }
                }
            }
        } else {
            const int tc = p.tile_c;
            const int ntask = nrows * tc;
            for (int base = threadIdx.x; base < ntask; base += kThreads * kUnroll) {
                T val[kUnroll];
                bool ok[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int t = base + u * kThreads;
                    ok[u] = false;
                    if (t < ntask) {
                        const int row = t / tc;
                        const int j = t - row * tc;
                        const int64_t c = p.col_offset + j;
                        if (((valid >> row) & 1u) && c >= 0 && c < p.cols) {
                            val[u] = ld_elem<ES>(p.src, (k0 + row) * p.ld_dense + j);
                            ok[u] = MM == kNoMask ? true : __ldg(p.mask + (k0 + row) * p.ld_mask + j) != 0;
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    if (!ok[u]) continue;
                    const int t = base + u * kThreads;
                    const int row = t / tc;
                    const int j = t - row * tc;
                    st_elem<ES>(p.dst, rows_of[row] * p.ld_arr + p.col_offset + j, val[u]);
                }
            }
        }
        if (stager) finish_index_stage(p, next, nchunks, next_raw, s_row[buf ^ 1], &s_valid[buf ^ 1]);
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------- column gather (axis 1)

constexpr int kColChunk = 256;  // indices per unit (one output column per thread)
constexpr int kColRows = 32;    // output rows per unit

struct ColParams {
    const char* src;
    char* out;
    const int32_t* idx;
    int64_t rows, cols, ld_src, ld_out, n_idx, row_offset, col_offset;
    int32_t tile_r;
    int64_t n_kchunks, units;
    uint32_t pad_word;
};

template <int ES>
__global__ void __launch_bounds__(kThreads) k_gather_cols(const ColParams p) {
    typedef typename sbt_elem<ES>::T T;
    for (int64_t unit = blockIdx.x; unit < p.units; unit += gridDim.x) {
        const int64_t kc = unit % p.n_kchunks, rb = unit / p.n_kchunks;
        const int64_t k = kc * kColChunk + threadIdx.x;
        int64_t c = -1;
        if (k < p.n_idx) {
            c = (int64_t)__ldg(p.idx + k) + p.col_offset;
            if (c < 0 || c >= p.cols) c = -1;
        }
        const int i0 = (int)(rb * kColRows);
        const int nr = p.tile_r - i0 < kColRows ? p.tile_r - i0 : kColRows;
        if (k < p.n_idx) {
            const int64_t col = c;  // this thread's column, checked once for all its rows
            for (int ib = 0; ib < nr; ib += 8) {
                T v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int64_t r = p.row_offset + i0 + ib + u;
                    v[u] = (T)p.pad_word;
                    if (ib + u < nr && col >= 0 && r >= 0 && r < p.rows)
                        v[u] = __ldg(reinterpret_cast<const T*>(p.src) + r * p.ld_src + col);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (ib + u < nr) reinterpret_cast<T*>(p.out)[(int64_t)(i0 + ib + u) * p.ld_out + k] = v[u];
            }
        }
    }
}

// ---------------------------------------------------------------------------- scatter-add (gather backward)

// Element-type additions done by the L2 (red = reduction without a return value).
// KIND: 4 = fp32, 2 = bf16, 3 = fp16; rounding to nearest even, no flush of subnormals
// for the 16-bit types.
template <int KIND>
__device__ __forceinline__ void red_add_v4(char* p, const uint4& v) {
    if (KIND == 4)
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(__uint_as_float(v.x)),
                     "f"(__uint_as_float(v.y)), "f"(__uint_as_float(v.z)), "f"(__uint_as_float(v.w))
                     : "memory");
    else if (KIND == 2)
        asm volatile("red.global.add.noftz.v4.bf16x2 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
    else
        asm volatile("red.global.add.noftz.v4.f16x2 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
}

template <int KIND>
__device__ __forceinline__ void red_add_elem(char* p, uint32_t bits) {
    if (KIND == 4)
        asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(__uint_as_float(bits)) : "memory");
    else if (KIND == 2)
        asm volatile("red.global.add.noftz.bf16 [%0], %1;" ::"l"(p), "h"((unsigned short)bits) : "memory");
    else
        asm volatile("red.global.add.noftz.f16 [%0], %1;" ::"l"(p), "h"((unsigned short)bits) : "memory");
}

template <int KIND, bool VEC>
__global__ void __launch_bounds__(kThreads) k_scatter_add_rows(const RowParams p) {
    __shared__ int64_t s_row[2][kChunkRows];
    __shared__ uint32_t s_valid[2];
    constexpr int ES = KIND == 4 ? 4 : 2;
    constexpr int V = 16 / ES;
    typedef typename sbt_elem<ES>::T T;
    const int64_t nchunks = (p.n_idx + kChunkRows - 1) / kChunkRows;
    const bool stager = threadIdx.x < 32;
    if (stager) finish_index_stage(p, blockIdx.x, nchunks, issue_index_load(p, blockIdx.x, nchunks), s_row[0], &s_valid[0]);
    __syncthreads();
    int buf = 0;
    for (int64_t chunk = blockIdx.x; chunk < nchunks; chunk += gridDim.x, buf ^= 1) {
        const int64_t next = chunk + gridDim.x;
        const int32_t next_raw = stager ? issue_index_load(p, next, nchunks) : 0;
        const int64_t k0 = chunk * kChunkRows;
        const int nrows = (int)(p.n_idx - k0 < kChunkRows ? p.n_idx - k0 : kChunkRows);
        const uint32_t valid = s_valid[buf];
        const int64_t* rows_of = s_row[buf];
        const int per_row = VEC ? p.nvec : p.tile_c;
        // vectors: one per thread and trip (bf16 1 KiB rows: 0.466 ms at 1, 0.484 at 2, 0.486 at 8)
        constexpr int UA = VEC ? 1 : kUnroll;
        const int ntask = nrows * per_row;
        for (int base = threadIdx.x; base < ntask; base += kThreads * UA) {
            uint4 val[UA];
            T sv[UA];
#pragma unroll
            for (int u = 0; u < UA; ++u) {
                const int t = base + u * kThreads;
                if (t < ntask) {
                    const int row = t / per_row;
                    const int j = (t - row * per_row) * (VEC ? V : 1);
                    if ((valid >> row) & 1u) {
                        if (VEC)
                            val[u] = sbt_ld_nc_v4(p.src + ((k0 + row) * p.ld_dense + j) * ES);
                        else
                            sv[u] = ld_elem<ES>(p.src, (k0 + row) * p.ld_dense + j);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < UA; ++u) {
                const int t = base + u * kThreads;
                if (t >= ntask) continue;
                const int row = t / per_row;
                if (!((valid >> row) & 1u)) continue;
                const int j = (t - row * per_row) * (VEC ? V : 1);
                const int64_t c0 = p.col_offset + j;
                char* drow = p.dst + rows_of[row] * p.ld_arr * ES;
                if (VEC) {
                    if (c0 >= 0 && c0 + V <= p.cols) {
                        red_add_v4<KIND>(drow + c0 * ES, val[u]);
                    } else {
#pragma unroll
                        for (int e = 0; e < V; ++e) {
                            const int64_t c = c0 + e;
                            if (c >= 0 && c < p.cols) red_add_elem<KIND>(drow + c * ES, sbt_vec_get<ES>(val[u], e));
                        }
                    }
                } else if (c0 >= 0 && c0 < p.cols) {
                    red_add_elem<KIND>(drow + c0 * ES, (uint32_t)sv[u]);
                }
            }
        }
        if (stager) finish_index_stage(p, next, nchunks, next_raw, s_row[buf ^ 1], &s_valid[buf ^ 1]);
        __syncthreads();
    }
}

template <int KIND, bool VEC>
sbt_status launch_scatter_add_t(sbt_context* ctx, const RowParams& p, cudaStream_t stream) {
    auto kern = k_scatter_add_rows<KIND, VEC>;
    const int grid = sbt_persistent_grid(ctx, (const void*)kern, kThreads, 0, sbt_cdiv(p.n_idx, kChunkRows));
    kern<<<grid, kThreads, 0, stream>>>(p);
    return sbt_after_launch(ctx, "scatter_add_rows");
}

template <int ES, bool VEC, int MM>
sbt_status launch_gather_t(sbt_context* ctx, const RowParams& p, cudaStream_t stream) {
    auto kern = k_gather_rows<ES, VEC, MM>;
    const int64_t nchunks = sbt_cdiv(p.n_idx, kChunkRows);
    const int grid = sbt_persistent_grid(ctx, (const void*)kern, kThreads, 0, nchunks);
    kern<<<grid, kThreads, 0, stream>>>(p);
    return sbt_after_launch(ctx, "gather_rows");
}

template <int ES, bool VEC, int MM>
sbt_status launch_scatter_t(sbt_context* ctx, const RowParams& p, cudaStream_t stream) {
    auto kern = k_scatter_rows<ES, VEC, MM>;
    const int64_t nchunks = sbt_cdiv(p.n_idx, kChunkRows);
    const int grid = sbt_persistent_grid(ctx, (const void*)kern, kThreads, 0, nchunks);
    kern<<<grid, kThreads, 0, stream>>>(p);
    return sbt_after_launch(ctx, "scatter_rows_masked");
}

template <int ES>
sbt_status dispatch_rows(sbt_context* ctx, bool gather, bool vec, int mm, const RowParams& p, cudaStream_t s) {
#define SBT_ROWS_CASE(VEC_, MM_) \
    return gather ? launch_gather_t<ES, VEC_, MM_>(ctx, p, s) : launch_scatter_t<ES, VEC_, MM_>(ctx, p, s)
    if (vec) {
        if (mm == kNoMask) SBT_ROWS_CASE(true, kNoMask);
        if (mm == kMaskVec) SBT_ROWS_CASE(true, kMaskVec);
        SBT_ROWS_CASE(true, kMaskBytes);
    }
    if (mm == kNoMask) SBT_ROWS_CASE(false, kNoMask);
    SBT_ROWS_CASE(false, kMaskBytes);
#undef SBT_ROWS_CASE
}

// The vector path needs every 16-byte vector of both sides aligned: the
// indexed array at (row r, column col_offset + 16*v bytes) for every r, and
// the dense side at (row k, 16*v bytes) for every k.
bool rows_vector_ok(int es, const void* arr, int64_t ld_arr, int64_t col_offset, const void* dense,
                    int64_t ld_dense, int32_t tile_c) {
    const int V = 16 / es;
    if (tile_c % V) return false;
    if (!sbt_mul16(ld_arr, es) || !sbt_mul16(ld_dense, es) || !sbt_mul16(col_offset, es)) return false;
    if (!sbt_aligned16(dense)) return false;
    if (arr && !sbt_aligned16(arr)) return false;
    return true;
}

int pick_mask_mode(int es, bool vec, const uint8_t* mask, int64_t ld_mask) {
    if (!mask) return kNoMask;
    const int V = 16 / es;
    if (vec && (reinterpret_cast<uintptr_t>(mask) % V) == 0 && (ld_mask % V) == 0) return kMaskVec;
    return kMaskBytes;
}

}  // namespace

sbt_status sbt_launch_gather(sbt_context* ctx, int es, const void* src, int64_t rows, int64_t cols, int64_t ld_src,
                             const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                             int32_t tile_c, const uint8_t* mask, int64_t ld_mask, void* out, int64_t ld_out,
                             uint32_t pad_word, cudaStream_t stream) {
    RowParams p;
    p.src = (const char*)src;
    p.dst = (char*)out;
    p.idx = idx;
    p.mask = mask;
    p.rows = (src && cols > 0) ? rows : 0;  // an empty table makes every row invalid
    p.cols = cols;
    p.ld_arr = ld_src;
    p.ld_dense = ld_out;
    p.ld_mask = ld_mask;
    p.n_idx = n_idx;
    p.row_offset = row_offset;
    p.col_offset = col_offset;
    p.tile_c = tile_c;
    p.pad_word = pad_word;
    // The bulk-copy gather is taken only on request: on the 1 KiB-row workload the
    // register-staged vector path below moves ~3% more bytes per second.
    if (ctx->path == SBT_PATH_TMA && p.rows > 0 &&
        sbt_gather_bulk_ok(es, src, cols, ld_src, col_offset, tile_c, mask, out, ld_out))
        return sbt_launch_gather_bulk(ctx, es, src, rows, ld_src, idx, n_idx, row_offset, col_offset, tile_c, out,
                                      ld_out, pad_word, stream);
    bool vec = rows_vector_ok(es, src, ld_src, col_offset, out, ld_out, tile_c);
    if (ctx->path == SBT_PATH_SCALAR) vec = false;
    p.nvec = vec ? tile_c / (16 / es) : 0;
    const int mm = pick_mask_mode(es, vec, mask, ld_mask);
    return es == 4 ? dispatch_rows<4>(ctx, true, vec, mm, p, stream) : dispatch_rows<2>(ctx, true, vec, mm, p, stream);
}

sbt_status sbt_launch_scatter(sbt_context* ctx, int es, void* dst, int64_t rows, int64_t cols, int64_t ld_dst,
                              const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                              const void* src, int64_t ld_src, int32_t tile_c, const uint8_t* mask, int64_t ld_mask,
                              cudaStream_t stream) {
    RowParams p;
    p.src = (const char*)src;
    p.dst = (char*)dst;
    p.idx = idx;
    p.mask = mask;
    p.rows = rows;
    p.cols = cols;
    p.ld_arr = ld_dst;
    p.ld_dense = ld_src;
    p.ld_mask = ld_mask;
    p.n_idx = n_idx;
    p.row_offset = row_offset;
    p.col_offset = col_offset;
    p.tile_c = tile_c;
    p.pad_word = 0;
    if ((ctx->path == SBT_PATH_AUTO || ctx->path == SBT_PATH_TMA) &&
        sbt_scatter_bulk_ok(es, src, ld_src, tile_c, mask, ld_mask))
        return sbt_launch_scatter_bulk(ctx, es, dst, rows, cols, ld_dst, idx, n_idx, row_offset, col_offset, src,
                                       ld_src, tile_c, mask, ld_mask, stream);
    bool vec = rows_vector_ok(es, dst, ld_dst, col_offset, src, ld_src, tile_c);
    if (ctx->path == SBT_PATH_SCALAR) vec = false;
    p.nvec = vec ? tile_c / (16 / es) : 0;
    const int mm = pick_mask_mode(es, vec, mask, ld_mask);
    return es == 4 ? dispatch_rows<4>(ctx, false, vec, mm, p, stream)
                   : dispatch_rows<2>(ctx, false, vec, mm, p, stream);
}

sbt_status sbt_launch_scatter_add(sbt_context* ctx, int kind, void* dst, int64_t rows, int64_t cols, int64_t ld_dst,
                                  const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                                  const void* src, int64_t ld_src, int32_t tile_c, cudaStream_t stream) {
    const int es = kind == 4 ? 4 : 2;
    RowParams p;
    p.src = (const char*)src;
    p.dst = (char*)dst;
    p.idx = idx;
    p.mask = nullptr;
    p.rows = rows;
    p.cols = cols;
    p.ld_arr = ld_dst;
    p.ld_dense = ld_src;
    p.ld_mask = 0;
    p.n_idx = n_idx;
    p.row_offset = row_offset;
    p.col_offset = col_offset;
    p.tile_c = tile_c;
    p.pad_word = 0;
    bool vec = rows_vector_ok(es, dst, ld_dst, col_offset, src, ld_src, tile_c);
    if (ctx->path == SBT_PATH_SCALAR) vec = false;
    p.nvec = vec ? tile_c / (16 / es) : 0;
#define SBT_SA(K_) return vec ? launch_scatter_add_t<K_, true>(ctx, p, stream) : launch_scatter_add_t<K_, false>(ctx, p, stream)
    if (kind == 4) SBT_SA(4);
    if (kind == 2) SBT_SA(2);
    SBT_SA(3);
#undef SBT_SA
}

sbt_status sbt_launch_gather_cols(sbt_context* ctx, int es, const void* src, int64_t rows, int64_t cols, int64_t ld_src,
                                  const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                                  int32_t tile_r, void* out, int64_t ld_out, uint32_t pad_word, cudaStream_t stream) {
    ColParams p;
    p.src = (const char*)src;
    p.out = (char*)out;
    p.idx = idx;
    p.rows = (src && cols > 0) ? rows : 0;
    p.cols = cols;
    p.ld_src = ld_src;
    p.ld_out = ld_out;
    p.n_idx = n_idx;
    p.row_offset = row_offset;
    p.col_offset = col_offset;
    p.tile_r = tile_r;
    p.n_kchunks = sbt_cdiv(n_idx, kColChunk);
    p.units = p.n_kchunks * sbt_cdiv(tile_r, kColRows);
    p.pad_word = pad_word;
    if (es == 4) {
        const int grid = sbt_persistent_grid(ctx, (const void*)k_gather_cols<4>, kThreads, 0, p.units);
        k_gather_cols<4><<<grid, kThreads, 0, stream>>>(p);
    } else {
        const int grid = sbt_persistent_grid(ctx, (const void*)k_gather_cols<2>, kThreads, 0, p.units);
        k_gather_cols<2><<<grid, kThreads, 0, stream>>>(p);
    }
    return sbt_after_launch(ctx, "gather_cols");
}
