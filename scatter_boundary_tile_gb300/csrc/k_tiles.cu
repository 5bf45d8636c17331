// Padded tile load, clipped tile store (grids of tiles) and the ragged 3D
// tile load.
//
// Tile load/store: one task per 16-byte vector of the contiguous tile side
// (or per element on the scalar path), grid-stride over all tiles of the
// grid.  A vector wholly inside the array takes one 16-byte access; a
// partial vector is handled element by element and no address is formed for
// an element outside the array; a vector wholly outside reads the pad value
// (load) or writes nothing (store).  This is the copy-plan split of Tylo.jl
// "Boundary tiles" (full aligned vectors vs scalar zero-fill), applied per
// vector of the tile; cuTile.jl "Memory", "Bounds checking" fixes padding on
// load and clipping on store.
//
// Ragged load: one block per (sequence, head, 128-row tile) work unit, the
// unit's valid-row count taken once from cu_seqlens (Mojo "RaggedTMA3DTile":
// only `dynamic_dim` rows of a tile are valid); rows past the sequence are
// written as zeros, so the padded output is defined everywhere.
#include "sbt_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

struct TileParams {
    const char* arr;  // load: source array; store: unused
    char* arr_w;      // store: destination array
    const char* tiles_r;  // store: source tiles
    char* tiles_w;        // load: destination tiles
    int64_t rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c;
    int32_t grid_c, tile_r, tile_c;
    int32_t nvc;       // vectors per tile row (vector path)
    int64_t total;     // tasks: vectors (vector path) or elements
    uint32_t pad_word;
};

struct TaskPos {
    int64_t r, c;  // array coordinates of the task's first element
};

// Task t of the contiguous tile side -> array coordinates.  `per_row` is the
// number of tasks per tile row and `w` the elements each task covers.
__device__ __forceinline__ TaskPos tile_task_pos(const TileParams& p, int64_t t, int per_row, int w) {
    const int64_t per_tile = (int64_t)p.tile_r * per_row;
    const int64_t tile = t / per_tile;
    const int within = (int)(t - tile * per_tile);
    const int i = within / per_row;
    const int j = (within - i * per_row) * w;
    const int64_t ti = tile / p.grid_c;
    const int64_t tj = tile - ti * p.grid_c;
    TaskPos q;
    q.r = p.origin_r + ti * p.step_r + i;
    q.c = p.origin_c + tj * p.step_c + j;
    return q;
}

template <int ES>
__device__ __forceinline__ typename sbt_elem<ES>::T ld_elem(const char* base, int64_t off) {
    return __ldg(reinterpret_cast<const typename sbt_elem<ES>::T*>(base) + off);
}

template <int ES>
__device__ __forceinline__ void st_elem(char* base, int64_t off, typename sbt_elem<ES>::T v) {
    reinterpret_cast<typename sbt_elem<ES>::T*>(base)[off] = v;
}

template <int ES, bool VEC>
__global__ void __launch_bounds__(kThreads) k_tile_load(const TileParams p) {
    constexpr int V = 16 / ES;
    typedef typename sbt_elem<ES>::T T;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t base = (int64_t)blockIdx.x * kThreads + threadIdx.x; base < p.total; base += stride * kUnroll) {
        if (VEC) {
            uint4 val[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t t = base + u * stride;
                const uint4 padv = make_uint4(p.pad_word, p.pad_word, p.pad_word, p.pad_word);
                val[u] = padv;
                if (t < p.total) {
                    const TaskPos q = tile_task_pos(p, t, p.nvc, V);
                    if (q.r >= 0 && q.r < p.rows) {
                        if (q.c >= 0 && q.c + V <= p.cols) {
                            val[u] = sbt_ld_nc_v4(p.arr + (q.r * p.stride_r + q.c) * ES);
                        } else if (q.c + V > 0 && q.c < p.cols) {
#pragma unroll
                            for (int e = 0; e < V; ++e) {
                                const int64_t c = q.c + e;
                                if (c >= 0 && c < p.cols)
                                    sbt_vec_set<ES>(val[u], e, ld_elem<ES>(p.arr, q.r * p.stride_r + c));
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t t = base + u * stride;
                if (t < p.total) sbt_st_v4(p.tiles_w + t * 16, val[u]);
            }
        } else {
            T val[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t t = base + u * stride;
                val[u] = (T)p.pad_word;
                if (t < p.total) {
                    const TaskPos q = tile_task_pos(p, t, p.tile_c, 1);
                    if (q.r >= 0 && q.r < p.rows && q.c >= 0 && q.c < p.cols)
                        val[u] = ld_elem<ES>(p.arr, q.r * p.stride_r + q.c * p.stride_c);
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t t = base + u * stride;
                if (t < p.total) st_elem<ES>(p.tiles_w, t, val[u]);
            }
        }
    }
}

template <int ES, bool VEC>
__global__ void __launch_bounds__(kThreads) k_tile_store(const TileParams p) {
    constexpr int V = 16 / ES;
    typedef typename sbt_elem<ES>::T T;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t base = (int64_t)blockIdx.x * kThreads + threadIdx.x; base < p.total; base += stride * kUnroll) {
        if (VEC) {
            uint4 val[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t t = base + u * stride;
                if (t < p.total) val[u] = sbt_ld_nc_v4(p.tiles_r + t * 16);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t t = base + u * stride;
                if (t >= p.total) continue;
                const TaskPos q = tile_task_pos(p, t, p.nvc, V);
                if (q.r < 0 || q.r >= p.rows) continue;
                if (q.c >= 0 && q.c + V <= p.cols) {
                    sbt_st_v4(p.arr_w + (q.r * p.stride_r + q.c) * ES, val[u]);
                } else if (q.c + V > 0 && q.c < p.cols) {
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const int64_t c = q.c + e;
                        if (c >= 0 && c < p.cols) st_elem<ES>(p.arr_w, q.r * p.stride_r + c, sbt_vec_get<ES>(val[u], e));
                    }
                }
            }
        } else {
            T val[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t t = base + u * stride;
                if (t < p.total) val[u] = ld_elem<ES>(p.tiles_r, t);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t t = base + u * stride;
                if (t >= p.total) continue;
                const TaskPos q = tile_task_pos(p, t, p.tile_c, 1);
                if (q.r >= 0 && q.r < p.rows && q.c >= 0 && q.c < p.cols)
                    st_elem<ES>(p.arr_w, q.r * p.stride_r + q.c * p.stride_c, val[u]);
            }
        }
    }
}

// ---------------------------------------------------------------------------- ragged

constexpr int kRaggedRows = 128;
constexpr int kRaggedUnroll = 8;

struct RaggedParams {
    const char* x;
    char* out;
    const int32_t* cu;
    int64_t total_rows, ld_row, ld_head;
    int32_t heads, depth, batch, t_pad;
    int32_t n_rt;      // row tiles per (sequence, head)
    int32_t per_row;   // tasks per output row: depth/V (vector path) or depth
    int64_t units;     // batch * heads * n_rt
};

template <int ES, bool VEC>
__global__ void __launch_bounds__(kThreads) k_ragged_load(const RaggedParams p) {
    constexpr int V = VEC ? 16 / ES : 1;
    typedef typename sbt_elem<ES>::T T;
    for (int64_t unit = blockIdx.x; unit < p.units; unit += gridDim.x) {
        const int rt = (int)(unit % p.n_rt);
        const int64_t bh = unit / p.n_rt;
        const int h = (int)(bh % p.heads);
        const int b = (int)(bh / p.heads);
        const int64_t off = __ldg(p.cu + b);
        const int64_t len = (int64_t)__ldg(p.cu + b + 1) - off;
        const int r0 = rt * kRaggedRows;
        const int nrows = p.t_pad - r0 < kRaggedRows ? p.t_pad - r0 : kRaggedRows;
        // rows [r0, r0 + nvalid) of this tile are inside the sequence
        int64_t nvalid = len - r0;
        nvalid = nvalid < 0 ? 0 : (nvalid > nrows ? nrows : nvalid);
        char* out_tile = p.out + ((bh * p.t_pad + r0) * (int64_t)p.depth) * ES;
        const int ntask = nrows * p.per_row;
        for (int base = threadIdx.x; base < ntask; base += kThreads * kRaggedUnroll) {
            uint4 vv[kRaggedUnroll];
            T sv[kRaggedUnroll];
#pragma unroll
            for (int u = 0; u < kRaggedUnroll; ++u) {
                const int t = base + u * kThreads;
                const int i = t / p.per_row;
                const int j = (t - i * p.per_row) * V;
                const int64_t row = off + r0 + i;
                const bool ok = t < ntask && i < nvalid && row >= 0 && row < p.total_rows;
                const int64_t src = row * p.ld_row + (int64_t)h * p.ld_head + j;
                if (VEC) {
                    vv[u] = ok ? sbt_ld_nc_v4(p.x + src * ES) : make_uint4(0, 0, 0, 0);
                } else {
                    sv[u] = ok ? ld_elem<ES>(p.x, src) : (T)0;
                }
            }
#pragma unroll
            for (int u = 0; u < kRaggedUnroll; ++u) {
                const int t = base + u * kThreads;
                if (t >= ntask) continue;
                if (VEC)
                    sbt_st_v4(out_tile + (int64_t)t * 16, vv[u]);
                else
                    st_elem<ES>(out_tile, t, sv[u]);
            }
        }
    }
}

template <int ES, bool VEC>
sbt_status launch_tile_load_t(sbt_context* ctx, const TileParams& p, cudaStream_t s) {
    auto kern = k_tile_load<ES, VEC>;
    const int grid = sbt_persistent_grid(ctx, (const void*)kern, kThreads, 0, sbt_cdiv(p.total, kThreads));
    kern<<<grid, kThreads, 0, s>>>(p);
    return sbt_after_launch(ctx, "tile_load_padded");
}

template <int ES, bool VEC>
sbt_status launch_tile_store_t(sbt_context* ctx, const TileParams& p, cudaStream_t s) {
    auto kern = k_tile_store<ES, VEC>;
    const int grid = sbt_persistent_grid(ctx, (const void*)kern, kThreads, 0, sbt_cdiv(p.total, kThreads));
    kern<<<grid, kThreads, 0, s>>>(p);
    return sbt_after_launch(ctx, "tile_store_clipped");
}

template <int ES, bool VEC>
sbt_status launch_ragged_t(sbt_context* ctx, const RaggedParams& p, cudaStream_t s) {
    auto kern = k_ragged_load<ES, VEC>;
    const int grid = sbt_persistent_grid(ctx, (const void*)kern, kThreads, 0, p.units);
    kern<<<grid, kThreads, 0, s>>>(p);
    return sbt_after_launch(ctx, "ragged_tile_load");
}

// Every vector of every tile 16-byte aligned on both sides.
bool tiles_vector_ok(int es, const void* arr, int64_t stride_r, int64_t stride_c, int64_t origin_c, int64_t step_c,
                     int32_t grid_c, int32_t tile_c, const void* tiles) {
    const int V = 16 / es;
    if (stride_c != 1 || tile_c % V) return false;
    if (!sbt_mul16(stride_r, es) || !sbt_mul16(origin_c, es)) return false;
    if (grid_c > 1 && !sbt_mul16(step_c, es)) return false;
    if (!sbt_aligned16(tiles)) return false;
    if (arr && !sbt_aligned16(arr)) return false;
    return true;
}

TileParams make_tile_params(int64_t rows, int64_t cols, int64_t stride_r, int64_t stride_c, int64_t origin_r,
                            int64_t origin_c, int64_t step_r, int64_t step_c, int32_t grid_r, int32_t grid_c,
                            int32_t tile_r, int32_t tile_c, bool vec, int es) {
    TileParams p;
    p.arr = nullptr;
    p.arr_w = nullptr;
    p.tiles_r = nullptr;
    p.tiles_w = nullptr;
    p.rows = rows;
    p.cols = cols;
    p.stride_r = stride_r;
    p.stride_c = stride_c;
    p.origin_r = origin_r;
    p.origin_c = origin_c;
    p.step_r = step_r;
    p.step_c = step_c;
    p.grid_c = grid_c;
    p.tile_r = tile_r;
    p.tile_c = tile_c;
    p.nvc = vec ? tile_c / (16 / es) : 0;
    const int64_t elems = (int64_t)grid_r * grid_c * tile_r * tile_c;
    p.total = vec ? elems / (16 / es) : elems;
    p.pad_word = 0;
    return p;
}

}  // namespace

sbt_status sbt_launch_tile_load(sbt_context* ctx, int es, const void* src, int64_t rows, int64_t cols,
                                int64_t stride_r, int64_t stride_c, int64_t origin_r, int64_t origin_c,
                                int64_t step_r, int64_t step_c, int32_t grid_r, int32_t grid_c, int32_t tile_r,
                                int32_t tile_c, void* dst, uint32_t pad_word, cudaStream_t stream) {
    bool vec = tiles_vector_ok(es, src, stride_r, stride_c, origin_c, step_c, grid_c, tile_c, dst);
    if (ctx->path == SBT_PATH_SCALAR) vec = false;
    TileParams p = make_tile_params(src ? rows : 0, src ? cols : 0, stride_r, stride_c, origin_r, origin_c, step_r,
                                    step_c, grid_r, grid_c, tile_r, tile_c, vec, es);
    p.arr = (const char*)src;
    p.tiles_w = (char*)dst;
    p.pad_word = pad_word;
    if (es == 4) return vec ? launch_tile_load_t<4, true>(ctx, p, stream) : launch_tile_load_t<4, false>(ctx, p, stream);
    return vec ? launch_tile_load_t<2, true>(ctx, p, stream) : launch_tile_load_t<2, false>(ctx, p, stream);
}

sbt_status sbt_launch_tile_store(sbt_context* ctx, int es, const void* src_tiles, int32_t grid_r, int32_t grid_c,
                                 int32_t tile_r, int32_t tile_c, void* dst, int64_t rows, int64_t cols,
                                 int64_t stride_r, int64_t stride_c, int64_t origin_r, int64_t origin_c,
                                 int64_t step_r, int64_t step_c, cudaStream_t stream) {
    bool vec = tiles_vector_ok(es, dst, stride_r, stride_c, origin_c, step_c, grid_c, tile_c, src_tiles);
    if (ctx->path == SBT_PATH_SCALAR) vec = false;
    TileParams p = make_tile_params(rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c, grid_r,
                                    grid_c, tile_r, tile_c, vec, es);
    p.arr_w = (char*)dst;
    p.tiles_r = (const char*)src_tiles;
    if (es == 4)
        return vec ? launch_tile_store_t<4, true>(ctx, p, stream) : launch_tile_store_t<4, false>(ctx, p, stream);
    return vec ? launch_tile_store_t<2, true>(ctx, p, stream) : launch_tile_store_t<2, false>(ctx, p, stream);
}

sbt_status sbt_launch_ragged(sbt_context* ctx, int es, const void* x, int64_t total_rows, int32_t heads,
                             int32_t depth, int64_t ld_row, int64_t ld_head, const int32_t* cu_seqlens,
                             int32_t batch, int32_t t_pad, void* out, cudaStream_t stream) {
    const int V = 16 / es;
    bool vec = (depth % V) == 0 && sbt_aligned16(out) && (!x || sbt_aligned16(x)) && sbt_mul16(ld_row, es) &&
               sbt_mul16(ld_head, es);
    if (ctx->path == SBT_PATH_SCALAR) vec = false;
    RaggedParams p;
    p.x = (const char*)x;
    p.out = (char*)out;
    p.cu = cu_seqlens;
    p.total_rows = x ? total_rows : 0;
    p.ld_row = ld_row;
    p.ld_head = ld_head;
    p.heads = heads;
    p.depth = depth;
    p.batch = batch;
    p.t_pad = t_pad;
    p.n_rt = (int32_t)sbt_cdiv(t_pad, kRaggedRows);
    p.per_row = vec ? depth / V : depth;
    p.units = (int64_t)batch * heads * p.n_rt;
    if (es == 4) return vec ? launch_ragged_t<4, true>(ctx, p, stream) : launch_ragged_t<4, false>(ctx, p, stream);
    return vec ? launch_ragged_t<2, true>(ctx, p, stream) : launch_ragged_t<2, false>(ctx, p, stream);
}
