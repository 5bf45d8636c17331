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
// Ragged load: one block per (sequence, 128-row tile, head) work unit, the
// unit's valid-row count taken once from cu_seqlens (Mojo "RaggedTMA3DTile":
// only `dynamic_dim` rows of a tile are valid); rows past the sequence are
// written as zeros, so the padded output is defined everywhere.
#include "sbt_internal.cuh"

namespace {

constexpr int kThreads = 256;

// Copy paths of the tile kernels (chosen per call on the host):
//   kAligned -- every vector of the call is 16-byte aligned on both sides;
//   kRealign -- the tile side is aligned, the array's rows are not: a vector
//               of the array is assembled from the two aligned 16-byte chunks
//               that cover it (only when both chunks lie inside the array's
//               byte span, so nothing outside the caller's buffer is read);
//   kElem    -- element by element (column stride != 1, odd tile widths, or
//               unaligned stores; the store's element path is one warp per
//               tile, k_tile_store_rows).
enum TileMode { kAligned = 0, kRealign = 1, kElem = 2 };

struct TileParams {
    const char* arr;      // load: source array
    char* arr_w;          // store: destination array
    const char* tiles_r;  // store: source tiles
    char* tiles_w;        // load: destination tiles
    int64_t rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c;
    int32_t grid_c, tile_r, tile_c;
    uint32_t per_row;      // tasks per tile row: vectors or elements
    uint32_t per_tile;     // tile_r * per_row
    sbt_fastdiv div_per_tile, div_per_row, div_grid_c;
    uint32_t tile0;        // first tile of this launch
    uint32_t ntasks;       // tasks of this launch (< 2^31)
    uint32_t pad_word;
    uint64_t arr_lo, arr_hi;  // byte span [lo, hi) of the array (realign path)
};

struct TaskPos {
    int64_t r, c;      // array coordinates of the task's first element
    int64_t linear;    // index of the task in the whole contiguous tile array
};

// Task t of this launch -> array coordinates, with 32-bit multiply-shift divisions.
__device__ __forceinline__ TaskPos tile_task_pos(const TileParams& p, uint32_t t, int w) {
    const uint32_t tile_rel = sbt_div(p.div_per_tile, t);
    const uint32_t within = t - tile_rel * p.per_tile;
    const uint32_t i = sbt_div(p.div_per_row, within);
    const uint32_t j = (within - i * p.per_row) * (uint32_t)w;
    const uint32_t tile = p.tile0 + tile_rel;
    const uint32_t ti = sbt_div(p.div_grid_c, tile);
    const uint32_t tj = tile - ti * (uint32_t)p.grid_c;
    TaskPos q;
    q.r = p.origin_r + (int64_t)ti * p.step_r + i;
    q.c = p.origin_c + (int64_t)tj * p.step_c + j;
    q.linear = (int64_t)p.tile0 * p.per_tile + t;
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

__device__ __forceinline__ uint32_t sel4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t q) {
    return q == 0 ? a : q == 1 ? b : q == 2 ? c : d;
}

// Bytes [d, d + 16) of the 32 bytes (lo, hi) for an even d, 0 < d < 16: word
// selects, then (2-byte elements only) one 16-bit funnel shift per word.
template <int ES>
__device__ __forceinline__ uint4 realign16_even(const uint4& lo, const uint4& hi, uint32_t d) {
    const uint32_t q = d >> 2;
    const uint32_t s0 = sel4(lo.x, lo.y, lo.z, lo.w, q);
    const uint32_t s1 = sel4(lo.y, lo.z, lo.w, hi.x, q);
    const uint32_t s2 = sel4(lo.z, lo.w, hi.x, hi.y, q);
    const uint32_t s3 = sel4(lo.w, hi.x, hi.y, hi.z, q);
    if (ES == 4) return make_uint4(s0, s1, s2, s3);
    const uint32_t s4 = sel4(hi.x, hi.y, hi.z, hi.w, q);
    const uint32_t b = (d & 2u) * 8u;  // 0 or 16 bits
    return make_uint4(__funnelshift_r(s0, s1, b), __funnelshift_r(s1, s2, b), __funnelshift_r(s2, s3, b),
                      __funnelshift_r(s3, s4, b));
}

// One 16-byte vector of array row r starting at column c (the whole vector in bounds).
template <int ES, int MODE>
__device__ __forceinline__ uint4 load_row_vector(const TileParams& p, int64_t r, int64_t c) {
    const char* a = p.arr + (r * p.stride_r + c) * ES;
    if (MODE == kAligned) return sbt_ld_nc_v4(a);
    const uint64_t addr = reinterpret_cast<uint64_t>(a);
    const uint32_t s = (uint32_t)(addr & 15u);
    if (s == 0) return sbt_ld_nc_v4(a);
    const uint64_t base = addr - s;
    if (base >= p.arr_lo && base + 32 <= p.arr_hi) {
        const uint4 lo = sbt_ld_nc_v4_l1(reinterpret_cast<const void*>(base));
        const uint4 hi = sbt_ld_nc_v4_l1(reinterpret_cast<const void*>(base + 16));
        return realign16_even<ES>(lo, hi, s);
    }
    uint4 v = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int e = 0; e < 16 / ES; ++e) sbt_vec_set<ES>(v, e, ld_elem<ES>(p.arr, r * p.stride_r + c + e));
    return v;
}

template <int ES, int MODE>
__global__ void __launch_bounds__(kThreads) k_tile_load(const TileParams p) {
    constexpr int V = 16 / ES;
    // Vectors per thread and loop trip: one.  With more, the realign path's
    // chunk pairs overflow L1 before neighbouring lanes reuse them (unaligned fp32
    // 16,381 x 16,411: 0.373 ms at 1, 0.400 at 2, 0.427 at 4, 0.486 at 8), and the
    // aligned path gains nothing either (0.349 / 0.351 / 0.357 ms at 1 / 2 / 4).
    constexpr int U = MODE == kElem ? 8 : 1;
    typedef typename sbt_elem<ES>::T T;
    const uint32_t stride = gridDim.x * kThreads;
    for (uint32_t base = blockIdx.x * kThreads + threadIdx.x; base < p.ntasks; base += stride * U) {
        if (MODE != kElem) {
            uint4 val[U];
            int64_t lin[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t t = base + u * stride;
                val[u] = make_uint4(p.pad_word, p.pad_word, p.pad_word, p.pad_word);
                lin[u] = -1;
                if (t < p.ntasks) {
                    const TaskPos q = tile_task_pos(p, t, V);
                    lin[u] = q.linear;
                    if (q.r >= 0 && q.r < p.rows) {
                        if (q.c >= 0 && q.c + V <= p.cols) {
                            val[u] = load_row_vector<ES, MODE>(p, q.r, q.c);
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
            for (int u = 0; u < U; ++u) {
                if (lin[u] < 0) continue;
                // aligned path: streaming stores (tiles not read again here; 0.349 -> 0.337 ms on the
                // 16,384 x 16,416 fp32 grid); the realign path measured 2% slower with them
                if (MODE == kAligned)
                    sbt_st_v4_cs(p.tiles_w + lin[u] * 16, val[u]);
                else
                    sbt_st_v4(p.tiles_w + lin[u] * 16, val[u]);
            }
        } else {
            T val[U];
            int64_t lin[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t t = base + u * stride;
                val[u] = (T)p.pad_word;
                lin[u] = -1;
                if (t < p.ntasks) {
                    const TaskPos q = tile_task_pos(p, t, 1);
                    lin[u] = q.linear;
                    if (q.r >= 0 && q.r < p.rows && q.c >= 0 && q.c < p.cols)
                        val[u] = ld_elem<ES>(p.arr, q.r * p.stride_r + q.c * p.stride_c);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (lin[u] >= 0) st_elem<ES>(p.tiles_w, lin[u], val[u]);
        }
    }
}

// Vector path of the clipped store (every vector 16-byte aligned on both
// sides); the element path is k_tile_store_rows below.
template <int ES>
__global__ void __launch_bounds__(kThreads) k_tile_store(const TileParams p) {
    constexpr int V = 16 / ES;
    constexpr int U = 1;  // vectors per thread and trip (aligned fp32 store: 0.337 ms at 1, 0.351 at 2, 0.354 at 4, 0.365 at 8)
    const uint32_t stride = gridDim.x * kThreads;
    for (uint32_t base = blockIdx.x * kThreads + threadIdx.x; base < p.ntasks; base += stride * U) {
        uint4 val[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t t = base + u * stride;
            if (t < p.ntasks) val[u] = sbt_ld_nc_v4(p.tiles_r + ((int64_t)p.tile0 * p.per_tile + t) * 16);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t t = base + u * stride;
            if (t >= p.ntasks) continue;
            const TaskPos q = tile_task_pos(p, t, V);
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
    }
}

// Element path of the clipped store, one warp per tile.  A tile's rows are
// contiguous on the tile side, so lane j moves column j (then j + 32, ...) of
// every row with one 2- or 4-byte load and store.  The tile's array origin,
// its in-bounds row range and each lane's column test are worked out once
// per tile, so a row costs a few address additions; rows outside the array
// are not visited.  (One task per element, each decoding its own tile, row and
// column, was instruction-bound at 0.62 ms on the unaligned fp32 workload.
// A vector kernel that passed each tile vector one lane up and wrote aligned
// 16-byte destination chunks, the row ends element by element, took 0.70 ms
// there: its many partial-sector writes cost more than this kernel's 4-byte
// ones.)
template <int ES>
__global__ void __launch_bounds__(kThreads) k_tile_store_rows(const TileParams p, uint32_t ntiles) {
    typedef typename sbt_elem<ES>::T T;
    constexpr int U = 32;  // rows in flight per lane (8: 0.51 ms, 16: 0.49, 32: 0.445, 64: 0.53 on the unaligned fp32 workload)
    const int lane = threadIdx.x & 31;
    const uint32_t nwarps = gridDim.x * (kThreads / 32);
    const int64_t tile_elems = (int64_t)p.tile_r * p.tile_c;
    for (uint32_t t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); t < ntiles; t += nwarps) {
        const uint32_t tr = sbt_div(p.div_grid_c, t);
        const uint32_t tc = t - tr * (uint32_t)p.grid_c;
        const int64_t r0 = p.origin_r + (int64_t)tr * p.step_r;
        const int64_t c0 = p.origin_c + (int64_t)tc * p.step_c;
        // tile rows i with 0 <= r0 + i < rows
        const int i_lo = r0 >= 0 ? 0 : (int)(-r0 < p.tile_r ? -r0 : p.tile_r);
        const int i_hi = p.rows - r0 <= 0 ? 0 : (int)(p.rows - r0 < p.tile_r ? p.rows - r0 : p.tile_r);
        const T* src = reinterpret_cast<const T*>(p.tiles_r) + (int64_t)t * tile_elems;
        T* dst = reinterpret_cast<T*>(p.arr_w);
        for (int j = lane; j < p.tile_c; j += 32) {
            const int64_t c = c0 + j;
            const bool col_ok = c >= 0 && c < p.cols;
            const int64_t col_off = c * p.stride_c;
            for (int i0 = i_lo; i0 < i_hi; i0 += U) {
                T v[U];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    v[u] = i0 + u < i_hi ? src[(int64_t)(i0 + u) * p.tile_c + j] : T(0);
                if (col_ok) {
                    const int64_t row_off = (r0 + i0) * p.stride_r + col_off;
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (i0 + u < i_hi) dst[row_off + (int64_t)u * p.stride_r] = v[u];
                }
            }
        }
    }
}

template <int ES>
sbt_status launch_tile_store_rows(sbt_context* ctx, const TileParams& p, int64_t ntiles, cudaStream_t s) {
    auto kern = k_tile_store_rows<ES>;
    const int grid = sbt_persistent_grid(ctx, (const void*)kern, kThreads, 0, sbt_cdiv(ntiles, kThreads / 32));
    kern<<<grid, kThreads, 0, s>>>(p, (uint32_t)ntiles);
    return sbt_after_launch(ctx, "tile_store_clipped (element rows)");
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
        // heads vary fastest, so blocks running together cover whole packed rows
        const int h = (int)(unit % p.heads);
        const int64_t brt = unit / p.heads;
        const int rt = (int)(brt % p.n_rt);
        const int b = (int)(brt / p.n_rt);
        const int64_t bh = (int64_t)b * p.heads + h;
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

// Launches `kern` over all tiles, splitting so that each launch has fewer than 2^31 tasks.
template <typename Kern>
sbt_status launch_tiles(sbt_context* ctx, Kern kern, TileParams p, int64_t ntiles, const char* what, cudaStream_t s) {
    const int64_t max_tiles = ((int64_t)1 << 31) / 2 / p.per_tile;
    for (int64_t t0 = 0; t0 < ntiles; t0 += max_tiles) {
        const int64_t nt = ntiles - t0 < max_tiles ? ntiles - t0 : max_tiles;
        p.tile0 = (uint32_t)t0;
        p.ntasks = (uint32_t)(nt * p.per_tile);
        const int grid = sbt_persistent_grid(ctx, (const void*)kern, kThreads, 0, sbt_cdiv(p.ntasks, kThreads));
        kern<<<grid, kThreads, 0, s>>>(p);
        sbt_status st = sbt_after_launch(ctx, what);
        if (st) return st;
    }
    return SBT_OK;
}

// Inverse of k_ragged_load: only the unit's valid rows are read from the
// tiles and written to the packed array; rows past the sequence are skipped.
template <int ES, bool VEC>
__global__ void __launch_bounds__(kThreads) k_ragged_store(const RaggedParams p) {
    constexpr int V = VEC ? 16 / ES : 1;
    typedef typename sbt_elem<ES>::T T;
    for (int64_t unit = blockIdx.x; unit < p.units; unit += gridDim.x) {
        // heads vary fastest, so blocks running together cover whole packed rows
        const int h = (int)(unit % p.heads);
        const int64_t brt = unit / p.heads;
        const int rt = (int)(brt % p.n_rt);
        const int b = (int)(brt / p.n_rt);
        const int64_t bh = (int64_t)b * p.heads + h;
        const int64_t off = __ldg(p.cu + b);
        const int64_t len = (int64_t)__ldg(p.cu + b + 1) - off;
        const int r0 = rt * kRaggedRows;
        const int nrows = p.t_pad - r0 < kRaggedRows ? p.t_pad - r0 : kRaggedRows;
        int64_t nvalid = len - r0;
        nvalid = nvalid < 0 ? 0 : (nvalid > nrows ? nrows : nvalid);
        if (nvalid == 0) continue;
        const char* in_tile = p.x + ((bh * p.t_pad + r0) * (int64_t)p.depth) * ES;
        const int ntask = (int)nvalid * p.per_row;
        for (int base = threadIdx.x; base < ntask; base += kThreads * kRaggedUnroll) {
            uint4 vv[kRaggedUnroll];
            T sv[kRaggedUnroll];
#pragma unroll
            for (int u = 0; u < kRaggedUnroll; ++u) {
                const int t = base + u * kThreads;
                if (t < ntask) {
                    if (VEC)
                        vv[u] = sbt_ld_nc_v4(in_tile + (int64_t)t * 16);
                    else
                        sv[u] = ld_elem<ES>(in_tile, t);
                }
            }
#pragma unroll
            for (int u = 0; u < kRaggedUnroll; ++u) {
                const int t = base + u * kThreads;
                if (t >= ntask) continue;
                const int i = t / p.per_row;
                const int j = (t - i * p.per_row) * V;
                const int64_t row = off + r0 + i;
                if (row < 0 || row >= p.total_rows) continue;
                const int64_t dst = row * p.ld_row + (int64_t)h * p.ld_head + j;
                if (VEC)
                    sbt_st_v4(p.out + dst * ES, vv[u]);
                else
                    st_elem<ES>(p.out, dst, sv[u]);
            }
        }
    }
}

template <int ES, bool VEC>
sbt_status launch_ragged_store_t(sbt_context* ctx, const RaggedParams& p, cudaStream_t s) {
    auto kern = k_ragged_store<ES, VEC>;
    const int grid = sbt_persistent_grid(ctx, (const void*)kern, kThreads, 0, p.units);
    kern<<<grid, kThreads, 0, s>>>(p);
    return sbt_after_launch(ctx, "ragged_tile_store");
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

sbt_status make_tile_params(TileParams* pp, int64_t rows, int64_t cols, int64_t stride_r, int64_t stride_c,
                            int64_t origin_r, int64_t origin_c, int64_t step_r, int64_t step_c, int32_t grid_r,
                            int32_t grid_c, int32_t tile_r, int32_t tile_c, bool vec, int es, int64_t* ntiles) {
    TileParams& p = *pp;
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
    p.per_row = vec ? (uint32_t)(tile_c / (16 / es)) : (uint32_t)tile_c;
    p.per_tile = (uint32_t)tile_r * p.per_row;
    p.div_per_tile = sbt_make_fastdiv(p.per_tile);
    p.div_per_row = sbt_make_fastdiv(p.per_row);
    p.div_grid_c = sbt_make_fastdiv((uint32_t)grid_c);
    p.tile0 = 0;
    p.ntasks = 0;
    p.pad_word = 0;
    p.arr_lo = p.arr_hi = 0;
    *ntiles = (int64_t)grid_r * grid_c;
    if (*ntiles >= ((int64_t)1 << 31)) return sbt_fail(SBT_ERR_UNSUPPORTED, "tile grid with 2^31 or more tiles");
    return SBT_OK;
}

// The realign path: column stride 1, rows moving forward, the tile side aligned.
bool tiles_realign_ok(int es, int64_t stride_r, int64_t stride_c, int32_t tile_c, const void* tiles) {
    return stride_c == 1 && stride_r > 0 && tile_c % (16 / es) == 0 && sbt_aligned16(tiles);
}

}  // namespace

sbt_status sbt_launch_tile_load(sbt_context* ctx, int es, const void* src, int64_t rows, int64_t cols,
                                int64_t stride_r, int64_t stride_c, int64_t origin_r, int64_t origin_c,
                                int64_t step_r, int64_t step_c, int32_t grid_r, int32_t grid_c, int32_t tile_r,
                                int32_t tile_c, void* dst, uint32_t pad_word, cudaStream_t stream) {
    if (!src) rows = cols = 0;  // an empty array: every element is padding
    // TMA tiles when asked, or by default for tiles of 16 KiB and more (measured: even with the
    // vector path at 8 KiB, ~2% ahead at 32 KiB on a 16,384 x 16,416 fp32 array).
    const bool big_tile = (int64_t)tile_r * tile_c * es >= 16384;
    if ((ctx->path == SBT_PATH_TMA || (ctx->path == SBT_PATH_AUTO && big_tile)) &&
        sbt_tile_tma_ok(es, src, rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c, grid_r, grid_c,
                        tile_r, tile_c, dst, false))
        return sbt_launch_tile_load_tma(ctx, es, src, rows, cols, stride_r, origin_r, origin_c, step_r, step_c, grid_r,
                                        grid_c, tile_r, tile_c, dst, pad_word, stream);
    int mode = tiles_vector_ok(es, src, stride_r, stride_c, origin_c, step_c, grid_c, tile_c, dst) ? kAligned
               : (src && tiles_realign_ok(es, stride_r, stride_c, tile_c, dst)) ? kRealign
                                                                                : kElem;
    if (ctx->path == SBT_PATH_SCALAR) mode = kElem;
    TileParams p;
    int64_t ntiles = 0;
    sbt_status st = make_tile_params(&p, rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c, grid_r,
                                     grid_c, tile_r, tile_c, mode != kElem, es, &ntiles);
    if (st) return st;
    p.arr = (const char*)src;
    p.tiles_w = (char*)dst;
    p.pad_word = pad_word;
    if (mode == kRealign) {
        p.arr_lo = reinterpret_cast<uint64_t>(src);
        p.arr_hi = p.arr_lo + (uint64_t)(((rows > 0 ? rows - 1 : 0) * stride_r + cols) * es);
    }
    const char* what = "tile_load_padded";
#define SBT_TL(ES_, M_) return launch_tiles(ctx, k_tile_load<ES_, M_>, p, ntiles, what, stream)
    if (es == 4) {
        if (mode == kAligned) SBT_TL(4, kAligned);
        if (mode == kRealign) SBT_TL(4, kRealign);
        SBT_TL(4, kElem);
    }
    if (mode == kAligned) SBT_TL(2, kAligned);
    if (mode == kRealign) SBT_TL(2, kRealign);
    SBT_TL(2, kElem);
#undef SBT_TL
}

sbt_status sbt_launch_tile_store(sbt_context* ctx, int es, const void* src_tiles, int32_t grid_r, int32_t grid_c,
                                 int32_t tile_r, int32_t tile_c, void* dst, int64_t rows, int64_t cols,
                                 int64_t stride_r, int64_t stride_c, int64_t origin_r, int64_t origin_c,
                                 int64_t step_r, int64_t step_c, cudaStream_t stream) {
    const bool big_tile = (int64_t)tile_r * tile_c * es >= 16384;
    if ((ctx->path == SBT_PATH_TMA || (ctx->path == SBT_PATH_AUTO && big_tile)) &&
        sbt_tile_tma_ok(es, dst, rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c, grid_r, grid_c,
                        tile_r, tile_c, src_tiles, true))
        return sbt_launch_tile_store_tma(ctx, es, src_tiles, grid_r, grid_c, tile_r, tile_c, dst, rows, cols, stride_r,
                                         origin_r, origin_c, step_r, step_c, stream);
    int mode = tiles_vector_ok(es, dst, stride_r, stride_c, origin_c, step_c, grid_c, tile_c, src_tiles) ? kAligned
                                                                                                         : kElem;
    if (ctx->path == SBT_PATH_SCALAR) mode = kElem;
    TileParams p;
    int64_t ntiles = 0;
    sbt_status st = make_tile_params(&p, rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c, grid_r,
                                     grid_c, tile_r, tile_c, mode != kElem, es, &ntiles);
    if (st) return st;
    p.arr_w = (char*)dst;
    p.tiles_r = (const char*)src_tiles;
    const char* what = "tile_store_clipped";
    if (mode == kElem)
        return es == 4 ? launch_tile_store_rows<4>(ctx, p, ntiles, stream)
                       : launch_tile_store_rows<2>(ctx, p, ntiles, stream);
    return es == 4 ? launch_tiles(ctx, k_tile_store<4>, p, ntiles, what, stream)
                   : launch_tiles(ctx, k_tile_store<2>, p, ntiles, what, stream);
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

sbt_status sbt_launch_ragged_store(sbt_context* ctx, int es, const void* tiles, int32_t batch, int32_t heads,
                                   int32_t depth, int32_t t_pad, const int32_t* cu_seqlens, void* x,
                                   int64_t total_rows, int64_t ld_row, int64_t ld_head, cudaStream_t stream) {
    const int V = 16 / es;
    bool vec = (depth % V) == 0 && sbt_aligned16(tiles) && sbt_aligned16(x) && sbt_mul16(ld_row, es) &&
               sbt_mul16(ld_head, es);
    if (ctx->path == SBT_PATH_SCALAR) vec = false;
    RaggedParams p;
    p.x = (const char*)tiles;  // the dense side is read here
    p.out = (char*)x;          // and the packed side written
    p.cu = cu_seqlens;
    p.total_rows = total_rows;
    p.ld_row = ld_row;
    p.ld_head = ld_head;
    p.heads = heads;
    p.depth = depth;
    p.batch = batch;
    p.t_pad = t_pad;
    p.n_rt = (int32_t)sbt_cdiv(t_pad, kRaggedRows);
    p.per_row = vec ? depth / V : depth;
    p.units = (int64_t)batch * heads * p.n_rt;
    if (es == 4)
        return vec ? launch_ragged_store_t<4, true>(ctx, p, stream) : launch_ragged_store_t<4, false>(ctx, p, stream);
    return vec ? launch_ragged_store_t<2, true>(ctx, p, stream) : launch_ragged_store_t<2, false>(ctx, p, stream);
}
