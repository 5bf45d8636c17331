// Clipped tile store into destination rows that are not 16-byte aligned, for
// grids whose tiles sit side by side along the array row (column step equal to
// the tile width), so that the tile rows of one grid row form one run of the
// destination row (cuTile.jl "Memory": clipped stores; Tylo.jl "Boundary
// tiles", section "Accumulator stores and GEMM": bounded stores).
//
// Tasks are 16-byte tile vectors numbered along whole destination rows (grid
// row, tile row, then vectors across all tiles of the grid row), so the 32
// lanes of a warp hold consecutive vectors of one row.  Each lane passes its
// vector one lane up; a lane whose left neighbour holds the previous vector of
// the same row, with both vectors inside the array, writes the aligned 16-byte
// destination chunk that starts inside the neighbour's vector.  The bytes
// before the first such chunk of a run, and after its last, go out element
// by element; a vector that crosses the array's edge stores its in-bounds
// elements one by one.  Every byte written belongs to an element in bounds, so
// the result equals element stores.  (SBT_PATH_VECTOR.)
//
// The default kernel (k_tile_store_runs_bulk) cuts each run into chunks of at
// most 1,024 vectors, one chunk per block at a time, and lets the TMA bulk-copy
// engine write it.  Word j of a chunk is the destination's aligned 16-byte
// word at B + 16 j, B = (address of the chunk's first vector) - sh, sh = that
// address mod 16: the last sh bytes of vector j - 1 and the first 16 - sh of
// vector j (the previous vector comes from the next lane down, through shared
// memory across warps, and from one extra load before the chunk).  Words whose
// bytes all belong to in-bounds elements collect in shared memory and leave in
// one cp.async.bulk shared -> global copy per chunk (both addresses 16-byte
// aligned, a multiple of 16 bytes); the other words (at the ends of a run's
// in-bounds span) and the bytes of a run's last vector past its last word go
// out element by element.
#include <algorithm>

#include "sbt_internal.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace sbt_ptx;

constexpr int kRunThreads = 256;
constexpr unsigned int kFull = 0xffffffffu;

struct RunParams {
    const char* tiles;  // [grid_r][grid_c][tile_r][tile_c], 16-byte aligned
    char* arr;          // destination element (0, 0)
    int64_t rows, cols, stride_r, origin_r, origin_c, step_r;
    uint32_t tile_r, per_row, grid_c;  // per_row: vectors per tile row
    uint32_t width;                    // vectors per destination run: grid_c * per_row
    uint32_t ntasks;                   // grid_r * tile_r * width, below 2^31
    sbt_fastdiv div_width, div_tile_r, div_per_row;
};

__device__ __forceinline__ uint32_t pick4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t q) {
    return q == 0 ? a : q == 1 ? b : q == 2 ? c : d;
}

// Bytes [d, d + 16) of the 32 bytes (lo, hi), d even, 0 < d < 16.
template <int ES>
__device__ __forceinline__ uint4 bytes_from(const uint4& lo, const uint4& hi, uint32_t d) {
    const uint32_t q = d >> 2;
    const uint32_t w0 = pick4(lo.x, lo.y, lo.z, lo.w, q);
    const uint32_t w1 = pick4(lo.y, lo.z, lo.w, hi.x, q);
    const uint32_t w2 = pick4(lo.z, lo.w, hi.x, hi.y, q);
    const uint32_t w3 = pick4(lo.w, hi.x, hi.y, hi.z, q);
    if (ES == 4) return make_uint4(w0, w1, w2, w3);
    const uint32_t w4 = pick4(hi.x, hi.y, hi.z, hi.w, q);
    const uint32_t b = (d & 2u) * 8u;
    return make_uint4(__funnelshift_r(w0, w1, b), __funnelshift_r(w1, w2, b), __funnelshift_r(w2, w3, b),
                      __funnelshift_r(w3, w4, b));
}

template <int ES>
__global__ void __launch_bounds__(kRunThreads) k_tile_store_runs(const RunParams p) {
    constexpr int V = 16 / ES;
    typedef typename sbt_elem<ES>::T T;
    const int lane = threadIdx.x & 31;
    const uint32_t stride = gridDim.x * kRunThreads;
    // the loop bound is the same for the whole warp: the shuffles see every lane
    for (uint32_t wbase = blockIdx.x * kRunThreads + (threadIdx.x & ~31u); wbase < p.ntasks; wbase += stride) {
        const uint32_t t = wbase + lane;
        const bool live = t < p.ntasks;
        uint32_t run = 0xffffffffu;  // destination run (grid row, tile row) of this lane
        int inside = 0;              // the whole vector lies inside the array
        uint4 v = make_uint4(0, 0, 0, 0);
        int64_t r = -1, c = 0;
        if (live) {
            run = sbt_div(p.div_width, t);
            const uint32_t vc = t - run * p.width;
            const uint32_t ti = sbt_div(p.div_tile_r, run);
            const uint32_t i = run - ti * p.tile_r;
            const uint32_t tj = sbt_div(p.div_per_row, vc);
            const uint32_t j = vc - tj * p.per_row;
            const uint64_t tile = (uint64_t)ti * p.grid_c + tj;
            v = sbt_ld_nc_v4(p.tiles + ((tile * p.tile_r + i) * p.per_row + j) * 16);
            r = p.origin_r + (int64_t)ti * p.step_r + i;
            c = p.origin_c + (int64_t)vc * V;
            inside = r >= 0 && r < p.rows && c >= 0 && c + V <= p.cols;
        }
        const uint32_t run_prev = __shfl_up_sync(kFull, run, 1);
        const uint32_t run_next = __shfl_down_sync(kFull, run, 1);
        const int in_prev = __shfl_up_sync(kFull, inside, 1);
        const int in_next = __shfl_down_sync(kFull, inside, 1);
        uint4 prev;
        prev.x = __shfl_up_sync(kFull, v.x, 1);
        prev.y = __shfl_up_sync(kFull, v.y, 1);
        prev.z = __shfl_up_sync(kFull, v.z, 1);
        prev.w = __shfl_up_sync(kFull, v.w, 1);
        if (!live || r < 0 || r >= p.rows) continue;
        if (inside) {
            char* a = p.arr + (r * p.stride_r + c) * ES;
            const uint32_t sh = (uint32_t)(reinterpret_cast<uintptr_t>(a) & 15u);  // the same along the run
            if (sh == 0) {
                sbt_st_v4(a, v);
                continue;
            }
            const bool prev_ok = lane > 0 && run_prev == run && in_prev;   // the chunk before a is written here
            const bool next_ok = lane < 31 && run_next == run && in_next;  // the chunk after is written next door
            if (prev_ok) sbt_st_v4(a - sh, bytes_from<ES>(prev, v, 16u - sh));
            const int head = (int)(16u - sh) / ES;  // elements before the next chunk boundary
#pragma unroll
            for (int e = 0; e < V; ++e) {
                const bool mine = e < head ? !prev_ok : !next_ok;
                if (mine) reinterpret_cast<T*>(a)[e] = sbt_vec_get<ES>(v, e);
            }
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) {
                const int64_t ce = c + e;
                if (ce >= 0 && ce < p.cols)
                    reinterpret_cast<T*>(p.arr)[r * p.stride_r + ce] = sbt_vec_get<ES>(v, e);
            }
        }
    }
}

constexpr int kBulkThreads = 256;
constexpr int kBulkPer = 4;                        // vectors per thread and chunk
constexpr int kBulkVec = kBulkThreads * kBulkPer;  // at most 1,024 vectors (16 KB) per chunk

struct BulkRunParams {
    const char* tiles;  // [grid_r][grid_c][tile_r][tile_c], 16-byte aligned
    char* arr;          // destination element (0, 0)
    int64_t rows, stride_r, origin_r, origin_c, step_r;
    int64_t lo, hi;                    // bytes of a run inside the array: [lo, hi) from the run's column 0
    uint32_t tile_r, per_row, grid_c;  // per_row: vectors per tile row
    uint32_t width;                    // vectors per run: grid_c * per_row
    uint32_t chunk, n_chunks;          // vectors per chunk (a multiple of 32, <= kBulkVec), chunks per run
    uint32_t n_items;                  // runs * n_chunks, below 2^31
    sbt_fastdiv div_chunks, div_tile_r, div_per_row;
};

template <int ES>
__global__ void __launch_bounds__(kBulkThreads) k_tile_store_runs_bulk(const BulkRunParams p) {
    constexpr int V = 16 / ES;
    constexpr int kWarps = kBulkThreads / 32;
    typedef typename sbt_elem<ES>::T T;
    __shared__ __align__(128) uint4 words[kBulkVec];
    __shared__ uint4 edge[kWarps][kBulkPer];  // each warp's lane-31 vectors, for the next warp's lane 0
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (uint32_t item = blockIdx.x; item < p.n_items; item += gridDim.x) {
        const uint32_t run = sbt_div(p.div_chunks, item);
        const uint32_t k = item - run * p.n_chunks;
        const uint32_t ti = sbt_div(p.div_tile_r, run);
        const uint32_t i = run - ti * p.tile_r;
        const int64_t r = p.origin_r + (int64_t)ti * p.step_r + i;
        if (r < 0 || r >= p.rows) continue;  // the same for the whole block
        const uint32_t v0 = k * p.chunk;
        const uint32_t nv = min(p.chunk, p.width - v0);
        // run column 0 as an address (it may lie before the array: only in-bounds bytes are written)
        char* const row = p.arr + (r * p.stride_r + p.origin_c) * ES;
        const uint32_t sh = (uint32_t)(reinterpret_cast<uintptr_t>(row) & 15u);
        const int64_t bo = 16 * (int64_t)v0 - sh;  // word 0 of this chunk, from the run's column 0
        // words j_lo .. j_hi - 1 hold in-bounds elements only
        const int64_t dlo = p.lo - bo, dhi = p.hi - bo;
        const int64_t lo_w = dlo <= 0 ? 0 : (dlo + 15) / 16, hi_w = dhi < 16 ? 0 : dhi / 16;
        const uint32_t j_lo = (uint32_t)(lo_w < nv ? lo_w : nv);
        uint32_t j_hi = (uint32_t)(hi_w < nv ? hi_w : nv);
        if (j_hi < j_lo) j_hi = j_lo;
        const uint64_t row0 = ((uint64_t)ti * p.grid_c * p.tile_r + i) * p.per_row;  // tile (ti, 0), row i
        auto src = [&](uint32_t q) {  // tile vector q of this run
            const uint32_t tj = sbt_div(p.div_per_row, q);
            return p.tiles + (row0 + (uint64_t)tj * p.tile_r * p.per_row + (q - tj * p.per_row)) * 16;
        };
        uint4 v[kBulkPer];
#pragma unroll
        for (int u = 0; u < kBulkPer; ++u) {
            const uint32_t j = tid + kBulkThreads * u;
            v[u] = j < nv ? sbt_ld_nc_v4(src(v0 + j)) : make_uint4(0, 0, 0, 0);
        }
        uint4 before = make_uint4(0, 0, 0, 0);  // vector v0 - 1, for word 0
        if (tid == 0 && sh != 0 && v0 > 0) before = sbt_ld_nc_v4(src(v0 - 1));
        if (lane == 31) {
#pragma unroll
            for (int u = 0; u < kBulkPer; ++u) edge[warp][u] = v[u];
        }
        if (tid == 0) bulk_wait_read<0>();  // the previous chunk's copy has read `words`
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kBulkPer; ++u) {
            const uint32_t j = tid + kBulkThreads * u;
            uint4 prev;
            prev.x = __shfl_up_sync(kFull, v[u].x, 1);
            prev.y = __shfl_up_sync(kFull, v[u].y, 1);
            prev.z = __shfl_up_sync(kFull, v[u].z, 1);
            prev.w = __shfl_up_sync(kFull, v[u].w, 1);
            if (lane == 0) prev = warp > 0 ? edge[warp - 1][u] : u > 0 ? edge[kWarps - 1][u - 1] : before;
            if (j >= nv) continue;
            const uint4 w = sh == 0 ? v[u] : bytes_from<ES>(prev, v[u], 16u - sh);
            if (j >= j_lo && j < j_hi) {
                words[j] = w;
            } else {
                const int64_t wo = bo + 16 * (int64_t)j;
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const int64_t o = wo + e * ES;
                    if (o >= p.lo && o < p.hi) *reinterpret_cast<T*>(row + o) = sbt_vec_get<ES>(w, e);
                }
            }
            if (sh != 0 && v0 + j == p.width - 1) {  // the run's last bytes, past its last word
                const int64_t vo = 16 * (int64_t)(v0 + j);
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const int64_t o = vo + e * ES;
                    if (e * ES >= (int)(16u - sh) && o >= p.lo && o < p.hi)
                        *reinterpret_cast<T*>(row + o) = sbt_vec_get<ES>(v[u], e);
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && j_hi > j_lo) {
            bulk_s2g(row + bo + 16 * (int64_t)j_lo, smem_u32(&words[j_lo]), 16u * (j_hi - j_lo));
            bulk_commit();
        }
    }
    if (tid == 0) bulk_wait<0>();
}

}  // namespace

bool sbt_tile_store_runs_ok(sbt_context* ctx, int es, const void* src_tiles, int32_t grid_r, int32_t grid_c,
                            int32_t tile_r, int32_t tile_c, const void* dst, int64_t stride_r, int64_t stride_c,
                            int64_t origin_c, int64_t step_c) {
    const int V = 16 / es;
    if (ctx->path == SBT_PATH_SCALAR || (es != 2 && es != 4)) return false;
    if (stride_c != 1 || step_c != tile_c || tile_c % V != 0 || !sbt_aligned16(src_tiles)) return false;
    // rows that are 16-byte aligned take the vector and TMA paths
    const bool rows_aligned = ((reinterpret_cast<uintptr_t>(dst) + (uintptr_t)(origin_c * es)) & 15u) == 0 &&
                              ((stride_r * es) & 15) == 0;
    if (rows_aligned) return false;
    const int64_t width = (int64_t)grid_c * (tile_c / V);
    return width < ((int64_t)1 << 31) && (int64_t)grid_r * tile_r * width < ((int64_t)1 << 31);
}

sbt_status sbt_launch_tile_store_runs(sbt_context* ctx, int es, const void* src_tiles, int32_t grid_r,
                                      int32_t grid_c, int32_t tile_r, int32_t tile_c, void* dst, int64_t rows,
                                      int64_t cols, int64_t stride_r, int64_t origin_r, int64_t origin_c,
                                      int64_t step_r, cudaStream_t stream) {
    if (ctx->path != SBT_PATH_VECTOR) {
        BulkRunParams b;
        b.tiles = (const char*)src_tiles;
        b.arr = (char*)dst;
        b.rows = rows;
        b.stride_r = stride_r;
        b.origin_r = origin_r;
        b.origin_c = origin_c;
        b.step_r = step_r;
        b.tile_r = (uint32_t)tile_r;
        b.per_row = (uint32_t)(tile_c / (16 / es));
        b.grid_c = (uint32_t)grid_c;
        b.width = b.grid_c * b.per_row;
        const int64_t run_cols = (int64_t)b.width * (16 / es);
        b.lo = std::max<int64_t>(0, -origin_c) * es;
        b.hi = std::max<int64_t>(std::min<int64_t>(run_cols, cols - origin_c), 0) * es;
        // as few chunks as 1,024-vector chunks need, of equal size rounded up to whole warps
        const uint32_t n = (uint32_t)sbt_cdiv(b.width, kBulkVec);
        b.chunk = (uint32_t)std::min<int64_t>(kBulkVec, (sbt_cdiv(b.width, n) + 31) / 32 * 32);
        b.n_chunks = (uint32_t)sbt_cdiv(b.width, b.chunk);
        b.n_items = (uint32_t)((int64_t)grid_r * tile_r * b.n_chunks);
        b.div_chunks = sbt_make_fastdiv(b.n_chunks);
        b.div_tile_r = sbt_make_fastdiv(b.tile_r);
        b.div_per_row = sbt_make_fastdiv(b.per_row);
        const void* kern = es == 4 ? (const void*)k_tile_store_runs_bulk<4> : (const void*)k_tile_store_runs_bulk<2>;
        const int grid = sbt_persistent_grid(ctx, kern, kBulkThreads, 0, b.n_items);
        if (es == 4)
            k_tile_store_runs_bulk<4><<<grid, kBulkThreads, 0, stream>>>(b);
        else
            k_tile_store_runs_bulk<2><<<grid, kBulkThreads, 0, stream>>>(b);
        return sbt_after_launch(ctx, "tile_store_clipped (row runs, bulk copies)");
    }
    RunParams p;
    p.tiles = (const char*)src_tiles;
    p.arr = (char*)dst;
    p.rows = rows;
    p.cols = cols;
    p.stride_r = stride_r;
    p.origin_r = origin_r;
    p.origin_c = origin_c;
    p.step_r = step_r;
    p.tile_r = (uint32_t)tile_r;
    p.per_row = (uint32_t)(tile_c / (16 / es));
    p.grid_c = (uint32_t)grid_c;
    p.width = p.grid_c * p.per_row;
    p.ntasks = (uint32_t)((int64_t)grid_r * tile_r * p.width);
    p.div_width = sbt_make_fastdiv(p.width);
    p.div_tile_r = sbt_make_fastdiv(p.tile_r);
    p.div_per_row = sbt_make_fastdiv(p.per_row);
    const void* kern = es == 4 ? (const void*)k_tile_store_runs<4> : (const void*)k_tile_store_runs<2>;
    const int grid = sbt_persistent_grid(ctx, kern, kRunThreads, 0, sbt_cdiv(p.ntasks, kRunThreads));
    if (es == 4)
        k_tile_store_runs<4><<<grid, kRunThreads, 0, stream>>>(p);
    else
        k_tile_store_runs<2><<<grid, kRunThreads, 0, stream>>>(p);
    return sbt_after_launch(ctx, "tile_store_clipped (row runs)");
}
