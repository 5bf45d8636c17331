// Padded tile load and clipped tile store through TMA tensor copies.
//
// Taken for aligned tiles (cuTile.jl "Memory": loads and stores take a TMA
// hint; the host decides here from alignment): column stride 1, row stride,
// base and row width (cols * element size) 16-byte aligned, tile width a
// multiple of 16 bytes, every tile's first column 16-byte aligned, tiles of at
// most 32 KiB.  The row width matters because the hardware bounds the inner
// dimension in whole 16-byte chunks: a store box that ends inside a chunk
// writes the whole chunk.
//  - load: a 2D tensor-map tile load brings the whole box into shared memory;
//    the hardware fills every element outside the array with zero bits
//    (cuTile.jl "Memory", "Bounds checking": loads are padded).  When the pad
//    value is not zero, the warp rewrites the outside elements of edge tiles
//    in shared memory.  The tile then leaves with one bulk shared->global copy
//    into the contiguous tile array.
//  - store: one bulk copy brings the contiguous tile into shared memory and a
//    2D tensor-map store writes it; the hardware drops every element outside
//    the array (stores are clipped).  Used only when every tile origin is
//    non-negative.
// One warp per block drives a ring of kStages tiles; lane 0 issues the copies.
// Every wait is bounded; a timeout sets the device status flag and the warp
// leaves together after draining (bounded) its copies in flight.
#include <string>

#include "sbt_internal.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace sbt_ptx;

constexpr int kStages = 4;
constexpr uint32_t kMaxTileBytes = 32768;
constexpr unsigned int kCodeTileTma = 0x2000;

struct TileTmaParams {
    char* tiles_w;         // load: destination tiles
    const char* tiles_r;   // store: source tiles
    int64_t rows, cols;
    int64_t origin_r, origin_c, step_r, step_c;
    int32_t grid_c, tile_r, tile_c;
    int64_t ntiles;
    uint32_t tile_bytes, stage_bytes;
    uint32_t pad_word;
    int pad_fix;           // load: rewrite outside elements with the pad value
    unsigned int* status;
    uint64_t wait_ns;
};

__device__ __forceinline__ void tile_origin(const TileTmaParams& p, int64_t tile, int32_t* r, int32_t* c) {
    const int64_t ti = tile / p.grid_c, tj = tile - ti * p.grid_c;
    *r = (int32_t)(p.origin_r + ti * p.step_r);
    *c = (int32_t)(p.origin_c + tj * p.step_c);
}

template <int ES>
__global__ void __launch_bounds__(32) k_tile_load_tma(const __grid_constant__ CUtensorMap map, const TileTmaParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[kStages];
    __shared__ int s_abort;
    typedef typename sbt_elem<ES>::T T;
    const int lane = threadIdx.x;
    const int64_t my_tiles = p.ntiles > blockIdx.x ? (p.ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t full0 = smem_u32(full), stage0 = smem_u32(smem);
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(full0 + 8 * s, 1);
        s_abort = 0;
        fence_mbar_init();
        prefetch_tmap(&map);
    }
    __syncwarp();
    auto tile_of = [&](int64_t i) { return (int64_t)blockIdx.x + i * gridDim.x; };
    auto issue = [&](int64_t i, int st) {
        int32_t r, c;
        tile_origin(p, tile_of(i), &r, &c);
        mbar_arrive_expect_tx(full0 + 8 * st, p.tile_bytes);
        tma_load_2d(stage0 + st * p.stage_bytes, &map, c, r, full0 + 8 * st);
    };
    if (lane == 0)
        for (int64_t i = 0; i < kStages - 1 && i < my_tiles; ++i) issue(i, (int)i);
    int64_t i = 0;
    for (; i < my_tiles; ++i) {
        const int st = (int)(i % kStages);
        const bool ok = mbar_wait_bounded(full0 + 8 * st, (uint32_t)((i / kStages) & 1), p.wait_ns, &s_abort,
                                          p.status, kCodeTileTma);
        if (__any_sync(0xffffffffu, !ok)) break;  // the warp leaves together
        const int64_t tile = tile_of(i);
        int32_t r0, c0;
        tile_origin(p, tile, &r0, &c0);
        if (p.pad_fix && (r0 < 0 || c0 < 0 || r0 + p.tile_r > p.rows || c0 + p.tile_c > p.cols)) {
            T* t = reinterpret_cast<T*>(smem + (size_t)st * p.stage_bytes);
            for (int e = lane; e < p.tile_r * p.tile_c; e += 32) {
                const int ii = e / p.tile_c, jj = e - ii * p.tile_c;
                const int64_t r = (int64_t)r0 + ii, c = (int64_t)c0 + jj;
                if (r < 0 || r >= p.rows || c < 0 || c >= p.cols) t[e] = (T)p.pad_word;
            }
            fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
            bulk_s2g(p.tiles_w + tile * (int64_t)p.tile_bytes, stage0 + st * p.stage_bytes, p.tile_bytes);
            bulk_commit();
            const int64_t j = i + kStages - 1;
            if (j < my_tiles) {
                if (i >= 1) bulk_wait_read<1>();  // the store of tile i-1 has read its stage
                issue(j, (int)(j % kStages));
            }
        }
        __syncwarp();
    }
    if (lane == 0) {
        bulk_wait<0>();
        for (int64_t k = i; k < my_tiles && k < i + kStages - 1; ++k) {  // stopped early: loads in flight
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(full0 + 8 * (k % kStages), (uint32_t)((k / kStages) & 1)) &&
                   globaltimer() - t0 < p.wait_ns) {
            }
        }
    }
}

__global__ void __launch_bounds__(32) k_tile_store_tma(const __grid_constant__ CUtensorMap map, const TileTmaParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[kStages];
    __shared__ int s_abort;
    const int lane = threadIdx.x;
    const int64_t my_tiles = p.ntiles > blockIdx.x ? (p.ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t full0 = smem_u32(full), stage0 = smem_u32(smem);
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(full0 + 8 * s, 1);
        s_abort = 0;
        fence_mbar_init();
        prefetch_tmap(&map);
    }
    __syncwarp();
    auto tile_of = [&](int64_t i) { return (int64_t)blockIdx.x + i * gridDim.x; };
    auto issue = [&](int64_t i, int st) {
        mbar_arrive_expect_tx(full0 + 8 * st, p.tile_bytes);
        bulk_g2s(stage0 + st * p.stage_bytes, p.tiles_r + tile_of(i) * (int64_t)p.tile_bytes, p.tile_bytes,
                 full0 + 8 * st);
    };
    if (lane == 0)
        for (int64_t i = 0; i < kStages - 1 && i < my_tiles; ++i) issue(i, (int)i);
    int64_t i = 0;
    for (; i < my_tiles; ++i) {
        const int st = (int)(i % kStages);
        const bool ok = mbar_wait_bounded(full0 + 8 * st, (uint32_t)((i / kStages) & 1), p.wait_ns, &s_abort,
                                          p.status, kCodeTileTma);
        if (__any_sync(0xffffffffu, !ok)) break;
        if (lane == 0) {
            int32_t r0, c0;
            tile_origin(p, tile_of(i), &r0, &c0);
            if (r0 < p.rows && c0 < p.cols) tma_store_2d(&map, c0, r0, stage0 + st * p.stage_bytes);
            bulk_commit();
            const int64_t j = i + kStages - 1;
            if (j < my_tiles) {
                if (i >= 1) bulk_wait_read<1>();  // the store of tile i-1 has read its stage
                issue(j, (int)(j % kStages));
            }
        }
        __syncwarp();
    }
    if (lane == 0) {
        bulk_wait<0>();
        for (int64_t k = i; k < my_tiles && k < i + kStages - 1; ++k) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(full0 + 8 * (k % kStages), (uint32_t)((k / kStages) & 1)) &&
                   globaltimer() - t0 < p.wait_ns) {
            }
        }
    }
}

bool fits_i32(int64_t v) { return v >= INT32_MIN && v <= INT32_MAX; }

// Aligned tiles whose every coordinate fits the tensor map (int32) and the
// TMA rule that a box's first column starts on a 16-byte boundary.
bool tiles_tma_ok(int es, const void* arr, int64_t rows, int64_t cols, int64_t stride_r, int64_t stride_c,
                  int64_t origin_r, int64_t origin_c, int64_t step_r, int64_t step_c, int32_t grid_r, int32_t grid_c,
                  int32_t tile_r, int32_t tile_c, const void* tiles, bool store) {
    if (!arr || rows <= 0 || cols <= 0 || stride_c != 1 || stride_r < cols) return false;
    // The tensor copy bounds the inner dimension in whole 16-byte chunks (a store box
    // ending inside a chunk writes the whole chunk), so the row must end on one.
    if ((cols * es) % 16) return false;
    if (((uintptr_t)arr % 16) || ((uintptr_t)tiles % 16) || (stride_r * es) % 16) return false;
    if ((tile_c * es) % 16 || (int64_t)tile_r * tile_c * es > kMaxTileBytes) return false;
    if ((origin_c * es) % 16 || (grid_c > 1 && (step_c * es) % 16)) return false;
    if (rows > INT32_MAX || cols > INT32_MAX) return false;
    const int64_t r_last = origin_r + (int64_t)(grid_r - 1) * step_r, c_last = origin_c + (int64_t)(grid_c - 1) * step_c;
    if (!fits_i32(origin_r) || !fits_i32(origin_c) || !fits_i32(r_last + tile_r) || !fits_i32(c_last + tile_c) ||
        !fits_i32(r_last) || !fits_i32(c_last))
        return false;
    if (store && (origin_r < 0 || origin_c < 0 || r_last < 0 || c_last < 0)) return false;  // stores never start below 0
    return true;
}

sbt_status encode_tile_map(sbt_context* ctx, CUtensorMap* map, int es, const void* arr, int64_t rows, int64_t cols,
                           int64_t stride_r, int32_t tile_r, int32_t tile_c) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(stride_r * es)};
    cuuint32_t box[2] = {(cuuint32_t)tile_c, (cuuint32_t)tile_r};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = ctx->encode_tiled(map, es == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                                   const_cast<void*>(arr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return sbt_fail(SBT_ERR_TENSOR_MAP, "cuTensorMapEncodeTiled (tile) failed (" + std::to_string((int)r) + ")");
    return SBT_OK;
}

TileTmaParams make_params(sbt_context* ctx, int es, int64_t rows, int64_t cols, int64_t origin_r, int64_t origin_c,
                          int64_t step_r, int64_t step_c, int32_t grid_r, int32_t grid_c, int32_t tile_r,
                          int32_t tile_c) {
    TileTmaParams p = {};
    p.rows = rows;
    p.cols = cols;
    p.origin_r = origin_r;
    p.origin_c = origin_c;
    p.step_r = step_r;
    p.step_c = step_c;
    p.grid_c = grid_c;
    p.tile_r = tile_r;
    p.tile_c = tile_c;
    p.ntiles = (int64_t)grid_r * grid_c;
    p.tile_bytes = (uint32_t)((int64_t)tile_r * tile_c * es);
    p.stage_bytes = (p.tile_bytes + 127u) & ~127u;
    p.status = ctx->status;
    p.wait_ns = ctx->wait_limit_ns;
    return p;
}

template <typename Kern>
sbt_status launch(sbt_context* ctx, Kern kern, const CUtensorMap& map, const TileTmaParams& p, const char* what,
                  cudaStream_t stream) {
    const size_t smem = (size_t)kStages * p.stage_bytes;
    sbt_status st = sbt_cuda_check(
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kStages * kMaxTileBytes)),
        "cudaFuncSetAttribute(tile tma)");
    if (st) return st;
    const int grid = sbt_persistent_grid(ctx, (const void*)kern, 32, smem, p.ntiles);
    kern<<<grid, 32, smem, stream>>>(map, p);
    return sbt_after_launch(ctx, what);
}

}  // namespace

bool sbt_tile_tma_ok(int es, const void* arr, int64_t rows, int64_t cols, int64_t stride_r, int64_t stride_c,
                     int64_t origin_r, int64_t origin_c, int64_t step_r, int64_t step_c, int32_t grid_r,
                     int32_t grid_c, int32_t tile_r, int32_t tile_c, const void* tiles, bool store) {
    return tiles_tma_ok(es, arr, rows, cols, stride_r, stride_c, origin_r, origin_c, step_r, step_c, grid_r, grid_c,
                        tile_r, tile_c, tiles, store);
}

sbt_status sbt_launch_tile_load_tma(sbt_context* ctx, int es, const void* src, int64_t rows, int64_t cols,
                                    int64_t stride_r, int64_t origin_r, int64_t origin_c, int64_t step_r,
                                    int64_t step_c, int32_t grid_r, int32_t grid_c, int32_t tile_r, int32_t tile_c,
                                    void* dst, uint32_t pad_word, cudaStream_t stream) {
    CUtensorMap map;
    sbt_status st = encode_tile_map(ctx, &map, es, src, rows, cols, stride_r, tile_r, tile_c);
    if (st) return st;
    TileTmaParams p = make_params(ctx, es, rows, cols, origin_r, origin_c, step_r, step_c, grid_r, grid_c, tile_r, tile_c);
    p.tiles_w = (char*)dst;
    p.pad_word = pad_word;
    p.pad_fix = (es == 4 ? pad_word : (pad_word & 0xFFFFu)) != 0;
    return es == 4 ? launch(ctx, k_tile_load_tma<4>, map, p, "tile_load_padded (tma)", stream)
                   : launch(ctx, k_tile_load_tma<2>, map, p, "tile_load_padded (tma)", stream);
}

sbt_status sbt_launch_tile_store_tma(sbt_context* ctx, int es, const void* src_tiles, int32_t grid_r, int32_t grid_c,
                                     int32_t tile_r, int32_t tile_c, void* dst, int64_t rows, int64_t cols,
                                     int64_t stride_r, int64_t origin_r, int64_t origin_c, int64_t step_r,
                                     int64_t step_c, cudaStream_t stream) {
    CUtensorMap map;
    sbt_status st = encode_tile_map(ctx, &map, es, dst, rows, cols, stride_r, tile_r, tile_c);
    if (st) return st;
    TileTmaParams p = make_params(ctx, es, rows, cols, origin_r, origin_c, step_r, step_c, grid_r, grid_c, tile_r, tile_c);
    p.tiles_r = (const char*)src_tiles;
    return launch(ctx, k_tile_store_tma, map, p, "tile_store_clipped (tma)", stream);
}
