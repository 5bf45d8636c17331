// Row gather and masked row scatter through the TMA bulk-copy engine.
//
// Taken by the host when whole rows can move as 16-byte-aligned blocks: the
// gathered column window lies inside the table, and every row start (source,
// destination, mask) is 16-byte aligned with a byte length that is a multiple
// of 16.  Data in flight then lives in shared memory, not in registers, so
// the number of bytes in flight per SM no longer trades against occupancy.
//
// Each block is persistent and owns a ring of kStages shared-memory stages of
// R rows.  Warp 0 is the producer: its lanes load the next chunk's indices
// one chunk ahead, check them (64-bit, offset first -- warp.tile_load_indexed,
// description), ballot the valid rows, and issue one cp.async.bulk per row
// (gather) or per contiguous block of rows (scatter), all completing on the
// stage's mbarrier.
//  - gather: rows whose index is outside read the pad value -- the block
//    fills them in shared memory -- and the whole chunk leaves with one
//    shared->global bulk copy (or one per row when the output rows are not
//    contiguous).  A stage is refilled only after the bulk store that read it
//    has finished reading (bulk async-group wait).
//  - scatter: the block reads source vectors and mask bytes from shared
//    memory and writes the destination row with a 16-byte store when all of
//    the vector's mask bits are set, element stores otherwise; out-of-range
//    rows and columns are skipped (cuTile.jl "Memory": masked, clipped).
// Every mbarrier wait is bounded; on a timeout the block sets the device
// status flag, stops, and waits (bounded) for its copies in flight.
#include "sbt_internal.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace sbt_ptx;

constexpr int kStages = 4;          // gather ring: 4 stages of up to 16 KB
constexpr int kGatherThreads = 128;
constexpr int kScatterThreads = 256;
// Scatter ring: 6 stages of up to 12 KB, three blocks per SM.  Measured on
// the fp32 masked workload (1 KiB rows + 256 B mask): 0.526 ms, against 0.574
// with the gather's 4 x 16 KB and 0.53-0.63 for other splits of the same
// shared memory.
constexpr int kScatterStages = 6;
constexpr uint32_t kScatterChunkBytes = 12288;
constexpr unsigned int kCodeBulk = 0x1000;

struct BulkRowsParams {
    const char* arr;          // gather: table at column col_offset of row 0; scatter: dst at column col_offset
    char* arr_w;
    int64_t arr_row_bytes;    // row stride of the indexed array, bytes
    int64_t rows;             // rows of the indexed array
    int64_t cols_valid;       // scatter: columns of the window inside [0, cols) start at first_col, count cols_valid
    int64_t first_col;        // scatter: first in-bounds column of the window (relative to the window start)
    const int32_t* idx;
    int64_t n_idx, row_offset;
    const char* dense;        // gather: unused; scatter: source rows
    char* dense_w;            // gather: output rows
    int64_t dense_row_bytes;  // row stride of the dense side, bytes
    const uint8_t* mask;      // scatter only (may be NULL)
    int64_t mask_row_bytes;
    uint32_t row_bytes;       // bytes moved per row (tile_c * es)
    uint32_t mask_bytes;      // mask bytes per row (tile_c) or 0
    int R;                    // rows per chunk (<= 32)
    uint32_t stage_bytes;     // R * (row_bytes + mask_bytes), rounded to 128
    int dense_contiguous;     // dense_row_bytes == row_bytes
    int mask_contiguous;      // mask_row_bytes == mask_bytes
    uint32_t pad_word;
    int es;
    unsigned int* status;
    uint64_t wait_ns;
    int withhold_first_load;  // test hook: block 0 never issues its first chunk
};

__device__ __forceinline__ int64_t chunk_of(int64_t i) { return (int64_t)blockIdx.x + i * gridDim.x; }

// -------------------------------------------------------------------------------- gather

__global__ void __launch_bounds__(kGatherThreads) k_gather_bulk(const BulkRowsParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[kStages];
    __shared__ uint32_t s_valid[kStages];
    __shared__ int s_abort;
    const int lane = threadIdx.x & 31;
    const bool producer = threadIdx.x < 32;
    const int64_t nchunks = (p.n_idx + p.R - 1) / p.R;
    const int64_t my_chunks = nchunks > blockIdx.x ? (nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t full0 = smem_u32(full);
    const uint32_t stage0 = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(full0 + 8 * s, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    auto rows_in = [&](int64_t i) -> int {
        const int64_t k0 = chunk_of(i) * p.R;
        const int64_t left = p.n_idx - k0;
        return (int)(left < p.R ? left : p.R);
    };
    auto load_idx = [&](int64_t i) -> int32_t {
        return (i < my_chunks && lane < rows_in(i)) ? __ldg(p.idx + chunk_of(i) * p.R + lane) : 0;
    };
    // Warp 0: issue the copies of chunk i into stage st (indices already loaded: `raw`).
    auto issue = [&](int64_t i, int st, int32_t raw) {
        if (p.withhold_first_load && blockIdx.x == 0 && i == 0) return;  // test hook
        const int nrows = rows_in(i);
        const int64_t r = (int64_t)raw + p.row_offset;
        const bool valid = lane < nrows && r >= 0 && r < p.rows;
        const uint32_t ballot = __ballot_sync(0xffffffffu, valid);
        if (lane == 0) {
            s_valid[st] = ballot;
            mbar_arrive_expect_tx(full0 + 8 * st, (uint32_t)__popc(ballot) * p.row_bytes);
        }
        __syncwarp();
        if (valid)
            bulk_g2s(stage0 + st * p.stage_bytes + lane * p.row_bytes, p.arr + r * p.arr_row_bytes, p.row_bytes,
                     full0 + 8 * st);
    };

    int32_t raw_next = 0;
    if (producer) {
        for (int64_t i = 0; i < kStages - 1 && i < my_chunks; ++i) issue(i, (int)i, load_idx(i));
        raw_next = load_idx(kStages - 1);
    }
    const uint4 padv = make_uint4(p.pad_word, p.pad_word, p.pad_word, p.pad_word);
    const int vec_per_row = (int)(p.row_bytes / 16);
    int64_t i = 0;
    for (; i < my_chunks; ++i) {
        const int st = (int)(i % kStages);
        const bool ok = mbar_wait_bounded(full0 + 8 * st, (uint32_t)((i / kStages) & 1), p.wait_ns, &s_abort,
                                          p.status, kCodeBulk);
        if (__syncthreads_or(!ok)) break;  // every thread leaves together
        const int nrows = rows_in(i);
        const uint32_t valid = s_valid[st];
        const uint32_t all = nrows >= 32 ? 0xffffffffu : ((1u << nrows) - 1u);
        uint8_t* stage = smem + (size_t)st * p.stage_bytes;
        if (valid != all) {
            for (int t = threadIdx.x; t < nrows * vec_per_row; t += blockDim.x) {
                const int row = t / vec_per_row;
                if (!((valid >> row) & 1u))
                    *reinterpret_cast<uint4*>(stage + (size_t)row * p.row_bytes + (t - row * vec_per_row) * 16) = padv;
            }
            fence_proxy_async_smem();
        }
        __syncthreads();
        if (producer) {
            const int64_t k0 = chunk_of(i) * p.R;
            if (p.dense_contiguous) {
                if (lane == 0) bulk_s2g(p.dense_w + k0 * p.dense_row_bytes, stage0 + st * p.stage_bytes,
                                        (uint32_t)nrows * p.row_bytes);
            } else if (lane < nrows) {
                bulk_s2g(p.dense_w + (k0 + lane) * p.dense_row_bytes, stage0 + st * p.stage_bytes + lane * p.row_bytes,
                         p.row_bytes);
            }
            bulk_commit();
            const int64_t j = i + kStages - 1;
            if (j < my_chunks) {
                if (i >= 1) bulk_wait_read<1>();  // the store of chunk i-1 has read its stage
                issue(j, (int)(j % kStages), raw_next);
                raw_next = load_idx(j + 1);
            }
        }
    }
    if (producer) {
        bulk_wait<0>();
        if (i < my_chunks) {
            // Stopped early: wait (bounded) for the loads still in flight before the block exits.
            for (int64_t k = i; k < my_chunks && k < i + kStages - 1; ++k) {
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(full0 + 8 * (k % kStages), (uint32_t)((k / kStages) & 1)) &&
                       globaltimer() - t0 < p.wait_ns) {
                }
            }
        }
    }
}

// -------------------------------------------------------------------------------- scatter

template <int ES, bool MASK, bool VEC_DST>
__global__ void __launch_bounds__(kScatterThreads) k_scatter_bulk(const BulkRowsParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[kScatterStages];
    __shared__ int64_t s_row[kScatterStages][32];
    __shared__ uint32_t s_valid[kScatterStages];
    __shared__ int s_abort;
    constexpr int V = 16 / ES;
    constexpr uint32_t kAll = (1u << V) - 1u;
    typedef typename sbt_elem<ES>::T T;
    const int lane = threadIdx.x & 31;
    const bool producer = threadIdx.x < 32;
    const int64_t nchunks = (p.n_idx + p.R - 1) / p.R;
    const int64_t my_chunks = nchunks > blockIdx.x ? (nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t full0 = smem_u32(full);
    const uint32_t stage0 = smem_u32(smem);
    const uint32_t src_block = (uint32_t)p.R * p.row_bytes;  // mask block follows the source block

    if (threadIdx.x == 0) {
        for (int s = 0; s < kScatterStages; ++s) mbar_init(full0 + 8 * s, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    auto rows_in = [&](int64_t i) -> int {
        const int64_t k0 = chunk_of(i) * p.R;
        const int64_t left = p.n_idx - k0;
        return (int)(left < p.R ? left : p.R);
    };
    auto load_idx = [&](int64_t i) -> int32_t {
        return (i < my_chunks && lane < rows_in(i)) ? __ldg(p.idx + chunk_of(i) * p.R + lane) : 0;
    };
    auto issue = [&](int64_t i, int st, int32_t raw) {
        if (p.withhold_first_load && blockIdx.x == 0 && i == 0) return;  // test hook
        const int nrows = rows_in(i);
        const int64_t k0 = chunk_of(i) * p.R;
        const int64_t r = (int64_t)raw + p.row_offset;
        const bool valid = lane < nrows && r >= 0 && r < p.rows;
        const uint32_t ballot = __ballot_sync(0xffffffffu, valid);
        s_row[st][lane] = r;
        const uint32_t sbase = stage0 + st * p.stage_bytes;
        if (lane == 0) {
            s_valid[st] = ballot;
            mbar_arrive_expect_tx(full0 + 8 * st, (uint32_t)nrows * (p.row_bytes + (MASK ? p.mask_bytes : 0)));
            if (p.dense_contiguous)
                bulk_g2s(sbase, p.dense + k0 * p.dense_row_bytes, (uint32_t)nrows * p.row_bytes, full0 + 8 * st);
            if (MASK && p.mask_contiguous)
                bulk_g2s(sbase + src_block, p.mask + k0 * p.mask_row_bytes, (uint32_t)nrows * p.mask_bytes,
                         full0 + 8 * st);
        }
        __syncwarp();
        if (lane < nrows) {
            if (!p.dense_contiguous)
                bulk_g2s(sbase + lane * p.row_bytes, p.dense + (k0 + lane) * p.dense_row_bytes, p.row_bytes,
                         full0 + 8 * st);
            if (MASK && !p.mask_contiguous)
                bulk_g2s(sbase + src_block + lane * p.mask_bytes, p.mask + (k0 + lane) * p.mask_row_bytes,
                         p.mask_bytes, full0 + 8 * st);
        }
    };

    int32_t raw_next = 0;
    if (producer) {
        for (int64_t i = 0; i < kScatterStages && i < my_chunks; ++i) issue(i, (int)i, load_idx(i));
        raw_next = load_idx(kScatterStages);
    }
    const int vec_per_row = (int)(p.row_bytes / 16);
    int64_t i = 0;
    for (; i < my_chunks; ++i) {
        const int st = (int)(i % kScatterStages);
        // the producer loads the indices of chunk i + kScatterStages while this chunk moves
        const int32_t raw_after = producer ? load_idx(i + kScatterStages + 1) : 0;
        const bool ok = mbar_wait_bounded(full0 + 8 * st, (uint32_t)((i / kScatterStages) & 1), p.wait_ns, &s_abort,
                                          p.status, kCodeBulk);
        if (__syncthreads_or(!ok)) break;  // every thread leaves together
        const int nrows = rows_in(i);
        const uint32_t valid = s_valid[st];
        const uint8_t* src_s = smem + (size_t)st * p.stage_bytes;
        const uint8_t* msk_s = src_s + src_block;
        for (int t = threadIdx.x; t < nrows * vec_per_row; t += blockDim.x) {
            const int row = t / vec_per_row;
            if (!((valid >> row) & 1u)) continue;
            const int vc = t - row * vec_per_row;
            const int64_t j0 = (int64_t)vc * V;  // column within the window
            if (j0 + V <= p.first_col || j0 >= p.first_col + p.cols_valid) continue;
            const uint4 v = *reinterpret_cast<const uint4*>(src_s + (size_t)row * p.row_bytes + vc * 16);
            uint32_t mb = kAll;
            if (MASK) {
                const uint8_t* m = msk_s + (size_t)row * p.mask_bytes + j0;
                mb = 0;
                if (V == 4) {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(m);
#pragma unroll
                    for (int e = 0; e < 4; ++e) mb |= ((w >> (8 * e)) & 0xFFu) ? (1u << e) : 0u;
                } else {
                    const uint2 w = *reinterpret_cast<const uint2*>(m);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        mb |= ((w.x >> (8 * e)) & 0xFFu) ? (1u << e) : 0u;
                        mb |= ((w.y >> (8 * e)) & 0xFFu) ? (1u << (e + 4)) : 0u;
                    }
                }
                if (!mb) continue;
            }
            char* drow = p.arr_w + s_row[st][row] * p.arr_row_bytes;
            const bool inside = j0 >= p.first_col && j0 + V <= p.first_col + p.cols_valid;
            if (VEC_DST && mb == kAll && inside) {
                sbt_st_v4(drow + j0 * ES, v);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const int64_t j = j0 + e;
                    if (((mb >> e) & 1u) && j >= p.first_col && j < p.first_col + p.cols_valid)
                        reinterpret_cast<T*>(drow)[j] = sbt_vec_get<ES>(v, e);
                }
            }
        }
        __syncthreads();
        if (producer && i + kScatterStages < my_chunks) {
            issue(i + kScatterStages, st, raw_next);
            raw_next = raw_after;
        }
    }
    if (producer && i < my_chunks) {
        for (int64_t k = i; k < my_chunks && k < i + kScatterStages; ++k) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(full0 + 8 * (k % kScatterStages), (uint32_t)((k / kScatterStages) & 1)) &&
                   globaltimer() - t0 < p.wait_ns) {
            }
        }
    }
}

int rows_per_chunk(uint32_t bytes_per_row, uint32_t chunk_bytes = 16384) {
    int r = (int)(chunk_bytes / (bytes_per_row ? bytes_per_row : 1));
    return r < 1 ? 1 : (r > 32 ? 32 : r);
}

uint32_t round128(uint32_t x) { return (x + 127u) & ~127u; }

}  // namespace

// Whole rows of the gather window move as aligned 16-byte blocks.
bool sbt_gather_bulk_ok(int es, const void* src, int64_t cols, int64_t ld_src, int64_t col_offset, int32_t tile_c,
                        const uint8_t* mask, const void* out, int64_t ld_out) {
    const int64_t row_bytes = (int64_t)tile_c * es;
    if (mask || !src) return false;
    if (col_offset < 0 || col_offset + tile_c > cols) return false;
    if (row_bytes % 16 || row_bytes > 16384) return false;
    if (((uintptr_t)src + col_offset * es) % 16 || (ld_src * es) % 16) return false;
    if (((uintptr_t)out) % 16 || (ld_out * es) % 16) return false;
    return true;
}

bool sbt_scatter_bulk_ok(int es, const void* src, int64_t ld_src, int32_t tile_c, const uint8_t* mask,
                         int64_t ld_mask) {
    const int64_t row_bytes = (int64_t)tile_c * es;
    if (row_bytes % 16 || row_bytes > 16384) return false;
    if (((uintptr_t)src) % 16 || (ld_src * es) % 16) return false;
    if (mask && ((tile_c % 16) || ((uintptr_t)mask) % 16 || ld_mask % 16)) return false;
    return true;
}

sbt_status sbt_launch_gather_bulk(sbt_context* ctx, int es, const void* src, int64_t rows, int64_t ld_src,
                                  const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                                  int32_t tile_c, void* out, int64_t ld_out, uint32_t pad_word, cudaStream_t stream) {
    BulkRowsParams p = {};
    p.arr = (const char*)src + col_offset * es;
    p.arr_row_bytes = ld_src * es;
    p.rows = rows;
    p.idx = idx;
    p.n_idx = n_idx;
    p.row_offset = row_offset;
    p.dense_w = (char*)out;
    p.dense_row_bytes = ld_out * es;
    p.row_bytes = (uint32_t)tile_c * es;
    p.R = rows_per_chunk(p.row_bytes);
    p.stage_bytes = round128((uint32_t)p.R * p.row_bytes);
    p.dense_contiguous = p.dense_row_bytes == (int64_t)p.row_bytes;
    p.pad_word = pad_word;
    p.es = es;
    p.status = ctx->status;
    p.wait_ns = ctx->wait_limit_ns;
    p.withhold_first_load = ctx->test_hook == SBT_TEST_WITHHOLD_LOAD;
    const size_t smem = (size_t)kStages * p.stage_bytes;
    static bool attr_done[64] = {false};
    if (!attr_done[ctx->device & 63]) {
        sbt_status st = sbt_cuda_check(
            cudaFuncSetAttribute(k_gather_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize, kStages * 16384 + 512),
            "cudaFuncSetAttribute(gather bulk)");
        if (st) return st;
        attr_done[ctx->device & 63] = true;
    }
    const int grid = sbt_persistent_grid(ctx, (const void*)k_gather_bulk, kGatherThreads, smem, sbt_cdiv(n_idx, p.R));
    k_gather_bulk<<<grid, kGatherThreads, smem, stream>>>(p);
    return sbt_after_launch(ctx, "gather_rows (bulk)");
}

sbt_status sbt_launch_scatter_bulk(sbt_context* ctx, int es, void* dst, int64_t rows, int64_t cols, int64_t ld_dst,
                                   const int32_t* idx, int64_t n_idx, int64_t row_offset, int64_t col_offset,
                                   const void* src, int64_t ld_src, int32_t tile_c, const uint8_t* mask,
                                   int64_t ld_mask, cudaStream_t stream) {
    BulkRowsParams p = {};
    p.arr_w = (char*)dst + col_offset * es;
    p.arr_row_bytes = ld_dst * es;
    p.rows = rows;
    // window columns j in [first_col, first_col + cols_valid) land inside [0, cols)
    const int64_t lo = col_offset < 0 ? -col_offset : 0;
    const int64_t hi = (cols - col_offset) < tile_c ? (cols - col_offset) : tile_c;
    p.first_col = lo;
    p.cols_valid = hi > lo ? hi - lo : 0;
    p.idx = idx;
    p.n_idx = n_idx;
    p.row_offset = row_offset;
    p.dense = (const char*)src;
    p.dense_row_bytes = ld_src * es;
    p.mask = mask;
    p.mask_row_bytes = ld_mask;
    p.row_bytes = (uint32_t)tile_c * es;
    p.mask_bytes = mask ? (uint32_t)tile_c : 0u;
    p.R = rows_per_chunk(p.row_bytes + p.mask_bytes, kScatterChunkBytes);
    p.stage_bytes = round128((uint32_t)p.R * (p.row_bytes + p.mask_bytes));
    p.dense_contiguous = p.dense_row_bytes == (int64_t)p.row_bytes;
    p.mask_contiguous = mask && p.mask_row_bytes == (int64_t)p.mask_bytes;
    p.es = es;
    p.status = ctx->status;
    p.wait_ns = ctx->wait_limit_ns;
    p.withhold_first_load = ctx->test_hook == SBT_TEST_WITHHOLD_LOAD;
    const bool vec_dst = ((uintptr_t)p.arr_w % 16) == 0 && (p.arr_row_bytes % 16) == 0;
    const size_t smem = (size_t)kScatterStages * p.stage_bytes;
#define SBT_SB(ES_, M_, VD_)                                                                                        \
    do {                                                                                                           \
        auto kern = k_scatter_bulk<ES_, M_, VD_>;                                                                  \
        sbt_status st = sbt_cuda_check(                                                                            \
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),                        \
            "cudaFuncSetAttribute(scatter bulk)");                                                                 \
        if (st) return st;                                                                                         \
        const int grid = sbt_persistent_grid(ctx, (const void*)kern, kScatterThreads, smem, sbt_cdiv(n_idx, p.R)); \
        kern<<<grid, kScatterThreads, smem, stream>>>(p);                                                          \
        return sbt_after_launch(ctx, "scatter_rows_masked (bulk)");                                                \
    } while (0)
    if (es == 4) {
        if (mask) {
            if (vec_dst) SBT_SB(4, true, true);
            SBT_SB(4, true, false);
        }
        if (vec_dst) SBT_SB(4, false, true);
        SBT_SB(4, false, false);
    }
    if (mask) {
        if (vec_dst) SBT_SB(2, true, true);
        SBT_SB(2, true, false);
    }
    if (vec_dst) SBT_SB(2, false, true);
    SBT_SB(2, false, false);
#undef SBT_SB
}
