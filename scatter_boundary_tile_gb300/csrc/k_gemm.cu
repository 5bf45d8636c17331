// Boundary-tile bf16 GEMM  C = A * B  on tcgen05 tensor cores.
//
// cuTile.jl "Operations", muladd: (M,K) x (K,N) -> (M,N), bf16 inputs with an
// fp32 accumulator.  Tylo.jl "Boundary tiles", section "Accumulator stores
// and GEMM": ceiling-division K loop and output grid; boundary tiles are
// zero-filled; the accumulator is converted to the output type at the store
// and stores outside M x N are suppressed.
//
// Pipeline (all on the caller's stream):
//  1. Operand staging (the bounded copy of Tylo.jl "Boundary tiles"): A and
//     B may have any leading dimension (odd ones included), which TMA cannot
//     address (its row strides are multiples of 16 bytes).  Two kernels copy
//     A -> A' [Mp][Kp] and B -> B' [Np][Kp] (B transposed, so both operands
//     are K-major), zero-filling every element past M, N or K, with
//     Mp, Np, Kp rounded up to whole tiles.  A' and B' live in the caller's
//     workspace.
//  2. A persistent, warp-specialised kernel: warp 0 issues TMA tile loads
//     into a 4-stage shared-memory ring (128-byte swizzle), warp 1 issues
//     tcgen05.mma (M=128, N<=256, K=16, fp32 accumulator in TMEM, two
//     256-column accumulators so the epilogue of one tile overlaps the main
//     loop of the next), warps 2-5 drain TMEM with tcgen05.ld, round to bf16
//     (or keep fp32) and store through a shared-memory transpose so that
//     each store instruction writes one contiguous row segment.
//  Every mbarrier wait is bounded; a wait that runs out sets the device
//  status word, and the kernel drains and returns.
#include <cuda_bf16.h>

#include <algorithm>
#include <string>

#include "sbt_internal.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace sbt_ptx;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kGemmThreads = 192;  // warp 0: TMA, warp 1: MMA, warps 2..5: epilogue
constexpr uint32_t kABytes = BM * BK * 2;
constexpr int kEpiWarps = 4;
constexpr int kEpiWords = 32 * 33;  // per-warp 32x32 transpose buffer, padded rows
constexpr int kNumBars = 2 * kStages + 5;
// MN-major B in shared memory: one TMA box of 64 columns x BK rows (128-byte rows) per 64 columns.
constexpr uint32_t kMnAtomBytes = 64 * BK * 2;  // 8 KB: next 64 columns
constexpr uint32_t kMnKStepBytes = 16 * 128;     // one K = 16 step: 16 rows of 128 B
// Single-CTA kernel with BM x BN_ tiles (BN_ = 256, 128 or 64: narrower tiles
// spread a small problem over more SMs).
template <int BN_>
struct TcShape {
    static constexpr uint32_t kBBytes = BN_ * BK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;  // a multiple of 1024: swizzle atoms stay aligned
    static constexpr uint32_t kTmemCols = 2 * BN_;              // two accumulators; a power of two >= 32
    static constexpr size_t kSmem =
        1024 + (size_t)kStages * kStageBytes + (size_t)kEpiWarps * kEpiWords * 4 + kNumBars * 8 + 16;
};

enum : unsigned int { kCodeProducer = 0x100, kCodeMma = 0x200, kCodeEpilogue = 0x400, kCodeTeardown = 0x800 };

struct GemmParams {
    char* C;
    int64_t ldc;
    int c_f32;
    const float* acc;  // fp32 C only: added to the product before the store (NULL: nothing added)
    int64_t ld_acc;
    int M, N, K;
    int m_tiles, n_tiles, k_blocks;
    unsigned int* status;
    uint64_t wait_ns;
    int withhold_first_load;  // test hook: block 0 never issues its first stage
};

// Tile order: groups of kGroupM M-tiles are walked N column by N column, so the
// tiles running at the same time share a few A row blocks and B column blocks
// (a working set of tens of MB that stays in L2) instead of sweeping all of A
// for every N column.
constexpr int kGroupM = 8;
__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int* mt, int* nt) {
    const int per_group = kGroupM * n_tiles;
    const int g = tile / per_group;
    const int within = tile - g * per_group;
    const int first_m = g * kGroupM;
    const int gm = min(kGroupM, m_tiles - first_m);
    *mt = first_m + within % gm;
    *nt = within / gm;
}

// Drain one 128 x BN_ accumulator from TMEM (this warp's 32-lane quarter `q`),
// round (or keep fp32) and store rows row0.. of C through a padded shared
// transpose so that each store instruction covers 32 consecutive columns.
// A bf16 C is rounded before the transpose, which then moves half the bytes
// (shared memory is the resource the main loop competes for).  This epilogue
// runs under the next tile's main loop; a version that stored 16 rows at a
// time with the next TMEM load in flight slowed the 256 x 256 pair kernel
// with an fp32 C from 0.338 to 0.375 ms (its stores contend with the loop).
template <int BN_>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t tmem_acc, int q, int lane, float* buf,
                                              int row0, int n0) {
    const int n_valid = min(BN_, p.N - n0);
    const int chunks = (n_valid + 31) / 32;
    for (int c = 0; c < chunks; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_acc + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), r);
        tmem_ld_wait();
        if (!p.c_f32) {
            // [32 rows][17 words]: row `lane` packs its 32 columns as bf16 pairs; odd padding keeps
            // the row-wise writes and the column-wise reads free of bank conflicts.
            uint32_t* wb = reinterpret_cast<uint32_t*>(buf);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                wb[lane * 17 + j] = *reinterpret_cast<const uint32_t*>(&v);
            }
            __syncwarp();
            const int col = n0 + c * 32 + lane;
            if (col < p.N) {
                uint16_t* Cp = reinterpret_cast<uint16_t*>(p.C);
                for (int rr = 0; rr < 32 && row0 + rr < p.M; ++rr) {
                    const uint32_t w = wb[rr * 17 + (lane >> 1)];
                    Cp[(int64_t)(row0 + rr) * p.ldc + col] = (uint16_t)((lane & 1) ? (w >> 16) : (w & 0xFFFFu));
                }
            }
            __syncwarp();
            continue;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) buf[lane * 33 + j] = __uint_as_float(r[j]);
        __syncwarp();
        const int col = n0 + c * 32 + lane;
        if (col < p.N) {  // fp32 C
            float* Cp = reinterpret_cast<float*>(p.C);
            if (p.acc) {
                for (int rr = 0; rr < 32 && row0 + rr < p.M; ++rr)
                    Cp[(int64_t)(row0 + rr) * p.ldc + col] =
                        buf[rr * 33 + lane] + __ldg(p.acc + (int64_t)(row0 + rr) * p.ld_acc + col);
            } else {
                for (int rr = 0; rr < 32 && row0 + rr < p.M; ++rr)
                    Cp[(int64_t)(row0 + rr) * p.ldc + col] = buf[rr * 33 + lane];
            }
        }
        __syncwarp();
    }
}

// BMN: B is read MN-major (TMA boxes of 64 columns), else K-major rows of B'^T.  A template
// parameter, not a kernel argument: a branch on it in the single-thread TMA and MMA issue
// loops measured ~6% slower on the 256 x 256 pair kernel.
template <int BN_, bool BMN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm_bf16_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
    typedef TcShape<BN_> S;
    constexpr uint32_t kStageBytes = S::kStageBytes;
    constexpr uint32_t kTmemCols = S::kTmemCols;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* epi = reinterpret_cast<float*>(smem + (size_t)kStages * kStageBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi + kEpiWarps * kEpiWords);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
    const uint32_t mma_done_bar = bar0 + 8u * (2 * kStages + 4);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0);
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), kEpiWarps * 32);
        }
        mbar_init(mma_done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Set-up above overlaps the end of the staging kernel ahead in the stream (launched as a
    // programmatic dependent); from here on the staged operands are read and C is written.
    griddep_wait();
    const int num_tiles = p.m_tiles * p.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                int mt, nt;
                tile_coords(tile, p.m_tiles, p.n_tiles, &mt, &nt);
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, p.wait_ns, abort_flag, p.status,
                                           kCodeProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes);
                    if (p.withhold_first_load && blockIdx.x == 0 && issued == 0) {
                        // test hook: this stage's full barrier is never armed, so the MMA
                        // warp's bounded wait on it runs out
                        ++issued;
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    mbar_arrive_expect_tx(full_bar(stage), kStageBytes);
                    tma_load_2d(sa, &tmA, kb * BK, mt * BM, full_bar(stage));
                    if (BMN) {
#pragma unroll
                        for (int a = 0; a < BN_ / 64; ++a)
                            tma_load_2d(sa + kABytes + a * kMnAtomBytes, &tmB, nt * BN_ + 64 * a, kb * BK,
                                        full_bar(stage));
                    } else {
                        tma_load_2d(sa + kABytes, &tmB, kb * BK, nt * BN_, full_bar(stage));
                    }
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Drain: wait (bounded) until the copies still in flight have landed.
                uint32_t s = stage, ph = phase;
                for (int64_t j = 0; j < issued && j < kStages; ++j) {
                    if (s == 0) {
                        s = kStages - 1;
                        ph ^= 1u;
                    } else {
                        --s;
                    }
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(full_bar(s), ph) && globaltimer() - t0 < p.wait_ns) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t use = (uint32_t)(local >> 1);
                int mt_unused, nt;
                tile_coords(tile, p.m_tiles, p.n_tiles, &mt_unused, &nt);
                const int n_valid = min(BN_, p.N - nt * BN_);
                const uint32_t idesc =
                    idesc_bf16_f32(BM, (uint32_t)((n_valid + 15) & ~15)) | (BMN ? kIdescBMnMajor : 0u);
                if (!mbar_wait_bounded(tempty_bar(acc), (use & 1u) ^ 1u, p.wait_ns, abort_flag, p.status,
                                       kCodeMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN_);
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait_bounded(full_bar(stage), phase, p.wait_ns, abort_flag, p.status, kCodeMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int k_rem = p.K - kb * BK;
                    const int k_steps = k_rem >= BK ? BK / 16 : (k_rem + 15) / 16;
                    const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes);
                    const uint32_t sb = sa + kABytes;
                    for (int ks = 0; ks < k_steps; ++ks) {
                        const uint64_t bd = BMN ? smem_desc_mn_sw128(sb + kMnKStepBytes * ks, kMnAtomBytes)
                                                   : smem_desc_sw128(sb + 32u * ks);
                        tc_mma_f16(d_tmem, smem_desc_sw128(sa + 32u * ks), bd, idesc,
                                   (kb | ks) != 0 ? 1u : 0u);
                    }
                    tc_commit(empty_bar(stage));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit(tfull_bar(acc));
            }
            // every MMA this thread issued has completed once mma_done flips
            tc_commit(mma_done_bar);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(mma_done_bar, 0)) {
                if (globaltimer() - t0 > p.wait_ns) {
                    atomicOr(p.status, (unsigned int)kCodeTeardown);
                    break;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;  // TMEM lane quarter this warp may read
        float* buf = epi + (warp - 2) * kEpiWords;
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            int mt, nt;
                tile_coords(tile, p.m_tiles, p.n_tiles, &mt, &nt);
            if (!mbar_wait_bounded(tfull_bar(acc), use & 1u, p.wait_ns, abort_flag, p.status, kCodeEpilogue)) break;
            tc_fence_after();
            epilogue_tile<BN_>(p, tmem_base + (uint32_t)(acc * BN_), q, lane, buf, mt * BM + q * 32, nt * BN_);
            tc_fence_before();
            mbar_arrive(tempty_bar(acc));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------- CTA-pair kernel
//
// Two CTAs of a cluster compute one 256 x 256 tile with tcgen05.mma.cta_group::2
// (M = 256: 128 rows in each CTA's TMEM; B split 128 + 128 rows between the
// CTAs' shared memory).  Each CTA loads only its own half of B, so a CTA
// pulls 32 KB per 64-deep K step instead of 48 KB.  A stage holds two K steps
// (two 128-byte swizzle atoms of A and of B per CTA, 64 KB) and the ring three
// stages: one barrier round trip per 128 of K measured 0.409 ms for the
// 8191 x 8193 x 4097 call against 0.439 with six single-step stages of the same
// 192 KB.  Each CTA's TMA completes on the leader's
// full barrier; the leader's MMA commits are multicast to both CTAs' empty and
// TMEM-full barriers; both epilogues arrive on the leader's TMEM-empty barrier.

constexpr int kStages2 = 3;
constexpr uint32_t kHalfBytes = 128 * BK * 2;          // A rows or B rows of one CTA, one K step
constexpr int kKB2 = 2;                                // K steps per stage
constexpr uint32_t kStageBytes2 = 2 * kKB2 * kHalfBytes;  // per CTA: A atoms, then B atoms
constexpr uint32_t kTmemCols2 = 2 * BN;                    // two 128 x 256 accumulators per CTA
constexpr int kNumBars2 = 2 * kStages2 + 5;
constexpr size_t kGemmSmem2 = 1024 + (size_t)kStages2 * kStageBytes2 + (size_t)kEpiWarps * kEpiWords * 4 +
                              kNumBars2 * 8 + 16;

template <bool BMN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    k_gemm_bf16_tc_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* epi = reinterpret_cast<float*>(smem + (size_t)kStages2 * kStageBytes2);
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi + kEpiWarps * kEpiWords);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages2 + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages2 + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages2 + 2 + a); };
    const uint32_t mma_done_bar = bar0 + 8u * (2 * kStages2 + 4);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0);
    const int lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages2; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * kEpiWarps * 32);
        }
        mbar_init(mma_done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols2);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Set-up above overlaps the end of the staging kernel ahead in the stream (launched as a
    // programmatic dependent); from here on the staged operands are read and C is written.
    griddep_wait();
    const int num_tiles = p.m_tiles * p.n_tiles;  // 256 x 256 tiles

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (each CTA, own halves)
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            int64_t issued = 0;
            for (int tile = cluster; ok && tile < num_tiles; tile += nclusters) {
                int mt, nt;
                tile_coords(tile, p.m_tiles, p.n_tiles, &mt, &nt);
                for (int kb0 = 0; kb0 < p.k_blocks; kb0 += kKB2) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, p.wait_ns, abort_flag, p.status,
                                           kCodeProducer)) {
                        ok = false;
                        break;
                    }
                    const bool withhold = p.withhold_first_load && blockIdx.x == 0 && issued == 0;
                    ++issued;
                    if (!withhold) {
                        const int nkb = p.k_blocks - kb0 < kKB2 ? p.k_blocks - kb0 : kKB2;
                        const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes2);
                        const uint32_t leader_full = mapa_shared(full_bar(stage), 0);
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * nkb * 2 * kHalfBytes);
                        for (int j = 0; j < nkb; ++j) {
                            tma_load_2d_pair(sa + j * kHalfBytes, &tmA, (kb0 + j) * BK, mt * 256 + (int)rank * 128, leader_full);
                            if (BMN) {
                                for (int a = 0; a < 2; ++a)
                                    tma_load_2d_pair(sa + (kKB2 + j) * kHalfBytes + a * kMnAtomBytes, &tmB,
                                                     nt * 256 + (int)rank * 128 + 64 * a, (kb0 + j) * BK, leader_full);
                            } else {
                                tma_load_2d_pair(sa + (kKB2 + j) * kHalfBytes, &tmB, (kb0 + j) * BK,
                                                 nt * 256 + (int)rank * 128, leader_full);
                            }
                        }
                    }
                    if (++stage == kStages2) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader CTA only)
        if (lane == 0 && rank == 0) {
            uint32_t stage = 0, phase = 0;
            int local = 0;
            bool ok = true;
            const uint32_t idesc = idesc_bf16_f32(256, 256) | (BMN ? kIdescBMnMajor : 0u);
            for (int tile = cluster; ok && tile < num_tiles; tile += nclusters, ++local) {
                const int acc = local & 1;
                const uint32_t use = (uint32_t)(local >> 1);
                if (!mbar_wait_bounded(tempty_bar(acc), (use & 1u) ^ 1u, p.wait_ns, abort_flag, p.status,
                                       kCodeMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb0 = 0; kb0 < p.k_blocks; kb0 += kKB2) {
                    if (!mbar_wait_bounded(full_bar(stage), phase, p.wait_ns, abort_flag, p.status, kCodeMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nkb = p.k_blocks - kb0 < kKB2 ? p.k_blocks - kb0 : kKB2;
                    const uint32_t sa0 = smem_u32(smem + (size_t)stage * kStageBytes2);
                    for (int j = 0; j < nkb; ++j) {
                    const int kb = kb0 + j;
                    const int k_rem = p.K - kb * BK;
                    const int k_steps = k_rem >= BK ? BK / 16 : (k_rem + 15) / 16;
                    const uint32_t sa = sa0 + j * kHalfBytes;
                    const uint32_t sb = sa0 + (kKB2 + j) * kHalfBytes;
                    for (int ks = 0; ks < k_steps; ++ks) {
                        const uint64_t bd = BMN ? smem_desc_mn_sw128(sb + kMnKStepBytes * ks, kMnAtomBytes)
                                                   : smem_desc_sw128(sb + 32u * ks);
                        tc_mma_f16_pair(d_tmem, smem_desc_sw128(sa + 32u * ks), bd,
                                        idesc, (kb | ks) != 0 ? 1u : 0u);
                    }
                    }
                    tc_commit_pair_multicast(empty_bar(stage), 0x3);
                    if (++stage == kStages2) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit_pair_multicast(tfull_bar(acc), 0x3);
            }
            tc_commit_pair_multicast(mma_done_bar, 0x1);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(mma_done_bar, 0)) {
                if (globaltimer() - t0 > p.wait_ns) {
                    atomicOr(p.status, (unsigned int)kCodeTeardown);
                    break;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..5 of each CTA)
        const int q = warp & 3;
        float* buf = epi + (warp - 2) * kEpiWords;
        const uint32_t leader_tempty0 = mapa_shared(tempty_bar(0), 0);
        int local = 0;
        for (int tile = cluster; tile < num_tiles; tile += nclusters, ++local) {
            const int acc = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            int mt, nt;
                tile_coords(tile, p.m_tiles, p.n_tiles, &mt, &nt);
            if (!mbar_wait_bounded(tfull_bar(acc), use & 1u, p.wait_ns, abort_flag, p.status, kCodeEpilogue)) break;
            tc_fence_after();
            epilogue_tile<BN>(p, tmem_base + (uint32_t)(acc * BN), q, lane, buf, mt * 256 + (int)rank * 128 + q * 32,
                          nt * BN);
            tc_fence_before();
            mbar_arrive_cluster(leader_tempty0 + 8u * acc);
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the leader's MMAs into the peer's TMEM are complete before either CTA frees it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols2);
    }
}

// ---------------------------------------------------------------------------- CTA-pair kernel, 512 x 256 tiles
//
// The 256 x 256 pair tile above asks each SM for 512 B of operands per K
// element (128 rows of A, 128 columns of B); measured per-stage timelines show
// an SM taking in about 45 B per cycle from L2 through TMA whatever the stage
// size, against 64 B per cycle for the tensor pipe at full rate, so that
// kernel waits on its loads ~30% of the time.  Here each CTA of the pair holds
// 256 rows of A and 128 columns of B (768 B per K element for twice the
// MMAs, 48 B per cycle at full rate): every K = 16 step issues two
// tcgen05.mma.cta_group::2 of M = 256, N = 256 (the pair's row halves h = 0,
// 1), accumulating into TMEM columns h*256 .. h*256 + 255 of each CTA.  The
// two accumulators fill TMEM, so the epilogue of a tile (twelve warps, three
// per TMEM lane quarter; bf16 C only) runs between tiles instead of under the
// next main loop.

constexpr int kStages3 = 4;
constexpr uint32_t kA3Bytes = 2 * kHalfBytes;            // this CTA's 256 rows of A, one K step
constexpr uint32_t kStageBytes3 = kA3Bytes + kHalfBytes; // + its 128 columns of B: 48 KB
constexpr int kEpiWarps3 = 12;
constexpr int kEpiWords3 = 32 * 17;  // bf16 C only: a [32][17-word] transpose buffer per warp
constexpr int kGemmThreads3 = 64 + 32 * kEpiWarps3;
constexpr int kNumBars3 = 2 * kStages3 + 3;
constexpr size_t kGemmSmem3 = 1024 + (size_t)kStages3 * kStageBytes3 + (size_t)kEpiWarps3 * kEpiWords3 * 4 +
                              kNumBars3 * 8 + 16;

template <bool BMN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads3, 1)
    k_gemm_bf16_tc_pair512(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* epi = reinterpret_cast<float*>(smem + (size_t)kStages3 * kStageBytes3);
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi + kEpiWarps3 * kEpiWords3);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages3 + s); };
    const uint32_t tfull_bar = bar0 + 8u * (2 * kStages3);
    const uint32_t tempty_bar = bar0 + 8u * (2 * kStages3 + 1);
    const uint32_t mma_done_bar = bar0 + 8u * (2 * kStages3 + 2);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0);
    const int lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages3; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, 2 * kEpiWarps3 * 32);
        mbar_init(mma_done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();
    const int num_tiles = p.m_tiles * p.n_tiles;  // 512 x 256 tiles

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (each CTA, own rows and columns)
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            int64_t issued = 0;
            for (int tile = cluster; ok && tile < num_tiles; tile += nclusters) {
                int mt, nt;
                tile_coords(tile, p.m_tiles, p.n_tiles, &mt, &nt);
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, p.wait_ns, abort_flag, p.status,
                                           kCodeProducer)) {
                        ok = false;
                        break;
                    }
                    const bool withhold = p.withhold_first_load && blockIdx.x == 0 && issued == 0;
                    ++issued;
                    if (!withhold) {
                        const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes3);
                        const uint32_t leader_full = mapa_shared(full_bar(stage), 0);
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * kStageBytes3);
                        for (int h = 0; h < 2; ++h)
                            tma_load_2d_pair(sa + h * kHalfBytes, &tmA, kb * BK, mt * 512 + (int)rank * 256 + h * 128,
                                             leader_full);
                        if (BMN) {
                            for (int a = 0; a < 2; ++a)
                                tma_load_2d_pair(sa + kA3Bytes + a * kMnAtomBytes, &tmB, nt * 256 + (int)rank * 128 + 64 * a,
                                                 kb * BK, leader_full);
                        } else {
                            tma_load_2d_pair(sa + kA3Bytes, &tmB, kb * BK, nt * 256 + (int)rank * 128, leader_full);
                        }
                    }
                    if (++stage == kStages3) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader CTA only)
        if (lane == 0 && rank == 0) {
            uint32_t stage = 0, phase = 0;
            int local = 0;
            bool ok = true;
            const uint32_t idesc = idesc_bf16_f32(256, 256) | (BMN ? kIdescBMnMajor : 0u);
            for (int tile = cluster; ok && tile < num_tiles; tile += nclusters, ++local) {
                // both accumulators are free once the previous tile's epilogue has read them
                if (!mbar_wait_bounded(tempty_bar, ((uint32_t)local & 1u) ^ 1u, p.wait_ns, abort_flag, p.status,
                                       kCodeMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait_bounded(full_bar(stage), phase, p.wait_ns, abort_flag, p.status, kCodeMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int k_rem = p.K - kb * BK;
                    const int k_steps = k_rem >= BK ? BK / 16 : (k_rem + 15) / 16;
                    const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes3);
                    const uint32_t sb = sa + kA3Bytes;
                    for (int ks = 0; ks < k_steps; ++ks) {
                        const uint64_t bd = BMN ? smem_desc_mn_sw128(sb + kMnKStepBytes * ks, kMnAtomBytes)
                                                   : smem_desc_sw128(sb + 32u * ks);
                        for (int h = 0; h < 2; ++h)
                            tc_mma_f16_pair(tmem_base + (uint32_t)(h * 256), smem_desc_sw128(sa + h * kHalfBytes + 32u * ks),
                                            bd, idesc, (kb | ks) != 0 ? 1u : 0u);
                    }
                    tc_commit_pair_multicast(empty_bar(stage), 0x3);
                    if (++stage == kStages3) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit_pair_multicast(tfull_bar, 0x3);
            }
            tc_commit_pair_multicast(mma_done_bar, 0x1);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(mma_done_bar, 0)) {
                if (globaltimer() - t0 > p.wait_ns) {
                    atomicOr(p.status, (unsigned int)kCodeTeardown);
                    break;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..13 of each CTA)
        // warp w reads TMEM lane quarter w % 4 (rows q*32 .. q*32 + 31 of each row half); the
        // quarter's 16 chunks of 32 columns (8 per accumulator) are dealt to its three warps in
        // turn.  Per chunk: tcgen05.ld, RNE to bf16 pairs, a padded shared transpose, then 32
        // independent row stores (rows >= M and columns >= N masked).  Twelve warps measured
        // 0.351 against 0.359 ms for eight on the (8191, 8193, 4097) call.
        const int q = warp & 3;
        const int slice = (warp - 2) >> 2;  // 0..2: chunks ci = slice, slice + 3, ... of the 16 per quarter
        uint32_t* wb = reinterpret_cast<uint32_t*>(epi) + (warp - 2) * kEpiWords3;
        int local = 0;
        for (int tile = cluster; tile < num_tiles; tile += nclusters, ++local) {
            int mt, nt;
            tile_coords(tile, p.m_tiles, p.n_tiles, &mt, &nt);
            if (!mbar_wait_bounded(tfull_bar, (uint32_t)local & 1u, p.wait_ns, abort_flag, p.status, kCodeEpilogue))
                break;
            tc_fence_after();
#pragma unroll 1
            for (int ci = slice; ci < 16; ci += 3) {
                const int h = ci >> 3, c = ci & 7;
                const int row0 = mt * 512 + (int)rank * 256 + h * 128 + q * 32;
                const int col = nt * 256 + c * 32 + lane;
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 256 + c * 32), r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                    wb[lane * 17 + j] = *reinterpret_cast<const uint32_t*>(&v);
                }
                __syncwarp();
                const bool col_ok = col < p.N;
                const int rows = p.M - row0;
                uint16_t* Cp = reinterpret_cast<uint16_t*>(p.C) + (int64_t)row0 * p.ldc + col;
                const int sh = (lane & 1) * 16;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = wb[(16 * hh + i) * 17 + (lane >> 1)];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if (col_ok && 16 * hh + i < rows) *Cp = (uint16_t)(w[i] >> sh);
                        Cp += p.ldc;
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            mbar_arrive_cluster(mapa_shared(tempty_bar, 0));
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the leader's MMAs into the peer's TMEM are complete before either CTA frees it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 512);
    }
}

// ---------------------------------------------------------------------------- operand staging

// A' [Mp][Kp] <- A [M][K] (row stride lda), zero past M or K.  One 16-byte vector of A' per task.
__global__ void __launch_bounds__(256) k_stage_a(const uint16_t* __restrict__ A, int64_t lda, int M, int K,
                                                 uint16_t* __restrict__ Ap, int Kp, int64_t total_vecs) {
    const int kv = Kp / 8;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total_vecs;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = v / kv;
        const int k0 = (int)(v - m * kv) * 8;
        uint32_t w[4] = {0, 0, 0, 0};
        if (m < M) {
            const uint16_t* row = A + m * lda;
            if (k0 + 8 <= K) {  // whole vector inside the row: aligned 8-byte loads (lda may be odd)
                const uint64_t lo = sbt_load8_any(row + k0), hi = sbt_load8_any(row + k0 + 4);
                w[0] = (uint32_t)lo;
                w[1] = (uint32_t)(lo >> 32);
                w[2] = (uint32_t)hi;
                w[3] = (uint32_t)(hi >> 32);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int k = k0 + e;
                    const uint32_t x = k < K ? (uint32_t)__ldg(row + k) : 0u;
                    w[e >> 1] |= x << (16 * (e & 1));
                }
            }
        }
        sbt_st_v4(Ap + m * Kp + k0, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// B' [Np][Kp] <- transpose of B [K][N] (row stride ldb), zero past K or N.
// 64 x 64 tiles: each thread loads two 16-byte row pieces (8 values along n,
// through aligned 8-byte loads since ldb may be odd) into shared words, then
// reads an 8 (k) x 2 (n) block as eight words, transposes its 2 x 2 blocks of
// 16-bit values with byte permutes and writes two 16-byte vectors along k.
__global__ void __launch_bounds__(256) k_stage_bt(const uint16_t* __restrict__ B, int64_t ldb, int K, int N,
                                                  uint16_t* __restrict__ Bp, int Kp) {
    __shared__ uint32_t t[64][33];  // [k][n pair]
    const int k0 = blockIdx.x * 64, n0 = blockIdx.y * 64;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int v = i * 256 + threadIdx.x;  // 64 rows x 8 pieces
        const int kk = v >> 3, nh = (v & 7) * 8;
        const int k = k0 + kk, n = n0 + nh;
        uint64_t lo = 0, hi = 0;
        if (k < K && n < N) {
            const uint16_t* row = B + (int64_t)k * ldb;
            if (n + 8 <= N) {
                lo = sbt_load8_any(row + n);
                hi = sbt_load8_any(row + n + 4);
            } else {
                for (int e = 0; e < 8 && n + e < N; ++e) {
                    const uint64_t x = __ldg(row + n + e);
                    if (e < 4) lo |= x << (16 * e);
                    else hi |= x << (16 * (e - 4));
                }
            }
        }
        uint32_t* w = &t[kk][nh >> 1];
        w[0] = (uint32_t)lo;
        w[1] = (uint32_t)(lo >> 32);
        w[2] = (uint32_t)hi;
        w[3] = (uint32_t)(hi >> 32);
    }
    __syncthreads();
    // n = 2 np, 2 np + 1; k = kv .. kv + 7 (eight lanes cover one 128-byte run of a B' row)
    const int np = threadIdx.x >> 3, kv = (threadIdx.x & 7) * 8;
    uint32_t o0[4], o1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t w0 = t[kv + 2 * e][np], w1 = t[kv + 2 * e + 1][np];
        o0[e] = __byte_perm(w0, w1, 0x5410);  // (k, k+1) of n = 2 np
        o1[e] = __byte_perm(w0, w1, 0x7632);  // (k, k+1) of n = 2 np + 1
    }
    sbt_st_v4(Bp + (int64_t)(n0 + 2 * np) * Kp + k0 + kv, make_uint4(o0[0], o0[1], o0[2], o0[3]));
    sbt_st_v4(Bp + (int64_t)(n0 + 2 * np + 1) * Kp + k0 + kv, make_uint4(o1[0], o1[1], o1[2], o1[3]));
}

// One padded operand copy: dst [rows_p][cols_p] <- src [rows][cols] (row stride ld),
// zero past rows or cols; cols_p is a multiple of 8, so every 16-byte vector of dst
// is aligned.  The source rows are only 2-byte aligned when ld is odd: whole
// vectors come from aligned 8-byte words (each holds an element of the vector),
// the ragged end of a row element by element.
struct RowCopy {
    const uint16_t* src;
    int64_t ld;
    int rows, cols;
    uint16_t* dst;
    int cols_p;
    int64_t vecs;  // rows_p * cols_p / 8
};

__device__ __forceinline__ void row_copy_vector(const RowCopy& c, int64_t v) {
    const int kv = c.cols_p / 8;
    const int64_t r = v / kv;
    const int k0 = (int)(v - r * kv) * 8;
    uint32_t w[4] = {0, 0, 0, 0};
    if (r < c.rows && k0 < c.cols) {
        const uint16_t* row = c.src + r * c.ld;
        if (k0 + 8 <= c.cols) {
            const uint64_t lo = sbt_load8_any(row + k0), hi = sbt_load8_any(row + k0 + 4);
            w[0] = (uint32_t)lo;
            w[1] = (uint32_t)(lo >> 32);
            w[2] = (uint32_t)hi;
            w[3] = (uint32_t)(hi >> 32);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (k0 + e < c.cols) w[e >> 1] |= (uint32_t)__ldg(row + k0 + e) << (16 * (e & 1));
        }
    }
    sbt_st_v4(c.dst + r * c.cols_p + k0, make_uint4(w[0], w[1], w[2], w[3]));
}

// Both operand copies of one GEMM call in one launch: A' [Mp][Kp] (K-major) and
// B'' [Kp][Np] (B's own layout, read MN-major by the tensor-core kernel); either
// may be empty (vecs = 0) when TMA reads that operand where it lies.
__global__ void __launch_bounds__(256) k_stage_ab(const RowCopy a, const RowCopy b) {
    const int64_t total = a.vecs + b.vecs;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
        if (v < a.vecs)
            row_copy_vector(a, v);
        else
            row_copy_vector(b, v - a.vecs);
    }
}

// C[m][n] = acc[m][n] (fp32 C), or 0 without acc, for m < M, n < N: the K = 0 result.
__global__ void k_zero_c(char* C, int64_t ldc, int M, int N, int es, const float* acc, int64_t ld_acc) {
    const int64_t total = (int64_t)M * N;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / N, n = i - m * N;
        if (es == 4)
            reinterpret_cast<float*>(C)[m * ldc + n] = acc ? acc[m * ld_acc + n] : 0.f;
        else
            reinterpret_cast<uint16_t*>(C)[m * ldc + n] = 0;
    }
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

sbt_gemm_layout gemm_dims(int64_t M, int64_t N, int64_t K) {
    sbt_gemm_layout d;
    d.Mp = sbt_cdiv(M, 256) * 256;  // whole 256-row tiles for the CTA-pair kernel
    d.Np = sbt_cdiv(N, BN) * BN;
    d.Kp = sbt_cdiv(K, BK) * BK;
    d.a_bytes = round_up((size_t)d.Mp * d.Kp * 2, 256);
    d.b_bytes = round_up((size_t)d.Np * d.Kp * 2, 256);
    return d;
}

sbt_status encode_kmajor(sbt_context* ctx, CUtensorMap* map, void* base, int64_t rows, int64_t kp, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)kp, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kp * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = ctx->encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return sbt_fail(SBT_ERR_TENSOR_MAP, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    return SBT_OK;
}

// Tensor map over the caller's A itself, for rows that are 16-byte aligned:
// elements past K or M lie outside the tensor and TMA fills them with zeros,
// so the boundary tiles come out zero-filled without a staged copy.
sbt_status encode_direct_a(sbt_context* ctx, CUtensorMap* map, const void* A, int64_t lda, int64_t M, int64_t K) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)lda * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)BM};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = ctx->encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(A), dims, strides,
                                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return sbt_fail(SBT_ERR_TENSOR_MAP, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    return SBT_OK;
}

// Tensor map over the caller's B itself (rows 16-byte aligned), read MN-major:
// boxes of 64 columns x BK rows; columns past N and rows past K are zero-filled.
sbt_status encode_direct_b(sbt_context* ctx, CUtensorMap* map, const void* B, int64_t ldb, int64_t K, int64_t N) {
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)K};
    cuuint64_t strides[1] = {(cuuint64_t)ldb * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)BK};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = ctx->encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(B), dims, strides,
                                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return sbt_fail(SBT_ERR_TENSOR_MAP, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    return SBT_OK;
}

sbt_status launch_main(sbt_context* ctx, const CUtensorMap* tmA_direct, const CUtensorMap* tmB_direct,
                       const uint16_t* Ap, const uint16_t* Bp, const sbt_gemm_layout& d, void* C, int64_t ldc,
                       bool c_f32, const float* acc, int64_t ld_acc, int64_t M, int64_t N, int64_t K,
                       cudaStream_t stream);

}  // namespace

size_t sbt_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const sbt_gemm_layout d = gemm_dims(M, N, K);
    return d.a_bytes + d.b_bytes;
}

sbt_gemm_layout sbt_gemm_layout_of(int64_t M, int64_t N, int64_t K) { return gemm_dims(M, N, K); }

sbt_status sbt_launch_gemm_zero_k(sbt_context* ctx, void* C, int64_t ldc, bool c_f32, const float* acc,
                                  int64_t ld_acc, int64_t M, int64_t N, cudaStream_t stream) {
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sbt_cdiv(M * N, 256), (int64_t)ctx->sm_count * 8));
    k_zero_c<<<grid, 256, 0, stream>>>((char*)C, ldc, (int)M, (int)N, c_f32 ? 4 : 2, acc, ld_acc);
    return sbt_after_launch(ctx, "gemm (K=0)");
}

sbt_status sbt_launch_gemm(sbt_context* ctx, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                           int64_t ldc, sbt_dtype c_dtype, int64_t M, int64_t N, int64_t K, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
    (void)workspace_bytes;
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2)
        return sbt_fail(SBT_ERR_INVALID_ARG, "gemm_bounded: extents must be below 2^30");
    if (K == 0) return sbt_launch_gemm_zero_k(ctx, C, ldc, c_dtype == SBT_F32, nullptr, 0, M, N, stream);
    const sbt_gemm_layout d = gemm_dims(M, N, K);
    if (d.Np / 64 > 65535 || d.Kp / 64 > INT32_MAX)
        return sbt_fail(SBT_ERR_INVALID_ARG, "gemm_bounded: N too large for the staging grid");
    uint16_t* Ap = (uint16_t*)workspace;
    uint16_t* Bp = (uint16_t*)((char*)workspace + d.a_bytes);

    if (ctx->path == SBT_PATH_SCALAR) {
        // 1'. the transposing staging: A' [Mp][Kp] and B'^T [Np][Kp], both K-major
        const int64_t vecs = d.Mp * (d.Kp / 8);
        const int grid = (int)std::min<int64_t>(sbt_cdiv(vecs, 256), (int64_t)ctx->sm_count * 8);
        k_stage_a<<<grid, 256, 0, stream>>>((const uint16_t*)A, lda, (int)M, (int)K, Ap, (int)d.Kp, vecs);
        sbt_status st = sbt_after_launch(ctx, "gemm_bounded (stage A)");
        if (st) return st;
        dim3 g2((unsigned)(d.Kp / 64), (unsigned)(d.Np / 64));
        k_stage_bt<<<g2, 256, 0, stream>>>((const uint16_t*)B, ldb, (int)K, (int)N, Bp, (int)d.Kp);
        if ((st = sbt_after_launch(ctx, "gemm_bounded (stage B)"))) return st;
        return launch_main(ctx, nullptr, nullptr, Ap, Bp, d, C, ldc, c_dtype == SBT_F32, nullptr, 0, M, N, K, stream);
    }
    // 1. operand staging.  An operand whose rows are 16-byte aligned is read by TMA where it
    //    lies (SBT_PATH_AUTO / SBT_PATH_TMA); the others are copied, realigned and zero-padded,
    //    by one launch: A' [Mp][Kp], and B'' [Kp][Np] in B's own orientation (the tensor-core
    //    kernel reads B MN-major in both cases, so B needs no transpose).
    const bool tma_ok = ctx->path == SBT_PATH_AUTO || ctx->path == SBT_PATH_TMA;
    const bool direct_a = tma_ok && lda % 8 == 0 && (reinterpret_cast<uintptr_t>(A) & 15u) == 0;
    const bool direct_b = tma_ok && ldb % 8 == 0 && (reinterpret_cast<uintptr_t>(B) & 15u) == 0;
    CUtensorMap tmA, tmB;
    sbt_status st = SBT_OK;
    RowCopy ca = {}, cb = {};
    if (direct_a) {
        if ((st = encode_direct_a(ctx, &tmA, A, lda, M, K))) return st;
    } else {
        ca = {(const uint16_t*)A, lda, (int)M, (int)K, Ap, (int)d.Kp, d.Mp * (d.Kp / 8)};
    }
    if (direct_b) {
        if ((st = encode_direct_b(ctx, &tmB, B, ldb, K, N))) return st;
    } else {
        cb = {(const uint16_t*)B, ldb, (int)K, (int)N, Bp, (int)d.Np, d.Kp * (d.Np / 8)};
        if ((st = encode_direct_b(ctx, &tmB, Bp, d.Np, d.Kp, d.Np))) return st;
    }
    if (ca.vecs + cb.vecs > 0) {
        const int grid = (int)std::min<int64_t>(sbt_cdiv(ca.vecs + cb.vecs, 256), (int64_t)ctx->sm_count * 8);
        k_stage_ab<<<grid, 256, 0, stream>>>(ca, cb);
        if ((st = sbt_after_launch(ctx, "gemm_bounded (stage A, B)"))) return st;
    }
    return launch_main(ctx, direct_a ? &tmA : nullptr, &tmB, Ap, Bp, d, C, ldc, c_dtype == SBT_F32, nullptr, 0, M, N,
                       K, stream);
}

sbt_status sbt_launch_gemm_main(sbt_context* ctx, const uint16_t* Ap, const uint16_t* Bp, const sbt_gemm_layout& d,
                                void* C, int64_t ldc, bool c_f32, const float* acc, int64_t ld_acc, int64_t M,
                                int64_t N, int64_t K, cudaStream_t stream) {
    return launch_main(ctx, nullptr, nullptr, Ap, Bp, d, C, ldc, c_f32, acc, ld_acc, M, N, K, stream);
}

namespace {
sbt_status launch_main(sbt_context* ctx, const CUtensorMap* tmA_direct, const CUtensorMap* tmB_direct,
                       const uint16_t* Ap, const uint16_t* Bp, const sbt_gemm_layout& d, void* C, int64_t ldc,
                       bool c_f32, const float* acc, int64_t ld_acc, int64_t M, int64_t N, int64_t K,
                       cudaStream_t stream) {
    // 2. tensor-core main kernel
    // CTA pairs when there are at least as many 256 x 256 tiles as SM pairs;
    // single CTAs for smaller problems, with 128 x 256 tiles when those give
    // three quarters of the SMs work, else 128 x 128 or 128 x 64 tiles.
    const bool pair = ctx->sm_count >= 2 && (d.Mp / 256) * (d.Np / 256) >= ctx->sm_count / 2;
    const int64_t m_tiles1 = sbt_cdiv(M, BM);
    int bn1 = 64;
    for (int w : {256, 128})
        if (m_tiles1 * sbt_cdiv(N, w) * 4 >= (int64_t)ctx->sm_count * 3) {
            bn1 = w;
            break;
        }
    CUtensorMap tmA, tmB;
    sbt_status st = SBT_OK;
    if (tmA_direct)
        tmA = *tmA_direct;
    else if ((st = encode_kmajor(ctx, &tmA, (void*)Ap, d.Mp, d.Kp, BM)))
        return st;
    if (tmB_direct)
        tmB = *tmB_direct;
    else if ((st = encode_kmajor(ctx, &tmB, (void*)Bp, d.Np, d.Kp, pair ? 128 : bn1)))
        return st;
    GemmParams p;
    p.C = (char*)C;
    p.ldc = ldc;
    p.c_f32 = c_f32;
    p.acc = acc;
    p.ld_acc = ld_acc;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.m_tiles = (int)(d.Mp / BM);
    p.n_tiles = (int)(d.Np / BN);
    p.k_blocks = (int)(d.Kp / BK);
    p.status = ctx->status;
    p.wait_ns = ctx->wait_limit_ns;
    p.withhold_first_load = ctx->test_hook == SBT_TEST_WITHHOLD_LOAD;
    const bool bmn = tmB_direct != nullptr;
    static bool attr_set[64] = {false};
    if (!attr_set[ctx->device & 63]) {
        cudaError_t e = cudaSuccess;
        auto smem = [&](const void* f, size_t bytes) {
            if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        };
        smem((const void*)k_gemm_bf16_tc<256, false>, TcShape<256>::kSmem);
        smem((const void*)k_gemm_bf16_tc<128, false>, TcShape<128>::kSmem);
        smem((const void*)k_gemm_bf16_tc<64, false>, TcShape<64>::kSmem);
        smem((const void*)k_gemm_bf16_tc<256, true>, TcShape<256>::kSmem);
        smem((const void*)k_gemm_bf16_tc<128, true>, TcShape<128>::kSmem);
        smem((const void*)k_gemm_bf16_tc<64, true>, TcShape<64>::kSmem);
        smem((const void*)k_gemm_bf16_tc_pair<false>, kGemmSmem2);
        smem((const void*)k_gemm_bf16_tc_pair<true>, kGemmSmem2);
        smem((const void*)k_gemm_bf16_tc_pair512<false>, kGemmSmem3);
        smem((const void*)k_gemm_bf16_tc_pair512<true>, kGemmSmem3);
        if (e != cudaSuccess) return sbt_cuda_check(e, "cudaFuncSetAttribute(gemm smem)");
        attr_set[ctx->device & 63] = true;
    }
    if (pair) {
        // 512 x 256 tiles (two row halves per CTA) for a bf16 C, unless that leaves fewer tiles than
        // CTA pairs.  Their epilogue runs between tiles; an fp32 C (twice the bytes to store, an odd
        // row stride) measured faster on the 256 x 256 kernel, whose epilogue overlaps the next tile.
        const bool wide = !c_f32 && sbt_cdiv(d.Mp, 512) * (d.Np / 256) >= ctx->sm_count / 2;
        p.m_tiles = (int)(wide ? sbt_cdiv(d.Mp, 512) : d.Mp / 256);
        const int tiles = p.m_tiles * p.n_tiles;
        // as many CTA pairs as can be resident at once (queried once per device and kernel)
        static int max_clusters[2][64] = {{0}};
        int& mc = max_clusters[wide ? 1 : 0][ctx->device & 63];
        if (!mc) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = 2;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.gridDim = dim3(2 * (unsigned)(ctx->sm_count / 2), 1, 1);
            cfg.blockDim = dim3(wide ? kGemmThreads3 : kGemmThreads, 1, 1);
            cfg.dynamicSmemBytes = wide ? kGemmSmem3 : kGemmSmem2;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int n = 0;
            const cudaError_t qe = wide ? cudaOccupancyMaxActiveClusters(&n, k_gemm_bf16_tc_pair512<true>, &cfg)
                                        : cudaOccupancyMaxActiveClusters(&n, k_gemm_bf16_tc_pair<true>, &cfg);
            if (qe != cudaSuccess || n < 1) {
                (void)cudaGetLastError();
                n = ctx->sm_count / 2;
            }
            mc = n;
        }
        const int clusters = std::min(tiles, mc);
        cudaError_t e;
        if (wide)
            e = bmn ? sbt_launch_dependent(k_gemm_bf16_tc_pair512<true>, dim3(2 * clusters), dim3(kGemmThreads3),
                                           kGemmSmem3, stream, tmA, tmB, p)
                    : sbt_launch_dependent(k_gemm_bf16_tc_pair512<false>, dim3(2 * clusters), dim3(kGemmThreads3),
                                           kGemmSmem3, stream, tmA, tmB, p);
        else
            e = bmn ? sbt_launch_dependent(k_gemm_bf16_tc_pair<true>, dim3(2 * clusters), dim3(kGemmThreads),
                                           kGemmSmem2, stream, tmA, tmB, p)
                    : sbt_launch_dependent(k_gemm_bf16_tc_pair<false>, dim3(2 * clusters), dim3(kGemmThreads),
                                           kGemmSmem2, stream, tmA, tmB, p);
        if (e != cudaSuccess) return sbt_cuda_check(e, "gemm_bounded (tcgen05, CTA pairs)");
        return sbt_after_launch(ctx, "gemm_bounded (tcgen05, CTA pairs)");
    }
    // single CTAs: only the tiles that hold rows < M and columns < N
    p.m_tiles = (int)m_tiles1;
    p.n_tiles = (int)sbt_cdiv(N, bn1);
    const int tiles = p.m_tiles * p.n_tiles;
    const int grid = std::min(tiles, ctx->sm_count);
    cudaError_t e;
    auto launch1 = [&](auto kern, size_t smem_bytes) {
        return sbt_launch_dependent(kern, dim3(grid), dim3(kGemmThreads), smem_bytes, stream, tmA, tmB, p);
    };
    if (bn1 == 256)
        e = bmn ? launch1(k_gemm_bf16_tc<256, true>, TcShape<256>::kSmem) : launch1(k_gemm_bf16_tc<256, false>, TcShape<256>::kSmem);
    else if (bn1 == 128)
        e = bmn ? launch1(k_gemm_bf16_tc<128, true>, TcShape<128>::kSmem) : launch1(k_gemm_bf16_tc<128, false>, TcShape<128>::kSmem);
    else
        e = bmn ? launch1(k_gemm_bf16_tc<64, true>, TcShape<64>::kSmem) : launch1(k_gemm_bf16_tc<64, false>, TcShape<64>::kSmem);
    if (e != cudaSuccess) return sbt_cuda_check(e, "gemm_bounded (tcgen05)");
    return sbt_after_launch(ctx, "gemm_bounded (tcgen05)");
}
}  // namespace
