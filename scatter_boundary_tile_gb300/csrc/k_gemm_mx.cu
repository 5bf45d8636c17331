// Block-scaled GEMM on the tensor cores' own block scaling.
//
// cuTile.jl "Operations", muladd_scaled: its microscaling forms run on
// tcgen05.mma's block scaling with fp32 accumulation in TMEM, in three forms:
//  - kind::mxf8f6f4 (scale_vec::1X): E4M3 / E5M2 / E2M1 operands (E2M1 one
//    code per byte, see the staging below), one E8M0 scale per row of A and
//    per column of B for each K = 32 instruction;
//  - kind::mxf4 (scale_vec::2X): packed E2M1 x E2M1 (two codes per byte) with
//    E8M0 scales over blocks of 32; K = 64 per instruction, two scales each;
//  - kind::mxf4nvf4 (scale_vec::4X): packed E2M1 x E2M1 with E4M3 scales over
//    blocks of 16; K = 64 per instruction, four scales each.  The tensor cores
//    read these scales unsigned (UE4M3), so staging moves the sign of a
//    negative scale onto the 16 codes it multiplies (negating an E2M1 code
//    flips its bit 3, exactly), writes a NaN scale as zero and marks its row
//    of A or column of B; the epilogue writes NaN there.
// The packed forms carry half the operand bytes of the 8-bit form per element
// of K; what bounds each form is noted with its constants below.
//
// Pipeline (all on the caller's stream):
//  1. Staging (the bounded copy of Tylo.jl "Boundary tiles"): A -> A8 [Mp][Kb]
//     and B -> B8^T [Np][Kb], K-major, Kb bytes per row (8-bit codes or packed
//     E2M1 pairs), zero past M, N, K; the scales packed per (row or column
//     tile, four scales along K) into chunks in the order the tensor memory
//     wants them (below), neutral past the extents.  kind::mxf4 reads a packed
//     A whose rows start on 16-byte boundaries where it lies instead (the
//     tensor map's fill gives the zeros past M and K).
//  2. A persistent kernel on clusters of two CTAs (M = 256 per pair, N = 208
//     per tile): warp 0 of each CTA TMA-loads its 128 rows of A8, its 104 rows
//     of B8^T and the scale chunks of the stage's K blocks into a ring (a K
//     block is one 128-byte swizzled row of each operand: 128 8-bit codes or
//     256 packed E2M1 codes); the leader's warp 1 copies the scale chunks into
//     TMEM (tcgen05.cp.cta_group::2, each CTA's own chunk to its own TMEM) and
//     issues four block-scaled MMAs per K block, 32 bytes of K each, each
//     choosing its chunk and scale bytes; the epilogue warps of each CTA (four
//     for the 8-bit form, twelve for the packed ones) add acc and store fp32 D
//     inside M x N.
//
// Scale placement in TMEM (per CTA, 32-bit columns, 4 scale bytes each): a
// chunk holds four consecutive scales along K (entries 4c .. 4c + 3 of chunk
// c).  Entry s of row m (of this CTA's 128 rows of A) sits in lane m, column
// sfa + m / 32, byte s; that of column n of B (all 208 columns, in both CTAs)
// in lanes n % 32 + 32 q of every quarter q, column sfb + n / 32, byte s.  An
// instruction reads byte sf_id (1X), bytes sf_id and sf_id + 1 (2X) or all
// four (4X).  Scale addresses must be multiples of 4 columns.  A's chunk comes
// with one tcgen05.cp 32x128b.warpx4 (row r of a [32][16-byte] chunk to lane r
// of every quarter: byte 16 r + 4 j + s = entry s of row 32 j + r), or, in the
// packed forms, two chunks at once with one tcgen05.cp 128x256b; B's with one
// tcgen05.cp 128x256b from a 4 KB chunk that repeats the same 32 rows for the
// four quarters.  Each copy costs about the same in the MMA stream
// whatever its size (three 512-byte copies per 8-bit K block cost ~57 us of
// the 8191 x 8193 x 4096 call, two copies ~39 us), so B's eight columns take
// one larger copy.
//
// TMEM: two 208-column fp32 accumulators (the epilogue of one tile overlaps
// the main loop of the next) and a 12-column scale slot per chunk of each K
// block in the ring (at most 96 columns beside the accumulators).  A slot is
// rewritten only after the stage's previous MMAs completed: its new data
// arrives after the producer saw the stage's empty barrier, which those MMAs'
// commit signals.  8-bit form: two K blocks per stage halve the barrier round
// trips (0.334 -> 0.327 ms for the 8191 x 8193 x 4096 call); the scale slots
// of three such stages do not fit beside two 224-column accumulators, hence
// N = 208 (224 with two stages: 0.331 ms; 208 with five one-block stages:
// 0.352 ms).  The packed forms need two (mxf4) or four (mxf4nvf4) chunks per
// K block, hence four and two one-block stages.
#include <algorithm>
#include <string>

#include "sbt_internal.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace sbt_ptx;

constexpr int MX_BN = 208;   // columns per tile
constexpr int kMxFmtE2M1 = 3;  // sbt_lowp_format code of E2M1 (E4M3 = 0 and E5M2 = 1 are the MMA codes too)
constexpr int kMxFmtE8M0 = 2;  // sbt_lowp_format code of E8M0

// Operand type field of the kind::mxf8f6f4 instruction descriptor.
uint32_t mma_format(int fmt) { return fmt == kMxFmtE2M1 ? 5u : (uint32_t)fmt; }
constexpr int MX_BK = 128;   // bytes of one operand row per K block (one 128-byte swizzle row)
constexpr uint32_t kMxABytes = 128 * MX_BK;
constexpr uint32_t kMxBBytes = (MX_BN / 2) * MX_BK;
constexpr uint32_t kMxSfCol0 = 2 * MX_BN;              // scale slots after the two accumulators
constexpr uint32_t kMxSfCols = 12;                      // per chunk: 4 columns of A scales + 8 of B scales

// The three MMA forms (see the top of the file).
enum { kKindF8F6F4 = 0, kKindF4 = 1, kKindNvF4 = 2 };

template <int KIND>
struct MxCfg {
    static constexpr int kScalesPerStep = KIND == kKindF8F6F4 ? 1 : KIND == kKindF4 ? 2 : 4;
    static constexpr int kChunks = kScalesPerStep;  // per K block: 4 steps x scales per step / 4 per chunk
    static constexpr int kKPerStep = KIND == kKindF8F6F4 ? 32 : 64;   // elements of K per instruction
    static constexpr int kKPerBlock = 4 * kKPerStep;                   // elements of K per K block
    static constexpr int kStages = KIND == kKindF8F6F4 ? 3 : KIND == kKindF4 ? 4 : 2;
    static constexpr int kKB = KIND == kKindF8F6F4 ? 2 : 1;           // K blocks per stage
    // A's scales: with two or more chunks per K block, pairs of chunks travel in one
    // 4 KB tcgen05.cp 128x256b source (see the staging); else one 512 B chunk each.
    static constexpr bool kPairA = kChunks >= 2;
    static constexpr uint32_t kSfaBytes = kPairA ? (kChunks / 2) * 4096 : kChunks * 512;  // per K block
    // Stage layout per CTA: the K blocks' A atoms, then their B atoms, then their
    // B scale chunks (4 KB each) and A scale chunks; every piece 1024-aligned.
    static constexpr uint32_t kBOff = kKB * kMxABytes;
    static constexpr uint32_t kSfbOff = kBOff + kKB * kMxBBytes;
    static constexpr uint32_t kSfaOff = kSfbOff + kKB * kChunks * 4096;
    static constexpr uint32_t kTxBytes = kMxABytes + kMxBBytes + kChunks * 4096 + kSfaBytes;  // one CTA, one K block
    static constexpr uint32_t kStageBytes = (kSfaOff + kKB * kSfaBytes + 1023u) & ~1023u;
    // Epilogue: kEpiSlices warps per TMEM lane quarter, each draining every kEpiSlices-th
    // 32-column chunk; warp 0 loads, warp 1 issues the MMAs.
    // (Three for the packed forms: their main loop is short enough for four warps' fp32 stores to
    // set the pace, 0.206 -> 0.188 ms for the 8191 x 8193 x 4096 mxf4 kernel; the 8-bit form has
    // no shared memory left for more, and two stages with twelve warps were slower.)
    static constexpr int kEpiSlices = KIND == kKindF8F6F4 ? 1 : 3;
    // The 8-bit form transposes half a chunk (16 columns) at a time, each store covering two
    // rows: 0.324 -> 0.316 ms for the call (the packed forms ran 6-7% slower that way).
    static constexpr bool kHalfEpi = KIND == kKindF8F6F4;
    static constexpr int kEpiWords = kHalfEpi ? 32 * 17 : 32 * 33;  // one warp's transpose buffer (padded)
    static constexpr int kEpiWarps = 4 * kEpiSlices;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    static constexpr int kNumBars = 2 * kStages + 5;
    static constexpr size_t kSmemUsed =
        1024 + (size_t)kStages * kStageBytes + (size_t)kEpiWarps * kEpiWords * 4 + kNumBars * 8 + 16;
    // Every CTA allocates all 512 TMEM columns, so two CTAs of different pairs on one SM could each
    // hold one half of the other's pair waiting: ask for more than half the SM's shared memory
    // (228 KB, 1 KB of it reserved per CTA) so that only one fits.
    static constexpr size_t kSmemOneCta = 233472 / 2;
    static constexpr size_t kSmem = kSmemUsed > kSmemOneCta ? kSmemUsed : kSmemOneCta;
    static_assert(kMxSfCol0 + kStages * kKB * kChunks * kMxSfCols <= 512, "TMEM columns");
    static_assert(kMxBBytes % 1024 == 0 && kStageBytes % 1024 == 0 && kMxSfCol0 % 4 == 0, "layout");
    static_assert(kSmem <= 232448, "shared memory");
};

enum : unsigned int { kCodeProducer = 0x1100, kCodeMma = 0x1200, kCodeEpilogue = 0x1400, kCodeTeardown = 0x1800 };

struct MxParams {
    float* D;
    int64_t ldd;
    const float* acc;
    int64_t ld_acc;
    int M, N, K;
    int m_tiles, n_tiles, k_blocks;  // 256-row tiles, 208-column tiles, K blocks
    int n_chunks;                    // scale chunks along K per row / column tile
    const uint8_t* nan_a;            // mxf4nvf4: rows of A (Mp) and columns of B (Np) with a NaN
    const uint8_t* nan_b;            //   scale; unused by the other forms
    uint32_t idesc;                  // formats, M = 256, N = 208; the scale bytes are or-ed in per step
    unsigned int* status;
    uint64_t wait_ns;
    int withhold_first_load;
};

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

// Drain this warp's 32 rows of one 128 x 208 accumulator, add acc and store
// columns < N of rows < M through a padded shared transpose (one contiguous
// 32-column segment per store instruction).  mxf4nvf4: NaN in the rows and
// columns whose scales held a NaN.
template <int KIND>
__device__ __forceinline__ void mx_epilogue_tile(const MxParams& p, uint32_t tmem_acc, int q, int slice, int lane,
                                                 float* buf, int row0, int n0) {
    const int n_valid = min(MX_BN, p.N - n0);  // columns of this tile inside N (MX_BN is not a multiple of 32)
    const int chunks = (n_valid + 31) / 32;
    uint32_t nan_rows = 0;  // bit rr: row row0 + rr (< Mp) had a NaN scale
    if constexpr (KIND == kKindNvF4) nan_rows = __ballot_sync(0xffffffffu, p.nan_a[row0 + lane] != 0);
    for (int c = slice; c < chunks; c += MxCfg<KIND>::kEpiSlices) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_acc + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), r);
        tmem_ld_wait();
        if constexpr (MxCfg<KIND>::kHalfEpi) {
            // columns 16 h .. 16 h + 15 through a [32][17] buffer; lanes 0-15 store row 2 i,
            // lanes 16-31 row 2 i + 1 (the 8-bit form carries no NaN marks)
            const int rows = min(32, p.M - row0);
            const int cl = lane & 15, rh = lane >> 4;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int j = 0; j < 16; ++j) buf[lane * 17 + j] = __uint_as_float(r[16 * h + j]);
                __syncwarp();
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = buf[(2 * i + rh) * 17 + cl];
                const int col = n0 + c * 32 + 16 * h + cl;
                if (c * 32 + 16 * h + cl < n_valid) {
                    if (p.acc) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (2 * i + rh < rows) v[i] += __ldg(p.acc + (int64_t)(row0 + 2 * i + rh) * p.ld_acc + col);
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (2 * i + rh < rows) p.D[(int64_t)(row0 + 2 * i + rh) * p.ldd + col] = v[i];
                }
                __syncwarp();
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) buf[lane * 33 + j] = __uint_as_float(r[j]);
            __syncwarp();
            const int col = n0 + c * 32 + lane;
            if (c * 32 + lane < n_valid) {
                bool nan_col = false;
                if constexpr (KIND == kKindNvF4) nan_col = p.nan_b[col] != 0;
                const int rows = min(32, p.M - row0);
                // two halves of 16 rows: all loads of a half issue before its stores (a loop carrying
                // each store behind its own shared load ran at ~90 cycles a row)
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = buf[(16 * h + i) * 33 + lane];
                    if (p.acc) {
                        const float* a = p.acc + (int64_t)(row0 + 16 * h) * p.ld_acc + col;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (16 * h + i < rows) v[i] += __ldg(a + (int64_t)i * p.ld_acc);
                    }
                    if constexpr (KIND == kKindNvF4) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (nan_col || ((nan_rows >> (16 * h + i)) & 1u)) v[i] = __uint_as_float(0x7FC00000u);
                    }
                    float* d = p.D + (int64_t)(row0 + 16 * h) * p.ldd + col;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (16 * h + i < rows) d[(int64_t)i * p.ldd] = v[i];
                }
            }
            __syncwarp();
        }
    }
}

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MxCfg<KIND>::kThreads, 1)
    k_gemm_mx_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                   const MxParams p) {
    using C = MxCfg<KIND>;
    constexpr int kMxStages = C::kStages, kMxKB = C::kKB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* epi = reinterpret_cast<float*>(smem + (size_t)kMxStages * C::kStageBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi + C::kEpiWarps * C::kEpiWords);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kMxStages + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kMxStages + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kMxStages + 2 + a); };
    const uint32_t mma_done_bar = bar0 + 8u * (2 * kMxStages + 4);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0);
    const int lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMxStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * C::kEpiWarps * 32);
        }
        mbar_init(mma_done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmSA);
        prefetch_tmap(&tmSB);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Set-up above overlaps the end of the staging kernel ahead in the stream (launched as a
    // programmatic dependent); from here on the staged operands are read and C is written.
    griddep_wait();
    const int num_tiles = p.m_tiles * p.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (each CTA, own halves)
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            int64_t issued = 0;
            for (int tile = cluster; ok && tile < num_tiles; tile += nclusters) {
                int mt, nt;
                tile_coords(tile, p.m_tiles, p.n_tiles, &mt, &nt);
                for (int kb0 = 0; kb0 < p.k_blocks; kb0 += kMxKB) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, p.wait_ns, abort_flag, p.status,
                                           kCodeProducer)) {
                        ok = false;
                        break;
                    }
                    const bool withhold = p.withhold_first_load && blockIdx.x == 0 && issued == 0;
                    ++issued;
                    if (!withhold) {
                        const int nkb = p.k_blocks - kb0 < kMxKB ? p.k_blocks - kb0 : kMxKB;
                        const uint32_t sa = smem_u32(smem + (size_t)stage * C::kStageBytes);
                        const uint32_t leader_full = mapa_shared(full_bar(stage), 0);
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * (uint32_t)nkb * C::kTxBytes);
                        for (int j = 0; j < nkb; ++j) {
                            const int kb = kb0 + j;
                            const int c0 = kb * C::kChunks;  // first scale chunk of this K block
                            tma_load_2d_pair(sa + j * kMxABytes, &tmA, kb * MX_BK, mt * 256 + (int)rank * 128,
                                             leader_full);
                            tma_load_2d_pair(sa + C::kBOff + j * kMxBBytes, &tmB, kb * MX_BK,
                                             nt * MX_BN + (int)rank * (MX_BN / 2), leader_full);
                            // scale chunks viewed as rows of 256 B: B 4 KB per (tile, chunk), A 512 B per
                            // (128-row group, chunk); the K block's chunks are adjacent
                            tma_load_2d_pair(sa + C::kSfbOff + j * C::kChunks * 4096, &tmSB, 0,
                                             (nt * p.n_chunks + c0) * 16, leader_full);
                            if constexpr (C::kPairA)
                                tma_load_2d_pair(sa + C::kSfaOff + j * C::kSfaBytes, &tmSA, 0,
                                                 ((mt * 2 + (int)rank) * (p.n_chunks / 2) + c0 / 2) * 16,
                                                 leader_full);
                            else
                                tma_load_2d_pair(sa + C::kSfaOff + j * C::kSfaBytes, &tmSA, 0,
                                                 ((mt * 2 + (int)rank) * p.n_chunks + c0) * 2, leader_full);
                        }
                    }
                    if (++stage == kMxStages) {
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
            for (int tile = cluster; ok && tile < num_tiles; tile += nclusters, ++local) {
                const int acc = local & 1;
                const uint32_t use = (uint32_t)(local >> 1);
                if (!mbar_wait_bounded(tempty_bar(acc), (use & 1u) ^ 1u, p.wait_ns, abort_flag, p.status,
                                       kCodeMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * MX_BN);
                for (int kb0 = 0; kb0 < p.k_blocks; kb0 += kMxKB) {
                    if (!mbar_wait_bounded(full_bar(stage), phase, p.wait_ns, abort_flag, p.status, kCodeMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nkb = p.k_blocks - kb0 < kMxKB ? p.k_blocks - kb0 : kMxKB;
                    const uint32_t sa = smem_u32(smem + (size_t)stage * C::kStageBytes);
                    for (int j = 0; j < nkb; ++j) {
                        const int kb = kb0 + j;
                        const int k_rem = p.K - kb * C::kKPerBlock;
                        const int k_steps =
                            k_rem >= C::kKPerBlock ? 4 : (k_rem + C::kKPerStep - 1) / C::kKPerStep;
                        const int n_ch = (k_steps * C::kScalesPerStep + 3) / 4;  // chunks these steps read
                        const uint32_t slot0 =
                            tmem_base + kMxSfCol0 + kMxSfCols * (uint32_t)((stage * kMxKB + j) * C::kChunks);
                        // slot of chunk c: A's four columns at sf_a(c), B's eight at sf_b(c); paired
                        // chunks keep A's eight columns (two chunks) first, then B's two sets of eight
                        auto sf_a = [&](int c) {
                            return C::kPairA ? slot0 + 24u * (uint32_t)(c >> 1) + 4u * (uint32_t)(c & 1)
                                             : slot0 + kMxSfCols * (uint32_t)c;
                        };
                        auto sf_b = [&](int c) {
                            return C::kPairA ? slot0 + 24u * (uint32_t)(c >> 1) + 8u + 8u * (uint32_t)(c & 1)
                                             : slot0 + kMxSfCols * (uint32_t)c + 4u;
                        };
                        for (int c = 0; c < n_ch; ++c) {
                            const uint32_t ch = (uint32_t)(j * C::kChunks + c);
                            if constexpr (C::kPairA) {
                                if ((c & 1) == 0)
                                    tc_cp_pair_128x256b(sf_a(c), smem_desc_rows32(sa + C::kSfaOff + j * C::kSfaBytes +
                                                                                  (uint32_t)(c >> 1) * 4096));
                            } else {
                                tc_cp_pair_32x128b_warpx4(sf_a(c), smem_desc_rows16(sa + C::kSfaOff + ch * 512));
                            }
                            tc_cp_pair_128x256b(sf_b(c), smem_desc_rows32(sa + C::kSfbOff + ch * 4096));
                        }
                        const uint32_t a_s = sa + j * kMxABytes, b_s = sa + C::kBOff + j * kMxBBytes;
                        for (int ks = 0; ks < k_steps; ++ks) {
                            const int e = ks * C::kScalesPerStep;  // first scale entry of this step
                            const uint32_t sfa = sf_a(e >> 2), sfb = sf_b(e >> 2);
                            const uint32_t sf_id = (uint32_t)(e & 3);
                            const uint32_t idesc = p.idesc | (sf_id << 4) | (sf_id << 29);
                            const uint64_t ad = smem_desc_sw128(a_s + 32u * ks), bd = smem_desc_sw128(b_s + 32u * ks);
                            const uint32_t accum = (kb | ks) != 0 ? 1u : 0u;
                            if constexpr (KIND == kKindF8F6F4)
                                tc_mma_mx_pair(d_tmem, ad, bd, idesc, sfa, sfb, accum);
                            else if constexpr (KIND == kKindF4)
                                tc_mma_mxf4_pair(d_tmem, ad, bd, idesc, sfa, sfb, accum);
                            else
                                tc_mma_mxf4nvf4_pair(d_tmem, ad, bd, idesc, sfa, sfb, accum);
                        }
                    }
                    tc_commit_pair_multicast(empty_bar(stage), 0x3);
                    if (++stage == kMxStages) {
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
        // ------------------------------------------------------------ epilogue (warps 2.. of each CTA)
        const int q = warp & 3, slice = (warp - 2) >> 2;  // TMEM lane quarter (warp % 4), chunk slice
        float* buf = epi + (warp - 2) * C::kEpiWords;
        const uint32_t leader_tempty0 = mapa_shared(tempty_bar(0), 0);
        int local = 0;
        for (int tile = cluster; tile < num_tiles; tile += nclusters, ++local) {
            const int acc = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            int mt, nt;
            tile_coords(tile, p.m_tiles, p.n_tiles, &mt, &nt);
            if (!mbar_wait_bounded(tfull_bar(acc), use & 1u, p.wait_ns, abort_flag, p.status, kCodeEpilogue)) break;
            tc_fence_after();
            mx_epilogue_tile<KIND>(p, tmem_base + (uint32_t)(acc * MX_BN), q, slice, lane, buf, mt * 256 + (int)rank * 128 + q * 32,
                             nt * MX_BN);
            tc_fence_before();
            mbar_arrive_cluster(leader_tempty0 + 8u * acc);
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

// ---------------------------------------------------------------------------- staging

// E2M1 operands: kind::mxf8f6f4 reads a 4-bit type from each 16-byte piece of
// a K-major row as 16 packed codes in the first 8 bytes (even element in the
// low nibble, as in the caller's arrays) followed by 8 bytes of padding.
// (Found by running one-K-block products with the codes one per byte: the
// results matched this reading exactly and no other.)

// Eight 4-bit codes (code i in bits 4i..4i+3) spread to one code per byte.
__device__ __forceinline__ uint64_t spread_nibbles(uint32_t x) {
    uint64_t v = x;
    v = (v | (v << 16)) & 0x0000FFFF0000FFFFull;
    v = (v | (v << 8)) & 0x00FF00FF00FF00FFull;
    v = (v | (v << 4)) & 0x0F0F0F0F0F0F0F0Full;
    return v;
}

// The inverse: eight bytes holding one code each (low nibble) packed into 32 bits.
__device__ __forceinline__ uint32_t pack_nibbles(uint64_t v) {
    v = (v | (v >> 4)) & 0x00FF00FF00FF00FFull;
    v = (v | (v >> 8)) & 0x0000FFFF0000FFFFull;
    v = (v | (v >> 16)) & 0x00000000FFFFFFFFull;
    return (uint32_t)v;
}

// Sixteen codes of a row starting at element e0 (a multiple of 16), one per
// byte: bytes of an 8-bit format, or the nibbles of packed E2M1 (two per
// byte, even element low); `avail` codes are inside the row, the rest zero.
template <bool P4>
__device__ __forceinline__ void load16_codes(const uint8_t* row, int e0, int avail, uint64_t* lo, uint64_t* hi) {
    *lo = 0;
    *hi = 0;
    if (avail >= 16) {
        if (P4) {
            const uint64_t c = sbt_load8_any(row + e0 / 2);
            *lo = spread_nibbles((uint32_t)c);
            *hi = spread_nibbles((uint32_t)(c >> 32));
        } else {
            *lo = sbt_load8_any(row + e0);
            *hi = sbt_load8_any(row + e0 + 8);
        }
        return;
    }
    for (int e = 0; e < 16 && e < avail; ++e) {
        uint64_t b;
        if (P4) b = (uint64_t)((__ldg(row + (e0 + e) / 2) >> (4 * ((e0 + e) & 1))) & 15u);
        else b = __ldg(row + e0 + e);
        if (e < 8) *lo |= b << (8 * e);
        else *hi |= b << (8 * (e - 8));
    }
}

// A8 [Mp][Kp] <- A [M][K] (row stride lda elements), zero past M or K; 16 codes per task.
template <bool P4>
__global__ void __launch_bounds__(256) k_mx_stage_a(const uint8_t* __restrict__ A, int64_t lda, int M, int K,
                                                    uint8_t* __restrict__ Ap, int Kp, int64_t tasks) {
    const int kv = Kp / 16;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < tasks; t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = t / kv;
        const int k0 = (int)(t - m * kv) * 16;
        uint64_t lo = 0, hi = 0;
        if (m < M && k0 < K) load16_codes<P4>(A + (P4 ? m * lda / 2 : m * lda), k0, K - k0, &lo, &hi);
        if (P4) {  // 16 packed codes, then 8 bytes of padding
            lo = (uint64_t)pack_nibbles(lo) | ((uint64_t)pack_nibbles(hi) << 32);
            hi = 0;
        }
        sbt_st_v4(Ap + m * Kp + k0, make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32)));
    }
}

// A4 [Mp][Kb] <- packed E2M1 A [M][K] (two codes per byte, row stride lda / 2
// bytes), zero past M or K; 16 bytes (32 codes) per task.  NV: the codes of a
// block of 16 whose E4M3 scale is negative are negated (bit 3 of each code),
// and the first nan_n tasks clear the NaN marks the scale staging sets.
template <bool NV>
__global__ void __launch_bounds__(256) k_mx4_stage_a(const uint8_t* __restrict__ A, int64_t lda,
                                                     const uint8_t* __restrict__ SA, int64_t ld_sa, int M, int K,
                                                     uint8_t* __restrict__ Ap, int Kb, int64_t tasks,
                                                     uint8_t* __restrict__ nan_marks, int64_t nan_n) {
    const int kv = Kb / 16;
    const int kbytes = K / 2;  // a multiple of 8: K is a multiple of the scale block (16 or 32)
    const int64_t n = NV && nan_n > tasks ? nan_n : tasks;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
        if (NV && t < nan_n) nan_marks[t] = 0;
        if (t >= tasks) continue;
        const int64_t m = t / kv;
        const int b0 = (int)(t - m * kv) * 16;
        uint64_t lo = 0, hi = 0;
        if (m < M && b0 < kbytes) {  // then b0 + 8 <= kbytes
            const uint8_t* row = A + m * (lda / 2);
            lo = sbt_load8_any(row + b0);
            if (b0 + 16 <= kbytes) hi = sbt_load8_any(row + b0 + 8);
            if constexpr (NV) {
                const uint8_t* sc = SA + m * ld_sa + b0 / 8;  // scales of the two blocks of 16 codes
                if (__ldg(sc) & 0x80u) lo ^= 0x8888888888888888ull;
                if (b0 + 16 <= kbytes && (__ldg(sc + 1) & 0x80u)) hi ^= 0x8888888888888888ull;
            }
        }
        sbt_st_v4(Ap + m * Kb + b0, make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32)));
    }
}

// B8^T [Np][Kp] <- transpose of B [K][N] (row stride ldb bytes), zero past K or N.
// 64 (k) x 208 (n) tiles (a whole N tile of the main kernel, so each B row
// piece read is 208 bytes long), 208 threads.  Loads: four 16-byte row pieces
// per thread into shared words; stores: each thread reads a 16 (k) x 4 (n)
// block as sixteen words, transposes its four 4 x 4 byte blocks with byte
// permutes and writes four 16-byte vectors (one per n row).  The four threads
// of an n group are adjacent lanes, so each row's 64 bytes leave in one warp
// store as two whole sectors; rows k >= 32 of the shared tile sit 8 words to
// the right, which with the odd pitch puts the four k quarters a warp reads in
// four different bank octets.
constexpr int kBtK = 64, kBtN = MX_BN, kBtThreads = (kBtN / 4) * (kBtK / 16), kBtPitch = kBtN / 4 + 9;
static_assert(kBtK * kBtN / 16 % kBtThreads == 0, "load split");
//
// PACKED (E2M1 for kind::mxf4 / mxf4nvf4): rows of Kp / 2 bytes, 16 codes in
// 8 bytes with no padding; NV: the 16 codes of a block whose E4M3 scale is
// negative are negated.
template <bool P4, bool PACKED, bool NV>
__global__ void __launch_bounds__(kBtThreads) k_mx_stage_bt(const uint8_t* __restrict__ B, int64_t ldb, int K, int N,
                                                            uint8_t* __restrict__ Bp, int Kp,
                                                            const uint8_t* __restrict__ SB, int64_t ld_sb) {
    __shared__ uint32_t t[kBtK][kBtPitch];
    const int k0 = blockIdx.x * kBtK, n0 = blockIdx.y * kBtN;
#pragma unroll
    for (int i = 0; i < kBtK * kBtN / 16 / kBtThreads; ++i) {
        const int v = i * kBtThreads + threadIdx.x;
        const int kk = v / (kBtN / 16), nh = (v % (kBtN / 16)) * 16;
        const int k = k0 + kk, n = n0 + nh;
        uint64_t lo = 0, hi = 0;
        if (k < K && n < N) load16_codes<P4>(B + (P4 ? (int64_t)k * ldb / 2 : (int64_t)k * ldb), n, N - n, &lo, &hi);
        uint32_t* w = &t[kk][(nh >> 2) + ((kk >> 5) << 3)];
        w[0] = (uint32_t)lo;
        w[1] = (uint32_t)(lo >> 32);
        w[2] = (uint32_t)hi;
        w[3] = (uint32_t)(hi >> 32);
    }
    __syncthreads();
    const int nw = threadIdx.x >> 2, kv = (threadIdx.x & 3) * 16;  // n = 4 nw .. + 3, k = kv .. + 15
    const int col = nw + ((kv >> 5) << 3);
    if (k0 + kv >= Kp) return;
    uint32_t out[4][4];  // out[j][g]: bytes k = kv + 4 g .. + 3 of row n = 4 nw + j
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t w0 = t[kv + 4 * g][col], w1 = t[kv + 4 * g + 1][col];
        const uint32_t w2 = t[kv + 4 * g + 2][col], w3 = t[kv + 4 * g + 3][col];
        const uint32_t a0 = __byte_perm(w0, w1, 0x5140), a1 = __byte_perm(w0, w1, 0x7362);
        const uint32_t a2 = __byte_perm(w2, w3, 0x5140), a3 = __byte_perm(w2, w3, 0x7362);
        out[0][g] = __byte_perm(a0, a2, 0x5410);
        out[1][g] = __byte_perm(a0, a2, 0x7632);
        out[2][g] = __byte_perm(a1, a3, 0x5410);
        out[3][g] = __byte_perm(a1, a3, 0x7632);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 v = make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]);
        if (P4)  // 16 packed codes (then 8 bytes of padding unless PACKED)
            v = make_uint4(pack_nibbles((uint64_t)v.x | ((uint64_t)v.y << 32)),
                           pack_nibbles((uint64_t)v.z | ((uint64_t)v.w << 32)), 0u, 0u);
        const int64_t n = n0 + 4 * nw + j;
        if constexpr (PACKED) {
            if constexpr (NV) {
                if (k0 + kv < K && n < N && (__ldg(SB + (int64_t)((k0 + kv) / 16) * ld_sb + n) & 0x80u)) {
                    v.x ^= 0x88888888u;
                    v.y ^= 0x88888888u;
                }
            }
            *reinterpret_cast<uint2*>(Bp + n * (Kp / 2) + (k0 + kv) / 2) = make_uint2(v.x, v.y);
        } else {
            sbt_st_v4(Bp + n * Kp + k0 + kv, v);
        }
    }
}

// Scale chunks: chunk c of a row / column holds its scales 4c .. 4c + 3.
//  SA8 chunk (g, c), 512 B in the source form of tcgen05.cp 32x128b.warpx4
//    (row r of [32][16 B] goes to lane r of every lane quarter): byte
//    16 r + 4 j + s is scale 4c + s of A row 128 g + 32 j + r (lane quarter q
//    reads column sfa + q, so quarter q finds its rows in column j = q).
//  SB8 chunk (t, c), 4 KB in the source form of tcgen05.cp 128x256b (row r to
//    lane r, 8 columns of 4 scale bytes; byte b of row r at (r / 8) * 256 +
//    (b / 16) * 128 + (r % 8) * 16 + b % 16): every lane quarter alike, row
//    32 q + i column c' holding the scales of B column 208 t + 32 c' + i.
//  PAIR_A (forms with two or more chunks per K block): A's chunks 2 cp and
//    2 cp + 1 of row group g share one 4 KB source of that same form, so one
//    copy fills eight columns: lane 32 q + i, column j (j < 4) holds chunk
//    2 cp's entries of A row 128 g + 32 j + i, column 4 + j chunk 2 cp + 1's.
// E8M0 scales are copied; UE4M3 (mxf4nvf4) takes the magnitude of an E4M3
// scale (its sign went to the operand codes), zero for NaN with the row of A
// or column of B marked in nan_a / nan_b.  Past the extents 2^0 (127, or 0x38
// in UE4M3): those operand codes are zero.  A task forms one lane's 16 bytes;
// the 4 KB sources repeat them for the four lane quarters.
template <bool UE4M3>
__device__ __forceinline__ uint32_t stage_scale(uint32_t code, bool* nan) {
    if (!UE4M3) return code;
    if ((code & 0x7Fu) == 0x7Fu) {
        *nan = true;
        return 0u;
    }
    return code & 0x7Fu;
}

template <bool UE4M3, bool PAIR_A>
__global__ void __launch_bounds__(256) k_mx_stage_scales(const uint8_t* __restrict__ SA, int64_t ld_sa,
                                                         const uint8_t* __restrict__ SB, int64_t ld_sb, int M, int N,
                                                         int Ks, int n_chunks, uint8_t* __restrict__ SAp,
                                                         int64_t tasks_a, uint8_t* __restrict__ SBp, int64_t tasks_b,
                                                         uint8_t* __restrict__ nan_a, uint8_t* __restrict__ nan_b) {
    constexpr uint32_t kOne = UE4M3 ? 0x38u : 127u;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < tasks_a + tasks_b;
         t += (int64_t)gridDim.x * blockDim.x) {
        uint32_t w[4];
        uint8_t* dst;
        if (t < tasks_a) {
            int r;
            int64_t g;
            int kb;
            int half = 0;
            int64_t pair = 0;
            if (PAIR_A) {  // lane i (of every quarter), columns 4 half .. + 3 of the source of chunks 2 cp, 2 cp + 1
                pair = t >> 6;
                const int n_pairs = n_chunks / 2;
                g = pair / n_pairs;
                const int cp = (int)(pair - g * n_pairs);
                r = (int)(t & 31);
                half = (int)((t >> 5) & 1);
                kb = 2 * cp + half;
            } else {
                r = (int)(t & 31);
                const int64_t chunk = t >> 5;
                g = chunk / n_chunks;
                kb = (int)(chunk - g * n_chunks);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t m = 128 * g + 32 * j + r;
                uint32_t v = 0;
                bool nan = false;
#pragma unroll
                for (int st = 0; st < 4; ++st) {
                    const int ks = 4 * kb + st;
                    v |= ((m < M && ks < Ks) ? stage_scale<UE4M3>(__ldg(SA + m * ld_sa + ks), &nan) : kOne)
                         << (8 * st);
                }
                if (UE4M3 && nan) nan_a[m] = 1;
                w[j] = v;
            }
            if (PAIR_A) {  // the same 16 bytes for lane r of each of the four quarters
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int lane = 32 * q + r;
                    sbt_st_v4(SAp + pair * 4096 + ((lane >> 3) * 256 + half * 128 + (lane & 7) * 16),
                              make_uint4(w[0], w[1], w[2], w[3]));
                }
                continue;
            }
            dst = SAp + t * 16;
        } else {
            // lane i (of every quarter), columns c0 .. c0 + 3 of the 4 KB chunk
            const int64_t u = t - tasks_a;
            const int64_t chunk = u >> 6;
            const int i = (int)(u & 31);
            const int half = (int)((u >> 5) & 1);
            const int c0 = 4 * half;
            const int64_t tile = chunk / n_chunks;
            const int kb = (int)(chunk - tile * n_chunks);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int within = 32 * (c0 + e) + i;
                const int64_t n = tile * MX_BN + within;
                uint32_t v = 0;
                bool nan = false;
#pragma unroll
                for (int st = 0; st < 4; ++st) {
                    const int ks = 4 * kb + st;
                    const bool in = within < MX_BN && n < N && ks < Ks;
                    v |= (in ? stage_scale<UE4M3>(__ldg(SB + (int64_t)ks * ld_sb + n), &nan) : kOne) << (8 * st);
                }
                if (UE4M3 && nan) nan_b[n] = 1;
                w[e] = v;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // the same 16 bytes for lane i of each of the four quarters
                const int lane = 32 * q + i;
                sbt_st_v4(SBp + chunk * 4096 + ((lane >> 3) * 256 + half * 128 + (lane & 7) * 16),
                          make_uint4(w[0], w[1], w[2], w[3]));
            }
            continue;
        }
        sbt_st_v4(dst, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// Workspace layout of one call: A8 [Mp][Kb], B8^T [Np][Kb] (Kb bytes per row:
// k_blocks 128-byte K blocks), the scale chunks, and (mxf4nvf4) the NaN marks
// of the rows of A and columns of B.
struct MxLayout {
    int64_t Mp, Np, Kb, k_blocks, n_chunks, m_tiles, n_tiles;
    size_t a_off, b_off, sa_off, sb_off, nan_off, total;
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

MxLayout mx_layout(int64_t M, int64_t N, int64_t K, int kind) {
    const int k_per_block = kind == kKindF8F6F4 ? MxCfg<kKindF8F6F4>::kKPerBlock : MxCfg<kKindF4>::kKPerBlock;
    const int chunks = kind == kKindF8F6F4 ? 1 : kind == kKindF4 ? 2 : 4;
    MxLayout L;
    L.k_blocks = sbt_cdiv(K, k_per_block);
    L.Kb = L.k_blocks * MX_BK;
    L.n_chunks = L.k_blocks * chunks;
    L.m_tiles = sbt_cdiv(M, 256);
    L.Mp = L.m_tiles * 256;
    L.n_tiles = sbt_cdiv(N, MX_BN);
    L.Np = L.n_tiles * MX_BN;
    L.a_off = 0;
    L.b_off = round256((size_t)L.Mp * L.Kb);
    L.sa_off = L.b_off + round256((size_t)L.Np * L.Kb);
    // A's chunks: 512 B each, or (two or more per K block) 4 KB per pair
    L.sb_off = L.sa_off + round256((size_t)(L.Mp / 128) * L.n_chunks * (chunks >= 2 ? 2048 : 512));
    L.nan_off = L.sb_off + round256((size_t)L.n_tiles * L.n_chunks * 4096);
    L.total = L.nan_off + (kind == kKindNvF4 ? round256((size_t)(L.Mp + L.Np)) : 0);
    return L;
}

// Bytes [rows][inner] with row stride `stride` (0: inner), read in boxes of
// box_rows x box_inner; reads past the extents fill zeros.
sbt_status encode_u8(sbt_context* ctx, CUtensorMap* map, void* base, int64_t inner, int64_t rows, int box_inner,
                     int box_rows, bool swizzle, int64_t stride = 0) {
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(stride ? stride : inner)};
    cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = ctx->encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                                   swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return sbt_fail(SBT_ERR_TENSOR_MAP, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    return SBT_OK;
}

}  // namespace

size_t sbt_gemm_mx_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    size_t most = 0;
    for (int kind = kKindF8F6F4; kind <= kKindNvF4; ++kind) most = std::max(most, mx_layout(M, N, K, kind).total);
    return most;
}

namespace {

// Shared-memory attribute and resident clusters of one form of the kernel, once per device.
template <int KIND>
sbt_status mx_kernel_setup(sbt_context* ctx, int* clusters_out) {
    static bool attr_set[64] = {false};
    static int max_clusters[64] = {0};
    const int dev = ctx->device & 63;
    constexpr size_t smem = MxCfg<KIND>::kSmem;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_mx_pair<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return sbt_cuda_check(e, "cudaFuncSetAttribute(gemm mx smem)");
        attr_set[dev] = true;
    }
    if (!max_clusters[dev]) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * (unsigned)(ctx->sm_count / 2), 1, 1);
        cfg.blockDim = dim3(MxCfg<KIND>::kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_gemm_mx_pair<KIND>, &cfg) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            n = ctx->sm_count / 2;
        }
        max_clusters[dev] = n;
    }
    *clusters_out = max_clusters[dev];
    return SBT_OK;
}

template <int KIND>
sbt_status mx_launch(sbt_context* ctx, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSA,
                     const CUtensorMap& tmSB, const MxParams& p, cudaStream_t stream) {
    int max_clusters = 0;
    sbt_status st = mx_kernel_setup<KIND>(ctx, &max_clusters);
    if (st) return st;
    const int clusters = std::min(p.m_tiles * p.n_tiles, max_clusters);
    const cudaError_t e = sbt_launch_dependent(k_gemm_mx_pair<KIND>, dim3(2 * clusters), dim3(MxCfg<KIND>::kThreads),
                                               MxCfg<KIND>::kSmem, stream, tmA, tmB, tmSA, tmSB, p);
    if (e != cudaSuccess) return sbt_cuda_check(e, "gemm_block_scaled (tcgen05 block-scaled, CTA pairs)");
    return sbt_after_launch(ctx, "gemm_block_scaled (tcgen05 block-scaled, CTA pairs)");
}

}  // namespace

sbt_status sbt_launch_gemm_mx(sbt_context* ctx, int a_fmt, const void* A, int64_t lda, int b_fmt, const void* B,
                              int64_t ldb, int s_fmt, const void* SA, int64_t ld_sa, const void* SB, int64_t ld_sb,
                              const float* acc, int64_t ld_acc, float* D, int64_t ldd, int64_t M, int64_t N,
                              int64_t K, void* workspace, cudaStream_t stream) {
    // packed E2M1 x E2M1 takes the 4-bit forms; everything else kind::mxf8f6f4
    const bool packed = a_fmt == kMxFmtE2M1 && b_fmt == kMxFmtE2M1;
    const int kind = !packed ? kKindF8F6F4 : s_fmt == kMxFmtE8M0 ? kKindF4 : kKindNvF4;
    const int block = kind == kKindNvF4 ? 16 : 32;
    const MxLayout L = mx_layout(M, N, K, kind);
    const int64_t Kp = L.Kb * (packed ? 2 : 1);  // elements of K per staged row
    if (L.Np / kBtN > 65535 || Kp / 64 > INT32_MAX)
        return sbt_fail(SBT_ERR_INVALID_ARG, "gemm_block_scaled: N too large for the staging grid");
    uint8_t* ws = (uint8_t*)workspace;
    uint8_t *Ap = ws + L.a_off, *Bp = ws + L.b_off, *SAp = ws + L.sa_off, *SBp = ws + L.sb_off;
    uint8_t* nan_a = kind == kKindNvF4 ? ws + L.nan_off : nullptr;
    uint8_t* nan_b = nan_a ? nan_a + L.Mp : nullptr;
    const int Ks = (int)(K / block);
    const uint8_t *A8 = (const uint8_t*)A, *B8 = (const uint8_t*)B, *SA8 = (const uint8_t*)SA,
                  *SB8 = (const uint8_t*)SB;
    // kind::mxf4 reads packed A where it lies when its rows start on 16-byte boundaries (the
    // tensor map zero-fills past K and M, as the staging would); kind::mxf4nvf4 must stage A to
    // move scale signs onto its codes, and kind::mxf8f6f4's 8-bit A is staged as before
    const bool direct_a = kind == kKindF4 && lda % 32 == 0 && (reinterpret_cast<uintptr_t>(A) & 15u) == 0;

    // 1. staging
    {
        const int64_t tasks = L.Mp * (L.Kb / 16);
        const int64_t nan_n = nan_a ? L.Mp + L.Np : 0;
        const int grid = (int)std::min<int64_t>(sbt_cdiv(std::max(tasks, nan_n), 256), (int64_t)ctx->sm_count * 8);
        if (kind == kKindNvF4)
            k_mx4_stage_a<true><<<grid, 256, 0, stream>>>(A8, lda, SA8, ld_sa, (int)M, (int)K, Ap, (int)L.Kb, tasks,
                                                          nan_a, nan_n);
        else if (kind == kKindF4 && !direct_a)
            k_mx4_stage_a<false><<<grid, 256, 0, stream>>>(A8, lda, SA8, ld_sa, (int)M, (int)K, Ap, (int)L.Kb, tasks,
                                                           nullptr, 0);
        else if (kind == kKindF8F6F4 && a_fmt == kMxFmtE2M1)
            k_mx_stage_a<true><<<grid, 256, 0, stream>>>(A8, lda, (int)M, (int)K, Ap, (int)L.Kb, tasks);
        else if (kind == kKindF8F6F4)
            k_mx_stage_a<false><<<grid, 256, 0, stream>>>(A8, lda, (int)M, (int)K, Ap, (int)L.Kb, tasks);
        sbt_status st = direct_a ? SBT_OK : sbt_after_launch(ctx, "gemm_block_scaled (stage A)");
        if (st) return st;
        dim3 g2((unsigned)sbt_cdiv(Kp, kBtK), (unsigned)(L.Np / kBtN));
        if (kind == kKindNvF4)
            k_mx_stage_bt<true, true, true><<<g2, kBtThreads, 0, stream>>>(B8, ldb, (int)K, (int)N, Bp, (int)Kp, SB8,
                                                                          ld_sb);
        else if (kind == kKindF4)
            k_mx_stage_bt<true, true, false><<<g2, kBtThreads, 0, stream>>>(B8, ldb, (int)K, (int)N, Bp, (int)Kp,
                                                                           nullptr, 0);
        else if (b_fmt == kMxFmtE2M1)
            k_mx_stage_bt<true, false, false><<<g2, kBtThreads, 0, stream>>>(B8, ldb, (int)K, (int)N, Bp, (int)Kp,
                                                                            nullptr, 0);
        else
            k_mx_stage_bt<false, false, false><<<g2, kBtThreads, 0, stream>>>(B8, ldb, (int)K, (int)N, Bp, (int)Kp,
                                                                             nullptr, 0);
        if ((st = sbt_after_launch(ctx, "gemm_block_scaled (stage B)"))) return st;
        // one task per lane of a quarter and half of a 4 KB source (stored to all four quarters),
        // or per lane of a 512 B A chunk
        const int64_t ta = (L.Mp / 128) * L.n_chunks * 32, tb = L.n_tiles * L.n_chunks * 64;
        const int g3 = (int)std::min<int64_t>(sbt_cdiv(ta + tb, 256), (int64_t)ctx->sm_count * 8);
        if (kind == kKindNvF4)
            k_mx_stage_scales<true, true><<<g3, 256, 0, stream>>>(SA8, ld_sa, SB8, ld_sb, (int)M, (int)N, Ks,
                                                                  (int)L.n_chunks, SAp, ta, SBp, tb, nan_a, nan_b);
        else if (kind == kKindF4)
            k_mx_stage_scales<false, true><<<g3, 256, 0, stream>>>(SA8, ld_sa, SB8, ld_sb, (int)M, (int)N, Ks,
                                                                   (int)L.n_chunks, SAp, ta, SBp, tb, nullptr,
                                                                   nullptr);
        else
            k_mx_stage_scales<false, false><<<g3, 256, 0, stream>>>(SA8, ld_sa, SB8, ld_sb, (int)M, (int)N, Ks,
                                                                    (int)L.n_chunks, SAp, ta, SBp, tb, nullptr,
                                                                    nullptr);
        if ((st = sbt_after_launch(ctx, "gemm_block_scaled (stage scales)"))) return st;
    }

    // 2. block-scaled tensor-core kernel
    const int chunks = (int)(L.n_chunks / L.k_blocks);
    CUtensorMap tmA, tmB, tmSA, tmSB;
    sbt_status st = direct_a ? encode_u8(ctx, &tmA, const_cast<void*>(A), K / 2, M, MX_BK, 128, true, lda / 2)
                             : encode_u8(ctx, &tmA, Ap, L.Kb, L.Mp, MX_BK, 128, true);
    if (st) return st;
    if ((st = encode_u8(ctx, &tmB, Bp, L.Kb, L.Np, MX_BK, MX_BN / 2, true))) return st;
    if (chunks >= 2) {  // 4 KB per pair of A's chunks, as 16 rows of 256 B
        if ((st = encode_u8(ctx, &tmSA, SAp, 256, (L.Mp / 128) * (L.n_chunks / 2) * 16, 256, 8 * chunks, false)))
            return st;
    } else if ((st = encode_u8(ctx, &tmSA, SAp, 256, (L.Mp / 128) * L.n_chunks * 2, 256, 2 * chunks, false))) {
        return st;
    }
    if ((st = encode_u8(ctx, &tmSB, SBp, 256, L.n_tiles * L.n_chunks * 16, 256, 16 * chunks, false))) return st;
    MxParams p;
    p.D = D;
    p.ldd = ldd;
    p.acc = acc;
    p.ld_acc = ld_acc;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.m_tiles = (int)L.m_tiles;
    p.n_tiles = (int)L.n_tiles;
    p.k_blocks = (int)L.k_blocks;
    p.n_chunks = (int)L.n_chunks;
    p.nan_a = nan_a;
    p.nan_b = nan_b;
    p.idesc = kind == kKindF8F6F4 ? idesc_mx_e8m0(mma_format(a_fmt), mma_format(b_fmt), 256, MX_BN, 0)
                                  : idesc_mxf4(256, MX_BN, kind == kKindF4);
    p.status = ctx->status;
    p.wait_ns = ctx->wait_limit_ns;
    p.withhold_first_load = ctx->test_hook == SBT_TEST_WITHHOLD_LOAD;
    if (kind == kKindF4) return mx_launch<kKindF4>(ctx, tmA, tmB, tmSA, tmSB, p, stream);
    if (kind == kKindNvF4) return mx_launch<kKindNvF4>(ctx, tmA, tmB, tmSA, tmSB, p, stream);
    return mx_launch<kKindF8F6F4>(ctx, tmA, tmB, tmSA, tmSB, p, stream);
}
